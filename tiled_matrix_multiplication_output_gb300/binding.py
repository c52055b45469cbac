"""ctypes binding of the C ABI in include/tiled_gemm.h.

Argument marshalling only: every step of the product runs in the CUDA
library.  The functions named like the C entry points take raw pointers
(ints), sizes and enum values and return the C status code.  `matmul` is the
convenience form for PyTorch CUDA tensors (PyTorch provides the device
memory and the stream); it raises GemmError on a non-zero status.

There is no fallback: if the library is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

F32, F16, BF16 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}

OK, ERR_INVALID_VALUE, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4

# The largest M, N or K the library accepts (GEMM_MAX_DIM).
MAX_DIM = (1 << 31) - 256

KERNELS = {
    "auto": 0,
    "simt": 1,
    "simt_tpb3": 2,
    "tc_128x128": 3,
    "tc_128x256": 4,
    "tc_256x256": 5,
    "tc_256x128": 6,
    "tc_small": 7,
    "tile16": 8,
}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}

HEADER = os.path.join(_build.ROOT, "include", "tiled_gemm.h")

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int

_SIGNATURES = {
    "gemm": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _p], _int),
    "gemm_ex": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _p], _int),
    "gemm_ex_kernel": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _int, _p], _int),
    "gemm_select_kernel": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int], _int),
    "gemm_ws_split_count": ([_i64, _i64, _i64, _int, _int, _int], _int),
    "gemm_general": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, ctypes.c_float, ctypes.c_float,
                      _int, _int, _int, _int, _p], _int),
    "gemm_ex_host": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _p, _p, _p, _p], _int),
    "gemm_ex_host_ws": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _p, _p, _p, _p,
                         ctypes.c_size_t, _p], _int),
    "gemm_host_panel_rows": ([_i64], _i64),
    "gemm_workspace_size": ([_i64, _i64, _i64], ctypes.c_size_t),
    "gemm_ex_ws": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _p, ctypes.c_size_t, _p],
                   _int),
    "gemm_splitk_workspace_size": ([_i64, _i64, _i64, _int], ctypes.c_size_t),
    "gemm_splitk": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _int, _p, ctypes.c_size_t,
                     _p], _int),
    "gemm_splitk_noalloc": ([_p, _p, _p, _i64, _i64, _i64, _int, _int, _int, _int, _p], _int),
    "gemm_device_status": ([_p], _int),
    "gemm_debug_config": ([_i64, _int], _int),
    "gemm_launch_count": ([], ctypes.c_uint64),
    "gemm_traffic_model": ([_i64] * 9 + [_p], _int),
    "gemm_error_string": ([_int], ctypes.c_char_p),
}


class GemmError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: status {code} ({error_string(code)})")


def header_functions() -> list[str]:
    """Names of the functions declared in include/tiled_gemm.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the CUDA library (optionally building it first)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is not built; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def gemm(A, B, C, M, N, K, in_dtype, acc_dtype, stream=None) -> int:
    return load_library().gemm(A, B, C, M, N, K, in_dtype, acc_dtype, stream)


def gemm_ex(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype, stream=None) -> int:
    return load_library().gemm_ex(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype, stream)


def gemm_ex_kernel(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype, kernel, stream=None) -> int:
    return load_library().gemm_ex_kernel(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype,
                                         kernel, stream)


def gemm_general(A, B, C, M, N, K, op_a, op_b, alpha, beta, in_dtype, acc_dtype, out_dtype,
                 kernel=0, stream=None) -> int:
    return load_library().gemm_general(A, B, C, M, N, K, op_a, op_b, alpha, beta, in_dtype,
                                       acc_dtype, out_dtype, kernel, stream)


def gemm_select_kernel(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype) -> int:
    return load_library().gemm_select_kernel(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype)


def gemm_ex_host(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype, out_dtype, dA, dB, dC,
                 stream=None) -> int:
    return load_library().gemm_ex_host(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype,
                                       out_dtype, dA, dB, dC, stream)


def gemm_ex_host_ws(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype, out_dtype, dA, dB, dC,
                    workspace, workspace_bytes, stream=None) -> int:
    return load_library().gemm_ex_host_ws(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype,
                                          out_dtype, dA, dB, dC, workspace, workspace_bytes,
                                          stream)


def gemm_host_panel_rows(M) -> int:
    return load_library().gemm_host_panel_rows(M)


def gemm_workspace_size(M, N, K) -> int:
    return load_library().gemm_workspace_size(M, N, K)


def gemm_ws_split_count(M, N, K, in_dtype, acc_dtype, out_dtype) -> int:
    return load_library().gemm_ws_split_count(M, N, K, in_dtype, acc_dtype, out_dtype)


def gemm_ex_ws(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype, workspace, workspace_bytes,
               stream=None) -> int:
    return load_library().gemm_ex_ws(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype, workspace,
                                     workspace_bytes, stream)


def matmul_ws(A, B, out_dtype=None, workspace=None, out=None, stream=None):
    """C = A @ B through gemm_ex_ws (last-wave balancing with a workspace,
    allocated by PyTorch unless given)."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[1]
    odt = torch.float32 if out_dtype is None else (
        torch_dtype(out_dtype) if isinstance(out_dtype, (str, int)) else out_dtype)
    C = out if out is not None else torch.empty((M, N), dtype=odt, device=A.device)
    if workspace is None:
        workspace = torch.empty(max(gemm_workspace_size(M, N, K), 16), dtype=torch.uint8,
                                device=A.device)
    nbytes = workspace.numel() * workspace.element_size()
    rc = gemm_ex_ws(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, dtype_code(A.dtype), F32,
                    dtype_code(C.dtype), workspace.data_ptr(), nbytes, _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, "gemm_ex_ws")
    return C


def gemm_splitk_workspace_size(M, N, K, splits) -> int:
    return load_library().gemm_splitk_workspace_size(M, N, K, splits)


def gemm_splitk(A, B, C, M, N, K, splits, in_dtype, acc_dtype, out_dtype, workspace,
                workspace_bytes, stream=None) -> int:
    return load_library().gemm_splitk(A, B, C, M, N, K, splits, in_dtype, acc_dtype, out_dtype,
                                      workspace, workspace_bytes, stream)


# Size of the library's fixed split-K scratch (GEMM_SPLITK_NOALLOC_MAX_BYTES).
SPLITK_NOALLOC_MAX_BYTES = 8 << 20


def gemm_splitk_noalloc(A, B, C, M, N, K, splits, in_dtype, acc_dtype, out_dtype,
                        stream=None) -> int:
    return load_library().gemm_splitk_noalloc(A, B, C, M, N, K, splits, in_dtype, acc_dtype,
                                              out_dtype, stream)


def matmul_splitk(A, B, splits: int, out_dtype=None, workspace=None, stream=None):
    """C = A @ B through gemm_splitk for contiguous CUDA tensors.  The FP32
    workspace is allocated by PyTorch unless given (a CUDA tensor of at
    least gemm_splitk_workspace_size bytes)."""
    torch = _torch()
    M, K = A.shape
    N = B.shape[1]
    odt = torch.float32 if out_dtype is None else (
        torch_dtype(out_dtype) if isinstance(out_dtype, (str, int)) else out_dtype)
    C = torch.empty((M, N), dtype=odt, device=A.device)
    need = gemm_splitk_workspace_size(M, N, K, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=A.device)
    nbytes = workspace.numel() * workspace.element_size()
    rc = gemm_splitk(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, int(splits),
                     dtype_code(A.dtype), F32, dtype_code(odt), workspace.data_ptr(), nbytes,
                     _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, "gemm_splitk")
    return C


def gemm_device_status(stream=None) -> int:
    return load_library().gemm_device_status(stream)


TRAFFIC_KEYS = ("a_elems", "b_elems", "c_elems", "bytes", "flops", "tiles", "steps",
                "ws_max", "ws_full")


def gemm_traffic_model(M, N, K, tm, tn, tk, in_bytes=2, acc_bytes=4, c_bytes=4) -> dict:
    """The library's closed-form traffic / working-set counts as a dict."""
    out = (ctypes.c_int64 * 9)()
    rc = load_library().gemm_traffic_model(M, N, K, tm, tn, tk, in_bytes, acc_bytes, c_bytes,
                                           out)
    if rc != OK:
        raise GemmError(rc, "gemm_traffic_model")
    return dict(zip(TRAFFIC_KEYS, list(out)))


def gemm_launch_count() -> int:
    return load_library().gemm_launch_count()


def gemm_debug_config(wait_budget_cycles: int = 0, fault_skip_kblock: int = -1) -> int:
    return load_library().gemm_debug_config(wait_budget_cycles, fault_skip_kblock)


def error_string(code: int) -> str:
    try:
        return load_library().gemm_error_string(code).decode()
    except RuntimeError:
        return "library not loaded"


gemm_error_string = error_string


# ------------------------------------------------------- PyTorch convenience

def _torch():
    import torch
    return torch


def dtype_code(dt) -> int:
    torch = _torch()
    if isinstance(dt, str):
        return DTYPE_CODES[dt]
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[dt]


def torch_dtype(code_or_name):
    torch = _torch()
    if isinstance(code_or_name, str):
        code_or_name = DTYPE_CODES[code_or_name]
    return {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[code_or_name]


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


OPS = {"n": 0, "t": 1}


def addmm(A, B, C=None, op_a="n", op_b="n", alpha=1.0, beta=0.0, out_dtype=None,
          kernel: str | int = "auto", stream=None):
    """C = alpha * op(A) @ op(B) + beta * C for contiguous CUDA tensors, in place
    in C when given (C is allocated, and beta must be 0, otherwise).

    op "n" takes an operand as stored, "t" its transpose (A stored K x M, B
    stored N x K).  Returns C without synchronizing."""
    torch = _torch()
    if A.dim() != 2 or B.dim() != 2 or A.dtype != B.dtype:
        raise ValueError("A and B must be 2-D tensors of one dtype")
    if not (A.is_cuda and B.is_cuda and A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous CUDA tensors")
    ta, tb = OPS[op_a], OPS[op_b]
    M, K = (A.shape[1], A.shape[0]) if ta else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if tb else (B.shape[0], B.shape[1])
    if K != K2:
        raise ValueError("inner dimensions differ")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs C")
        odt = torch.float32 if out_dtype is None else torch_dtype(out_dtype) \
            if isinstance(out_dtype, (str, int)) else out_dtype
        C = torch.empty((M, N), dtype=odt, device=A.device)
    elif tuple(C.shape) != (M, N) or not C.is_contiguous() or not C.is_cuda:
        raise ValueError("C must be a contiguous (M, N) CUDA tensor")
    kid = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    rc = gemm_general(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, ta, tb, float(alpha),
                      float(beta), dtype_code(A.dtype), F32, dtype_code(C.dtype), kid,
                      _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, "gemm_general")
    return C


def matmul(A, B, out_dtype=None, kernel: str | int = "auto", out=None, stream=None):
    """C = A @ B for contiguous row-major CUDA tensors (FP32 accumulation).

    out_dtype defaults to FP32 (the accumulator type); `out` may supply a
    preallocated contiguous (M, N) tensor of that type.  Runs on `stream`
    (default: PyTorch's current stream) and returns without synchronizing.
    """
    torch = _torch()
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"bad shapes {tuple(A.shape)} @ {tuple(B.shape)}")
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    if not (A.is_contiguous() and B.is_contiguous()):
        raise ValueError("A and B must be contiguous row-major")
    M, K = A.shape
    N = B.shape[1]
    odt = torch.float32 if out_dtype is None else (
        torch_dtype(out_dtype) if isinstance(out_dtype, (str, int)) else out_dtype)
    if out is None:
        out = torch.empty((M, N), dtype=odt, device=A.device)
    elif out.shape != (M, N) or out.dtype != odt or not out.is_contiguous():
        raise ValueError("out must be a contiguous (M, N) tensor of the output dtype")
    kid = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    rc = gemm_ex_kernel(A.data_ptr(), B.data_ptr(), out.data_ptr(), M, N, K,
                        dtype_code(A.dtype), F32, dtype_code(odt), kid, _stream_handle(stream))
    if rc != OK:
        raise GemmError(rc, "gemm_ex_kernel")
    return out
