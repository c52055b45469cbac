"""Python access to the plain CPU oracle in ``oracle.c``.

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  Nothing here imports the
GPU library, and the GPU library never imports this package.

The C file is compiled with gcc on first use (or by ``build()``) into
``oracle/_build/liboracle.so``; ``-ffp-contract=off`` keeps every FP64
multiply and add separately rounded on both x86 and Arm hosts.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

# The oracle's own storage-type numbering (see oracle.c).
_DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_CODE_TORCH = {v: k for k, v in _DTYPE_CODE.items()}
_NAME_TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

TRAFFIC_KEYS = ("a_elems", "b_elems", "c_elems", "bytes", "flops", "tiles",
                "steps", "ws_max", "ws_full")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def _build_cmd(out: str) -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
            "-pthread", "-Wall", "-Wextra", "-o", out, _SRC, "-lm"]


def _stamp() -> str:
    """SHA-256 of the source, the compiler command and the host architecture."""
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_build_cmd("<out>")).replace(_HERE, "<oracle>").encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library unless the one on disk was
    built from this source with this command; returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stamp = _stamp()
    stamp_path = _LIB_PATH + ".sha256"
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read().strip() == stamp:
                return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(_build_cmd(tmp), check=True)
    os.replace(tmp, _LIB_PATH)
    with open(stamp_path + f".{os.getpid()}", "w") as f:
        f.write(stamp + "\n")
    os.replace(stamp_path + f".{os.getpid()}", stamp_path)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.orc_widen.argtypes = [_p, ctypes.c_int, _i64, _p]
            lib.orc_round.argtypes = [_p, _i64, ctypes.c_int, _p]
            lib.orc_gemm.argtypes = [_p, _p, ctypes.c_int, _i64, _i64, _i64, _p, _p, ctypes.c_int]
            lib.orc_gemm_entries.argtypes = [_p, _p, ctypes.c_int, _i64, _i64, _i64,
                                             _p, _p, _i64, _p, _p]
            lib.orc_gemm_general.argtypes = [_p, _p, ctypes.c_int, _i64, _i64, _i64,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                             ctypes.c_double, _p, ctypes.c_int, _p, _p]
            lib.orc_tile_ranges.argtypes = [_i64, _i64, _p, _p, _i64]
            lib.orc_tile_ranges.restype = _i64
            lib.orc_traffic.argtypes = [_i64] * 9 + [_p]
            _lib = lib
    return _lib


def _torch_dtype(dtype) -> torch.dtype:
    if isinstance(dtype, str):
        return _NAME_TORCH[dtype]
    return dtype


def _raw(t: torch.Tensor) -> np.ndarray:
    """Contiguous CPU storage of a matrix as a numpy array of its bits."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a.size else None


def widen(t: torch.Tensor) -> np.ndarray:
    """Exact FP64 values of a FP32/FP16/BF16 tensor, decoded by the oracle."""
    raw = _raw(t)
    out = np.empty(raw.size, dtype=np.float64)
    rc = _load().orc_widen(_ptr(raw), _DTYPE_CODE[t.dtype], raw.size, _ptr(out))
    assert rc == 0, rc
    return out.reshape(tuple(t.shape))


def round_to(x: np.ndarray, dtype) -> torch.Tensor:
    """Correctly rounded (nearest-even) conversion of FP64 values to dtype."""
    dt = _torch_dtype(dtype)
    x = np.ascontiguousarray(x, dtype=np.float64)
    if dt == torch.float32:
        out = np.empty(x.size, dtype=np.float32)
    else:
        out = np.empty(x.size, dtype=np.int16)
    rc = _load().orc_round(_ptr(x), x.size, _DTYPE_CODE[dt], _ptr(out))
    assert rc == 0, rc
    t = torch.from_numpy(out)
    if dt != torch.float32:
        t = t.view(dt)
    return t.reshape(x.shape)


def gemm(A: torch.Tensor, B: torch.Tensor, nthreads: int | None = None):
    """(C, Cabs) in FP64: C = A @ B and Cabs[i,j] = sum_k |A[i,k] B[k,j]|."""
    if A.dtype != B.dtype:
        raise TypeError("A and B must share a storage type")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    a, b = _raw(A), _raw(B)
    C = np.empty((M, N), dtype=np.float64)
    Cabs = np.empty((M, N), dtype=np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().orc_gemm(_ptr(a), _ptr(b), _DTYPE_CODE[A.dtype], M, N, K,
                          _ptr(C), _ptr(Cabs), int(nthreads))
    assert rc == 0, rc
    return C, Cabs


def gemm_general(A: torch.Tensor, B: torch.Tensor, op_a: str = "n", op_b: str = "n",
                 alpha: float = 1.0, beta: float = 0.0, C_in: torch.Tensor | None = None):
    """(C, Cabs) in FP64 for C = alpha * op(A) @ op(B) + beta * C_in.

    op "n" uses a matrix as stored; "t" its transpose (A stored K x M, B
    stored N x K).  Cabs = |alpha| * sum_k |op(A)[i,k] op(B)[k,j]|."""
    if A.dtype != B.dtype:
        raise TypeError("A and B must share a storage type")
    ta, tb = op_a.lower() == "t", op_b.lower() == "t"
    M, K = (A.shape[1], A.shape[0]) if ta else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if tb else (B.shape[0], B.shape[1])
    if K != K2:
        raise ValueError("inner dimensions differ")
    a, b = _raw(A), _raw(B)
    if C_in is not None:
        c_in = _raw(C_in)
        c_code = _DTYPE_CODE[C_in.dtype]
        if tuple(C_in.shape) != (M, N):
            raise ValueError("C_in must be M x N")
    else:
        c_in, c_code = np.zeros(0, dtype=np.float32), 0
    C = np.empty((M, N), dtype=np.float64)
    Cabs = np.empty((M, N), dtype=np.float64)
    rc = _load().orc_gemm_general(_ptr(a), _ptr(b), _DTYPE_CODE[A.dtype], M, N, K, int(ta),
                                  int(tb), float(alpha), float(beta), _ptr(c_in), c_code,
                                  _ptr(C), _ptr(Cabs))
    assert rc == 0, rc
    return C, Cabs


def gemm_entries(A: torch.Tensor, B: torch.Tensor, rows, cols):
    """(values, abs sums) of C[rows[s], cols[s]] for each sample s."""
    M, K = A.shape
    _, N = B.shape
    a, b = _raw(A), _raw(B)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    out = np.empty(r.size, dtype=np.float64)
    out_abs = np.empty(r.size, dtype=np.float64)
    rc = _load().orc_gemm_entries(_ptr(a), _ptr(b), _DTYPE_CODE[A.dtype], M, N, K,
                                  _ptr(r), _ptr(c), r.size, _ptr(out), _ptr(out_abs))
    assert rc == 0, rc
    return out, out_abs


def tile_ranges(n: int, t: int) -> list[tuple[int, int]]:
    """[(start, stop), ...] slicing [0, n) into tiles of size t."""
    cap = max(1, -(-n // t)) if t > 0 else 1
    starts = np.zeros(cap, dtype=np.int64)
    lens = np.zeros(cap, dtype=np.int64)
    cnt = _load().orc_tile_ranges(n, t, _ptr(starts), _ptr(lens), cap)
    if cnt < 0:
        raise ValueError("bad tile range arguments")
    return [(int(starts[i]), int(starts[i] + lens[i])) for i in range(cnt)]


def traffic(M: int, N: int, K: int, tm: int, tn: int, tk: int,
            in_bytes: int = 2, acc_bytes: int = 4, c_bytes: int = 4) -> dict:
    """The tile-walking traffic / FLOP / working-set counts of the loop nest."""
    res = np.zeros(len(TRAFFIC_KEYS), dtype=np.int64)
    rc = _load().orc_traffic(M, N, K, tm, tn, tk, in_bytes, acc_bytes, c_bytes, _ptr(res))
    if rc != 0:
        raise ValueError("bad traffic arguments")
    return {k: int(v) for k, v in zip(TRAFFIC_KEYS, res)}


def tolerance(Cabs: np.ndarray) -> np.ndarray:
    """Element-wise acceptance bound for FP16/BF16 inputs with FP32
    accumulation: |C - C_ref| <= 1e-3 * sum_k |a_ik b_kj| + 1e-6."""
    return 1e-3 * Cabs + 1e-6
