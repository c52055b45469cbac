"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg

TC_KERNELS = ("tc_128x128", "tc_128x256", "tc_256x256", "tc_256x128", "tc_small")
# tile16 needs 16-byte aligned operand rows; the two SIMT kernels take any shape.
ALL_KERNELS = ("simt", "simt_tpb3", "tile16") + TC_KERNELS

# Half an ulp at 1.0 of each output type: the relative size of one
# round-to-nearest step when the FP32 accumulator is written out.  Used only
# for same-sign products (see tolerance_check).
HALF_ULP = {torch.float32: 2.0 ** -24, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def run_gpu(A: torch.Tensor, B: torch.Tensor, out_dtype=torch.float32, kernel="auto",
            device="cuda:0") -> torch.Tensor:
    """C from the CUDA library (through gemm_ex_kernel), copied to the host.
    Also checks the device status word (no watchdog timeout)."""
    dA = A.to(device)
    dB = B.to(device)
    C = tg.matmul(dA, dB, out_dtype=out_dtype, kernel=kernel)
    rc = tg.gemm_device_status(torch.cuda.current_stream().cuda_stream)
    assert rc == tg.binding.OK, tg.error_string(rc)
    return C.cpu()


def expect_exact(C_gpu: torch.Tensor, A: torch.Tensor, B: torch.Tensor):
    """Integer-valued inputs: the exact product rounded (nearest-even) to the
    output type, element for element."""
    C_ref, _ = oracle.gemm(A, B)
    want = oracle.round_to(C_ref, C_gpu.dtype)
    got = C_gpu.double().numpy()
    np.testing.assert_array_equal(got, want.double().numpy())


def tolerance_check(C_gpu: torch.Tensor, C_ref: np.ndarray, Cabs: np.ndarray,
                    same_sign: bool = False):
    """|C - C_ref| <= 1e-3 * sum|a b| + 1e-6 element for element: the stated
    bound, with nothing added, for every product whose terms differ in sign.

    same_sign=True is only for inputs whose products all share one sign, so
    that |C_ref| = sum|a b|.  There the final rounding of the FP32
    accumulator to a BF16 output alone (half an ulp, 2^-9 |C|) exceeds
    1e-3 * sum|a b|, so half an ulp of the output type at |C_ref| is added.
    Returns the worst ratio err / bound."""
    got = C_gpu.double().numpy()
    bound = oracle.tolerance(Cabs)
    if same_sign:
        bound = bound + HALF_ULP[C_gpu.dtype] * np.abs(C_ref)
    err = np.abs(got - C_ref)
    assert np.all(np.isfinite(got)), "non-finite output"
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{bad.sum()} elements out of bound, e.g. {idx.tolist()}: "
                             f"got {got[tuple(idx[0])]}, want {C_ref[tuple(idx[0])]}, "
                             f"bound {bound[tuple(idx[0])]}")
    return float(np.max(err / bound)) if err.size else 0.0


def expect_close(C_gpu: torch.Tensor, A: torch.Tensor, B: torch.Tensor, same_sign: bool = False):
    C_ref, Cabs = oracle.gemm(A, B)
    return tolerance_check(C_gpu, C_ref, Cabs, same_sign)


def sample_indices(M: int, N: int, count: int, seed: int, tile_m: int = 128, tile_n: int = 128):
    """Sampled output coordinates: random ones plus every corner and the
    first/last row and column of tiles along the edges."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, count))
    cols = list(rng.integers(0, N, count))
    edge_r = sorted({0, M - 1} | {min(M - 1, t) for t in range(tile_m - 1, M, tile_m)}
                    | {t for t in range(0, M, tile_m)})
    edge_c = sorted({0, N - 1} | {min(N - 1, t) for t in range(tile_n - 1, N, tile_n)}
                    | {t for t in range(0, N, tile_n)})
    for r in edge_r[:: max(1, len(edge_r) // 16)]:
        for c in edge_c[:: max(1, len(edge_c) // 16)]:
            rows.append(r)
            cols.append(c)
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)
