"""The five named workloads at their full sizes, through the C ABI in the
launch configuration bench.py times (automatic kernel choice).

Small workloads are compared with the oracle element by element; the 4096^3
and 8192^3 products are compared on sampled outputs (every tile corner and
edge plus random entries, each an oracle dot product) and by row and column
sums, which involve every output element."""
import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tests.conftest import load_golden
from tests.helpers import HALF_ULP, expect_exact, run_gpu, sample_indices, tolerance_check
from tiled_matrix_multiplication_output_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.gemm_debug_config(0, -1)


def _out(w):
    return binding.torch_dtype(w.out_dtype)


def test_worked_9x9():
    w = inputs.WORKLOADS["worked_9x9"]
    A, B = inputs.make(w)
    C = run_gpu(A, B, _out(w), "auto")
    expect_exact(C, A, B)
    assert C.sum().item() == 2420280


def test_square_128_f16_and_traffic_model():
    w = inputs.WORKLOADS["square_128_f16"]
    A, B = inputs.make(w)
    C_ref, Cabs = oracle.gemm(A, B)
    for kernel in ("auto", "tc_128x128", "tc_128x256", "tc_256x256", "tc_256x128", "simt"):
        tolerance_check(run_gpu(A, B, _out(w), kernel), C_ref, Cabs, with_output_rounding=False)
    g = load_golden("page_figures.txt")
    t = oracle.traffic(128, 128, 128, 16, 16, 32, in_bytes=2, acc_bytes=4, c_bytes=4)
    assert t["bytes"] == int(g["traffic_128_tile16x16x32_total_kib"]) * 1024
    assert t["flops"] == int(g["ops_128"]) == w.flops


def test_edge_96x200x1000_bf16_every_kernel():
    w = inputs.WORKLOADS["edge_96x200x1000_bf16"]
    A, B = inputs.make(w)
    C_ref, Cabs = oracle.gemm(A, B)
    for kernel in ("auto", "tc_128x128", "tc_128x256", "tc_256x256", "tc_256x128", "simt", "simt_tpb3"):
        tolerance_check(run_gpu(A, B, _out(w), kernel), C_ref, Cabs, with_output_rounding=False)


def _sums_check(C_gpu, A, B):
    """Row and column sums of C against FP64 sums of the products; the bound
    is the per-element bound summed (plus the output rounding of each
    element for 16-bit outputs)."""
    Ad, Bd = A.double(), B.double()
    Cd = C_gpu.double()
    rnd = HALF_ULP[C_gpu.dtype] if C_gpu.dtype != torch.float32 else 0.0
    # rows: sum_j C[i, j] = A[i, :] . (B 1)
    ref_r = (Ad @ Bd.sum(1)).numpy()
    abs_r = (Ad.abs() @ Bd.abs().sum(1)).numpy()
    got_r = Cd.sum(1).numpy()
    bound_r = 1e-3 * abs_r + 1e-6 * C_gpu.shape[1] + rnd * Cd.abs().sum(1).numpy()
    assert np.all(np.abs(got_r - ref_r) <= bound_r)
    # columns: sum_i C[i, j] = (1^T A) . B[:, j]
    ref_c = (Ad.sum(0) @ Bd).numpy()
    abs_c = (Ad.abs().sum(0) @ Bd.abs()).numpy()
    got_c = Cd.sum(0).numpy()
    bound_c = 1e-3 * abs_c + 1e-6 * C_gpu.shape[0] + rnd * Cd.abs().sum(0).numpy()
    assert np.all(np.abs(got_c - ref_c) <= bound_c)


@pytest.mark.parametrize("name", ["square_4096_f16", "square_8192_bf16"])
def test_large_workload_sampled(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.make(w)
    C = run_gpu(A, B, _out(w), "auto")
    assert C.shape == (w.M, w.N)
    assert torch.isfinite(C.float()).all()
    rows, cols = sample_indices(w.M, w.N, 3000, seed=w.seed, tile_m=256, tile_n=256)
    ref, ref_abs = oracle.gemm_entries(A, B, rows, cols)
    got = C[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
    # the stated bound, with no allowance for the output rounding
    assert np.all(np.abs(got - ref) <= oracle.tolerance(ref_abs))
    _sums_check(C, A, B)
    # run-to-run determinism at full size
    C2 = run_gpu(A, B, _out(w), "auto")
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))


def test_tall_product_many_tiles():
    """M = 131072 rows (512 pair tiles, 1024 single-CTA tiles) with a short K:
    sampled entries within the bound, row and column sums, on the automatic
    choice and on gemm_ex_ws."""
    A, B = inputs.draw(131072, 256, 136, "bf16", "normal", seed=30)
    for C in (run_gpu(A, B, torch.bfloat16, "auto"),
              tg.matmul_ws(A.cuda(), B.cuda(), out_dtype=torch.bfloat16).cpu()):
        rows, cols = sample_indices(131072, 256, 4000, seed=31, tile_m=256, tile_n=256)
        ref, ref_abs = oracle.gemm_entries(A, B, rows, cols)
        got = C[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
        half_ulp = HALF_ULP[torch.bfloat16] * np.abs(ref)
        assert np.all(np.abs(got - ref) <= oracle.tolerance(ref_abs) + half_ulp)
        _sums_check(C, A, B)


@pytest.mark.parametrize("M, N, K, out_dtype", [
    (2097152, 64, 64, torch.float32),      # 2^21 rows: 16384 tile rows, TMA row coordinates to 2^21
    (64, 2097152, 64, torch.bfloat16),     # 2^21 columns
    (128, 128, 1048576, torch.float32),    # 2^20 K steps of one element: one tile, 16384 K steps
])
def test_extreme_dimensions_sampled_exact(M, N, K, out_dtype):
    """Dimensions far beyond the named workloads, on the automatic choice and
    on gemm_ex_ws (split-K for the long-K case): integer inputs in [-1, 1]
    keep every sum exact in FP32 (|C| <= K <= 2^20), so sampled entries --
    every tile edge included -- must equal the oracle's, rounded to the
    output type."""
    A, B = inputs.draw(M, N, K, "bf16", "int", seed=40, lo=-1, hi=1)
    rows, cols = sample_indices(M, N, 3000, seed=41)
    ref, _ = oracle.gemm_entries(A, B, rows, cols)
    want = oracle.round_to(ref, out_dtype).double().numpy()
    for C in (run_gpu(A, B, out_dtype, "auto"),
              tg.matmul_ws(A.cuda(), B.cuda(), out_dtype=out_dtype).cpu()):
        got = C[torch.from_numpy(rows), torch.from_numpy(cols)].double().numpy()
        np.testing.assert_array_equal(got, want)
