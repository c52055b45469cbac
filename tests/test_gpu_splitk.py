"""Split-K (gemm_splitk) on the GPU: FP32 partials per K range in a caller
workspace, summed in split order.  Exact on integer inputs, within the bound
on random inputs, identical run to run, and argument checks."""
import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tests.helpers import expect_exact, tolerance_check
from tiled_matrix_multiplication_output_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.gemm_debug_config(0, -1)


def _splitk(A, B, splits, out_dtype=torch.float32):
    C = tg.matmul_splitk(A.cuda(), B.cuda(), splits, out_dtype=out_dtype)
    assert tg.gemm_device_status(torch.cuda.current_stream().cuda_stream) == 0
    return C.cpu()


@pytest.mark.parametrize("splits", [1, 2, 5, 16, 1000])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_splitk_exact_integers(splits, out_dtype):
    """The edge-tile workload's shape (96 x 200 x 1000): partial tiles in M, N
    and K; integer inputs, so every split count gives the exact product."""
    A, B = inputs.draw(96, 200, 1000, "bf16", "int", seed=70)
    expect_exact(_splitk(A, B, splits, out_dtype), A, B)


def test_splitk_edge_workload_within_bound():
    w = inputs.WORKLOADS["edge_96x200x1000_bf16"]
    A, B = inputs.make(w)
    ref, Cabs = oracle.gemm(A, B)
    for splits in (2, 4, 8, 16):
        tolerance_check(_splitk(A, B, splits), ref, Cabs)


def test_splitk_long_k_many_splits():
    A, B = inputs.draw(256, 264, 16392, "f16", "uniform", seed=71)
    ref, Cabs = oracle.gemm(A, B)
    C = _splitk(A, B, 48)
    tolerance_check(C, ref, Cabs)
    C2 = _splitk(A, B, 48)
    assert torch.equal(C, C2)


def test_workspace_size_and_checks():
    assert tg.gemm_splitk_workspace_size(96, 200, 1000, 4) == 4 * 96 * 200 * 4
    # 16 K steps into 5 ranges: 4 steps per range, 4 ranges used
    assert tg.gemm_splitk_workspace_size(96, 200, 1000, 5) == 4 * 96 * 200 * 4
    assert tg.gemm_splitk_workspace_size(96, 200, 1000, 1000) == 16 * 96 * 200 * 4
    assert tg.gemm_splitk_workspace_size(0, 200, 1000, 4) == 0
    A = torch.zeros(96, 1000, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1000, 200, dtype=torch.bfloat16, device="cuda")
    C = torch.empty(96, 200, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    rc = tg.gemm_splitk(A.data_ptr(), B.data_ptr(), C.data_ptr(), 96, 200, 1000, 4, tg.BF16,
                        tg.F32, tg.F32, ws.data_ptr(), 1024, None)
    assert rc == tg.binding.ERR_INVALID_VALUE       # workspace too small
    rc = tg.gemm_splitk(A.data_ptr(), B.data_ptr(), C.data_ptr(), 96, 200, 1000, 0, tg.BF16,
                        tg.F32, tg.F32, ws.data_ptr(), 1024, None)
    assert rc == tg.binding.ERR_INVALID_VALUE       # splits < 1


def test_splitk_unaligned_falls_back_exactly():
    A, B = inputs.draw(50, 37, 333, "f16", "int", seed=72)   # no TMA-legal pitches
    C = tg.matmul_splitk(A.cuda(), B.cuda(), 4)
    expect_exact(C.cpu(), A, B)


def test_gemm_ex_ws_splits_few_tile_products():
    """gemm_ex_ws takes split-K for few output tiles and a long K (32 K steps
    or more; 96 x 200 x 4000 here): two launches, bit for bit the result of
    gemm_splitk with the reported count, on integer and on random inputs;
    large products and shorter K are not split (the 96 x 200 x 1000
    workload, and up to K = 2048, run on the 16 x 16-tile kernel in a
    single launch)."""
    M, N, K = 96, 200, 4000
    count = tg.gemm_ws_split_count(M, N, K, tg.BF16, tg.F32, tg.F32)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert count == min(sms // 2, 8)      # 2 tiles, 63 K steps: up to one unit per SM, 8 ranges at most
    assert tg.gemm_ws_split_count(8192, 8192, 8192, tg.BF16, tg.F32, tg.BF16) == 0
    assert tg.gemm_ws_split_count(128, 128, 128, tg.F16, tg.F32, tg.F32) == 0
    assert tg.gemm_ws_split_count(96, 200, 1000, tg.BF16, tg.F32, tg.F32) == 0  # 16 K steps
    assert tg.gemm_ws_split_count(96, 200, 2048, tg.BF16, tg.F32, tg.F32) == 0  # tile16 (K <= 2048)
    assert tg.gemm_ws_split_count(96, 200, 2056, tg.BF16, tg.F32, tg.F32) >= 2  # 33 K steps
    assert tg.gemm_ws_split_count(96, 200, 4000, tg.F32, tg.F32, tg.F32) == 0   # SIMT path
    assert tg.gemm_ws_split_count(-1, 200, 1000, tg.BF16, tg.F32, tg.F32) == -tg.binding.ERR_INVALID_VALUE
    A, B = inputs.draw(M, N, K, "bf16", "int", seed=31)
    dA, dB = A.cuda(), B.cuda()
    s = torch.cuda.current_stream().cuda_stream
    ws_bytes = tg.gemm_workspace_size(M, N, K)
    assert ws_bytes >= tg.gemm_splitk_workspace_size(M, N, K, count)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), float("nan"), device="cuda")
    n0 = tg.gemm_launch_count()
    rc = tg.gemm_ex_ws(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, tg.BF16, tg.F32,
                       tg.F32, ws.data_ptr(), ws_bytes, s)
    assert rc == 0
    assert tg.gemm_launch_count() - n0 == 2
    assert tg.gemm_device_status(s) == 0
    expect_exact(C.cpu(), A, B)
    ws2 = torch.empty(tg.gemm_splitk_workspace_size(M, N, K, count), dtype=torch.uint8, device="cuda")
    for dist in ("int", "normal"):
        A, B = inputs.draw(M, N, K, "bf16", dist, seed=32)
        dA, dB = A.cuda(), B.cuda()
        C = torch.empty((M, N), device="cuda")
        C2 = torch.empty((M, N), device="cuda")
        assert tg.gemm_ex_ws(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, tg.BF16, tg.F32,
                             tg.F32, ws.data_ptr(), ws_bytes, s) == 0
        rc = tg.gemm_splitk(dA.data_ptr(), dB.data_ptr(), C2.data_ptr(), M, N, K, count, tg.BF16,
                            tg.F32, tg.F32, ws2.data_ptr(), ws2.numel(), s)
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int32), C2.view(torch.int32)), dist


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [(96, 200, 3000), (100, 136, 2056), (384, 256, 4096)])
def test_gemm_ex_ws_few_tile_split_every_output_type(shape, out_dtype):
    """The few-tile split path of gemm_ex_ws on ragged shapes and every output
    type: exact on integer inputs, within the bound on random ones, and
    identical run to run (the partials are added in a fixed order)."""
    M, N, K = shape
    code = {torch.float32: tg.F32, torch.float16: tg.F16, torch.bfloat16: tg.BF16}[out_dtype]
    assert tg.gemm_ws_split_count(M, N, K, tg.F16, tg.F32, code) >= 2
    s = torch.cuda.current_stream().cuda_stream
    ws_bytes = tg.gemm_workspace_size(M, N, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for dist in ("int", "normal"):
        A, B = inputs.draw(M, N, K, "f16", dist, seed=33)
        dA, dB = A.cuda(), B.cuda()
        outs = []
        for _ in range(2):
            C = torch.empty((M, N), dtype=out_dtype, device="cuda")
            assert tg.gemm_ex_ws(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, tg.F16, tg.F32,
                                 code, ws.data_ptr(), ws_bytes, s) == 0
            outs.append(C)
        assert tg.gemm_device_status(s) == 0
        assert torch.equal(outs[0].view(torch.uint8), outs[1].view(torch.uint8))
        if dist == "int":
            expect_exact(outs[0].cpu(), A, B)
        else:
            C_ref, Cabs = oracle.gemm(A, B)
            tolerance_check(outs[0].cpu(), C_ref, Cabs)


def test_gemm_ex_ws_edge_workload_is_one_launch():
    """The 96 x 200 x 1000 workload through gemm_ex_ws: 16 K steps are short
    of the split threshold, so one launch of the single-tile kernel, exact
    on integer inputs."""
    M, N, K = 96, 200, 1000
    A, B = inputs.draw(M, N, K, "bf16", "int", seed=34)
    dA, dB = A.cuda(), B.cuda()
    s = torch.cuda.current_stream().cuda_stream
    ws_bytes = tg.gemm_workspace_size(M, N, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    C = torch.full((M, N), float("nan"), device="cuda")
    n0 = tg.gemm_launch_count()
    assert tg.gemm_ex_ws(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, tg.BF16, tg.F32,
                         tg.F32, ws.data_ptr(), ws_bytes, s) == 0
    assert tg.gemm_launch_count() - n0 == 1
    assert tg.gemm_device_status(s) == 0
    expect_exact(C.cpu(), A, B)
