"""gemm_ex_ws: the persistent CTA-pair kernel with the tiles of its last,
partial wave split along K (FP32 partials in a caller workspace, summed in K
order by a second kernel).  Exact on integer inputs, identical run to run,
and equal to gemm_ex wherever the plan does not split.  The full-size
workloads through this entry point are checked element by element in
test_gpu_workloads.py."""
import numpy as np
import pytest
import torch

import tiled_matrix_multiplication_output_gb300 as tg
from tests.helpers import expect_exact
from tiled_matrix_multiplication_output_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.gemm_debug_config(0, -1)


def _ws(A, B, out_dtype=torch.float32, workspace=None):
    C = tg.matmul_ws(A.cuda(), B.cuda(), out_dtype=out_dtype, workspace=workspace)
    assert tg.gemm_device_status(torch.cuda.current_stream().cuda_stream) == 0
    return C.cpu()


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_split_last_wave_exact_integers(out_dtype):
    """2048 x 3072: 96 pair tiles over the resident pairs leaves a partial
    last wave of 20 tiles, each split into 3 K ranges; ragged K
    (776 = 12 * 64 + 8)."""
    A, B = inputs.draw(2048, 3072, 776, "bf16", "int", seed=90)
    expect_exact(_ws(A, B, out_dtype), A, B)


def test_ragged_edges_exact():
    A, B = inputs.draw(2400, 2504, 776, "f16", "int", seed=91)
    expect_exact(_ws(A, B), A, B)


def test_small_or_missing_workspace_falls_back():
    A, B = inputs.draw(2560, 2560, 256, "bf16", "int", seed=92)
    tiny = torch.empty(64, dtype=torch.uint8, device="cuda")
    expect_exact(_ws(A, B, workspace=tiny), A, B)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(2560, 2560, device="cuda")
    rc = tg.gemm_ex_ws(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 2560, 2560, 256, tg.BF16,
                       tg.F32, tg.F32, None, 0, None)
    assert rc == 0
    torch.cuda.synchronize()
    expect_exact(C.cpu(), A, B)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    rc = tg.gemm_ex_ws(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 2560, 2560, 256, tg.BF16,
                       tg.F32, tg.F32, ws.data_ptr() + 4, 1 << 19, None)
    assert rc == tg.binding.ERR_INVALID_VALUE


def test_workspace_size_bound():
    n = tg.gemm_workspace_size(8192, 8192, 8192)
    props = torch.cuda.get_device_properties(0)
    assert n == (props.multi_processor_count // 2) * 256 * 256 * 4
    assert tg.gemm_workspace_size(0, 8, 8) == 0


def test_workspace_path_shape_fuzz_exact():
    """gemm_ex_ws on 12 seeded random shapes (M, N up to 2600, K up to 1200,
    every output type): whatever it picks -- whole waves, a split last wave,
    few-tile split-K or another tile shape -- the result is exact on integer
    inputs."""
    rng = np.random.default_rng(2026)
    odts = [torch.float32, torch.float16, torch.bfloat16]
    for i in range(12):
        M = int(rng.integers(25, 326)) * 8
        N = int(rng.integers(25, 326)) * 8
        K = int(rng.integers(8, 151)) * 8
        A, B = inputs.draw(M, N, K, "bf16" if i % 2 else "f16", "int", seed=200 + i)
        expect_exact(_ws(A, B, odts[i % 3]), A, B)
