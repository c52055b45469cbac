"""gemm_splitk_noalloc: split-K for callers that cannot allocate device
memory (code under a framework that owns every allocation, real-time paths
where cudaMalloc may synchronize the device, services that reserve all
memory up front).  Its partials live in the library's fixed
scratch array instead of a caller workspace.

Checked through the C ABI on two calls in a row (different shapes and split
counts, so the second call reuses the scratch the first one left behind):
each result equals, bit for bit, that of the existing entry point,
gemm_splitk with a caller workspace, at the same split count (the same
kernels summing the same partials in the same order), and lies within the
element-wise bound |C - C_ref| <= 1e-3 sum|ab| + 1e-6 of the oracle's
product, the tolerance the other tests use.  This file is collected last so
that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tiled_matrix_multiplication_output_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.load_library(build_if_missing=True)
    tg.gemm_debug_config(0, -1)


def _both(A, B, splits, out_dtype):
    """(no-allocation result, caller-workspace result), both on the GPU."""
    dA, dB = A.cuda(), B.cuda()
    M, K = A.shape
    N = B.shape[1]
    odt = binding.dtype_code(out_dtype)
    stream = torch.cuda.current_stream().cuda_stream
    C_na = torch.empty((M, N), dtype=out_dtype, device="cuda")
    rc = tg.gemm_splitk_noalloc(dA.data_ptr(), dB.data_ptr(), C_na.data_ptr(), M, N, K, splits,
                                binding.dtype_code(A.dtype), tg.F32, odt, stream)
    assert rc == tg.binding.OK, tg.error_string(rc)
    C_ws = torch.empty((M, N), dtype=out_dtype, device="cuda")
    ws = torch.empty(tg.gemm_splitk_workspace_size(M, N, K, splits) + 16, dtype=torch.uint8,
                     device="cuda")
    rc = tg.gemm_splitk(dA.data_ptr(), dB.data_ptr(), C_ws.data_ptr(), M, N, K, splits,
                        binding.dtype_code(A.dtype), tg.F32, odt, ws.data_ptr(), ws.numel(),
                        stream)
    assert rc == tg.binding.OK, tg.error_string(rc)
    assert tg.gemm_device_status(stream) == tg.binding.OK
    return C_na.cpu(), C_ws.cpu()


def _check(C_noalloc, C_workspace, A, B):
    """Bit for bit equal to the caller-workspace entry point, and within the
    stated bound of the oracle's product."""
    assert torch.equal(C_noalloc.view(torch.uint8), C_workspace.view(torch.uint8))
    C_ref, Cabs = oracle.gemm(A, B)
    err = np.abs(C_noalloc.double().numpy() - C_ref)
    assert np.all(err <= oracle.tolerance(Cabs))


def test_two_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle():
    # first call: the edge workload's shape, 8 splits, FP32 output
    A1, B1 = inputs.draw(96, 200, 1000, "bf16", "normal", seed=80)
    got1, want1 = _both(A1, B1, 8, torch.float32)
    _check(got1, want1, A1, B1)
    # second call: another shape, more splits and a BF16 output, reusing the
    # scratch the first call left behind
    A2, B2 = inputs.draw(256, 264, 8200, "bf16", "normal", seed=81)
    got2, want2 = _both(A2, B2, 24, torch.bfloat16)
    _check(got2, want2, A2, B2)


def test_requests_beyond_the_scratch_are_rejected():
    M, N, K, splits = 1024, 1024, 8192, 8           # 32 MiB of partials > 8 MiB
    assert tg.gemm_splitk_workspace_size(M, N, K, splits) > binding.SPLITK_NOALLOC_MAX_BYTES
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 5.0, device="cuda")
    rc = tg.gemm_splitk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, splits,
                                tg.BF16, tg.F32, tg.F32, None)
    assert rc == tg.binding.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(C == 5.0)                       # nothing was launched
