"""The bounded-wait watchdog of the tensor-core kernel, exercised without any
GPU fault: the producer is told to skip the loads of one K step, so the MMA
warp's wait on that stage runs out of its (short) budget.  The kernel must
report GEMM_ERR_TIMEOUT through the status word, leave the context usable,
and the next product must be correct."""
import pytest
import torch

import tiled_matrix_multiplication_output_gb300 as tg
from tests.helpers import TC_KERNELS, expect_close, run_gpu
from tiled_matrix_multiplication_output_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _restore():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.gemm_debug_config(0, -1)
    yield
    tg.gemm_debug_config(0, -1)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_timeout_is_reported_and_context_survives(kernel):
    A, B = inputs.draw(512, 512, 1024, "bf16", "normal", seed=21)
    dA, dB = A.cuda(), B.cuda()
    sh = torch.cuda.current_stream().cuda_stream
    assert tg.gemm_device_status(sh) == tg.binding.OK
    # ~10 ms of SM clock per wait; K step 2 is never loaded
    tg.gemm_debug_config(20_000_000, 2)
    tg.matmul(dA, dB, kernel=kernel)
    assert tg.gemm_device_status(sh) == tg.binding.ERR_TIMEOUT
    tg.gemm_debug_config(0, -1)
    # the status word was cleared by the read
    assert tg.gemm_device_status(sh) == tg.binding.OK
    # the context still works and the next product is right
    expect_close(run_gpu(A, B, torch.float32, kernel), A, B)


def test_skip_beyond_k_changes_nothing():
    """A skip index past the last K step never fires."""
    A, B = inputs.draw(256, 256, 128, "f16", "int", seed=22)
    tg.gemm_debug_config(20_000_000, 1000)
    from tests.helpers import expect_exact
    expect_exact(run_gpu(A, B, torch.float32, "tc_128x128"), A, B)
