"""gemm_general on the GPU: transposed operands (A stored K x M, B stored
N x K) and the alpha * op(A) op(B) + beta * C epilogue, on every kernel,
against the oracle's general form."""
import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tests.helpers import HALF_ULP, TC_KERNELS, tolerance_check
from tiled_matrix_multiplication_output_gb300 import inputs

pytestmark = pytest.mark.gpu

OPS = [("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.gemm_debug_config(0, -1)


def _stored(A0, B0, op_a, op_b):
    A = A0.t().contiguous() if op_a == "t" else A0
    B = B0.t().contiguous() if op_b == "t" else B0
    return A, B


def _run(A, B, op_a, op_b, kernel, alpha=1.0, beta=0.0, C_in=None, out_dtype=torch.float32):
    C = C_in.clone().cuda() if C_in is not None else None
    C = tg.addmm(A.cuda(), B.cuda(), C, op_a=op_a, op_b=op_b, alpha=alpha, beta=beta,
                 out_dtype=out_dtype, kernel=kernel)
    assert tg.gemm_device_status(torch.cuda.current_stream().cuda_stream) == 0
    return C.cpu()


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("kernel", TC_KERNELS + ("simt", "tile16", "auto"))
def test_transposes_exact(op_a, op_b, kernel):
    """Integer inputs, several tiles with ragged edges (304 x 264 x 520: all
    pitches multiples of 8 so every layout is tensor-core eligible)."""
    A0, B0 = inputs.draw(304, 264, 520, "bf16", "int", seed=60)
    A, B = _stored(A0, B0, op_a, op_b)
    C = _run(A, B, op_a, op_b, kernel)
    ref, _ = oracle.gemm_general(A, B, op_a, op_b)
    np.testing.assert_array_equal(C.double().numpy(), oracle.round_to(ref, torch.float32).double().numpy())


@pytest.mark.parametrize("op_a,op_b", OPS)
def test_transposes_random_tolerance(op_a, op_b):
    A0, B0 = inputs.draw(520, 392, 1032, "f16", "normal", seed=61)
    A, B = _stored(A0, B0, op_a, op_b)
    ref, Cabs = oracle.gemm_general(A, B, op_a, op_b)
    for kernel in TC_KERNELS + ("simt", "tile16"):
        for out in (torch.float32, torch.bfloat16):
            tolerance_check(_run(A, B, op_a, op_b, kernel, out_dtype=out), ref, Cabs)


@pytest.mark.parametrize("kernel", TC_KERNELS + ("simt", "simt_tpb3", "tile16"))
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_addmm_exact_integers(kernel, out_dtype):
    """alpha = 2, beta = -1 with integer C_in: exact in every output type
    (all values stay below 2^11)."""
    A0, B0 = inputs.draw(136, 200, 72, "f16", "int", lo=-2, hi=2, seed=62)
    C_in = torch.randint(-50, 51, (136, 200), generator=torch.Generator().manual_seed(1)).to(out_dtype)
    C = _run(A0, B0, "n", "n", kernel, alpha=2.0, beta=-1.0, C_in=C_in, out_dtype=out_dtype)
    ref, _ = oracle.gemm_general(A0, B0, alpha=2.0, beta=-1.0, C_in=C_in)
    np.testing.assert_array_equal(C.double().numpy(), oracle.round_to(ref, out_dtype).double().numpy())


@pytest.mark.parametrize("kernel", TC_KERNELS + ("simt", "tile16"))
def test_addmm_random_and_transposed(kernel):
    A0, B0 = inputs.draw(304, 264, 776, "bf16", "normal", seed=63)
    A, B = _stored(A0, B0, "t", "t")
    C_in = torch.randn(304, 264, generator=torch.Generator().manual_seed(2))
    C = _run(A, B, "t", "t", kernel, alpha=0.5, beta=1.5, C_in=C_in)
    ref, Cabs = oracle.gemm_general(A, B, "t", "t", alpha=0.5, beta=1.5, C_in=C_in)
    # the product's bound, plus FP32 rounding of the beta * C_in term
    bound = oracle.tolerance(Cabs) + 2.0 ** -22 * np.abs(1.5 * C_in.double().numpy())
    assert np.all(np.abs(C.double().numpy() - ref) <= bound)


def test_beta_zero_ignores_nan_in_c():
    A0, B0 = inputs.draw(256, 256, 64, "bf16", "int", seed=64)
    C_in = torch.full((256, 256), float("nan"))
    for kernel in TC_KERNELS + ("simt", "tile16"):
        C = _run(A0, B0, "n", "n", kernel, beta=0.0, C_in=C_in)
        assert torch.isfinite(C).all()


def test_k0_general_is_beta_c():
    A = torch.zeros(64, 0, dtype=torch.bfloat16)
    B = torch.zeros(0, 48, dtype=torch.bfloat16)
    C_in = torch.randint(-5, 6, (64, 48)).float()
    C = _run(A, B, "n", "n", "auto", alpha=3.0, beta=2.0, C_in=C_in)
    assert torch.equal(C, 2.0 * C_in)


def test_bad_op_rejected():
    rc = tg.gemm_general(16, 16, 16, 4, 4, 4, 7, 0, 1.0, 0.0, tg.BF16, tg.F32, tg.F32, 0, None)
    assert rc == tg.binding.ERR_INVALID_VALUE


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("kernel", TC_KERNELS)
@pytest.mark.parametrize("shape", [(304, 320, 192), (136, 192, 320), (520, 640, 1152)])
def test_half_full_last_stage_exact(op_a, op_b, kernel, shape):
    """K a multiple of 64 with an odd number of 64-wide K steps, so on the
    kernels whose stages hold two K steps the last stage is half full; N a
    multiple of 64 but not of the tile width; M ragged.  Integer inputs."""
    M, N, K = shape
    A0, B0 = inputs.draw(M, N, K, "f16", "int", seed=62)
    A, B = _stored(A0, B0, op_a, op_b)
    C = _run(A, B, op_a, op_b, kernel)
    ref, _ = oracle.gemm_general(A, B, op_a, op_b)
    np.testing.assert_array_equal(C.double().numpy(), oracle.round_to(ref, torch.float32).double().numpy())
