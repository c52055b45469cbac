"""The latency-path kernel (tile16: one 16 x 16 output tile per block, the
tile's whole K range copied at once and split between the block's eight
warps; warp-level MMA for 16-bit inputs, FFMA for FP32) against the CPU
oracle: bit-exact on integer inputs in every layout and type, within the
stated bound on random ones, with its operand rules enforced."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tests.helpers import tolerance_check
from tiled_matrix_multiplication_output_gb300 import inputs

pytestmark = pytest.mark.gpu

OUT_TYPES = (torch.float32, torch.float16, torch.bfloat16)
OPS = (("n", "n"), ("t", "n"), ("n", "t"), ("t", "t"))
# sizes whose rows are a multiple of 16 bytes, for each input type
ALIGNED = {"f32": (4, 8, 12, 16), "f16": (8, 16), "bf16": (8, 16)}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.load_library()
    tg.gemm_debug_config(0, -1)
    yield


def _stored(A0, B0, op_a, op_b):
    A = A0.t().contiguous() if op_a == "t" else A0
    B = B0.t().contiguous() if op_b == "t" else B0
    return A, B


def _exact_batch(cases):
    """Each (M, N, K, in_dtype, out_dtype, op_a, op_b, seed) case launched on
    tile16 before one synchronisation, then compared bit for bit with
    the oracle's exact product of the integer inputs."""
    runs = []
    for M, N, K, in_dt, out_dt, op_a, op_b, seed in cases:
        A0, B0 = inputs.draw(M, N, K, in_dt, "int", seed=seed)
        A, B = _stored(A0, B0, op_a, op_b)
        C = tg.addmm(A.cuda(), B.cuda(), op_a=op_a, op_b=op_b, out_dtype=out_dt,
                     kernel="tile16")
        runs.append((A, B, op_a, op_b, C))
    assert tg.gemm_device_status(torch.cuda.current_stream().cuda_stream) == tg.binding.OK
    for A, B, op_a, op_b, C in runs:
        ref, _ = oracle.gemm_general(A, B, op_a, op_b)
        want = oracle.round_to(ref, C.dtype).double().numpy()
        got = C.cpu().double().numpy()
        if not np.array_equal(got, want):
            raise AssertionError(f"not exact: {tuple(A.shape)} {op_a}, {tuple(B.shape)} {op_b}, "
                                 f"{A.dtype} -> {C.dtype}")


def test_every_tiny_shape_every_layout():
    """Every (M, N, K) in {1..17}^3 that the kernel takes, in each of the
    four layouts: the stored row length of A (K as stored, M transposed) and
    of B (N as stored, K transposed) a multiple of 16 bytes, the other sizes
    free.  K free (A transposed, B as stored) exercises the partial last
    16-byte word along K and the warps left with no K at all.  Inputs cycle
    F32, F16, BF16 and outputs F32, F16, BF16, integer values in [-4, 4]."""
    cases = []
    i = 0
    for in_dt in ("f32", "f16", "bf16"):
        al = ALIGNED[in_dt]
        for op_a, op_b in OPS:
            a_pitch_is_k = op_a == "n"
            b_pitch_is_k = op_b == "t"
            ms = range(1, 18) if a_pitch_is_k else al
            ns = al if not b_pitch_is_k else range(1, 18)
            ks = al if (a_pitch_is_k or b_pitch_is_k) else range(1, 18)
            for M, N, K in itertools.product(ms, ns, ks):
                cases.append((M, N, K, in_dt, OUT_TYPES[i % 3], op_a, op_b, 9000 + i))
                i += 1
    assert len(cases) > 1500
    for start in range(0, len(cases), 400):
        _exact_batch(cases[start:start + 400])


@pytest.mark.parametrize("in_dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("op_a,op_b", OPS)
def test_ragged_grid_with_block_restarts(in_dt, op_a, op_b):
    """1304 x 1000 outputs (82 x 63 tiles, both edges partial) is more tiles
    than the grid has blocks (eight per SM), so blocks go on to further
    tiles and reuse their shared memory; K = 40 and K = 1000 split unevenly
    between the warps.  Integer inputs, exact, every output type."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 82 * 63 > 8 * sms
    cases = [(1304, 1000, K, in_dt, out, op_a, op_b, 9800 + K + j)
             for K in (40, 1000) for j, out in enumerate(OUT_TYPES)]
    _exact_batch(cases)


@pytest.mark.parametrize("in_dt,k_max,k_over", [("f16", 3392, 4096), ("bf16", 3392, 4096),
                                                 ("f32", 1696, 2048)])
def test_longest_k_and_the_shared_memory_limit(in_dt, k_max, k_over):
    """K near the largest the kernel takes (the K slices of one tile and the
    warps' partials in one block's shared memory, 227 KiB): exact; a K
    beyond it is refused with GEMM_ERR_UNSUPPORTED, and the automatic
    choice goes elsewhere."""
    _exact_batch([(40, 24, k_max, in_dt, torch.float32, op_a, op_b, 9900 + j)
                  for j, (op_a, op_b) in enumerate(OPS)])
    A = torch.zeros(40, k_over, dtype=tg.binding.torch_dtype(in_dt), device="cuda")
    B = torch.zeros(k_over, 24, dtype=A.dtype, device="cuda")
    with pytest.raises(tg.GemmError) as e:
        tg.matmul(A, B, kernel="tile16")
    assert e.value.code == tg.binding.ERR_UNSUPPORTED
    C = torch.empty(40, 24, device="cuda")
    k = tg.gemm_select_kernel(A.data_ptr(), B.data_ptr(), C.data_ptr(), 40, 24, k_over,
                              tg.binding.dtype_code(A.dtype), tg.F32, tg.F32)
    assert tg.KERNEL_NAMES[k] != "tile16"


def test_unaligned_operands_are_refused():
    """Rows of 10 BF16 elements (20 bytes), or an A that starts 4 bytes
    into its allocation: GEMM_ERR_UNSUPPORTED when forced; the automatic
    choice takes the tiled SIMT kernel, exact."""
    A, B = inputs.draw(64, 64, 10, "bf16", "int", seed=9950)
    with pytest.raises(tg.GemmError) as e:
        tg.matmul(A.cuda(), B.cuda(), kernel="tile16")
    assert e.value.code == tg.binding.ERR_UNSUPPORTED
    A2, B2 = inputs.draw(64, 64, 64, "bf16", "int", seed=9951)
    base = torch.zeros(64 * 64 + 2, dtype=torch.bfloat16, device="cuda")
    dA = base[2:].view(64, 64)
    dA.copy_(A2.cuda())
    with pytest.raises(tg.GemmError) as e:
        tg.matmul(dA, B2.cuda(), kernel="tile16")
    assert e.value.code == tg.binding.ERR_UNSUPPORTED
    C = tg.matmul(dA, B2.cuda())
    ref, _ = oracle.gemm(A2, B2, nthreads=1)
    np.testing.assert_array_equal(C.cpu().double().numpy(), ref)


@pytest.mark.parametrize("in_dt", ["f16", "bf16"])
def test_named_edge_workload_random_values(in_dt):
    """96 x 200 x 1000 (the edge workload's shape) with N(0, 1) inputs, every
    output type: within the stated bound 1e-3 sum|ab| + 1e-6 as it stands
    (random signs: the output rounding is far inside it)."""
    A, B = inputs.draw(96, 200, 1000, in_dt, "normal", seed=9960)
    C_ref, Cabs = oracle.gemm(A, B)
    for out in OUT_TYPES:
        C = tg.matmul(A.cuda(), B.cuda(), out_dtype=out, kernel="tile16").cpu()
        tolerance_check(C, C_ref, Cabs)


def test_fp32_random_values_and_run_to_run():
    """FP32 100 x 200 x 1000 and 520 x 392 x 1032 on N(0, 1): within the
    stated bound, and two runs bit-identical (a fixed split of K between
    the warps and a fixed order of their partials)."""
    for M, N, K, seed in ((100, 200, 1000, 9970), (520, 392, 1032, 9971)):
        A, B = inputs.draw(M, N, K, "f32", "normal", seed=seed)
        C_ref, Cabs = oracle.gemm(A, B)
        dA, dB = A.cuda(), B.cuda()
        C1 = tg.matmul(dA, dB, kernel="tile16").cpu()
        C2 = tg.matmul(dA, dB, kernel="tile16").cpu()
        tolerance_check(C1, C_ref, Cabs)
        assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


def test_k0_and_beta():
    """K = 0: C = beta * C (zeros when beta = 0, and C is not read)."""
    A = torch.zeros(40, 0, dtype=torch.float16, device="cuda")
    B = torch.zeros(0, 24, dtype=torch.float16, device="cuda")
    C = torch.full((40, 24), float("nan"), device="cuda")
    tg.addmm(A, B, C, beta=0.0, kernel="tile16")
    torch.cuda.synchronize()
    assert not C.any()
    C_in = torch.randint(-5, 6, (40, 24), device="cuda").float()
    C = C_in.clone()
    tg.addmm(A, B, C, alpha=3.0, beta=2.0, kernel="tile16")
    torch.cuda.synchronize()
    assert torch.equal(C, 2.0 * C_in)


@pytest.mark.parametrize("in_dt", ["f32", "bf16"])
@pytest.mark.parametrize("op_a,op_b", OPS)
def test_addmm_every_layout_and_output(in_dt, op_a, op_b):
    """C = 2 op(A) op(B) - C_in on tile16 with integer inputs and an integer
    C_in: exact in every output type (values stay below 2^11), every
    layout, FP32 and BF16 inputs; ragged 136 x 200 x 72."""
    M, N, K = 136, 200, 72
    A0, B0 = inputs.draw(M, N, K, in_dt, "int", lo=-2, hi=2, seed=9990)
    A, B = _stored(A0, B0, op_a, op_b)
    for j, out in enumerate(OUT_TYPES):
        C_in = torch.randint(-50, 51, (M, N), generator=torch.Generator().manual_seed(9991 + j)).to(out)
        C = tg.addmm(A.cuda(), B.cuda(), C_in.cuda(), op_a=op_a, op_b=op_b, alpha=2.0, beta=-1.0,
                     kernel="tile16").cpu()
        ref, _ = oracle.gemm_general(A, B, op_a, op_b, alpha=2.0, beta=-1.0, C_in=C_in)
        np.testing.assert_array_equal(C.double().numpy(),
                                      oracle.round_to(ref, out).double().numpy(),
                                      err_msg=f"{in_dt} {op_a}{op_b} -> {out}")
