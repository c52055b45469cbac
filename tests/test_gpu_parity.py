"""Parity of the CUDA path (through the C ABI) with the CPU oracle on seeded
inputs: bit-exact on integer-valued inputs, within the stated tolerance on
random FP16/BF16/FP32 inputs, on every kernel, at sizes spanning several
tiles with ragged tails in M, N and K."""
import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tests.conftest import load_worked_9x9
from tests.helpers import ALL_KERNELS, TC_KERNELS, expect_close, expect_exact, run_gpu
from tiled_matrix_multiplication_output_gb300 import inputs

pytestmark = pytest.mark.gpu

OUT_TYPES = (torch.float32, torch.float16, torch.bfloat16)


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    tg.load_library()
    tg.gemm_debug_config(0, -1)
    yield


# -------------------------------------------------- the worked 9x9 example

@pytest.mark.parametrize("kernel", ["simt_tpb3", "simt", "auto"])
def test_worked_example_bit_exact(kernel):
    A, B = load_worked_9x9()
    A = torch.tensor(A, dtype=torch.float32)
    B = torch.tensor(B, dtype=torch.float32)
    C = run_gpu(A, B, torch.float32, kernel)
    want = torch.tensor([[5832 * i + 162 * i * j + 72 * j + 3672 for j in range(9)]
                         for i in range(9)], dtype=torch.float32)
    assert torch.equal(C, want)
    expect_exact(C, A, B)


# ------------------------------------------- first tensor-core smoke cases

@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_tc_single_tile_exact(kernel):
    """One full tile, integer inputs: every element exact."""
    A, B = inputs.draw(128, 128, 64, "bf16", "int", seed=1)
    expect_exact(run_gpu(A, B, torch.float32, kernel), A, B)


@pytest.mark.parametrize("kernel", TC_KERNELS)
@pytest.mark.parametrize("in_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out_dtype", OUT_TYPES)
def test_tc_ragged_exact(kernel, in_dtype, out_dtype):
    """Several tiles, ragged in every dimension (300 = 2*128 + 44 rows,
    264 = 256 + 8 columns, 520 = 8*64 + 8 K), integer inputs."""
    A, B = inputs.draw(300, 264, 520, in_dtype, "int", seed=2)
    expect_exact(run_gpu(A, B, out_dtype, kernel), A, B)


@pytest.mark.parametrize("kernel", ["simt", "simt_tpb3"])
@pytest.mark.parametrize("in_dtype", ["f32", "f16", "bf16"])
def test_simt_ragged_exact(kernel, in_dtype):
    M, N, K = (70, 45, 101) if kernel == "simt_tpb3" else (150, 133, 77)
    A, B = inputs.draw(M, N, K, in_dtype, "int", seed=3)
    for out in OUT_TYPES:
        expect_exact(run_gpu(A, B, out, kernel), A, B)


# ------------------------------------------------- brute force, tiny shapes

def test_brute_force_tiny_shapes_all_kernels():
    """M, N in 1..17 and K in 1..17 sampled (plus a few tile edges), integer
    inputs: every kernel that accepts the shape is bit-exact."""
    rng = np.random.default_rng(5)
    dims = list(range(1, 18)) + [63, 64, 65, 127, 128, 129]
    for trial in range(40):
        M, N, K = (int(rng.choice(dims)) for _ in range(3))
        A, B = inputs.draw(M, N, K, "bf16", "int", seed=trial)
        for kernel in ("simt", "simt_tpb3"):
            expect_exact(run_gpu(A, B, torch.float32, kernel), A, B)
    # tensor-core kernels need N and K multiples of 8 (16-byte rows)
    for trial in range(24):
        M = int(rng.integers(1, 300))
        N = 8 * int(rng.integers(1, 40))
        K = 8 * int(rng.integers(1, 40))
        A, B = inputs.draw(M, N, K, "f16", "int", seed=100 + trial)
        for kernel in TC_KERNELS:
            expect_exact(run_gpu(A, B, torch.float32, kernel), A, B)


# ----------------------------------------------- random values, tolerance

@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_random_bf16_within_tolerance(kernel):
    M, N, K = (200, 136, 1000) if kernel != "simt_tpb3" else (40, 24, 300)
    A, B = inputs.draw(M, N, K, "bf16", "normal", seed=7)
    for out in OUT_TYPES:
        expect_close(run_gpu(A, B, out, kernel), A, B)


@pytest.mark.parametrize("kernel", ["simt", "auto"])
def test_random_f32_within_tolerance(kernel):
    A, B = inputs.draw(257, 129, 515, "f32", "normal", seed=8)
    expect_close(run_gpu(A, B, torch.float32, kernel), A, B, with_output_rounding=False)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_large_k_and_many_tiles(kernel):
    """K = 4104 (64 K steps + a ragged 8) and a 3 x 5 grid of tiles."""
    A, B = inputs.draw(520, 1160, 4104, "f16", "uniform", seed=9)
    expect_close(run_gpu(A, B, torch.float32, kernel), A, B, with_output_rounding=False)


# ---------------------------------------------------------- special cases

def test_k0_writes_zeros():
    for kernel in ("auto", "simt"):
        A = torch.zeros(37, 0, dtype=torch.bfloat16, device="cuda")
        B = torch.zeros(0, 24, dtype=torch.bfloat16, device="cuda")
        out = torch.full((37, 24), 7.0, device="cuda")
        tg.matmul(A, B, out=out, kernel=kernel)
        torch.cuda.synchronize()
        assert not out.any()


def test_m0_n0_noop():
    A = torch.zeros(0, 16, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(16, 8, dtype=torch.bfloat16, device="cuda")
    out = tg.matmul(A, B)
    assert out.shape == (0, 8)
    rc = tg.gemm_ex(0, 0, 0, 0, 0, 5, tg.BF16, tg.F32, tg.F32, None)
    assert rc == 0


def test_identity_and_gemv():
    A, _ = inputs.draw(256, 1, 256, "bf16", "normal", seed=10)
    eye = torch.eye(256, dtype=torch.bfloat16)
    for kernel in TC_KERNELS + ("simt",):
        C = run_gpu(A, eye, torch.float32, kernel)
        assert torch.equal(C, A.float())
    # M = 1: a row vector times a matrix
    a, b = inputs.draw(1, 512, 384, "bf16", "normal", seed=11)
    for kernel in TC_KERNELS:
        expect_close(run_gpu(a, b, torch.float32, kernel), a, b)


def test_deterministic_run_to_run():
    A, B = inputs.draw(640, 768, 2048, "bf16", "normal", seed=12)
    for kernel in TC_KERNELS:
        C1 = run_gpu(A, B, torch.bfloat16, kernel)
        C2 = run_gpu(A, B, torch.bfloat16, kernel)
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))


def test_forced_tc_rejects_unaligned():
    A = torch.zeros(64, 10, dtype=torch.bfloat16, device="cuda")   # K*2 = 20 bytes
    B = torch.zeros(10, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.GemmError) as e:
        tg.matmul(A, B, kernel="tc_128x128")
    assert e.value.code == tg.binding.ERR_UNSUPPORTED
    out = tg.matmul(A, B)   # auto picks the SIMT kernel
    torch.cuda.synchronize()
    assert not out.any()


def test_unaligned_shapes_route_to_simt_and_are_exact():
    A, B = inputs.draw(129, 131, 77, "f16", "int", seed=13)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty(129, 131, device="cuda")
    k = tg.gemm_select_kernel(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 129, 131, 77,
                              tg.F16, tg.F32, tg.F32)
    assert tg.KERNEL_NAMES[k] == "simt"
    expect_exact(run_gpu(A, B, torch.float32, "auto"), A, B)


def test_host_buffer_entry_point():
    A, B = inputs.draw(300, 264, 520, "bf16", "normal", seed=14)
    C = torch.empty(300, 264, dtype=torch.bfloat16).pin_memory()
    Ah, Bh = A.pin_memory(), B.pin_memory()
    dA = torch.empty_like(A, device="cuda")
    dB = torch.empty_like(B, device="cuda")
    dC = torch.empty_like(C, device="cuda")
    s = torch.cuda.current_stream()
    rc = tg.gemm_ex_host(Ah.data_ptr(), Bh.data_ptr(), C.data_ptr(), 300, 264, 520, tg.BF16,
                         tg.F32, tg.BF16, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                         s.cuda_stream)
    assert rc == 0
    s.synchronize()
    expect_close(C, A, B)


def test_stream_ordering_on_side_stream():
    A, B = inputs.draw(512, 512, 512, "bf16", "normal", seed=15)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA, dB = A.cuda(), B.cuda()
        C = tg.matmul(dA, dB, out_dtype=torch.float32)
        Ch = C.cpu()
    s.synchronize()
    expect_close(Ch, A, B, with_output_rounding=False)


def test_host_buffer_entry_point_pipelined():
    """More than 1024 rows: the host-buffer path runs in row panels on its
    own copy streams; the result is exact on integer inputs, and a second
    call right after the first (other inputs, same device buffers) sees its
    own inputs only."""
    M, N, K = 4100, 520, 264            # 5 panels of 1024 rows, the last one 4 rows
    s = torch.cuda.current_stream()
    dA = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(K, N, dtype=torch.bfloat16, device="cuda")
    dC = torch.empty(M, N, dtype=torch.float32, device="cuda")
    outs = []
    for seed in (15, 16):
        A, B = inputs.draw(M, N, K, "bf16", "int", seed=seed)
        Ah, Bh = A.pin_memory(), B.pin_memory()
        C = torch.empty(M, N, dtype=torch.float32).pin_memory()
        rc = tg.gemm_ex_host(Ah.data_ptr(), Bh.data_ptr(), C.data_ptr(), M, N, K, tg.BF16,
                             tg.F32, tg.F32, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                             s.cuda_stream)
        assert rc == 0
        outs.append((A, B, C, Ah, Bh))
    s.synchronize()
    for A, B, C, _, _ in outs:
        expect_exact(C, A, B)
    # work queued after the call on the same stream sees the finished product
    assert torch.equal(dC.cpu(), outs[-1][2])


def test_automatic_choice_on_the_named_workloads():
    """The cost model's picks on the named workloads: the single-CTA kernel
    for one-tile problems (lowest fixed latency), the CTA-pair kernel for the
    large squares, SIMT for FP32 and for shapes the tensor maps cannot take."""
    def pick(M, N, K, in_dt, out_dt, dtype=torch.bfloat16):
        A = torch.zeros(M, K, dtype=dtype, device="cuda")
        B = torch.zeros(K, N, dtype=dtype, device="cuda")
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        return tg.KERNEL_NAMES[tg.gemm_select_kernel(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                                     M, N, K, in_dt, tg.F32, out_dt)]
    assert pick(9, 9, 9, tg.F32, tg.F32, torch.float32) == "simt"
    assert pick(128, 128, 128, tg.F16, tg.F32, torch.float16) == "tc_128x128"
    assert pick(96, 200, 1000, tg.BF16, tg.F32) == "tc_128x128"
    assert pick(4096, 4096, 4096, tg.F16, tg.F16, torch.float16) == "tc_256x256"
    assert pick(8192, 8192, 8192, tg.BF16, tg.BF16) == "tc_256x256"


@pytest.mark.parametrize("in_dtype", ["f32", "f16"])
def test_simt_large_tile_kernel_exact(in_dtype):
    """Grids of at least one 128 x 128 tile per SM take the SIMT kernel's
    large-tile form: ragged in every dimension (2051 x 1283 x 77: 17 x 11
    tiles, 9 K tiles of 8 with a partial last one), integer inputs, every
    output type; exact."""
    A, B = inputs.draw(2051, 1283, 77, in_dtype, "int", seed=16)
    assert 17 * 11 >= torch.cuda.get_device_properties(0).multi_processor_count
    for out in OUT_TYPES:
        expect_exact(run_gpu(A, B, out, "simt"), A, B)


def test_simt_large_tile_kernel_transposed_and_addmm():
    """The large-tile SIMT kernel with transposed operands and the
    alpha/beta store, against the oracle's general form (integer inputs,
    exact)."""
    M, N, K = 2048, 1536, 40
    A0, B0 = inputs.draw(M, N, K, "f32", "int", seed=17)
    Cin = inputs.draw(M, 1, N, "f32", "int", seed=18)[0]          # an M x N integer matrix
    for op_a, op_b in (("t", "n"), ("n", "t"), ("t", "t")):
        A = A0.t().contiguous() if op_a == "t" else A0
        B = B0.t().contiguous() if op_b == "t" else B0
        C = tg.addmm(A.cuda(), B.cuda(), Cin.clone().cuda(), op_a=op_a, op_b=op_b, alpha=2.0,
                     beta=-1.0, out_dtype=torch.float32, kernel="simt").cpu()
        ref, _ = oracle.gemm_general(A, B, op_a, op_b, alpha=2.0, beta=-1.0, C_in=Cin)
        np.testing.assert_array_equal(C.double().numpy(), ref)


@pytest.mark.parametrize("op_a,op_b", [("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")])
def test_simt_large_tile_kernel_layouts_ragged_k_tiles(op_a, op_b):
    """The large-tile SIMT kernel in every operand layout, ragged in M, N
    and K, with 1, 2, 3 and 10 K tiles of 8: the counts at which its
    register prefetch (one K tile ahead, or two ahead for A transposed with
    B as stored) starts, runs and drains differently.  Integer inputs,
    exact against the oracle's general form; FP16 inputs on one case."""
    M, N = 2051, 1283
    for K, in_dtype, seed in ((5, "f32", 40), (13, "f32", 41), (21, "f32", 42),
                              (77, "f32", 43), (21, "f16", 44)):
        A0, B0 = inputs.draw(M, N, K, in_dtype, "int", seed=seed)
        A = A0.t().contiguous() if op_a == "t" else A0
        B = B0.t().contiguous() if op_b == "t" else B0
        C = tg.addmm(A.cuda(), B.cuda(), op_a=op_a, op_b=op_b, out_dtype=torch.float32,
                     kernel="simt").cpu()
        ref, _ = oracle.gemm_general(A, B, op_a, op_b)
        np.testing.assert_array_equal(C.double().numpy(), ref, err_msg=f"K={K} {in_dtype}")
