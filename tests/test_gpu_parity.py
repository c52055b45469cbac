"""Parity of the CUDA path (through the C ABI) with the CPU oracle on seeded
inputs: bit-exact on integer-valued inputs, within the stated tolerance on
random FP16/BF16/FP32 inputs, on every kernel, at sizes spanning several
tiles with ragged tails in M, N and K."""
import itertools

import numpy as np
import pytest
import torch

import oracle
import tiled_matrix_multiplication_output_gb300 as tg
from tests.conftest import load_worked_9x9
from tests.helpers import (ALL_KERNELS, TC_KERNELS, expect_close, expect_exact, run_gpu,
                           tolerance_check)
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

def _exact_cases(cases, kernels):
    """Each (M, N, K, in_dtype, out_dtype, seed) case on each kernel, all
    launched before one synchronisation, then compared bit for bit with the
    oracle's exact integer product rounded to the output type."""
    runs = []
    for M, N, K, in_dt, out_dt, seed in cases:
        A, B = inputs.draw(M, N, K, in_dt, "int", seed=seed)
        dA, dB = A.cuda(), B.cuda()
        outs = [(k, tg.matmul(dA, dB, out_dtype=out_dt, kernel=k)) for k in kernels]
        runs.append((A, B, outs))
    assert tg.gemm_device_status(torch.cuda.current_stream().cuda_stream) == tg.binding.OK
    for A, B, outs in runs:
        C_ref, _ = oracle.gemm(A, B, nthreads=1)
        for kernel, C in outs:
            want = oracle.round_to(C_ref, C.dtype).double().numpy()
            got = C.cpu().double().numpy()
            if not np.array_equal(got, want):
                raise AssertionError(f"{kernel} not exact at M, N, K = {tuple(A.shape) + (B.shape[1],)}")


OUT_CYCLE = (torch.float32, torch.float16, torch.bfloat16)


def test_brute_force_every_tiny_shape_simt():
    """Every (M, N, K) in {1..17}^3 (4913 shapes) on both SIMT kernels,
    integer inputs in [-4, 4]: bit-exact.  The input type cycles F32, F16,
    BF16 and the output type F32, F16, BF16 (offset), so every pair occurs."""
    in_cycle = ("f32", "f16", "bf16")
    cases = [(M, N, K, in_cycle[i % 3], OUT_CYCLE[(i // 3) % 3], i)
             for i, (M, N, K) in enumerate(itertools.product(range(1, 18), repeat=3))]
    for start in range(0, len(cases), 500):
        _exact_cases(cases[start:start + 500], ("simt", "simt_tpb3"))


def test_brute_force_every_tiny_shape_tensor_cores():
    """Every (M, 8n, 8k) in the {1..17}^3 cube -- M in 1..17, N and K in
    {8, 16}, the sizes whose 16-bit rows meet the 16-byte TMA rule -- on
    every tensor-core kernel, FP16 and BF16 inputs, every output type."""
    cases = [(M, N, K, "f16" if i % 2 else "bf16", OUT_CYCLE[i % 3], 5000 + i)
             for i, (M, N, K) in enumerate(itertools.product(range(1, 18), (8, 16), (8, 16)))]
    _exact_cases(cases, TC_KERNELS)


def test_brute_force_tile_edges_all_kernels():
    """Dimensions one below and one above a 64- and a 128-wide tile
    (63, 65, 127, 129) against tiny ones, on every kernel that accepts them:
    SIMT for any size, tensor cores for N and K multiples of 8."""
    dims = (1, 17, 63, 65, 127, 129)
    simt = [(M, N, K, "bf16", OUT_CYCLE[i % 3], 6000 + i)
            for i, (M, N, K) in enumerate(itertools.product(dims, repeat=3)) if max(M, N, K) >= 63]
    _exact_cases(simt, ("simt", "simt_tpb3"))
    tc = [(M, N, K, "f16", OUT_CYCLE[i % 3], 7000 + i)
          for i, (M, N, K) in enumerate(itertools.product(dims, (8, 64, 72, 136), (8, 56, 72, 136)))]
    _exact_cases(tc, TC_KERNELS)


def test_random_tensor_core_shapes_exact():
    """24 seeded random shapes up to 300 x 320 x 320 on every tensor-core
    kernel, integer inputs: bit-exact."""
    rng = np.random.default_rng(5)
    cases = []
    for trial in range(24):
        M = int(rng.integers(1, 300))
        N = 8 * int(rng.integers(1, 40))
        K = 8 * int(rng.integers(1, 40))
        cases.append((M, N, K, "f16", torch.float32, 100 + trial))
    _exact_cases(cases, TC_KERNELS)


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
    expect_close(run_gpu(A, B, torch.float32, kernel), A, B)


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_same_sign_products(kernel):
    """Inputs on U[0, 1]: every product positive, so |C_ref| = sum|ab|.  FP32
    and FP16 outputs meet the stated bound as it is; a BF16 output gets half
    an ulp of BF16 on top, because its final rounding alone (2^-9 |C|)
    exceeds 1e-3 sum|ab| when nothing cancels."""
    M, N, K = (200, 136, 1000) if kernel != "simt_tpb3" else (40, 24, 300)
    A, B = inputs.draw(M, N, K, "bf16", "positive", seed=16)
    C_ref, Cabs = oracle.gemm(A, B)
    for out in (torch.float32, torch.float16):
        tolerance_check(run_gpu(A, B, out, kernel), C_ref, Cabs)
    tolerance_check(run_gpu(A, B, torch.bfloat16, kernel), C_ref, Cabs, same_sign=True)


@pytest.mark.parametrize("kernel", TC_KERNELS)
def test_large_k_and_many_tiles(kernel):
    """K = 4104 (64 K steps + a ragged 8) and a 3 x 5 grid of tiles."""
    A, B = inputs.draw(520, 1160, 4104, "f16", "uniform", seed=9)
    expect_close(run_gpu(A, B, torch.float32, kernel), A, B)


# ---------------------------------------------------------- special cases

def test_k0_writes_zeros():
    for kernel in ("auto", "simt", "tile16"):
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
    for kernel in TC_KERNELS + ("simt", "tile16"):
        C = run_gpu(A, eye, torch.float32, kernel)
        assert torch.equal(C, A.float())
    # M = 1: a row vector times a matrix
    a, b = inputs.draw(1, 512, 384, "bf16", "normal", seed=11)
    for kernel in TC_KERNELS + ("tile16",):
        expect_close(run_gpu(a, b, torch.float32, kernel), a, b)


def test_deterministic_run_to_run():
    A, B = inputs.draw(640, 768, 2048, "bf16", "normal", seed=12)
    for kernel in TC_KERNELS + ("tile16",):
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
    expect_close(Ch, A, B)


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


@pytest.mark.parametrize("M, N, K, out_dtype", [
    (4100, 520, 264, torch.float32),     # 5 panels of 1024 rows, the last one 4 rows
    (8192, 2048, 776, torch.bfloat16),   # 8 panels of 1024 rows: 32 pair tiles each, one
                                         # partial wave split along K in every panel
    (700, 4096, 1024, torch.float16),    # a single piece
])
def test_host_buffer_entry_point_with_workspace(M, N, K, out_dtype):
    """gemm_ex_host_ws: each panel's product through the workspace path
    (last-wave split); exact on integer inputs, as gemm_ex_host is, and within
    the stated bound on random inputs."""
    s = torch.cuda.current_stream()
    dA = torch.empty(M, K, dtype=torch.float16, device="cuda")
    dB = torch.empty(K, N, dtype=torch.float16, device="cuda")
    dC = torch.empty(M, N, dtype=out_dtype, device="cuda")
    ws_bytes = tg.gemm_workspace_size(M, N, K)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    code = tg.binding.dtype_code(out_dtype)
    for dist in ("int", "normal"):
        A, B = inputs.draw(M, N, K, "f16", dist, seed=34)
        Ah, Bh = A.pin_memory(), B.pin_memory()
        C_ws = torch.empty(M, N, dtype=out_dtype).pin_memory()
        C_plain = torch.empty(M, N, dtype=out_dtype).pin_memory()
        rc = tg.gemm_ex_host_ws(Ah.data_ptr(), Bh.data_ptr(), C_ws.data_ptr(), M, N, K, tg.F16,
                                tg.F32, code, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                                ws.data_ptr(), ws_bytes, s.cuda_stream)
        assert rc == 0
        s.synchronize()
        rc = tg.gemm_ex_host(Ah.data_ptr(), Bh.data_ptr(), C_plain.data_ptr(), M, N, K, tg.F16,
                             tg.F32, code, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                             s.cuda_stream)
        assert rc == 0
        assert tg.gemm_device_status(s.cuda_stream) == 0
        if dist == "int":
            expect_exact(C_ws, A, B)
            expect_exact(C_plain, A, B)
        else:
            expect_close(C_ws, A, B)
    # a misaligned workspace is refused before anything is queued
    assert tg.gemm_ex_host_ws(Ah.data_ptr(), Bh.data_ptr(), C_ws.data_ptr(), M, N, K, tg.F16,
                              tg.F32, code, dA.data_ptr(), dB.data_ptr(), dC.data_ptr(),
                              ws.data_ptr() + 4, ws_bytes - 4, s.cuda_stream) == \
        tg.binding.ERR_INVALID_VALUE


def test_automatic_choice_on_the_named_workloads():
    """The automatic picks on the named workloads: the latency-path kernel
    when its 16 x 16 tiles' copies are short (one tile per SM up to K =
    2048, or up to three per SM and 1024 x SMs tile-K values; aligned FP32
    products of up to eleven tiles per SM), the non-persistent
    single-tile kernel when 128 x 64 tiles fit in one wave, the CTA-pair
    kernel for the large squares, the tiled SIMT kernel for the rest of FP32
    and for shapes the tensor maps cannot take."""
    def pick(M, N, K, in_dt, out_dt, dtype=torch.bfloat16):
        A = torch.zeros(M, K, dtype=dtype, device="cuda")
        B = torch.zeros(K, N, dtype=dtype, device="cuda")
        C = torch.empty(M, N, dtype=torch.float32, device="cuda")
        return tg.KERNEL_NAMES[tg.gemm_select_kernel(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                                     M, N, K, in_dt, tg.F32, out_dt)]
    assert pick(9, 9, 9, tg.F32, tg.F32, torch.float32) == "simt"
    assert pick(128, 128, 128, tg.F16, tg.F32, torch.float16) == "tile16"
    assert pick(96, 200, 1000, tg.BF16, tg.F32) == "tile16"
    assert pick(100, 200, 1000, tg.F32, tg.F32, torch.float32) == "tile16"
    assert pick(640, 640, 640, tg.F32, tg.F32, torch.float32) == "tile16"     # 10.5 tiles per SM
    assert pick(768, 768, 768, tg.F32, tg.F32, torch.float32) == "simt"       # 15.2 tiles per SM
    assert pick(1024, 1024, 1024, tg.F32, tg.F32, torch.float32) == "simt"
    assert pick(256, 256, 256, tg.BF16, tg.BF16) == "tile16"      # two tiles per SM, short K
    assert pick(128, 128, 2048, tg.BF16, tg.BF16) == "tile16"
    assert pick(256, 256, 1024, tg.BF16, tg.BF16) == "tc_small"
    assert pick(512, 512, 512, tg.BF16, tg.BF16) == "tc_small"
    assert pick(256, 256, 4096, tg.BF16, tg.F32) == "tc_128x128"   # split along K by gemm_ex_ws
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


def test_simt_large_tile_kernel_more_tiles_than_blocks():
    """More 128 x 128 tiles than the large-tile SIMT kernel has resident
    blocks (2600^2: 21 x 21 = 441 tiles against two blocks per SM), so blocks
    move on to a second output tile with their shared buffers and register
    prefetch restarted: every operand layout, ragged in M, N and K (1, 3 and
    10 K tiles of 8), integer inputs, exact against the oracle's general
    form."""
    M = N = 2600
    assert 21 * 21 > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    for K, seed in ((5, 50), (21, 51), (77, 52)):
        A0, B0 = inputs.draw(M, N, K, "f32", "int", seed=seed)
        for op_a, op_b in (("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")):
            A = A0.t().contiguous() if op_a == "t" else A0
            B = B0.t().contiguous() if op_b == "t" else B0
            C = tg.addmm(A.cuda(), B.cuda(), op_a=op_a, op_b=op_b, out_dtype=torch.float32,
                         kernel="simt").cpu()
            ref, _ = oracle.gemm_general(A, B, op_a, op_b)
            np.testing.assert_array_equal(C.double().numpy(), ref,
                                          err_msg=f"K={K} layout {op_a}{op_b}")


# ------------------------------------------------- IEEE special values

@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_nan_and_inf_propagate(kernel):
    """A NaN in A poisons its row of C; an infinity in A or B makes its row
    or column infinite with the sign of each product, except where it meets
    a zero (inf * 0 = NaN) or an infinity of the other sign (NaN).  Integer
    values elsewhere keep every finite partial sum exact, so the class of
    each result (finite value, +inf, -inf, NaN) does not depend on the
    summation order, and each element must equal the oracle's FP64 IEEE
    result rounded to the output type."""
    M, N, K = (136, 200, 72) if kernel != "simt_tpb3" else (20, 24, 18)
    for in_dt in ("f16", "bf16"):
        A, B = inputs.draw(M, N, K, in_dt, "int", seed=70)
        A[3, 5] = float("nan")
        A[7, 2] = float("inf")
        A[9, 4] = float("-inf")
        B[4, 11] = float("-inf")
        B[6, 13] = float("nan")
        B[2, 17] = 0.0                   # A[7, 2] = inf meets a zero: NaN at (7, 17)
        C_ref, _ = oracle.gemm(A, B)
        for out in OUT_TYPES:
            got = run_gpu(A, B, out, kernel).double().numpy()
            want = oracle.round_to(C_ref, out).double().numpy()
            assert np.isnan(want[3]).all() and np.isnan(want[:, 13]).all()
            assert np.isnan(want[7, 17])
            np.testing.assert_array_equal(got, want, err_msg=f"{in_dt} -> {out}")


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_f16_output_overflow_rounds_to_infinity(kernel):
    """FP32 sums around the binary16 limit, written as FP16: 65504 stays,
    65519 rounds down to 65504, 65520 (the midpoint to 65536) and beyond
    become +-inf, as IEEE nearest-even rounding gives.  C[i, j] = 65504 s +
    d with exact FP32 sums from an FP16 65504 and small integers."""
    M, N, K = (40, 64, 16) if kernel != "simt_tpb3" else (8, 16, 16)
    d = [0, 1, 15, 16, 17, 31, 32, 100, -16, -17, -1000, 0]
    A = torch.zeros(M, K, dtype=torch.float16)
    A[:, 0] = 1.0
    A[:, 1] = 1.0
    A[1::2, 0] = -1.0                          # odd rows: -65504 s + d
    B = torch.zeros(K, N, dtype=torch.float16)
    for j in range(N):
        B[0, j] = 65504.0
        B[1, j] = float(d[j % len(d)])
    C_ref, _ = oracle.gemm(A, B)
    want = oracle.round_to(C_ref, torch.float16)
    assert torch.isinf(want).any() and (want.abs() == 65504).any()
    got = run_gpu(A, B, torch.float16, kernel)
    np.testing.assert_array_equal(got.double().numpy(), want.double().numpy())
    # the FP32 and BF16 outputs of the same sums are finite and exact
    for out in (torch.float32, torch.bfloat16):
        np.testing.assert_array_equal(run_gpu(A, B, out, kernel).double().numpy(),
                                      oracle.round_to(C_ref, out).double().numpy())


@pytest.mark.parametrize("kernel", ALL_KERNELS)
def test_fp32_accumulator_overflow(kernel):
    """Products beyond the FP32 range (2^100 * 2^100 in BF16 inputs) overflow
    the FP32 accumulator to +-inf; the oracle's FP64 sum (2^200) rounds to
    +-inf in every output type, so both sides agree element for element."""
    M, N, K = (16, 32, 16) if kernel != "simt_tpb3" else (6, 8, 16)
    A = torch.zeros(M, K, dtype=torch.bfloat16)
    B = torch.zeros(K, N, dtype=torch.bfloat16)
    A[:, 0] = 2.0 ** 100
    A[::2, 0] = -(2.0 ** 100)
    B[0, : N // 2] = 2.0 ** 100
    B[1, :] = 3.0
    A[:, 1] = 1.0
    C_ref, _ = oracle.gemm(A, B)
    for out in OUT_TYPES:
        want = oracle.round_to(C_ref, out).double().numpy()
        assert np.isinf(want[:, : N // 2]).all() and np.isfinite(want[:, N // 2:]).all()
        np.testing.assert_array_equal(run_gpu(A, B, out, kernel).double().numpy(), want)


@pytest.mark.parametrize("op_a,op_b", [("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")])
def test_simt_f32_wide_load_kernel_exact(op_a, op_b):
    """FP32 operands whose stored rows are multiples of 4 elements take the
    large-tile SIMT kernel with 16-byte loads: ragged M and N (2060 = 16 *
    128 + 12 rows, 1292 = 10 * 128 + 12 columns) with 1, 2, 3 and 7 K tiles
    of 16, the last one partial; and 2600 x 2600 (441 tiles, more than the
    resident blocks) so blocks restart on a second tile.  Integer inputs,
    exact against the oracle's general form, every layout."""
    for M, N, K, seed in ((2060, 1292, 4, 90), (2060, 1292, 12, 91), (2060, 1292, 20, 92),
                          (2060, 1292, 36, 93), (2060, 1292, 100, 94), (2600, 2600, 36, 95)):
        A0, B0 = inputs.draw(M, N, K, "f32", "int", seed=seed)
        A = A0.t().contiguous() if op_a == "t" else A0
        B = B0.t().contiguous() if op_b == "t" else B0
        C = tg.addmm(A.cuda(), B.cuda(), op_a=op_a, op_b=op_b, out_dtype=torch.float32,
                     kernel="simt").cpu()
        ref, _ = oracle.gemm_general(A, B, op_a, op_b)
        np.testing.assert_array_equal(C.double().numpy(), ref,
                                      err_msg=f"{M}x{N}x{K} layout {op_a}{op_b}")


def test_simt_f32_wide_load_kernel_outputs_and_addmm():
    """The same kernel with 16-bit outputs (element stores), alpha and beta
    (C read back), and the 16-byte FP32 stores on full-width tiles beside
    element stores on the ragged last column of tiles."""
    M, N, K = 2048, 1548, 40                       # 1548 = 12 * 128 + 12
    A, B = inputs.draw(M, N, K, "f32", "int", seed=96)
    for out in (torch.float16, torch.bfloat16, torch.float32):
        expect_exact(run_gpu(A, B, out, "simt"), A, B)
    Cin = inputs.draw(M, 1, N, "f32", "int", seed=97)[0]
    C = tg.addmm(A.cuda(), B.cuda(), Cin.clone().cuda(), alpha=2.0, beta=-1.0,
                 out_dtype=torch.float32, kernel="simt").cpu()
    ref, _ = oracle.gemm_general(A, B, alpha=2.0, beta=-1.0, C_in=Cin)
    np.testing.assert_array_equal(C.double().numpy(), ref)
    # random FP32 inputs: within the stated bound
    A, B = inputs.draw(M, N, 1000, "f32", "normal", seed=98)
    expect_close(run_gpu(A, B, torch.float32, "simt"), A, B)


def test_large_products_with_k0_write_zeros_or_beta_c():
    """K = 0 on the large-tile SIMT kernels (FP32 with aligned rows, and BF16
    with an odd pitch) and on the tensor-core path's automatic choice: C =
    beta * C_in, zeros for beta = 0."""
    for dt in (torch.float32, torch.bfloat16):
        A = torch.zeros(2048, 0, dtype=dt, device="cuda")
        B = torch.zeros(0, 2052, dtype=dt, device="cuda")
        out = torch.full((2048, 2052), 7.0, device="cuda")
        tg.matmul(A, B, out=out, kernel="simt")
        torch.cuda.synchronize()
        assert not out.any()
        C_in = torch.full((2048, 2052), 3.0, device="cuda")
        tg.addmm(A, B, C_in, alpha=2.0, beta=-1.0, kernel="simt")
        torch.cuda.synchronize()
        assert torch.all(C_in == -3.0)
