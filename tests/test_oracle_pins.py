"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle restated.

Each group is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong index, a transposed operand, a bad rounding rule, a miscounted
edge tile) fails at least one test.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import load_golden, load_worked_9x9
from tiled_matrix_multiplication_output_gb300 import inputs


# --------------------------------------------------------------- worked 9x9

def test_worked_example_fixture_matches_generator():
    """The printed inputs (fixture) are A[i][j] = 9i + j and B = 2A."""
    A, B = load_worked_9x9()
    gA, gB = inputs.worked_example()
    assert A == gA.to(torch.int64).tolist()
    assert B == gB.to(torch.int64).tolist()


def test_worked_example_closed_form():
    """C[i][j] = 2 * sum_k (9i + k)(9k + j) = 5832 i + 162 i j + 72 j + 3672,
    from sum k = 36 and sum k^2 = 204 over k = 0..8.  Exact in FP64."""
    A, B = load_worked_9x9()
    C, Cabs = oracle.gemm(torch.tensor(A, dtype=torch.float32),
                          torch.tensor(B, dtype=torch.float32))
    for i in range(9):
        for j in range(9):
            want = 5832 * i + 162 * i * j + 72 * j + 3672
            assert C[i, j] == want
            assert Cabs[i, j] == want           # all products are >= 0
    assert C[0, 0] == 3672 and C[8, 8] == 61272 and C[8, 0] == 50328
    assert C.sum() == 2420280


# ----------------------------------------------------- brute force, integers

def _int_loop(A, B):
    """Independent reference: pure-Python integer triple loop."""
    M, K = len(A), len(A[0]) if A else 0
    N = len(B[0]) if B else 0
    return [[sum(A[i][k] * B[k][j] for k in range(K)) for j in range(N)] for i in range(M)]


def _check_against_int_loop(M, N, K, dtype, seed):
    A, B = inputs.draw(M, N, K, dtype, "int", seed=seed)
    C, Cabs = oracle.gemm(A, B, nthreads=1)
    Ai = A.to(torch.int64).tolist()
    Bi = B.to(torch.int64).tolist()
    want = np.array(_int_loop(Ai, Bi), dtype=np.float64)
    want_abs = np.array(_int_loop([[abs(v) for v in r] for r in Ai],
                                  [[abs(v) for v in r] for r in Bi]), dtype=np.float64)
    np.testing.assert_array_equal(C, want)
    np.testing.assert_array_equal(Cabs, want_abs)


def test_brute_force_every_tiny_shape():
    """Every (M, N, K) in {1..17}^3 (4913 shapes), integer inputs in [-4, 4]
    (exact in every storage type), against integer arithmetic; the storage
    type cycles F32, F16, BF16 from one shape to the next."""
    dtypes = ("f32", "f16", "bf16")
    for idx, (M, N, K) in enumerate(itertools.product(range(1, 18), repeat=3)):
        _check_against_int_loop(M, N, K, dtypes[idx % 3], seed=idx)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_brute_force_tile_edge_shapes(dtype):
    """Every (M, N, K) with each dimension in {63, 65, 129} or {1, 17}: one
    below and one above a 64-wide tile, and one past two of them."""
    dims = (1, 17, 63, 65, 129)
    for idx, (M, N, K) in enumerate(itertools.product(dims, repeat=3)):
        if max(M, N, K) < 63:
            continue
        _check_against_int_loop(M, N, K, dtype, seed=1000 + idx)


def test_not_transposed_and_not_symmetric():
    """A non-square, non-symmetric case where A @ B, A^T-ish and B @ A differ."""
    A = torch.tensor([[1., 2., 3.], [4., 5., 6.]])          # 2 x 3
    B = torch.tensor([[7., 8.], [9., 10.], [11., 12.]])     # 3 x 2
    C, _ = oracle.gemm(A, B)
    np.testing.assert_array_equal(C, [[58., 64.], [139., 154.]])


# ------------------------------------------------------------ special cases

def test_identity_gives_a():
    A, _ = inputs.draw(33, 1, 47, "bf16", "normal", seed=3)
    eye = torch.eye(47, dtype=torch.bfloat16)
    C, _ = oracle.gemm(A, eye)
    np.testing.assert_array_equal(C, A.double().numpy())


def test_permutation_permutes_columns():
    A, _ = inputs.draw(20, 1, 30, "f16", "uniform", seed=4)
    perm = torch.randperm(30, generator=torch.Generator().manual_seed(1))
    P = torch.zeros(30, 30, dtype=torch.float16)
    P[perm, torch.arange(30)] = 1                    # column j picks row perm[j]
    C, _ = oracle.gemm(A, P)
    np.testing.assert_array_equal(C, A.double().numpy()[:, perm.numpy()])


def test_k1_is_outer_product():
    A, B = inputs.draw(13, 17, 1, "f32", "normal", seed=5)
    C, Cabs = oracle.gemm(A, B)
    np.testing.assert_array_equal(C, np.outer(A.double().numpy()[:, 0], B.double().numpy()[0]))
    np.testing.assert_array_equal(Cabs, np.abs(C))


def test_k0_gives_zeros():
    A = torch.zeros(5, 0, dtype=torch.bfloat16)
    B = torch.zeros(0, 7, dtype=torch.bfloat16)
    C, Cabs = oracle.gemm(A, B)
    assert C.shape == (5, 7)
    assert not C.any() and not Cabs.any()


def test_library_cross_check_fp64():
    """Random FP32 inputs: agrees with numpy's FP64 matmul to ~1e-12."""
    A, B = inputs.draw(70, 90, 300, "f32", "normal", seed=6)
    C, Cabs = oracle.gemm(A, B, nthreads=4)
    ref = A.double().numpy() @ B.double().numpy()
    assert np.max(np.abs(C - ref) / (np.abs(ref) + Cabs)) < 1e-12
    ref_abs = np.abs(A.double().numpy()) @ np.abs(B.double().numpy())
    np.testing.assert_allclose(Cabs, ref_abs, rtol=1e-12)


def test_entries_match_full_product():
    A, B = inputs.draw(37, 41, 129, "bf16", "normal", seed=8)
    C, Cabs = oracle.gemm(A, B)
    rows = np.array([0, 36, 5, 17, 36])
    cols = np.array([0, 40, 40, 3, 0])
    v, va = oracle.gemm_entries(A, B, rows, cols)
    np.testing.assert_array_equal(v, C[rows, cols])
    np.testing.assert_array_equal(va, Cabs[rows, cols])


def test_entries_closed_form_worked_example():
    A, B = load_worked_9x9()
    rows = np.array([0, 8, 8, 3, 1])
    cols = np.array([0, 8, 0, 5, 1])
    v, va = oracle.gemm_entries(torch.tensor(A, dtype=torch.float32),
                                torch.tensor(B, dtype=torch.float32), rows, cols)
    want = [5832 * i + 162 * i * j + 72 * j + 3672 for i, j in zip(rows, cols)]
    np.testing.assert_array_equal(v, want)
    np.testing.assert_array_equal(va, want)


def test_thread_count_does_not_change_result():
    A, B = inputs.draw(31, 29, 77, "f16", "uniform", seed=9)
    C1, _ = oracle.gemm(A, B, nthreads=1)
    C7, _ = oracle.gemm(A, B, nthreads=7)
    np.testing.assert_array_equal(C1, C7)


# ------------------------------------------------------ widening / rounding

def test_widen_every_f16_pattern():
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.float16)
    got = oracle.widen(t)
    want = bits.numpy().view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_widen_every_bf16_pattern():
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    got = oracle.widen(t)
    want = (bits.to(torch.int32) << 16).view(torch.float32).double().numpy()
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], want[~nan])


def _nearest_even_reference(x, values, mant_lsb_of):
    """Brute force: the nearest finite grid value to x, ties to the one with
    an even last significand bit."""
    i = np.searchsorted(values, x)
    lo, hi = values[max(i - 1, 0)], values[min(i, len(values) - 1)]
    if x - lo < hi - x:
        return lo
    if hi - x < x - lo:
        return hi
    return lo if mant_lsb_of(lo) == 0 else hi


def _grid(dtype):
    bits = torch.arange(0, 32768, dtype=torch.int32).to(torch.int16)
    vals = bits.view(dtype).double().numpy()
    ok = np.isfinite(vals)
    vals, b = vals[ok], bits.numpy()[ok]
    full = np.concatenate([-vals[::-1], vals])
    fbits = np.concatenate([b[::-1], b])
    lsb = dict(zip(full.tolist(), (fbits & 1).tolist()))
    return np.unique(full), lambda v: lsb[float(v)]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_round_is_nearest_even(dtype):
    values, lsb = _grid(dtype)
    rng = np.random.default_rng(11)
    maxf = values[-1]
    # random values across the range, exact midpoints (ties), and subnormals
    xs = list(rng.uniform(-maxf, maxf, 400))
    xs += list(rng.normal(0, 1, 400))
    xs += list(rng.normal(0, 1e-6, 100))
    mids = (values[:-1] + values[1:]) / 2
    xs += list(mids[rng.choice(len(mids), 400)])
    xs = np.array(xs)
    got = oracle.round_to(xs, dtype).double().numpy()
    want = np.array([_nearest_even_reference(x, values, lsb) for x in xs])
    np.testing.assert_array_equal(got, want)


def test_round_matches_numpy_half_and_overflows():
    rng = np.random.default_rng(12)
    xs = np.concatenate([rng.normal(0, 300, 2000), rng.normal(0, 1e-5, 500),
                         [65504.0, 65519.99, 65520.0, -65520.0, 1e9, 0.0, -0.0]])
    got = oracle.round_to(xs, torch.float16).numpy().view(np.float16)
    want = xs.astype(np.float16)
    np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))


def test_round_f32_matches_numpy():
    rng = np.random.default_rng(13)
    xs = np.concatenate([rng.normal(0, 1, 3000) * 10.0 ** rng.integers(-40, 38, 3000),
                         [3.4028235677973366e38, 1e39, -1e39]])
    got = oracle.round_to(xs, torch.float32).numpy()
    with np.errstate(over="ignore"):
        want = xs.astype(np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_round_overflow_edges():
    got = oracle.round_to(np.array([65519.0, 65520.0, -65520.0]), torch.float16)
    assert got[0].item() == 65504.0
    assert math.isinf(got[1].item()) and got[1].item() > 0
    assert math.isinf(got[2].item()) and got[2].item() < 0


# ------------------------------------------------- traffic / tile walking

def test_traffic_matches_page_worked_count():
    g = load_golden("page_figures.txt")
    t = oracle.traffic(128, 128, 128, 16, 16, 32, in_bytes=2, acc_bytes=4, c_bytes=4)
    assert t["a_elems"] * 2 == int(g["traffic_128_tile16x16x32_a_kib"]) * 1024
    assert t["b_elems"] * 2 == int(g["traffic_128_tile16x16x32_b_kib"]) * 1024
    assert t["c_elems"] * 4 == int(g["traffic_128_tile16x16x32_c_kib"]) * 1024
    assert t["bytes"] == int(g["traffic_128_tile16x16x32_total_kib"]) * 1024
    assert t["flops"] == int(g["ops_128"])
    assert t["ws_full"] == int(g["working_set_16x16x32_kib"]) * 1024
    assert t["ws_max"] == t["ws_full"]


@pytest.mark.parametrize("tk", [1, 7, 32, 64, 200])
def test_traffic_tile_k_invariance(tk):
    """Changing only tile_k leaves the total traffic unchanged."""
    base = oracle.traffic(96, 200, 1000, 64, 128, 64)
    t = oracle.traffic(96, 200, 1000, 64, 128, tk)
    for key in ("a_elems", "b_elems", "c_elems", "bytes", "flops", "tiles"):
        assert t[key] == base[key]


def test_traffic_closed_form_on_ragged_shapes():
    """Summed actual extents equal M*K*ceil(N/tn), K*N*ceil(M/tm), M*N."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        M, N, K = (int(v) for v in rng.integers(1, 300, 3))
        tm, tn, tk = (int(v) for v in rng.integers(1, 70, 3))
        t = oracle.traffic(M, N, K, tm, tn, tk)
        assert t["a_elems"] == M * K * math.ceil(N / tn)
        assert t["b_elems"] == K * N * math.ceil(M / tm)
        assert t["c_elems"] == M * N
        assert t["flops"] == 2 * M * N * K
        assert t["tiles"] == math.ceil(M / tm) * math.ceil(N / tn)
        assert t["steps"] == t["tiles"] * math.ceil(K / tk)


def test_traffic_larger_tiles_read_less():
    small = oracle.traffic(1024, 1024, 1024, 64, 64, 64)
    big = oracle.traffic(1024, 1024, 1024, 128, 256, 64)
    assert big["a_elems"] < small["a_elems"] and big["b_elems"] < small["b_elems"]
    assert big["ws_full"] > small["ws_full"]


def test_edge_tile_working_set_counts_actual_extent():
    """96 rows with tile 64: the edge step's working set uses 32 rows."""
    t = oracle.traffic(96, 64, 64, 64, 64, 64, in_bytes=2, acc_bytes=4)
    assert t["ws_max"] == t["ws_full"]
    # a single partial tile: working set of the actual 32 x 64 x 64 step
    t2 = oracle.traffic(32, 64, 64, 64, 64, 64, in_bytes=2, acc_bytes=4)
    assert t2["ws_max"] == 32 * 64 * 2 + 64 * 64 * 2 + 32 * 64 * 4


def test_tile_ranges_page_examples():
    g = load_golden("page_figures.txt")
    want = [tuple(int(x) for x in s.split(":")) for s in g["slices_10_tile4"].split(",")]
    assert oracle.tile_ranges(10, 4) == want
    lens = [b - a for a, b in oracle.tile_ranges(96, 64)]
    assert lens == [int(x) for x in g["edge_96_tile64"].split(",")]
    assert len(oracle.tile_ranges(9, 3)) == int(g["tiles_9_tpb3"])
    assert 3 * 3 == int(g["threads_per_block_9x9"])
    assert oracle.tile_ranges(0, 4) == []


def test_tile_ranges_cover_exactly():
    for n, t in itertools.product(range(0, 40), range(1, 12)):
        r = oracle.tile_ranges(n, t)
        assert sum(b - a for a, b in r) == n
        assert all(r[i][1] == r[i + 1][0] for i in range(len(r) - 1))
        assert all(0 < b - a <= t for a, b in r)


# ------------------------------------------- transposed operands and addmm

@pytest.mark.parametrize("op_a,op_b", [("n", "n"), ("t", "n"), ("n", "t"), ("t", "t")])
def test_general_transposes_against_integer_loop(op_a, op_b):
    """op(A) @ op(B) with the stored matrices transposed as the op says, on
    integer inputs, against the pure-Python integer loop."""
    for trial, (M, N, K) in enumerate([(5, 7, 3), (17, 9, 33), (1, 13, 8), (12, 1, 1)]):
        A0, B0 = inputs.draw(M, N, K, "bf16", "int", seed=40 + trial)   # A0: M x K, B0: K x N
        A = A0.t().contiguous() if op_a == "t" else A0
        B = B0.t().contiguous() if op_b == "t" else B0
        C, Cabs = oracle.gemm_general(A, B, op_a, op_b)
        Ai, Bi = A0.to(torch.int64).tolist(), B0.to(torch.int64).tolist()
        np.testing.assert_array_equal(C, np.array(_int_loop(Ai, Bi), dtype=np.float64))
        C2, _ = oracle.gemm(A0, B0)
        np.testing.assert_array_equal(C, C2)


def test_general_transpose_is_not_identity():
    """A non-square case where the transposed read differs from the plain one."""
    A = torch.tensor([[1., 2.], [3., 4.], [5., 6.]])   # stored 3 x 2
    B = torch.tensor([[1., 0., 2.], [0., 1., 3.]])      # stored 2 x 3
    C_nn, _ = oracle.gemm_general(A, B, "n", "n")       # (3x2)(2x3)
    np.testing.assert_array_equal(C_nn, [[1, 2, 8], [3, 4, 18], [5, 6, 28]])
    C_tt, _ = oracle.gemm_general(A, B, "t", "t")       # (2x3)(3x2)
    np.testing.assert_array_equal(C_tt, [[11, 18], [14, 22]])


def test_general_alpha_beta_addmm():
    """alpha * A @ B + beta * C_in on integers, exact; beta = 0 ignores C_in
    (even NaN); A = 0 leaves beta * C_in."""
    A, B = inputs.draw(9, 11, 7, "f16", "int", seed=50)
    Cin = torch.randint(-9, 10, (9, 11), generator=torch.Generator().manual_seed(3)).to(torch.float32)
    C, Cabs = oracle.gemm_general(A, B, alpha=2.0, beta=-3.0, C_in=Cin)
    want = 2 * np.array(_int_loop(A.to(torch.int64).tolist(), B.to(torch.int64).tolist())) \
        - 3 * Cin.numpy().astype(np.int64)
    np.testing.assert_array_equal(C, want)
    plain, plain_abs = oracle.gemm(A, B)
    np.testing.assert_array_equal(Cabs, 2 * plain_abs)
    nan_in = torch.full((9, 11), float("nan"))
    C0, _ = oracle.gemm_general(A, B, beta=0.0, C_in=nan_in)
    np.testing.assert_array_equal(C0, plain)
    Z = torch.zeros_like(A)
    Cz, _ = oracle.gemm_general(Z, B, alpha=5.0, beta=0.5, C_in=Cin)
    np.testing.assert_array_equal(Cz, 0.5 * Cin.numpy())
