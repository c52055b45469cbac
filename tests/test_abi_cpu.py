"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/tiled_gemm.h declares, and rejects bad arguments on the
host before touching a device."""
import ctypes
import re

import pytest

import tiled_matrix_multiplication_output_gb300 as tg
from tiled_matrix_multiplication_output_gb300 import build as tgbuild


@pytest.fixture(scope="module")
def lib():
    if tgbuild.nvcc_path() is None:
        pytest.skip("nvcc not available")
    tgbuild.build()
    return tg.load_library()


def test_header_declares_the_boundary():
    names = tg.header_functions()
    for n in ("gemm", "gemm_ex", "gemm_ex_kernel", "gemm_select_kernel", "gemm_ex_host",
              "gemm_device_status", "gemm_debug_config", "gemm_error_string"):
        assert n in names


def test_library_exports_every_header_symbol(lib):
    raw = ctypes.CDLL(tg.library_path())
    for name in tg.header_functions():
        assert hasattr(raw, name), name


def test_invalid_arguments_rejected_on_host(lib):
    INV, UNS = tg.binding.ERR_INVALID_VALUE, tg.binding.ERR_UNSUPPORTED
    p = 16  # a dummy non-null address; never dereferenced on these paths
    assert tg.gemm(p, p, p, -1, 4, 4, tg.BF16, tg.F32) == INV
    assert tg.gemm(p, p, p, 4, -1, 4, tg.BF16, tg.F32) == INV
    assert tg.gemm(p, p, p, 4, 4, -1, tg.BF16, tg.F32) == INV
    assert tg.gemm(p, p, p, 1 << 31, 4, 4, tg.BF16, tg.F32) == INV
    # the size limit: 2^31 - 256, so that a tile's or a K tile's worth of
    # headroom above any accepted size still fits a 32-bit index
    big = (1 << 31) - 256
    assert tg.binding.MAX_DIM == big
    for dims in ((big + 1, 4, 4), (4, big + 1, 4), (4, 4, big + 1), ((1 << 31) - 1, 4, 4)):
        assert tg.gemm(p, p, p, *dims, tg.BF16, tg.F32) == INV, dims
        assert tg.gemm_general(p, p, p, *dims, 0, 0, 1.0, 0.0, tg.F32, tg.F32, tg.F32, 1,
                               None) == INV, dims
        assert tg.gemm_ex_ws(p, p, p, *dims, tg.BF16, tg.F32, tg.F32, None, 0, None) == INV
        assert tg.gemm_splitk_noalloc(p, p, p, *dims, 2, tg.BF16, tg.F32, tg.F32, None) == INV
    # at the limit itself a size is accepted (an empty product: nothing launches)
    assert tg.gemm(p, p, p, big, 0, 4, tg.BF16, tg.F32) == 0
    assert tg.gemm(p, p, p, 0, big, big, tg.BF16, tg.F32) == 0
    assert tg.gemm(p, p, None, 4, 4, 4, tg.BF16, tg.F32) == INV       # null C
    assert tg.gemm(None, p, p, 4, 4, 4, tg.BF16, tg.F32) == INV       # null A with K > 0
    assert tg.gemm(p, p, p, 4, 4, 4, 7, tg.F32) == INV                # unknown dtype
    assert tg.gemm_ex(p, p, p, 4, 4, 4, tg.BF16, tg.F32, 9) == INV
    assert tg.gemm(p, p, p, 4, 4, 4, tg.BF16, tg.F16) == UNS          # FP16 accumulation
    assert tg.gemm(p, p, p, 4, 4, 4, tg.F32, tg.BF16) == UNS
    assert tg.gemm_ex_kernel(p, p, p, 4, 4, 4, tg.BF16, tg.F32, tg.F32, 42) == INV
    assert tg.gemm_select_kernel(p, p, p, -3, 4, 4, tg.BF16, tg.F32, tg.F32) == -INV


def test_empty_products_are_noops_without_a_device(lib):
    assert tg.gemm(None, None, None, 0, 0, 0, tg.BF16, tg.F32) == 0
    assert tg.gemm(None, None, None, 0, 17, 5, tg.F16, tg.F32) == 0
    assert tg.gemm_ex(None, None, None, 9, 0, 5, tg.F32, tg.F32, tg.F32) == 0


def test_error_strings(lib):
    for code in range(5):
        assert tg.error_string(code)
    assert "unknown" in tg.error_string(99)


def test_debug_config_roundtrip(lib):
    assert tg.gemm_debug_config(1000, 3) == 0
    assert tg.gemm_debug_config(0, -1) == 0


def test_matmul_rejects_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        tg.matmul(torch.zeros(2, 2), torch.zeros(2, 2))


def test_library_traffic_model_matches_oracle_walker(lib):
    """The library's closed-form counts (used by the kernel choice) equal the
    oracle's tile-by-tile walk of the loop nest, edge tiles included."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(17)
    cases = [(128, 128, 128, 16, 16, 32), (96, 200, 1000, 128, 128, 64),
             (8192, 8192, 8192, 256, 256, 64), (1, 1, 1, 128, 256, 64)]
    cases += [tuple(int(v) for v in rng.integers(1, 400, 3)) + tuple(int(v) for v in rng.integers(1, 80, 3))
              for _ in range(150)]
    for M, N, K, tm, tn, tk in cases:
        for in_b, acc_b, c_b in ((2, 4, 4), (2, 4, 2), (4, 4, 4)):
            got = tg.gemm_traffic_model(M, N, K, tm, tn, tk, in_b, acc_b, c_b)
            want = oracle.traffic(M, N, K, tm, tn, tk, in_bytes=in_b, acc_bytes=acc_b, c_bytes=c_b)
            assert got == want, (M, N, K, tm, tn, tk)


def test_library_traffic_model_rejects_bad_tiles(lib):
    with pytest.raises(tg.GemmError):
        tg.gemm_traffic_model(8, 8, 8, 0, 8, 8)


def test_host_panel_rows(lib):
    # whole 256-row tile rows, about an eighth of M, at least 1024; one piece
    # when that leaves a single panel
    assert tg.gemm_host_panel_rows(8192) == 1024
    assert tg.gemm_host_panel_rows(4100) == 1024
    assert tg.gemm_host_panel_rows(20000) == 2560
    assert tg.gemm_host_panel_rows(1000) == 1000
    assert tg.gemm_host_panel_rows(1024) == 1024
    assert tg.gemm_host_panel_rows(0) == 0
    assert tg.gemm_host_panel_rows(-5) == 0
    assert tg.gemm_host_panel_rows(tg.binding.MAX_DIM + 1) == 0


def test_header_constants_match_the_binding():
    text = open(tg.binding.HEADER).read()
    assert "#define GEMM_MAX_DIM ((int64_t)2147483392)" in text
    assert 2147483392 == tg.binding.MAX_DIM
    # every gemm_kernel_t value, by name, is the binding's kernel code
    kernels = {m.group(1).lower(): int(m.group(2))
               for m in re.finditer(r"GEMM_KERNEL_(\w+)\s*=\s*(\d+)", text)}
    assert kernels == tg.KERNELS
