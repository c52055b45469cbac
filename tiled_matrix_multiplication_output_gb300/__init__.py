"""GB300-native output-stationary tiled matrix multiply, C = A @ B.

The product runs in the CUDA library `_build/libtiled_gemm.so` (hand-written
sm_103a kernels behind the C ABI of include/tiled_gemm.h); this package is
its ctypes binding plus the seeded input generator.  The library is loaded
on first use and there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    BF16, F16, F32, KERNEL_NAMES, KERNELS, GemmError, addmm, error_string, gemm, gemm_debug_config,
    gemm_device_status, gemm_error_string, gemm_ex, gemm_ex_host, gemm_ex_host_ws, gemm_ex_kernel,
    gemm_ex_ws, gemm_host_panel_rows,
    gemm_general, gemm_launch_count, gemm_traffic_model, gemm_workspace_size, matmul_ws,
    gemm_select_kernel, gemm_splitk, gemm_splitk_noalloc, gemm_splitk_workspace_size,
    gemm_ws_split_count,
    header_functions, library_path,
    load_library, matmul, matmul_splitk,
)
