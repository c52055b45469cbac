// Host side of the tensor-core GEMM: the driver entry point for tensor-map
// encoding and the dispatch over operand layouts.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace tmmo {

void* tensor_map_encoder()
{
    static void* fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
        else
            cudaGetLastError();  // leave no sticky error behind
    });
    return fn;
}

void tc_tile_shape(int variant, int* tile_m, int* tile_n)
{
    switch (variant) {
    case TC_128x128:
        *tile_m = 128;
        *tile_n = 128;
        break;
    case TC_128x256:
        *tile_m = 128;
        *tile_n = 256;
        break;
    case TC_256x128:
        *tile_m = 256;
        *tile_n = 128;
        break;
    default:
        *tile_m = 256;
        *tile_n = 256;
        break;
    }
}

cudaError_t tc_gemm_launch(const TcLaunch& l, cudaStream_t stream)
{
    if (l.op_a == 0 && l.op_b == 0)
        return tc_launch_nn(l, stream);
    if (l.op_a == 1 && l.op_b == 0)
        return tc_launch_tn(l, stream);
    if (l.op_a == 0 && l.op_b == 1)
        return tc_launch_nt(l, stream);
    return tc_launch_tt(l, stream);
}

}  // namespace tmmo
