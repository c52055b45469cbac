// Tensor-core kernels for op(A) op(B) with A as stored (M x K), B transposed (stored N x K).
#include "tc_launch.cuh"

namespace tmmo {

cudaError_t tc_launch_nt(const TcLaunch& l, cudaStream_t stream)
{
    return launch_layout<false, false>(l, stream);
}

}  // namespace tmmo
