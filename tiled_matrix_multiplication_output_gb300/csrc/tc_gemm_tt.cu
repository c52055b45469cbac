// Tensor-core kernels for op(A) op(B) with A transposed (stored K x M), B transposed (stored N x K).
#include "tc_launch.cuh"

namespace tmmo {

cudaError_t tc_launch_tt(const TcLaunch& l, cudaStream_t stream)
{
    return launch_layout<true, false>(l, stream);
}

}  // namespace tmmo
