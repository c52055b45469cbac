// Tensor-core kernels for op(A) op(B) with A transposed (stored K x M), B as stored (K x N).
#include "tc_launch.cuh"

namespace tmmo {

cudaError_t tc_launch_tn(const TcLaunch& l, cudaStream_t stream)
{
    return launch_layout<true, true>(l, stream);
}

}  // namespace tmmo
