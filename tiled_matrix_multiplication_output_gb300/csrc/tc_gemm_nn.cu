// Tensor-core kernels for op(A) op(B) with A as stored (M x K), B as stored (K x N).
#include "tc_launch.cuh"

namespace tmmo {

cudaError_t tc_launch_nn(const TcLaunch& l, cudaStream_t stream)
{
    return launch_layout<false, true>(l, stream);
}

}  // namespace tmmo
