// Tensor-core kernels for op(A) op(B) with A as stored (M x K), B as stored (K x N).
#include "tc_launch.cuh"

namespace tmmo {

cudaError_t tc_launch_nn(const TcLaunch& l, cudaStream_t stream)
{
    return launch_layout<false, true>(l, stream);
}

cudaError_t tc_hybrid_launch(const TcLaunch& l, cudaStream_t stream)
{
    int plan[8] = {};
    TcLaunch k = l;
    k.variant = TC_256x256;
    k.hybrid = true;
    k.plan = plan;
    cudaError_t err = launch_layout<false, true>(k, stream);
    if (err != cudaSuccess)
        return err;
    if (plan[2] == 0)
        return cudaSuccess;  // every tile was computed whole
    return tail_reduce_launch(k, plan, stream);
}

}  // namespace tmmo
