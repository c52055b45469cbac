// Split-K for products with few output tiles and a long K: the K steps of
// every output tile are divided into ranges, each range is a separate unit
// of work for the persistent tensor-core kernel (so more SMs share the
// reduction), its FP32 partial tile lands in a workspace, and a second
// kernel adds the partials in split order -- a fixed order, so the result is
// the same on every run -- and writes C.
//
// The reduction is a streaming pass over the workspace (HBM- or L2-bound):
// it reads splits * M * N FP32 values and writes M * N outputs, 16 bytes of
// workspace per thread and split in each step, grid-strided over the SMs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_launch.cuh"

namespace tmmo {
namespace {

__device__ __forceinline__ void store4(float* dst, float4 v)
{
    *reinterpret_cast<float4*>(dst) = v;
}
__device__ __forceinline__ void store4(__half* dst, float4 v)
{
    __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
    uint2 u = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    *reinterpret_cast<uint2*>(dst) = u;
}
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float4 v)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    *reinterpret_cast<uint2*>(dst) = u;
}

__device__ __forceinline__ float4 load4(const float* src)
{
    return *reinterpret_cast<const float4*>(src);
}
__device__ __forceinline__ float4 load4(const __half* src)
{
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* src)
{
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Launches a reduction kernel as a programmatic dependent of the tensor-core
// kernel before it on the stream: its blocks may be placed while that kernel
// still runs (it signals launch_dependents at its start) and start reading
// as soon as it completes, without a launch gap.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, cudaStream_t stream,
                             Args... args)
{
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

// out = alpha * acc + beta * C_old, four elements.
template <typename OutT>
__device__ __forceinline__ void finish4(OutT* dst, float4 acc, float alpha, float beta)
{
    acc.x *= alpha;
    acc.y *= alpha;
    acc.z *= alpha;
    acc.w *= alpha;
    if (beta != 0.0f) {
        const float4 c = load4(dst);
        acc.x = fmaf(beta, c.x, acc.x);
        acc.y = fmaf(beta, c.y, acc.y);
        acc.z = fmaf(beta, c.z, acc.z);
        acc.w = fmaf(beta, c.w, acc.w);
    }
    store4(dst, acc);
}

__device__ __forceinline__ void add4(float4& a, const float4 b)
{
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// C[i] = alpha * sum_s ws[s][i] + beta * C[i], four elements per step
// (M * N is a multiple of 4 because N is).  The partials are added in split
// order; the loads of eight splits are issued before they are added, so a
// thread waits for memory once per eight splits rather than once per split.
template <typename OutT>
__global__ void __launch_bounds__(256)
    splitk_reduce_kernel(const float* __restrict__ ws, OutT* __restrict__ C, long long mn,
                         int splits, float alpha, float beta)
{
    constexpr int BATCH = 8;
    grid_dep_wait();
    const long long n4 = mn / 4;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride) {
        const float* src = ws + 4 * i;
        float4 acc = load4(src);
        int s = 1;
        for (; s + BATCH <= splits; s += BATCH) {
            float4 v[BATCH];
#pragma unroll
            for (int j = 0; j < BATCH; ++j)
                v[j] = load4(src + static_cast<long long>(s + j) * mn);
#pragma unroll
            for (int j = 0; j < BATCH; ++j)
                add4(acc, v[j]);
        }
        for (; s < splits; ++s)
            add4(acc, load4(src + static_cast<long long>(s) * mn));
        finish4(C + 4 * i, acc, alpha, beta);
    }
}

template <typename OutT>
cudaError_t launch_reduce(const TcLaunch& l, int splits, cudaStream_t stream)
{
    const long long mn = static_cast<long long>(l.M) * l.N;
    const long long n4 = mn / 4;
    const long long cap = static_cast<long long>(std::max(l.num_sms, 1)) * 8;
    const int grid = static_cast<int>(std::max<long long>(1, std::min((n4 + 255) / 256, cap)));
    return launch_dependent(splitk_reduce_kernel<OutT>, dim3(grid), dim3(256), stream,
                            l.workspace, static_cast<OutT*>(l.C), mn, splits, l.alpha, l.beta);
}

// Tail reduction of the hybrid plan: block (x = tail tile, y = band of 16
// rows) sums the `splits` FP32 partials of its tile rows in split order and
// writes the part of C inside M x N.  Each thread owns TAIL_ITEMS groups of
// four columns and issues the loads of all of them before adding, so that
// many loads are in flight per thread.
constexpr int TAIL_BAND_ROWS = 16;
constexpr int TAIL_THREADS = 256;

template <typename OutT, int ITEMS>
__global__ void __launch_bounds__(TAIL_THREADS)
    tail_reduce_kernel(const float* __restrict__ ws, OutT* __restrict__ C, TcParams p, int tile_m,
                       int tile_n, int splits)
{
    grid_dep_wait();
    const int tail = blockIdx.x;
    int mb, nb;
    tc_tile_coords(p.dp_tiles + tail, p, mb, nb);
    const long long tile_elems = static_cast<long long>(tile_m) * tile_n;
    const float* base = ws + static_cast<long long>(tail) * splits * tile_elems;
    const int groups_per_row = tile_n / 4;
    long long off[ITEMS];
    long long dst[ITEMS];
    bool live[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
        const int g = threadIdx.x + i * TAIL_THREADS;
        const int r = blockIdx.y * TAIL_BAND_ROWS + g / groups_per_row;
        const int c = (g % groups_per_row) * 4;
        const int grow = mb * tile_m + r;
        const int gcol = nb * tile_n + c;
        // N is a multiple of 4, so a group lies wholly inside or outside C
        live[i] = g < TAIL_BAND_ROWS * groups_per_row && r < tile_m && grow < p.M && gcol < p.N;
        off[i] = static_cast<long long>(r) * tile_n + c;
        dst[i] = static_cast<long long>(grow) * p.N + gcol;
    }
    float4 acc[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
        acc[i] = live[i] ? load4(base + off[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 1; s < splits; ++s) {
        const float* part = base + static_cast<long long>(s) * tile_elems;
        float4 v[ITEMS];
#pragma unroll
        for (int i = 0; i < ITEMS; ++i)
            v[i] = live[i] ? load4(part + off[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < ITEMS; ++i)
            add4(acc[i], v[i]);
    }
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
        if (live[i])
            finish4(C + dst[i], acc[i], p.alpha, p.beta);
}

template <typename OutT>
cudaError_t launch_tail(const TcLaunch& l, const int* plan, cudaStream_t stream)
{
    TcParams p{};
    p.M = l.M;
    p.N = l.N;
    p.dp_tiles = plan[0];
    p.tiles_m = plan[3];
    p.tiles_n = plan[4];
    p.group_m = plan[5];
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.alpha = l.alpha;
    p.beta = l.beta;
    const int tile_m = plan[6], tile_n = plan[7];
    const dim3 grid(plan[2], (tile_m + TAIL_BAND_ROWS - 1) / TAIL_BAND_ROWS, 1);
    // groups of four columns per band, spread over the block's threads
    const int items = (TAIL_BAND_ROWS * (tile_n / 4) + TAIL_THREADS - 1) / TAIL_THREADS;
    if (items <= 2)
        return launch_dependent(tail_reduce_kernel<OutT, 2>, grid, dim3(TAIL_THREADS), stream,
                                l.workspace, static_cast<OutT*>(l.C), p, tile_m, tile_n, plan[1]);
    if (items <= 4)
        return launch_dependent(tail_reduce_kernel<OutT, 4>, grid, dim3(TAIL_THREADS), stream,
                                l.workspace, static_cast<OutT*>(l.C), p, tile_m, tile_n, plan[1]);
    return cudaErrorInvalidValue;  // tiles are at most 256 columns wide
}

}  // namespace

cudaError_t tail_reduce_launch(const TcLaunch& l, const int* plan, cudaStream_t stream)
{
    switch (l.out_dtype) {
    case DT_F32:
        return launch_tail<float>(l, plan, stream);
    case DT_F16:
        return launch_tail<__half>(l, plan, stream);
    default:
        return launch_tail<__nv_bfloat16>(l, plan, stream);
    }
}

int splitk_used_splits(int64_t K, int requested)
{
    const int64_t k_blocks = (K + TC_BK - 1) / TC_BK;
    if (k_blocks <= 0)
        return 1;
    const int64_t s = std::max<int64_t>(1, std::min<int64_t>(requested, k_blocks));
    const int64_t per = (k_blocks + s - 1) / s;
    return static_cast<int>((k_blocks + per - 1) / per);
}

cudaError_t tc_splitk_launch(const TcLaunch& l, int* used_splits, cudaStream_t stream)
{
    const int splits = splitk_used_splits(l.K, l.k_splits);
    TcLaunch k = l;
    k.k_splits = splits;
    k.alpha = 1.0f;  // alpha and beta are applied by the reduction
    k.beta = 0.0f;
    cudaError_t err = launch_variant<1, 128, 6, float, false, true, true>(k, stream);
    if (err != cudaSuccess)
        return err;
    if (used_splits)
        *used_splits = splits;
    switch (l.out_dtype) {
    case DT_F32:
        return launch_reduce<float>(l, splits, stream);
    case DT_F16:
        return launch_reduce<__half>(l, splits, stream);
    default:
        return launch_reduce<__nv_bfloat16>(l, splits, stream);
    }
}

}  // namespace tmmo
