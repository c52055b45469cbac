// Latency-path SIMT GEMM for small products: one 16 x 16 output tile per
// thread block, with the tile's whole K range of A rows and B columns
// staged in shared memory at once.
//
// A small product is a chain of latencies rather than work ("A memory count
// is not a latency estimate", Reading a matrix multiply through its tiles).
// The tensor-core kernels spend about a microsecond on barrier and
// accumulator set-up and tensor-map fetches before their first copy lands,
// and the tiled SIMT kernel pays one memory round trip per K tile.  This
// kernel avoids both: every thread issues all of its copies (cp.async, 16
// bytes, zero fill past the edges) before it waits for any, and the eight
// warps of a block split K between them, so a block's first multiply-add
// waits for one round trip and its warps meet only once, at the end.
//
//  * tile: a block owns 16 x 16 outputs and writes each of them once, from
//    one thread, after the last K term ("Keep one output tile resident");
//    every warp accumulates the whole tile over its own range of K (two
//    rows by four columns per lane), and the eight partials are summed
//    through shared memory in warp order;
//  * K is cut into 16-byte words (8 elements of 16-bit inputs, 4 of FP32);
//    warp w takes words [KV w / 8, KV (w + 1) / 8) of the KV words, copies
//    its own A and B slices in groups of four words and waits only for its
//    own copies (cp.async.wait_group, then __syncwarp for its lanes');
//  * edges: a word that crosses the end of K is copied in part and zero
//    filled, and rows past M or columns past N are zero filled, so each
//    output is the sum of exactly the definition's terms ("Edge tiles
//    still matter"), k ascending within a warp's range, then the warps'
//    partials in order;
//  * 16-bit inputs use the mixed-precision fused multiply-add
//    (fma.rn.f32.f16 / fma.rn.f32.bf16: a 16-bit product, exact in FP32,
//    added to an FP32 accumulator with one rounding), the same result as
//    widening both factors and calling fmaf;
//  * layouts: a k-contiguous slice (A as stored, B transposed) is kept with
//    its rows padded to 16 bytes past a multiple of 128, so the rows read
//    by one quarter-warp fall in different banks; an m- or n-contiguous
//    slice (A transposed, B as stored) is kept as 16-element rows along k.
//
// Requirements (simt_small_fits): 16-byte aligned A and B, each stored
// operand's row pitch a multiple of 16 bytes, and the K slices of one tile
// within the shared memory of a block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "launch.h"

namespace tmmo {
namespace {

constexpr int SS_TILE = 16;                  // output tile edge
constexpr int SS_WARPS = 8;                  // warps per block, each a range of K
constexpr int SS_THREADS = 32 * SS_WARPS;
constexpr int SS_GROUP = 4;                  // 16-byte words per commit group
constexpr int SS_SMEM_LIMIT = 227 * 1024;    // dynamic shared memory per block
constexpr int SS_MAX_DEVICES = 64;

// Shared-memory layout of one tile's K slices.
struct SsLayout {
    int kv;          // 16-byte words along K
    int pitch;       // row pitch (elements) of a k-contiguous slice
    int a_elems;     // elements of the A slice
    int b_elems;     // elements of the B slice
    long long bytes; // dynamic shared memory of a block
};

__host__ __device__ inline SsLayout ss_layout(long long K, int es, bool op_a, bool op_b)
{
    const int ve = 16 / es;
    SsLayout s{};
    const long long kv = (K + ve - 1) / ve;
    const long long kp = kv * ve;  // K rounded up to whole words
    const long long pitch = ((kp * es + 127) / 128) * 128 / es + 16 / es;
    const long long a = op_a ? kp * SS_TILE : SS_TILE * pitch;
    const long long b = op_b ? SS_TILE * pitch : kp * SS_TILE;
    s.bytes = (a + b) * es + static_cast<long long>(SS_WARPS) * SS_TILE * SS_TILE * 4;
    if (s.bytes > SS_SMEM_LIMIT)
        return s;  // too large; the other fields are not used
    s.kv = static_cast<int>(kv);
    s.pitch = static_cast<int>(pitch);
    s.a_elems = static_cast<int>(a);
    s.b_elems = static_cast<int>(b);
    return s;
}

// Raw elements: FP32, or the 16 bits of an F16 / BF16 value.
template <int DT>
struct SsElt {
    using T = uint16_t;
};
template <>
struct SsElt<DT_F32> {
    using T = float;
};

// Element e of a 16-byte word held as four 32-bit registers.
template <int ES>
__device__ __forceinline__ uint32_t ss_elt(const uint32_t (&w)[4], int e)
{
    if constexpr (ES == 4)
        return w[e];
    else
        return (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xffffu);
}

template <int DT>
__device__ __forceinline__ float ss_fma(uint32_t a, uint32_t b, float c)
{
    if constexpr (DT == DT_F32) {
        return fmaf(__uint_as_float(a), __uint_as_float(b), c);
    } else {
        const uint16_t ha = static_cast<uint16_t>(a), hb = static_cast<uint16_t>(b);
        if constexpr (DT == DT_F16)
            asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(c) : "h"(ha), "h"(hb));
        else
            asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(c) : "h"(ha), "h"(hb));
        return c;
    }
}

__device__ __forceinline__ void ss_copy16(void* dst, const void* src, int bytes)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(bytes)
                 : "memory");
}

template <int N>
__device__ __forceinline__ void ss_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Waits until at most `pending` of this thread's copy groups are in flight
// (at most SS_GROUP are waited for exactly; more pending waits for fewer).
__device__ __forceinline__ void ss_wait_pending(int pending)
{
    switch (pending) {
    case 0: ss_wait_group<0>(); break;
    case 1: ss_wait_group<1>(); break;
    case 2: ss_wait_group<2>(); break;
    case 3: ss_wait_group<3>(); break;
    default: ss_wait_group<4>(); break;
    }
}

__device__ __forceinline__ void ss_store(float* p, float v) { *p = v; }
__device__ __forceinline__ void ss_store(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void ss_store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ float ss_load(const float* p) { return *p; }
__device__ __forceinline__ float ss_load(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float ss_load(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <int DT, typename OutT, bool OP_A, bool OP_B>
__global__ void __launch_bounds__(SS_THREADS)
    simt_small_kernel(const void* __restrict__ Av, const void* __restrict__ Bv, OutT* C, int M,
                      int N, int K, float alpha, float beta)
{
    using T = typename SsElt<DT>::T;
    constexpr int ES = sizeof(T);
    constexpr int VE = 16 / ES;          // elements per 16-byte word
    constexpr int WPR = SS_TILE / VE;    // words per 16-element row
    extern __shared__ __align__(16) unsigned char ss_smem[];
    const T* A = static_cast<const T*>(Av);
    const T* B = static_cast<const T*>(Bv);
    const SsLayout L = ss_layout(K, ES, OP_A, OP_B);
    T* As = reinterpret_cast<T*>(ss_smem);
    T* Bs = As + L.a_elems;
    float* red = reinterpret_cast<float*>(Bs + L.b_elems);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int v0 = L.kv * warp / SS_WARPS, v1 = L.kv * (warp + 1) / SS_WARPS;
    const int groups = (v1 - v0 + SS_GROUP - 1) / SS_GROUP;
    const int r0 = (lane >> 2) * 2;  // this lane's rows: r0, r0 + 1
    const int q = lane & 3;          // and columns: col(j), j < 4
    auto col = [&](int j) { return OP_B ? q + 4 * j : 4 * q + j; };
    const int tiles_n = (N + SS_TILE - 1) / SS_TILE;
    const long long tiles = static_cast<long long>((M + SS_TILE - 1) / SS_TILE) * tiles_n;

    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int m0 = static_cast<int>(t / tiles_n) * SS_TILE;
        const int n0 = static_cast<int>(t % tiles_n) * SS_TILE;
        // Issue every copy of this warp's K range, one commit group per
        // SS_GROUP words.  A slice of nv words along K is 16 * nv words in
        // either layout, as is the B slice.
        for (int g = 0; g < groups; ++g) {
            const int va = v0 + g * SS_GROUP;
            const int nv = min(va + SS_GROUP, v1) - va;
            const int ka = va * VE;
            for (int i = lane; i < SS_TILE * nv; i += 32) {
                if (!OP_A) {  // A as stored, M x K: rows along k
                    const int row = i / nv, k = ka + (i % nv) * VE, m = m0 + row;
                    const int bytes = m < M ? max(0, min(VE, K - k)) * ES : 0;
                    ss_copy16(As + row * L.pitch + k,
                              bytes ? A + static_cast<long long>(m) * K + k : A, bytes);
                } else {      // A transposed, K x M: rows along m
                    const int k = ka + i / WPR, m = m0 + (i % WPR) * VE;
                    const int bytes = k < K ? max(0, min(VE, M - m)) * ES : 0;
                    ss_copy16(As + k * SS_TILE + (i % WPR) * VE,
                              bytes ? A + static_cast<long long>(k) * M + m : A, bytes);
                }
                if (!OP_B) {  // B as stored, K x N: rows along n
                    const int k = ka + i / WPR, n = n0 + (i % WPR) * VE;
                    const int bytes = k < K ? max(0, min(VE, N - n)) * ES : 0;
                    ss_copy16(Bs + k * SS_TILE + (i % WPR) * VE,
                              bytes ? B + static_cast<long long>(k) * N + n : B, bytes);
                } else {      // B transposed, N x K: rows along k
                    const int row = i / nv, k = ka + (i % nv) * VE, n = n0 + row;
                    const int bytes = n < N ? max(0, min(VE, K - k)) * ES : 0;
                    ss_copy16(Bs + row * L.pitch + k,
                              bytes ? B + static_cast<long long>(n) * K + k : B, bytes);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }

        float acc[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[i][j] = 0.0f;
        for (int g = 0; g < groups; ++g) {
            ss_wait_pending(groups - 1 - g);
            __syncwarp();
            const int va = v0 + g * SS_GROUP;
            const int vb = min(va + SS_GROUP, v1);
            for (int v = va; v < vb; ++v) {
                const int kw = v * VE;
                uint32_t a[2][VE], b[4][VE];
                if (!OP_A) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 w4 = *reinterpret_cast<const uint4*>(As + (r0 + i) * L.pitch + kw);
                        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < VE; ++e)
                            a[i][e] = ss_elt<ES>(w, e);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < VE; ++e) {
                        const T* p = As + (kw + e) * SS_TILE + r0;
                        if constexpr (ES == 4) {
                            const uint2 w2 = *reinterpret_cast<const uint2*>(p);
                            a[0][e] = w2.x;
                            a[1][e] = w2.y;
                        } else {
                            const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
                            a[0][e] = w & 0xffffu;
                            a[1][e] = w >> 16;
                        }
                    }
                }
                if (!OP_B) {
#pragma unroll
                    for (int e = 0; e < VE; ++e) {
                        const T* p = Bs + (kw + e) * SS_TILE + 4 * q;
                        uint32_t w[4];
                        if constexpr (ES == 4) {
                            const uint4 w4 = *reinterpret_cast<const uint4*>(p);
                            w[0] = w4.x; w[1] = w4.y; w[2] = w4.z; w[3] = w4.w;
                        } else {
                            const uint2 w2 = *reinterpret_cast<const uint2*>(p);
                            w[0] = w2.x; w[1] = w2.y; w[2] = 0u; w[3] = 0u;
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            b[j][e] = ss_elt<ES>(w, j);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 w4 = *reinterpret_cast<const uint4*>(Bs + col(j) * L.pitch + kw);
                        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < VE; ++e)
                            b[j][e] = ss_elt<ES>(w, e);
                    }
                }
#pragma unroll
                for (int e = 0; e < VE; ++e)
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            acc[i][j] = ss_fma<DT>(a[i][e], b[j][e], acc[i][j]);
            }
        }

        float* mine = red + warp * SS_TILE * SS_TILE;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                mine[(r0 + i) * SS_TILE + col(j)] = acc[i][j];
        __syncthreads();
        {
            const int r = threadIdx.x / SS_TILE, c = threadIdx.x % SS_TILE;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < SS_WARPS; ++w)
                sum += red[w * SS_TILE * SS_TILE + threadIdx.x];
            const int m = m0 + r, n = n0 + c;
            if (m < M && n < N) {
                OutT* p = C + static_cast<long long>(m) * N + n;
                float out = alpha * sum;
                if (beta != 0.0f)
                    out = fmaf(beta, ss_load(p), out);
                ss_store(p, out);
            }
        }
        __syncthreads();  // red is rewritten by the next tile
    }
}

int elem_size(int dt) { return dt == DT_F32 ? 4 : 2; }

template <int DT, typename OutT, bool OP_A, bool OP_B>
cudaError_t launch_layout(const SimtLaunch& l, long long smem, cudaStream_t stream)
{
    auto kern = simt_small_kernel<DT, OutT, OP_A, OP_B>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static bool ready[SS_MAX_DEVICES] = {};
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 0 || dev >= SS_MAX_DEVICES)
            return cudaErrorInvalidDevice;
        if (!ready[dev]) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SS_SMEM_LIMIT);
            if (err != cudaSuccess)
                return err;
            ready[dev] = true;
        }
    }
    const long long tiles =
        static_cast<long long>((l.M + SS_TILE - 1) / SS_TILE) * ((l.N + SS_TILE - 1) / SS_TILE);
    // One block per tile up to eight per SM; beyond that, blocks stride.
    const long long cap = static_cast<long long>(std::max(l.num_sms, 1)) * 8;
    const unsigned grid = static_cast<unsigned>(std::max<long long>(1, std::min(tiles, cap)));
    note_launch();
    kern<<<grid, SS_THREADS, static_cast<size_t>(smem), stream>>>(
        l.A, l.B, static_cast<OutT*>(l.C), l.M, l.N, l.K, l.alpha, l.beta);
    return cudaGetLastError();
}

template <int DT, typename OutT>
cudaError_t launch_out(const SimtLaunch& l, long long smem, cudaStream_t s)
{
    if (!l.op_a && !l.op_b)
        return launch_layout<DT, OutT, false, false>(l, smem, s);
    if (l.op_a && !l.op_b)
        return launch_layout<DT, OutT, true, false>(l, smem, s);
    if (!l.op_a && l.op_b)
        return launch_layout<DT, OutT, false, true>(l, smem, s);
    return launch_layout<DT, OutT, true, true>(l, smem, s);
}

template <int DT>
cudaError_t launch_in(const SimtLaunch& l, long long smem, cudaStream_t s)
{
    switch (l.out_dtype) {
    case DT_F32:
        return launch_out<DT, float>(l, smem, s);
    case DT_F16:
        return launch_out<DT, __half>(l, smem, s);
    default:
        return launch_out<DT, __nv_bfloat16>(l, smem, s);
    }
}

}  // namespace

bool simt_small_fits(const SimtLaunch& l)
{
    if (l.M <= 0 || l.N <= 0 || l.K < 0)
        return false;
    if (l.K == 0)
        return true;  // nothing is copied
    const int es = elem_size(l.in_dtype);
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(l.A) || !al(l.B))
        return false;
    const long long pitch_a = l.op_a ? l.M : l.K;
    const long long pitch_b = l.op_b ? l.K : l.N;
    if ((pitch_a * es) % 16 != 0 || (pitch_b * es) % 16 != 0)
        return false;
    return ss_layout(l.K, es, l.op_a != 0, l.op_b != 0).bytes <= SS_SMEM_LIMIT;
}

cudaError_t simt_small_launch(const SimtLaunch& l, cudaStream_t stream)
{
    if (!simt_small_fits(l))
        return cudaErrorNotSupported;
    const long long smem =
        ss_layout(l.K, elem_size(l.in_dtype), l.op_a != 0, l.op_b != 0).bytes;
    switch (l.in_dtype) {
    case DT_F32:
        return launch_in<DT_F32>(l, smem, stream);
    case DT_F16:
        return launch_in<DT_F16>(l, smem, stream);
    default:
        return launch_in<DT_BF16>(l, smem, stream);
    }
}

}  // namespace tmmo
