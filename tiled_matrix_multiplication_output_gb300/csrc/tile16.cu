// Latency-path GEMM for small products: one 16 x 16 output tile per thread
// block, with the tile's whole K range of A rows and B columns staged in
// shared memory at once and split between the block's eight warps.
//
// A small product is a chain of latencies rather than work ("A memory count
// is not a latency estimate", Reading a matrix multiply through its tiles).
// The tcgen05 kernels spend about a microsecond on barrier and accumulator
// set-up and tensor-map fetches before their first copy lands, and the
// tiled SIMT kernel pays one memory round trip per K tile.  This kernel
// avoids both: every thread issues all of its copies (cp.async, 16 bytes,
// zero fill past the edges) before it waits for any, and the eight warps of
// a block split K between them, so a block's first multiply waits for one
// round trip and its warps meet only once, at the end.
//
//  * tile: a block owns 16 x 16 outputs and writes each of them once, from
//    one thread, after the last K term ("Keep one output tile resident");
//    every warp accumulates the whole tile over its own range of K and the
//    eight partials are summed through shared memory in warp order;
//  * K is cut into 16-byte words (8 elements of 16-bit inputs, 4 of FP32);
//    warp w takes an eighth of them and copies its own A and B slices in
//    groups of four words, waiting only for its own copies
//    (cp.async.wait_group, then __syncwarp for its lanes');
//  * 16-bit inputs: each warp multiplies on the tensor cores with the
//    warp-level MMA (mma.sync m16n8k16, FP32 accumulation), two
//    instructions per 16 values of K for the whole 16 x 16 tile, fed from
//    the staged slices by ldmatrix; the warps' ranges are whole multiples
//    of 16 (the last word of K zero filled).  tcgen05.mma tiles start at 64
//    rows per CTA and bring TMEM allocation, an mbarrier handshake and a
//    tensor-map fetch -- the fixed costs this kernel exists to avoid;
//  * FP32 inputs: fused multiply-adds on the CUDA cores (fmaf), each lane
//    two rows by four columns of the tile, k ascending;
//  * edges: a word that crosses the end of K is copied in part and zero
//    filled, and rows past M or columns past N are zero filled, so each
//    output sums exactly the definition's terms ("Edge tiles still
//    matter"); the rows and columns past the edges are never stored;
//  * layouts: a k-contiguous slice (A as stored, B transposed) keeps its
//    rows padded to 16 bytes past a multiple of 128, so the eight rows of
//    one ldmatrix (or the rows of one quarter-warp) fall in different
//    banks; an m- or n-contiguous slice (A transposed, B as stored) is kept
//    as 16-element rows along k.
//
// Requirements (tile16_fits): 16-byte aligned A and B, each stored
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

constexpr int T16_TILE = 16;                 // output tile edge
constexpr int T16_WARPS = 8;                 // warps per block, each a range of K
constexpr int T16_THREADS = 32 * T16_WARPS;
constexpr int T16_GROUP = 4;                 // 16-byte words per commit group
constexpr int T16_SMEM_LIMIT = 227 * 1024;   // dynamic shared memory per block
constexpr int T16_MAX_DEVICES = 64;

// Shared-memory layout of one tile's K slices.
struct T16Layout {
    int kv;          // 16-byte words along K (even for 16-bit inputs)
    int pitch;       // row pitch (elements) of a k-contiguous slice
    int a_elems;     // elements of the A slice
    int b_elems;     // elements of the B slice
    long long bytes; // dynamic shared memory of a block
};

__host__ __device__ inline T16Layout t16_layout(long long K, int es, bool op_a, bool op_b)
{
    const int ve = 16 / es;
    const int unit = es == 2 ? 2 : 1;  // words per K step of a warp (16 values for the MMA)
    T16Layout s{};
    const long long kv = ((K + ve - 1) / ve + unit - 1) / unit * unit;
    const long long kp = kv * ve;  // K rounded up to whole steps
    const long long pitch = ((kp * es + 127) / 128) * 128 / es + 16 / es;
    const long long a = op_a ? kp * T16_TILE : T16_TILE * pitch;
    const long long b = op_b ? T16_TILE * pitch : kp * T16_TILE;
    s.bytes = (a + b) * es + static_cast<long long>(T16_WARPS) * T16_TILE * T16_TILE * 4;
    if (s.bytes > T16_SMEM_LIMIT)
        return s;  // too large; the other fields are not used
    s.kv = static_cast<int>(kv);
    s.pitch = static_cast<int>(pitch);
    s.a_elems = static_cast<int>(a);
    s.b_elems = static_cast<int>(b);
    return s;
}

// Raw elements: FP32, or the 16 bits of an F16 / BF16 value.
template <int DT>
struct T16Elt {
    using T = uint16_t;
};
template <>
struct T16Elt<DT_F32> {
    using T = float;
};

__device__ __forceinline__ void t16_copy16(void* dst, const void* src, int bytes)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(bytes)
                 : "memory");
}

template <int N>
__device__ __forceinline__ void t16_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Waits until at most `pending` of this thread's copy groups are in flight
// (more than four pending waits for four).
__device__ __forceinline__ void t16_wait_pending(int pending)
{
    switch (pending) {
    case 0: t16_wait_group<0>(); break;
    case 1: t16_wait_group<1>(); break;
    case 2: t16_wait_group<2>(); break;
    case 3: t16_wait_group<3>(); break;
    default: t16_wait_group<4>(); break;
    }
}

// Four 8 x 8 matrices of 16-bit elements from shared memory; each lane
// passes the address of one matrix row (lanes 8q .. 8q + 7: matrix q).
template <bool TRANS>
__device__ __forceinline__ void t16_ldmatrix4(const void* row, uint32_t (&r)[4])
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(row));
    if constexpr (TRANS)
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(a));
    else
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(a));
}

// d += a b for one 16 x 8 block: a the 16 x 16 A fragment, b0 b1 the
// 16 x 8 B fragment, FP32 accumulation.
template <int DT>
__device__ __forceinline__ void t16_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1)
{
    if constexpr (DT == DT_F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void t16_store(float* p, float v) { *p = v; }
__device__ __forceinline__ void t16_store(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void t16_store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ float t16_load(const float* p) { return *p; }
__device__ __forceinline__ float t16_load(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float t16_load(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <int DT, typename OutT, bool OP_A, bool OP_B>
__global__ void __launch_bounds__(T16_THREADS)
    tile16_kernel(const void* __restrict__ Av, const void* __restrict__ Bv, OutT* C, int M, int N,
                  int K, float alpha, float beta)
{
    using T = typename T16Elt<DT>::T;
    constexpr int ES = sizeof(T);
    constexpr bool MMA = ES == 2;
    constexpr int VE = 16 / ES;           // elements per 16-byte word
    constexpr int WPR = T16_TILE / VE;    // words per 16-element row
    constexpr int UNIT = MMA ? 2 : 1;     // words per K step of a warp
    extern __shared__ __align__(16) unsigned char t16_smem[];
    const T* A = static_cast<const T*>(Av);
    const T* B = static_cast<const T*>(Bv);
    const T16Layout L = t16_layout(K, ES, OP_A, OP_B);
    T* As = reinterpret_cast<T*>(t16_smem);
    T* Bs = As + L.a_elems;
    float* red = reinterpret_cast<float*>(Bs + L.b_elems);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int steps = L.kv / UNIT;
    const int v0 = UNIT * (steps * warp / T16_WARPS);
    const int v1 = UNIT * (steps * (warp + 1) / T16_WARPS);
    const int groups = (v1 - v0 + T16_GROUP - 1) / T16_GROUP;
    const int tiles_n = (N + T16_TILE - 1) / T16_TILE;
    const long long tiles = static_cast<long long>((M + T16_TILE - 1) / T16_TILE) * tiles_n;

    for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int m0 = static_cast<int>(t / tiles_n) * T16_TILE;
        const int n0 = static_cast<int>(t % tiles_n) * T16_TILE;
        // Issue every copy of this warp's K range, one commit group per
        // T16_GROUP words.  A group of nv words along K is 16 nv copies per
        // operand in either layout, at most 64: two slots per lane.
        for (int g = 0; g < groups; ++g) {
            const int va = v0 + g * T16_GROUP;
            const int nv = min(va + T16_GROUP, v1) - va;
            const int ka = va * VE;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int i = lane + 32 * x;
                if (!OP_A) {  // A as stored, M x K: 16 rows of nv words
                    const int row = i >> 2, w = i & 3;
                    if (w < nv) {
                        const int k = ka + w * VE, m = m0 + row;
                        const int bytes = m < M ? max(0, min(VE, K - k)) * ES : 0;
                        t16_copy16(As + row * L.pitch + k,
                                   bytes ? A + static_cast<long long>(m) * K + k : A, bytes);
                    }
                } else {      // A transposed, K x M: nv VE rows along k of WPR words
                    const int kr = i / WPR, w = i % WPR;
                    if (kr < nv * VE) {
                        const int k = ka + kr, m = m0 + w * VE;
                        const int bytes = k < K ? max(0, min(VE, M - m)) * ES : 0;
                        t16_copy16(As + k * T16_TILE + w * VE,
                                   bytes ? A + static_cast<long long>(k) * M + m : A, bytes);
                    }
                }
                if (!OP_B) {  // B as stored, K x N: nv VE rows along k of WPR words
                    const int kr = i / WPR, w = i % WPR;
                    if (kr < nv * VE) {
                        const int k = ka + kr, n = n0 + w * VE;
                        const int bytes = k < K ? max(0, min(VE, N - n)) * ES : 0;
                        t16_copy16(Bs + k * T16_TILE + w * VE,
                                   bytes ? B + static_cast<long long>(k) * N + n : B, bytes);
                    }
                } else {      // B transposed, N x K: 16 rows of nv words
                    const int row = i >> 2, w = i & 3;
                    if (w < nv) {
                        const int k = ka + w * VE, n = n0 + row;
                        const int bytes = n < N ? max(0, min(VE, K - k)) * ES : 0;
                        t16_copy16(Bs + row * L.pitch + k,
                                   bytes ? B + static_cast<long long>(n) * K + k : B, bytes);
                    }
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }

        float* mine = red + warp * T16_TILE * T16_TILE;
        if constexpr (MMA) {
            // Lanes 8q .. 8q + 7 address the rows of matrix q of each x4
            // ldmatrix.  A fragment: matrices (rows 0-7, k 0-7), (rows
            // 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15); B
            // fragment: (k 0-7, n 0-7), (k 8-15, n 0-7), (k 0-7, n 8-15),
            // (k 8-15, n 8-15), the first two for columns 0-7, the last two
            // for columns 8-15.
            const int mq = lane >> 3, mr = lane & 7;
            float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int g = 0; g < groups; ++g) {
                t16_wait_pending(groups - 1 - g);
                __syncwarp();
                const int va = v0 + g * T16_GROUP;
                const int vb = min(va + T16_GROUP, v1);
                for (int v = va; v < vb; v += UNIT) {
                    const int k0 = v * VE;
                    uint32_t a[4], b[4];
                    if (!OP_A)
                        t16_ldmatrix4<false>(As + ((mq & 1) * 8 + mr) * L.pitch + k0 + (mq >> 1) * 8, a);
                    else
                        t16_ldmatrix4<true>(As + (k0 + (mq >> 1) * 8 + mr) * T16_TILE + (mq & 1) * 8, a);
                    if (!OP_B)
                        t16_ldmatrix4<true>(Bs + (k0 + (mq & 1) * 8 + mr) * T16_TILE + (mq >> 1) * 8, b);
                    else
                        t16_ldmatrix4<false>(Bs + ((mq >> 1) * 8 + mr) * L.pitch + k0 + (mq & 1) * 8, b);
                    t16_mma<DT>(d[0], a, b[0], b[1]);
                    t16_mma<DT>(d[1], a, b[2], b[3]);
                }
            }
            // Accumulator of block nb: (row g, columns 2t, 2t + 1) and
            // (row g + 8, the same columns), g = lane / 4, t = lane % 4.
            const int gr = lane >> 2, tc = (lane & 3) * 2;
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                *reinterpret_cast<float2*>(mine + gr * T16_TILE + nb * 8 + tc) =
                    make_float2(d[nb][0], d[nb][1]);
                *reinterpret_cast<float2*>(mine + (gr + 8) * T16_TILE + nb * 8 + tc) =
                    make_float2(d[nb][2], d[nb][3]);
            }
        } else {
            // Each lane: rows r0, r0 + 1 and four columns (4q .. 4q + 3 of
            // B as stored, q, q + 4, q + 8, q + 12 of B transposed, so that
            // the rows of one quarter-warp's reads fall in different banks).
            const int r0 = (lane >> 2) * 2;
            const int q = lane & 3;
            auto col = [&](int j) { return OP_B ? q + 4 * j : 4 * q + j; };
            float acc[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[i][j] = 0.0f;
            for (int g = 0; g < groups; ++g) {
                t16_wait_pending(groups - 1 - g);
                __syncwarp();
                const int va = v0 + g * T16_GROUP;
                const int vb = min(va + T16_GROUP, v1);
                for (int v = va; v < vb; ++v) {
                    const int kw = v * VE;
                    float a[2][4], b[4][4];
                    if (!OP_A) {
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const float4 w = *reinterpret_cast<const float4*>(As + (r0 + i) * L.pitch + kw);
                            a[i][0] = w.x; a[i][1] = w.y; a[i][2] = w.z; a[i][3] = w.w;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 w = *reinterpret_cast<const float2*>(As + (kw + e) * T16_TILE + r0);
                            a[0][e] = w.x;
                            a[1][e] = w.y;
                        }
                    }
                    if (!OP_B) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 w = *reinterpret_cast<const float4*>(Bs + (kw + e) * T16_TILE + 4 * q);
                            b[0][e] = w.x; b[1][e] = w.y; b[2][e] = w.z; b[3][e] = w.w;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 w = *reinterpret_cast<const float4*>(Bs + col(j) * L.pitch + kw);
                            b[j][0] = w.x; b[j][1] = w.y; b[j][2] = w.z; b[j][3] = w.w;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e)
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                acc[i][j] = fmaf(a[i][e], b[j][e], acc[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mine[(r0 + i) * T16_TILE + col(j)] = acc[i][j];
        }
        __syncthreads();
        {
            const int r = threadIdx.x / T16_TILE, c = threadIdx.x % T16_TILE;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < T16_WARPS; ++w)
                sum += red[w * T16_TILE * T16_TILE + threadIdx.x];
            const int m = m0 + r, n = n0 + c;
            if (m < M && n < N) {
                OutT* p = C + static_cast<long long>(m) * N + n;
                float out = alpha * sum;
                if (beta != 0.0f)
                    out = fmaf(beta, t16_load(p), out);
                t16_store(p, out);
            }
        }
        __syncthreads();  // red is rewritten by the next tile
    }
}

int elem_size(int dt) { return dt == DT_F32 ? 4 : 2; }

template <int DT, typename OutT, bool OP_A, bool OP_B>
cudaError_t launch_layout(const SimtLaunch& l, long long smem, cudaStream_t stream)
{
    auto kern = tile16_kernel<DT, OutT, OP_A, OP_B>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static bool ready[T16_MAX_DEVICES] = {};
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 0 || dev >= T16_MAX_DEVICES)
            return cudaErrorInvalidDevice;
        if (!ready[dev]) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       T16_SMEM_LIMIT);
            if (err != cudaSuccess)
                return err;
            ready[dev] = true;
        }
    }
    const long long tiles = static_cast<long long>((l.M + T16_TILE - 1) / T16_TILE) *
                            ((l.N + T16_TILE - 1) / T16_TILE);
    // One block per tile up to eight per SM; beyond that, blocks stride.
    const long long cap = static_cast<long long>(std::max(l.num_sms, 1)) * 8;
    const unsigned grid = static_cast<unsigned>(std::max<long long>(1, std::min(tiles, cap)));
    note_launch();
    kern<<<grid, T16_THREADS, static_cast<size_t>(smem), stream>>>(
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

bool tile16_fits(const SimtLaunch& l)
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
    return t16_layout(l.K, es, l.op_a != 0, l.op_b != 0).bytes <= T16_SMEM_LIMIT;
}

cudaError_t tile16_launch(const SimtLaunch& l, cudaStream_t stream)
{
    if (!tile16_fits(l))
        return cudaErrorNotSupported;
    const long long smem = t16_layout(l.K, elem_size(l.in_dtype), l.op_a != 0, l.op_b != 0).bytes;
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
