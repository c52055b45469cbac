// Shared-memory tiled SIMT GEMM: FP32 fused multiply-adds on the CUDA cores.
//
// This is the kernel shape of "Tiled Matrix Multiplication" (manual tiled
// kernel): a thread block owns one BM x BN output tile, walks K in tiles of
// BK, stages an A tile and a B tile in shared memory behind a barrier,
// accumulates in registers, and writes its outputs once after the last K
// tile.  K tiles are ceil(K / BK) with guarded loads (zero fill past the
// edges, which adds exactly zero), so any M, N, K is exact, including the
// partial tiles the pages' idiomatic kernel would drop.
//
// Differences from the page's kernel, for sm_103a:
//  * each thread accumulates a TM x TN micro-tile (strided by the thread
//    grid, so consecutive threads touch consecutive columns: conflict-free
//    B reads and coalesced C writes); TM = TN = 1 with BM = BN = BK = 3 is
//    exactly the page's TPB = 3, one-thread-per-output kernel;
//  * the A tile is stored K-major in shared memory (As[k][m], padded by one
//    word) so a warp's row reads are broadcasts and its tile stores are
//    conflict-free -- the access pattern the page's bank-conflict note
//    recommends;
//  * inputs are widened to FP32 when staged, so FP32, FP16 and BF16 inputs
//    share the kernel; the FP32 result is rounded to the output type with
//    round-to-nearest-even;
//  * the grid is 1-D and each block strides over output tiles, so any M, N
//    fit the launch limits;
//  * the next K tile is fetched into registers while the current one is
//    multiplied from shared memory, so global latency is paid once per tile
//    and overlapped with the FMAs;
//  * transposed operands (A stored K x M, B stored N x K) are read through
//    strides, with the staging loop walking the contiguous dimension so
//    global reads stay coalesced; the store computes alpha * acc + beta * C
//    (C read only when beta != 0).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "launch.h"

namespace tmmo {
namespace {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__half* p, float v) { *p = __float2half_rn(v); }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float load_out(const float* p) { return *p; }
__device__ __forceinline__ float load_out(const __half* p) { return __half2float(*p); }
__device__ __forceinline__ float load_out(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <int BM, int BN, int BK, int TM, int TN, typename InT, typename OutT>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
    simt_gemm_kernel(const InT* __restrict__ A, const InT* __restrict__ B, OutT* C, int M, int N,
                     int K, int op_a, int op_b, float alpha, float beta)
{
    constexpr int TX = BN / TN;  // threads along N
    constexpr int TY = BM / TM;  // threads along M
    constexpr int NT = TX * TY;
    constexpr int LA = (BM * BK + NT - 1) / NT;  // A elements each thread stages per K tile
    constexpr int LB = (BK * BN + NT - 1) / NT;  // B elements each thread stages per K tile
    __shared__ float As[BK][BM + 1];
    __shared__ float Bs[BK][BN + 1];

    const int tid = threadIdx.x;
    const int tx = tid % TX;
    const int ty = tid / TX;
    const int tiles_n = (N + BN - 1) / BN;
    const int tiles_m = (M + BM - 1) / BM;
    const long long num_tiles = static_cast<long long>(tiles_m) * tiles_n;

    // The next K tile is read from global memory into registers (all of a
    // thread's loads in flight together) while the current one is used from
    // shared memory; it is widened and stored after the barrier that ends
    // that use (kept in the input type until then, so that no conversion
    // waits for a load before the multiplies).
    InT ra[LA], rb[LB];
    const InT zero = static_cast<InT>(0.0f);
    auto load_tile = [&](int m0, int n0, int k0) {
        // A tile (BM x BK): consecutive threads walk the dimension that is
        // contiguous in memory (k for A as stored, m for A transposed).
#pragma unroll
        for (int r = 0; r < LA; ++r) {
            const int e = tid + r * NT;
            const int i = op_a ? e % BM : e / BK;
            const int k = op_a ? e / BM : e % BK;
            const int gm = m0 + i, gk = k0 + k;
            const long long off = op_a ? static_cast<long long>(gk) * M + gm
                                       : static_cast<long long>(gm) * K + gk;
            ra[r] = (e < BM * BK && gm < M && gk < K) ? A[off] : zero;
        }
        // B tile (BK x BN): n contiguous for B as stored, k for B transposed.
#pragma unroll
        for (int r = 0; r < LB; ++r) {
            const int e = tid + r * NT;
            const int k = op_b ? e % BK : e / BN;
            const int j = op_b ? e / BK : e % BN;
            const int gk = k0 + k, gn = n0 + j;
            const long long off = op_b ? static_cast<long long>(gn) * K + gk
                                       : static_cast<long long>(gk) * N + gn;
            rb[r] = (e < BK * BN && gk < K && gn < N) ? B[off] : zero;
        }
    };
    auto store_tile = [&]() {
#pragma unroll
        for (int r = 0; r < LA; ++r) {
            const int e = tid + r * NT;
            if (e < BM * BK)
                As[op_a ? e / BM : e % BK][op_a ? e % BM : e / BK] = to_f32(ra[r]);
        }
#pragma unroll
        for (int r = 0; r < LB; ++r) {
            const int e = tid + r * NT;
            if (e < BK * BN)
                Bs[op_b ? e % BK : e / BN][op_b ? e / BK : e % BN] = to_f32(rb[r]);
        }
    };

    for (long long tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int m0 = static_cast<int>(tile / tiles_n) * BM;
        const int n0 = static_cast<int>(tile % tiles_n) * BN;

        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j)
                acc[i][j] = 0.0f;

        if (K > 0) {
            load_tile(m0, n0, 0);
            store_tile();
            __syncthreads();
        }
        for (int k0 = 0; k0 < K; k0 += BK) {
            const bool more = k0 + BK < K;
            if (more)
                load_tile(m0, n0, k0 + BK);
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i)
                    a[i] = As[k][ty + i * TY];
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    b[j] = Bs[k][tx + j * TX];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j)
                        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
            if (more) {
                store_tile();
                __syncthreads();
            }
        }

#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int gm = m0 + ty + i * TY;
            if (gm >= M)
                continue;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int gn = n0 + tx + j * TX;
                if (gn < N) {
                    OutT* dst = C + static_cast<long long>(gm) * N + gn;
                    const float v = (beta != 0.0f) ? fmaf(beta, load_out(dst), alpha * acc[i][j])
                                                   : alpha * acc[i][j];
                    store_out(dst, v);
                }
            }
        }
    }
}

// Large-tile variant for grids that fill the GPU: a 128 x 128 block tile,
// K tiles of 8, and an 8 x 8 micro-tile per thread (256 threads).  A
// thread's rows are {4 ty .. 4 ty + 3} and {64 + 4 ty .. 64 + 4 ty + 3} and
// its columns likewise with tx, so each K step reads its 8 A and 8 B values
// as four 16-byte shared-memory loads (64 FMAs per 4 loads, against 16 per 8
// in the 4 x 4 kernel); a warp's B reads are 16 consecutive 16-byte words
// and its A reads are broadcasts, so neither conflicts.  Staging, prefetch,
// edge guards, transposed operands and the alpha/beta store are those of
// simt_gemm_kernel.
template <typename InT, typename OutT, bool OP_A, bool OP_B>
__global__ void __launch_bounds__(256, 2)
    simt_gemm_big_kernel(const InT* __restrict__ A, const InT* __restrict__ B, OutT* C, int M,
                         int N, int K, float alpha, float beta)
{
    constexpr bool op_a = OP_A, op_b = OP_B;  // operand layouts fixed at compile time
    constexpr int BM = 128, BN = 128, BK = 8, NT = 256, PAD = 4;
    constexpr int LA = BM * BK / NT, LB = BK * BN / NT;  // 4 and 4
    // Two shared tiles: the K tile being multiplied and the next one, so a
    // single barrier per K tile separates a tile's stores from its reads.
    __shared__ __align__(16) float As[2][BK][BM + PAD];
    __shared__ __align__(16) float Bs[2][BK][BN + PAD];

    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int tiles_n = (N + BN - 1) / BN;
    const int tiles_m = (M + BM - 1) / BM;
    const long long num_tiles = static_cast<long long>(tiles_m) * tiles_n;

    // A thread stages elements tid + 256 r (r < 4) of each tile, counted
    // along the dimension that is contiguous in memory.  For A as stored
    // (M x K) element r is at row tid / 8 + 32 r, k = tid % 8; for A stored
    // transposed (K x M) at row tid % 128, k = tid / 128 + 2 r; B likewise,
    // with columns for rows.  So element r lies a fixed distance from
    // element 0 (32 rows or 2 k), and one offset plus one stride per operand
    // address all four.
    const int a_i = op_a ? tid % BM : tid / BK;  // tile row of element 0
    const int a_k = op_a ? tid / BM : tid % BK;  // tile k of element 0
    const int a_di = op_a ? 0 : NT / BK;         // rows from one element to the next
    const int a_dk = op_a ? NT / BM : 0;         // k from one element to the next
    const long long a_rs = op_a ? static_cast<long long>(a_dk) * M
                                : static_cast<long long>(a_di) * K;
    const long long a_ks = op_a ? M : 1;         // global distance of one k
    const int b_j = op_b ? tid / BK : tid % BN;
    const int b_k = op_b ? tid % BK : tid / BN;
    const int b_dj = op_b ? NT / BK : 0;
    const int b_dk = op_b ? 0 : NT / BN;
    const long long b_rs = op_b ? static_cast<long long>(b_dj) * K
                                : static_cast<long long>(b_dk) * N;
    const long long b_ks = op_b ? 1 : N;

    InT ra[LA], rb[LB];  // raw until stored, as in simt_gemm_kernel
    const InT zero = static_cast<InT>(0.0f);
    long long a_off = 0, b_off = 0;  // global offset of element 0 at k = 0
    unsigned a_rows = 0, b_cols = 0; // bit r: element r's row (column) is inside C
    auto set_tile = [&](int m0, int n0) {
        const int gm = m0 + a_i;
        a_off = op_a ? static_cast<long long>(a_k) * M + gm : static_cast<long long>(gm) * K + a_k;
        a_rows = 0;
#pragma unroll
        for (int r = 0; r < LA; ++r)
            a_rows |= (gm + r * a_di < M ? 1u : 0u) << r;
        const int gn = n0 + b_j;
        b_off = op_b ? static_cast<long long>(gn) * K + b_k : static_cast<long long>(b_k) * N + gn;
        b_cols = 0;
#pragma unroll
        for (int r = 0; r < LB; ++r)
            b_cols |= (gn + r * b_dj < N ? 1u : 0u) << r;
    };
    auto load_tile = [&](int k0) {
        const long long ka = a_off + static_cast<long long>(k0) * a_ks;
        const long long kb = b_off + static_cast<long long>(k0) * b_ks;
#pragma unroll
        for (int r = 0; r < LA; ++r)
            ra[r] = ((a_rows >> r) & 1u) && k0 + a_k + r * a_dk < K ? A[ka + r * a_rs] : zero;
#pragma unroll
        for (int r = 0; r < LB; ++r)
            rb[r] = ((b_cols >> r) & 1u) && k0 + b_k + r * b_dk < K ? B[kb + r * b_rs] : zero;
    };
    auto store_tile = [&](int buf) {
#pragma unroll
        for (int r = 0; r < LA; ++r)
            As[buf][a_k + r * a_dk][a_i + r * a_di] = to_f32(ra[r]);
#pragma unroll
        for (int r = 0; r < LB; ++r)
            Bs[buf][b_k + r * b_dk][b_j + r * b_dj] = to_f32(rb[r]);
    };

    for (long long tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int m0 = static_cast<int>(tile / tiles_n) * BM;
        const int n0 = static_cast<int>(tile % tiles_n) * BN;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc[i][j] = 0.0f;

        // One K tile multiplied from shared buffer `buf`.  Odd rows of the
        // micro-tile take its columns in reverse, so the FMAs on either side
        // of a row change share their B operand (measured 1-9 % faster than
        // the plain row order on every layout).
        auto multiply = [&](int buf) {
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][4 * ty]);
                const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][64 + 4 * ty]);
                const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][4 * tx]);
                const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + 4 * tx]);
                const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = (i & 1) ? 7 - jj : jj;
                        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    }
            }
        };

        // K tile t is multiplied from buffer t & 1, with one barrier per K
        // tile.  The previous output tile's last barrier follows all of its
        // shared-memory reads, so both buffers are free here.  Two schedules
        // of the register prefetch, chosen per operand layout by measurement
        // on GB300 (one tile ahead was the faster on three layouts, two
        // ahead on A transposed with B as stored, by about 12 %; measured
        // with FP32 operands, which now go to simt_gemm_f32v_kernel when
        // their rows are 16-byte aligned):
        //  - one ahead: tile t + 1 is loaded before the multiplies of tile t
        //    and stored into the other buffer after them;
        //  - two ahead: tile t + 1, loaded during iteration t - 1, is stored
        //    first, then the loads of tile t + 2 are issued before the
        //    multiplies, so a barrier lies between each load and its store.
        set_tile(m0, n0);
        if constexpr (OP_A && !OP_B) {
            // two ahead
            const int nk = (K + BK - 1) / BK;
            if (nk > 0) {
                load_tile(0);
                store_tile(0);
                if (nk > 1)
                    load_tile(BK);
                __syncthreads();
            }
            for (int t = 0; t < nk; ++t) {
                const int buf = t & 1;
                if (t + 1 < nk)
                    store_tile(buf ^ 1);
                if (t + 2 < nk)
                    load_tile((t + 2) * BK);
                multiply(buf);
                __syncthreads();
            }
        } else {
            // one ahead
            int buf = 0;
            if (K > 0) {
                load_tile(0);
                store_tile(0);
                __syncthreads();
            }
            for (int k0 = 0; k0 < K; k0 += BK) {
                const bool more = k0 + BK < K;
                if (more)
                    load_tile(k0 + BK);
                multiply(buf);
                // the other buffer was last read before the previous barrier
                if (more)
                    store_tile(buf ^ 1);
                __syncthreads();
                buf ^= 1;
            }
        }

#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int gm = m0 + (i < 4 ? 4 * ty + i : 64 + 4 * ty + i - 4);
            if (gm >= M)
                continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int gn = n0 + (j < 4 ? 4 * tx + j : 64 + 4 * tx + j - 4);
                if (gn < N) {
                    OutT* dst = C + static_cast<long long>(gm) * N + gn;
                    const float v = (beta != 0.0f) ? fmaf(beta, load_out(dst), alpha * acc[i][j])
                                                   : alpha * acc[i][j];
                    store_out(dst, v);
                }
            }
        }
    }
}

// FP32 operands whose rows start on 16-byte boundaries (base addresses
// 16-byte aligned; the contiguous dimension of each stored operand a
// multiple of 4): the large-tile kernel with 16-byte global loads.  A
// 128 x 128 block tile, K tiles of 16, an 8 x 8 micro-tile per thread laid
// out as in simt_gemm_big_kernel.  Each thread moves two 16-byte words of
// each operand per K tile.  Words that run along m or n in memory (A
// transposed, B as stored) land whole in the K-major shared tile and are
// copied there by cp.async, without passing through registers; words that
// run along k (A as stored, B transposed) are loaded into registers one K
// tile ahead and scattered as four 4-byte stores.  With K % 4 == 0 (or M,
// N % 4 == 0 for the transposed forms) a word is either wholly inside the
// matrix or wholly outside it, so one guard per word keeps ragged edges
// exact (cp.async reads nothing and writes zeros for a word outside).
//
// Measured on GB300 (FP32 4096^3, TFLOP/s, cp.async / register staging for
// the words that land whole): A, B as stored 59.2 / 56.6; A transposed
// 62.0 / 54.9; B transposed and both transposed unchanged (57.0, 54.8).
//
// The multiply-adds run in pairs (fma.rn.f32x2: two IEEE single-precision
// fused multiply-adds, columns 2p and 2p + 1 of a micro-tile row, in one
// instruction), so a K step issues 32 instructions for its 64 multiply-adds
// and leaves issue slots for the fragment loads; each result is the same
// fused multiply-add as fmaf, in the same order.  The one exception is A as
// stored with B transposed: both operands then go through registers, the
// pairs' extra registers spill, and single FMAs are faster.  Measured on
// GB300 (FP32 4096^3, TFLOP/s, paired / single), with every operand staged
// through registers: A, B as stored 56.7 / 50.3; A transposed 55.8 / 51.0;
// A as stored, B transposed 52.8 / 57.1.  Both transposed, with A copied by
// cp.async: 58.5 / 54.8.
template <typename OutT, bool OP_A, bool OP_B>
__global__ void __launch_bounds__(256, 2)
    simt_gemm_f32v_kernel(const float* __restrict__ A, const float* __restrict__ B, OutT* C,
                          int M, int N, int K, float alpha, float beta)
{
    constexpr int BM = 128, BN = 128, BK = 16, NT = 256, LD = BM + 4;
    constexpr bool PAIRED = !OP_B || OP_A;
    // Operands whose 16-byte words run along m or n in memory (A
    // transposed, B as stored) go global -> shared by cp.async; the others
    // are staged through registers and scattered into the K-major tile.
    constexpr bool ASYNC_A = OP_A, ASYNC_B = !OP_B;
    constexpr bool ASYNC = ASYNC_A || ASYNC_B;
    // words per thread per operand and K tile: BM * BK / 4 / NT
    constexpr int WA = BM * BK / 4 / NT, WB = BK * BN / 4 / NT;
    __shared__ __align__(16) float As3[2][BK][LD];
    __shared__ __align__(16) float Bs3[2][BK][LD];
    // Shared-memory addresses are spelled two ways below, which give the
    // same addresses but lead the compiler to different schedules: array
    // subscripts in the paired form, a flat offset (these lambdas) in the
    // single one.  Measured on GB300 (FP32 4096^3, TFLOP/s, with every
    // operand staged through registers): subscripts 56.6 against 53.0 with
    // A and B as stored; the flat offset 56.6 against 55.2 with B
    // transposed and 54.9 against 52.9 with both transposed.
    auto As = [&](int buf, int k, int m) -> float* { return &As3[0][0][0] + (buf * BK + k) * LD + m; };
    auto Bs = [&](int buf, int k, int n) -> float* { return &Bs3[0][0][0] + (buf * BK + k) * LD + n; };

    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int tiles_n = (N + BN - 1) / BN;
    const int tiles_m = (M + BM - 1) / BM;
    const long long num_tiles = static_cast<long long>(tiles_m) * tiles_n;

    // Word w of a thread is word tid + NT * w of the tile, counted along the
    // contiguous dimension.  A as stored (M x K): a row holds BK / 4 words,
    // so word w sits at row tid / 4 + 64 w, k (tid % 4) * 4.  A transposed
    // (K x M): a k-row holds 32 words, so word w sits at k-row tid / 32 +
    // 8 w, m (tid % 32) * 4.  B likewise (B as stored is like A transposed).
    constexpr int KW = BK / 4;                       // words per row along k
    const int a_r = OP_A ? tid / 32 : tid / KW;      // row (or k-row) of word 0
    const int a_c = OP_A ? (tid % 32) * 4 : (tid % KW) * 4;
    constexpr int A_DR = OP_A ? NT / 32 : NT / KW;   // rows from one word to the next
    const int b_r = OP_B ? tid / KW : tid / 32;
    const int b_c = OP_B ? (tid % KW) * 4 : (tid % 32) * 4;
    constexpr int B_DR = OP_B ? NT / KW : NT / 32;

    float4 ra[WA], rb[WB];
    const float* a_ptr = A;
    const float* b_ptr = B;
    unsigned a_ok = 0, b_ok = 0;  // bit w: word w's m (or n) range lies inside C
    const long long a_wstride = OP_A ? static_cast<long long>(A_DR) * M
                                     : static_cast<long long>(A_DR) * K;
    const long long b_wstride = OP_B ? static_cast<long long>(B_DR) * K
                                     : static_cast<long long>(B_DR) * N;
    const long long a_kstep = OP_A ? static_cast<long long>(BK) * M : BK;
    const long long b_kstep = OP_B ? BK : static_cast<long long>(BK) * N;

    auto set_tile = [&](int m0, int n0) {
        a_ok = 0;
        b_ok = 0;
        if (OP_A) {
            a_ptr = A + static_cast<long long>(a_r) * M + m0 + a_c;
            if (m0 + a_c < M)
                a_ok = (1u << WA) - 1;
        } else {
            a_ptr = A + static_cast<long long>(m0 + a_r) * K + a_c;
#pragma unroll
            for (int w = 0; w < WA; ++w)
                a_ok |= (m0 + a_r + w * A_DR < M ? 1u : 0u) << w;
        }
        if (OP_B) {
            b_ptr = B + static_cast<long long>(n0 + b_r) * K + b_c;
#pragma unroll
            for (int w = 0; w < WB; ++w)
                b_ok |= (n0 + b_r + w * B_DR < N ? 1u : 0u) << w;
        } else {
            b_ptr = B + static_cast<long long>(b_r) * N + n0 + b_c;
            if (n0 + b_c < N)
                b_ok = (1u << WB) - 1;
        }
    };
    // Loads K tile k0 (a_ptr, b_ptr already advanced to it).
    auto load_tile = [&](int k0) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < WA && !ASYNC_A; ++w) {
            const int kk = OP_A ? k0 + a_r + w * A_DR : k0 + a_c;
            ra[w] = ((a_ok >> w) & 1u) && kk < K
                        ? __ldg(reinterpret_cast<const float4*>(a_ptr + w * a_wstride))
                        : z;
        }
#pragma unroll
        for (int w = 0; w < WB && !ASYNC_B; ++w) {
            const int kk = OP_B ? k0 + b_c : k0 + b_r + w * B_DR;
            rb[w] = ((b_ok >> w) & 1u) && kk < K
                        ? __ldg(reinterpret_cast<const float4*>(b_ptr + w * b_wstride))
                        : z;
        }
    };
    // Operands whose 16-byte words land whole in the shared tile (A
    // transposed, B as stored), copied global -> shared without registers
    // (cp.async, 16 bytes, zero fill past the edges).
    auto copy_async = [&](int buf, int k0) {
#pragma unroll
        for (int w = 0; w < WA && ASYNC_A; ++w) {
            const int kk = k0 + a_r + w * A_DR;
            const bool in = ((a_ok >> w) & 1u) && kk < K;
            const float* src = in ? a_ptr + w * a_wstride : A;
            const uint32_t dst = static_cast<uint32_t>(
                __cvta_generic_to_shared(&As3[buf][a_r + w * A_DR][a_c]));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                         "r"(in ? 16 : 0)
                         : "memory");
        }
#pragma unroll
        for (int w = 0; w < WB && ASYNC_B; ++w) {
            const int kk = k0 + b_r + w * B_DR;
            const bool in = ((b_ok >> w) & 1u) && kk < K;
            const float* src = in ? b_ptr + w * b_wstride : B;
            const uint32_t dst = static_cast<uint32_t>(
                __cvta_generic_to_shared(&Bs3[buf][b_r + w * B_DR][b_c]));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                         "r"(in ? 16 : 0)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto store_tile = [&](int buf) {
#pragma unroll
        for (int w = 0; w < WA && !ASYNC_A; ++w) {
            if constexpr (PAIRED) {
                if (OP_A) {
                    *reinterpret_cast<float4*>(&As3[buf][a_r + w * A_DR][a_c]) = ra[w];
                } else {
                    const int r = a_r + w * A_DR;
                    As3[buf][a_c + 0][r] = ra[w].x;
                    As3[buf][a_c + 1][r] = ra[w].y;
                    As3[buf][a_c + 2][r] = ra[w].z;
                    As3[buf][a_c + 3][r] = ra[w].w;
                }
            } else if (OP_A) {
                *reinterpret_cast<float4*>(As(buf, a_r + w * A_DR, a_c)) = ra[w];
            } else {
                const int r = a_r + w * A_DR;
                *As(buf, a_c + 0, r) = ra[w].x;
                *As(buf, a_c + 1, r) = ra[w].y;
                *As(buf, a_c + 2, r) = ra[w].z;
                *As(buf, a_c + 3, r) = ra[w].w;
            }
        }
#pragma unroll
        for (int w = 0; w < WB && !ASYNC_B; ++w) {
            if (OP_B) {
                const int r = b_r + w * B_DR;
                *Bs(buf, b_c + 0, r) = rb[w].x;
                *Bs(buf, b_c + 1, r) = rb[w].y;
                *Bs(buf, b_c + 2, r) = rb[w].z;
                *Bs(buf, b_c + 3, r) = rb[w].w;
            } else {
                *reinterpret_cast<float4*>(&Bs3[buf][b_r + w * B_DR][b_c]) = rb[w];
            }
        }
    };

    for (long long tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int m0 = static_cast<int>(tile / tiles_n) * BM;
        const int n0 = static_cast<int>(tile % tiles_n) * BN;
        // acc holds the micro-tile for single FMAs; acc2[i][p] columns 2p,
        // 2p + 1 of row i for paired ones (only one of the two is used).
        float acc[8][8];
        float2 acc2[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                acc[i][j] = 0.0f;
            if constexpr (PAIRED) {
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    acc2[i][p] = make_float2(0.0f, 0.0f);
            }
        }

        // One K tile from shared buffer `buf`.  Odd micro-tile rows take the
        // columns in reverse (the zig-zag order of simt_gemm_big_kernel).
        auto multiply = [&](int buf) {
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                if constexpr (PAIRED) {
                    const float4 a0 = *reinterpret_cast<const float4*>(&As3[buf][k][4 * ty]);
                    const float4 a1 = *reinterpret_cast<const float4*>(&As3[buf][k][64 + 4 * ty]);
                    const float4 b0 = *reinterpret_cast<const float4*>(&Bs3[buf][k][4 * tx]);
                    const float4 b1 = *reinterpret_cast<const float4*>(&Bs3[buf][k][64 + 4 * tx]);
                    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                         make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                        for (int pp = 0; pp < 4; ++pp) {
                            const int p = (i & 1) ? 3 - pp : pp;
                            acc2[i][p] = __ffma2_rn(ai, b[p], acc2[i][p]);
                        }
                    }
                } else {
                    const float4 b0 = *reinterpret_cast<const float4*>(Bs(buf, k, 4 * tx));
                    const float4 b1 = *reinterpret_cast<const float4*>(Bs(buf, k, 64 + 4 * tx));
                    const float4 a0 = *reinterpret_cast<const float4*>(As(buf, k, 4 * ty));
                    const float4 a1 = *reinterpret_cast<const float4*>(As(buf, k, 64 + 4 * ty));
                    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const int j = (i & 1) ? 7 - jj : jj;
                            acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                        }
                }
            }
        };

        // K tile t is multiplied from buffer t & 1; tile t + 1 is loaded
        // into registers before those multiplies and stored into the other
        // buffer after them, one barrier per K tile (the previous output
        // tile's last barrier follows all of its shared-memory reads).
        set_tile(m0, n0);
        const int nk = (K + BK - 1) / BK;
        if (nk > 0) {
            if constexpr (ASYNC)
                copy_async(0, 0);
            load_tile(0);
            store_tile(0);
            if constexpr (ASYNC)
                asm volatile("cp.async.wait_all;" ::: "memory");
            __syncthreads();
        }
        for (int t = 0; t < nk; ++t) {
            const bool more = t + 1 < nk;
            if (more) {
                a_ptr += a_kstep;
                b_ptr += b_kstep;
                if constexpr (ASYNC)
                    copy_async((t + 1) & 1, (t + 1) * BK);
                load_tile((t + 1) * BK);
            }
            multiply(t & 1);
            if (more)
                store_tile((t + 1) & 1);
            if constexpr (ASYNC)
                asm volatile("cp.async.wait_all;" ::: "memory");
            __syncthreads();
        }

        if constexpr (PAIRED) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    acc[i][2 * p] = acc2[i][p].x;
                    acc[i][2 * p + 1] = acc2[i][p].y;
                }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int gm = m0 + (i < 4 ? 4 * ty + i : 64 + 4 * ty + i - 4);
            if (gm >= M)
                continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int gn = n0 + (j < 4 ? 4 * tx + j : 64 + 4 * tx + j - 4);
                if (gn < N) {
                    OutT* dst = C + static_cast<long long>(gm) * N + gn;
                    const float v = (beta != 0.0f) ? fmaf(beta, load_out(dst), alpha * acc[i][j])
                                                   : alpha * acc[i][j];
                    store_out(dst, v);
                }
            }
        }
    }
}

// Whether the 16-byte-load FP32 kernel can take these operands: FP32
// inputs, 16-byte aligned bases, and rows of every stored operand a
// multiple of 4 elements long.
inline bool simt_f32v_ok(const SimtLaunch& l)
{
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (l.in_dtype != DT_F32 || !al(l.A) || !al(l.B))
        return false;
    const int pitch_a = l.op_a ? l.M : l.K;
    const int pitch_b = l.op_b ? l.K : l.N;
    return pitch_a % 4 == 0 && pitch_b % 4 == 0;
}

template <int BM, int BN, int BK, int TM, int TN, typename InT, typename OutT>
cudaError_t launch_simt(const SimtLaunch& l, cudaStream_t stream)
{
    constexpr int NT = (BM / TM) * (BN / TN);
    // Grids that fill every SM with 128 x 128 tiles take the large-tile kernel.
    const long long big_tiles = static_cast<long long>((l.M + 127) / 128) * ((l.N + 127) / 128);
    if (BM == 64 && big_tiles >= l.num_sms) {
        const long long cap = static_cast<long long>(std::max(l.num_sms, 1)) * 2;
        const int grid = static_cast<int>(std::max<long long>(1, std::min(big_tiles, cap)));
        if constexpr (std::is_same<InT, float>::value) {
            if (simt_f32v_ok(l)) {
                note_launch();
                const float* A = static_cast<const float*>(l.A);
                const float* B = static_cast<const float*>(l.B);
                OutT* C = static_cast<OutT*>(l.C);
                if (!l.op_a && !l.op_b)
                    simt_gemm_f32v_kernel<OutT, false, false>
                        <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
                else if (l.op_a && !l.op_b)
                    simt_gemm_f32v_kernel<OutT, true, false>
                        <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
                else if (!l.op_a && l.op_b)
                    simt_gemm_f32v_kernel<OutT, false, true>
                        <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
                else
                    simt_gemm_f32v_kernel<OutT, true, true>
                        <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
                return cudaGetLastError();
            }
        }
        note_launch();
        const InT* A = static_cast<const InT*>(l.A);
        const InT* B = static_cast<const InT*>(l.B);
        OutT* C = static_cast<OutT*>(l.C);
        if (!l.op_a && !l.op_b)
            simt_gemm_big_kernel<InT, OutT, false, false>
                <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
        else if (l.op_a && !l.op_b)
            simt_gemm_big_kernel<InT, OutT, true, false>
                <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
        else if (!l.op_a && l.op_b)
            simt_gemm_big_kernel<InT, OutT, false, true>
                <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
        else
            simt_gemm_big_kernel<InT, OutT, true, true>
                <<<grid, 256, 0, stream>>>(A, B, C, l.M, l.N, l.K, l.alpha, l.beta);
        return cudaGetLastError();
    }
    const long long tiles = static_cast<long long>((l.M + BM - 1) / BM) * ((l.N + BN - 1) / BN);
    // Enough blocks for several resident per SM; each strides over tiles.
    const long long cap = static_cast<long long>(std::max(l.num_sms, 1)) * 16;
    const int grid = static_cast<int>(std::max<long long>(1, std::min(tiles, cap)));
    note_launch();
    simt_gemm_kernel<BM, BN, BK, TM, TN, InT, OutT><<<grid, NT, 0, stream>>>(
        static_cast<const InT*>(l.A), static_cast<const InT*>(l.B), static_cast<OutT*>(l.C), l.M,
        l.N, l.K, l.op_a, l.op_b, l.alpha, l.beta);
    return cudaGetLastError();
}

template <int BM, int BN, int BK, int TM, int TN, typename InT>
cudaError_t dispatch_out(const SimtLaunch& l, cudaStream_t s)
{
    switch (l.out_dtype) {
    case DT_F32:
        return launch_simt<BM, BN, BK, TM, TN, InT, float>(l, s);
    case DT_F16:
        return launch_simt<BM, BN, BK, TM, TN, InT, __half>(l, s);
    default:
        return launch_simt<BM, BN, BK, TM, TN, InT, __nv_bfloat16>(l, s);
    }
}

template <int BM, int BN, int BK, int TM, int TN>
cudaError_t dispatch_in(const SimtLaunch& l, cudaStream_t s)
{
    switch (l.in_dtype) {
    case DT_F32:
        return dispatch_out<BM, BN, BK, TM, TN, float>(l, s);
    case DT_F16:
        return dispatch_out<BM, BN, BK, TM, TN, __half>(l, s);
    default:
        return dispatch_out<BM, BN, BK, TM, TN, __nv_bfloat16>(l, s);
    }
}

}  // namespace

cudaError_t simt_gemm_launch(const SimtLaunch& l, cudaStream_t stream)
{
    if (l.tpb3)
        return dispatch_in<3, 3, 3, 1, 1>(l, stream);
    return dispatch_in<64, 64, 16, 4, 4>(l, stream);
}

}  // namespace tmmo
