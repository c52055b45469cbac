// Output-stationary tiled C = A @ B on the 5th-generation tensor cores.
//
// The loop nest is the one of "Reading a matrix multiply through its tiles"
// ("Keep one output tile resident"): for every output tile, the FP32
// accumulator starts at zero, A and B tiles stream along K into fast memory
// and are contracted into it, and the finished tile is written to C once.
// On sm_103a that becomes:
//
//   * a persistent grid (one CTA, or one CTA pair, per SM) that strides over
//     the output tiles in grouped raster order, so that concurrently running
//     tiles share A row-panels and B column-panels in L2;
//   * warp 0: the TMA producer.  It streams 128-byte-swizzled A boxes
//     (128 rows x 64 K, K-major) and B boxes (64 K x 64 N, N-major, i.e. B
//     stays row-major and is not transposed) into a STAGES-deep shared-memory
//     ring guarded by full/empty mbarriers;
//   * warp 1: the MMA issuer.  One thread issues tcgen05.mma (K = 16 per
//     instruction, four per 64-wide K step) into an FP32 accumulator held in
//     tensor memory (TMEM); the first MMA of a tile runs with accumulation
//     disabled, which is the "zero the accumulator" step.  Two accumulators
//     are kept so the epilogue of tile t overlaps the main loop of tile t+1;
//   * warps 2-5: the epilogue.  Each warp owns 32 TMEM lanes (32 output
//     rows), reads 32 columns at a time with tcgen05.ld, converts FP32 to the
//     output type with round-to-nearest-even, writes a 128-byte-swizzled
//     staging buffer and issues a TMA store.  The store clips rows >= M and
//     columns >= N, and TMA loads fill out-of-range A/B elements with zeros
//     (which add exactly nothing), so partial edge tiles in M, N and K are
//     exact ("Edge tiles still matter").
//
// Operands may also be given transposed ("Tiled Matrix Multiplication",
// "When would transposed loading be useful?"): op(A) = A^T is A stored K x M
// (M contiguous, an MN-major tcgen05 operand) and op(B) = B^T is B stored
// N x K (K contiguous, a K-major operand).  The template flags A_MN / B_MN
// select the box shapes and shared-memory descriptors; nothing is transposed
// in memory.  The epilogue can also compute alpha * acc + beta * C_in, the
// accumulate-into-C form of the helion kernel's torch.addmm ("Writing a
// matmul GPU kernel").
//
// Split-K (SPLIT = true): a unit of work is an output tile and one range of
// K steps; its FP32 partial goes to a workspace [split][M][N] through a 3-D
// TMA store, and a separate kernel sums the partials in split order.
//
// CG = 2 runs the same protocol on a CTA pair (cta_group::2): each CTA loads
// its own 128 rows of A and half of the B columns, the leader CTA issues
// M = 256 MMAs that read both CTAs' shared memory, and each CTA's TMEM holds
// its 128 rows of the 256 x BN accumulator.  No TMA multicast is used.
//
// Every mbarrier wait is bounded by a clock budget.  When one runs out the
// kernel records GEMM_ERR_TIMEOUT in the device status word, every role
// leaves its loop, in-flight copies and MMAs are drained (again bounded),
// TMEM is freed and the kernel returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "tc_params.h"

namespace tmmo {

constexpr int TC_BM = 128;       // accumulator rows per CTA (TMEM lanes)
constexpr int TC_BK = 64;        // K per stage: 64 x 2 bytes = one 128-byte swizzle row
constexpr int TC_UMMA_K = 16;    // K per tcgen05.mma for 16-bit inputs
constexpr int TC_THREADS = 192;  // 6 warps
constexpr int TC_EPI_WARP0 = 2;
constexpr int TC_STAGING_BYTES = 4096;  // 32 rows x 128 bytes per warp buffer
// Share of the next work item's main loop over which a finished tile's
// stores are spread (percent).  Every CTA finishes its tile at about the
// same time, and storing all of C's tiles at once delays the operand loads
// of the next tiles; a gap after each strip's store spreads the writes out.
// Measured on GB300 (BF16, the CTA-pair kernel, interleaved runs): 1-2 %
// off 8192^3 and 4096^3, 5 % off 12288 x 12288 x 2048, 3 % off
// 5120 x 5120 x 1024; spreading over 40 % or 60 % lost time at short K, and
// staggering the four epilogue warps against each other did not help.
#ifndef TMMO_STORE_SPREAD_PCT
#define TMMO_STORE_SPREAD_PCT 25
#endif

// KSUB 64-wide K steps share one shared-memory stage, released by one commit
// per KSUB * 4 MMAs; sub-step j of a stage sits at j * SUB_A / j * SUB_B.
// Each sub-step has its own full barrier, so the MMAs of the first K step
// start as soon as its copies land, while the stage's later copies are still
// in flight (measured on GB300: 4.5 % less time at 8192^3 and 4096^3 than
// one full barrier per stage).
template <int CG, int BN, int STAGES, int KSUB = 1>
struct TcLayout {
    static constexpr int SUB_A = TC_BM * TC_BK * 2;              // 16 KiB per K step
    static constexpr int A_STAGE = KSUB * SUB_A;
    static constexpr int B_COLS = BN / CG;                       // B columns held per CTA
    static constexpr int SUB_B = TC_BK * B_COLS * 2;
    static constexpr int B_STAGE = KSUB * SUB_B;
    static constexpr int B_BOXES = B_COLS / 64;                  // 64-column, 8 KiB boxes
    static constexpr int SUB_BYTES = SUB_A + SUB_B;              // bytes per K step per CTA
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_STAGING = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_BAR = OFF_STAGING + 4 * 2 * TC_STAGING_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5 + STAGES * (KSUB - 1);  // + full per later K step
    static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t TMEM_COLS = 2 * BN;    // two FP32 accumulators
    static_assert(B_COLS % 64 == 0, "B boxes are 64 columns wide");
    static_assert(TMEM_COLS == 32 || TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 ||
                      TMEM_COLS == 512,
                  "TMEM allocations are a power of two >= 32 columns");
    static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KiB of dynamic shared memory");
};

// Instruction descriptor of tcgen05.mma kind::f16: F32 accumulator (bits
// 4-5 = 1), A/B type F16 (0) or BF16 (1) in bits 7-9 / 10-12, A major-ness
// in bit 15 and B major-ness in bit 16 (0 = K-major, 1 = MN-major), N >> 3 in
// bits 17-22 and M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t tc_idesc(bool bf16, int m, int n, bool a_mn = false,
                                                bool b_mn = true)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Grouped raster order: tiles are taken `group_m` tile-rows at a time and,
// inside a group, down the rows of one tile-column before the next column.
__device__ __forceinline__ void tc_tile_coords(int t, const TcParams& p, int& mb, int& nb)
{
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int gm = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

// One unit of work: an output tile and the range of K steps it accumulates.
// Units t < dp_tiles are whole tiles (tile t, all of K), written to C.  The
// remaining units split the last num_tiles - dp_tiles tiles along K into
// k_splits ranges each (unit dp_tiles + j: tile dp_tiles + j / k_splits,
// range j % k_splits); their FP32 partials go to a workspace and are summed
// by a second kernel.  dp_tiles = num_tiles is the plain product, dp_tiles =
// 0 is split-K, anything between fills the last, partial wave of tiles with
// split pieces so that every CTA finishes at about the same time.
struct TcWork {
    int mb, nb;
    int kb_begin, kb_end;
    int split;    // K range within the tile
    int slot;     // index of the partial among all split units
    bool partial;
};

__device__ __forceinline__ TcWork tc_work(int t, const TcParams& p)
{
    TcWork w;
    int tile;
    if (t < p.dp_tiles) {
        tile = t;
        w.split = 0;
        w.slot = 0;
        w.partial = false;
        w.kb_begin = 0;
        w.kb_end = p.k_blocks;
    } else {
        const int j = t - p.dp_tiles;
        tile = p.dp_tiles + j / p.k_splits;
        w.split = j % p.k_splits;
        w.slot = j;
        w.partial = true;
        w.kb_begin = w.split * p.kb_per_split;
        w.kb_end = min(p.k_blocks, w.kb_begin + p.kb_per_split);
    }
    tc_tile_coords(tile, p, w.mb, w.nb);
    return w;
}

struct TcWatch {
    volatile int* abort_flag;  // shared memory, this CTA
    int* status;               // device status word
    long long budget;          // clock cycles per wait
};

__device__ __forceinline__ void tc_raise(const TcWatch& w)
{
    *w.abort_flag = 1;
    if (w.status)
        atomicCAS(w.status, 0, TC_STATUS_TIMEOUT);
}

// Bounded wait on an mbarrier phase.  Returns false if the budget ran out
// (and raises the abort) or another role already aborted.
template <bool CLUSTER_SCOPE = false>
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, const TcWatch& w)
{
    auto probe = [&]() {
        return CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (probe())
        return true;
    const long long t0 = clock64();
    while (true) {
        if (probe())
            return true;
        if (*w.abort_flag)
            return false;
        if (clock64() - t0 > w.budget) {
            tc_raise(w);
            return false;
        }
    }
}

template <typename OutT>
struct TcOut;
template <>
struct TcOut<float> {
    static constexpr int STRIP = 32;  // columns per 128-byte staging row
};
template <>
struct TcOut<__half> {
    static constexpr int STRIP = 64;
};
template <>
struct TcOut<__nv_bfloat16> {
    static constexpr int STRIP = 64;
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half*)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16*)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Read one 128-byte-wide strip (32 rows x STRIP columns) of the accumulator
// from TMEM, convert, and write it to a swizzled staging buffer: 16-byte
// chunk c of row r goes to chunk position c ^ (r % 8), the layout a
// SWIZZLE_128B TMA store expects, and conflict-free for 8 rows at a time.
__device__ __forceinline__ float out_to_f32(float v) { return v; }
__device__ __forceinline__ float out_to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float out_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// v[i] <- alpha * v[i] + beta * C_in[grow, gcol + i] for the `n` values of one
// 16-byte chunk of this thread's row (n = 4 FP32 or 8 16-bit values).  The
// chunk is read only if it lies inside C; N * sizeof(OutT) is a multiple of
// 16, so chunks never straddle the right edge.
template <typename OutT, int n>
__device__ __forceinline__ void tc_axpby_chunk(float* v, const TcParams& p, int grow, int gcol)
{
    if (p.beta != 0.0f && grow < p.M && gcol < p.N) {
        const OutT* src = static_cast<const OutT*>(p.C) + static_cast<long long>(grow) * p.N + gcol;
        const uint4 raw = *reinterpret_cast<const uint4*>(src);
        const OutT* e = reinterpret_cast<const OutT*>(&raw);
#pragma unroll
        for (int i = 0; i < n; ++i)
            v[i] = fmaf(p.beta, out_to_f32(e[i]), p.alpha * v[i]);
    } else {
#pragma unroll
        for (int i = 0; i < n; ++i)
            v[i] = p.alpha * v[i];
    }
}

template <typename OutT>
__device__ __forceinline__ void tc_strip_to_smem(uint32_t taddr, uint32_t staging, uint32_t row,
                                                 const TcParams& p, int grow, int gcol0)
{
    const uint32_t row_base = staging + row * 128;
    const uint32_t sw = row & 7;
    const bool scale = (p.alpha != 1.0f) || (p.beta != 0.0f);
    if constexpr (sizeof(OutT) == 4) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr, v);
        tmem_wait_ld();
        if (scale) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float f[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    f[i] = __uint_as_float(v[4 * c + i]);
                tc_axpby_chunk<OutT, 4>(f, p, grow, gcol0 + 4 * c);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    v[4 * c + i] = __float_as_uint(f[i]);
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
            st_shared_v4(row_base + ((c ^ sw) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                         v[4 * c + 3]);
    } else {
        uint32_t lo[32], hi[32];
        tmem_ld_32x32b_x32(taddr, lo);
        tmem_ld_32x32b_x32(taddr + 32, hi);
        tmem_wait_ld();
        OutT* tag = nullptr;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t* src = (c < 4) ? lo : hi;
            const int b = (c & 3) * 8;
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                f[i] = __uint_as_float(src[b + i]);
            if (scale)
                tc_axpby_chunk<OutT, 8>(f, p, grow, gcol0 + 8 * c);
            st_shared_v4(row_base + ((c ^ sw) << 4), pack2(f[0], f[1], tag), pack2(f[2], f[3], tag),
                         pack2(f[4], f[5], tag), pack2(f[6], f[7], tag));
        }
    }
}

template <int CG, int BN, int STAGES, typename OutT, bool A_MN, bool B_MN, bool SPLIT = false,
          int KSUB = 1>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
                   const TcParams p)
{
    using L = TcLayout<CG, BN, STAGES, KSUB>;
    constexpr int STRIP = TcOut<OutT>::STRIP;
    constexpr int TILE_M = TC_BM * CG;  // output rows per tile (per CTA pair)

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    // Full barrier of K step j of a stage: step 0 uses full_bar, later steps
    // their own, so the MMAs of a step can start before the stage's later
    // steps have landed.
    auto full_sub = [&](int s, int j) {
        return j == 0 ? full_bar(s) : bar0 + 8u * (2 * STAGES + 5 + s * (KSUB - 1) + (j - 1));
    };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0;
    const bool leader = (rank == 0);
    const int unit = (CG == 2) ? (blockIdx.x >> 1) : blockIdx.x;   // CTA or CTA pair index
    const int num_units = (CG == 2) ? (gridDim.x >> 1) : gridDim.x;
    const TcWatch watch{abort_flag, p.status, p.wait_budget};
    // A reduction launched after this kernel (split partials) may place its
    // blocks now; they wait for this grid to complete before reading.
    grid_dep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            for (int j = 0; j < KSUB; ++j)
                mbar_init(full_sub(s, j), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4 * CG);  // every epilogue warp of the pair
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t sA = sbase + L::OFF_A;
            const uint32_t sB = sbase + L::OFF_B;
            int stage = 0;
            uint32_t phase = 0;
            int issued[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                issued[s] = 0;
            bool ok = true;
            for (int t = unit; ok && t < p.num_work; t += num_units) {
                const TcWork w = tc_work(t, p);
                const int a_row = w.mb * TILE_M + static_cast<int>(rank) * TC_BM;
                const int b_col = w.nb * BN + static_cast<int>(rank) * L::B_COLS;
                for (int kb0 = w.kb_begin; kb0 < w.kb_end; kb0 += KSUB) {
                    const int nsub = min(KSUB, w.kb_end - kb0);
                    if (!tc_wait(empty_bar(stage), phase ^ 1, watch)) {
                        ok = false;
                        break;
                    }
                    // test hook (-1 in normal use): skip the stage holding that K step
                    if (p.fault_skip_kblock < kb0 || p.fault_skip_kblock >= kb0 + nsub) {
                        if (leader) {
#pragma unroll
                            for (int j = 0; j < KSUB; ++j) {
                                if (j < nsub)
                                    mbar_arrive_expect_tx(full_sub(stage, j), CG * L::SUB_BYTES);
                                else
                                    mbar_arrive(full_sub(stage, j));  // unused step: complete its phase
                            }
                        }
#pragma unroll
                        for (int sub = 0; sub < KSUB; ++sub) {
                        if (sub >= nsub)
                            break;
                        const int kb = kb0 + sub;
                        const uint32_t fb = (CG == 2) ? mapa_shared(full_sub(stage, sub), 0) : full_sub(stage, sub);
                        const uint32_t dA = sA + stage * L::A_STAGE + sub * L::SUB_A;
                        const uint32_t dB = sB + stage * L::B_STAGE + sub * L::SUB_B;
                        auto load = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
                            if constexpr (CG == 2)
                                tma_load_2d_pair(dst, map, fb, x, y);
                            else
                                tma_load_2d(dst, map, fb, x, y);
                        };
                        // A: K-major, one 128-row x 64-K box; or MN-major
                        // (A stored K x M), two 64-K x 64-M boxes.
                        if constexpr (A_MN) {
                            load(dA, &tmA, a_row, kb * TC_BK);
                            load(dA + 8192, &tmA, a_row + 64, kb * TC_BK);
                        } else {
                            load(dA, &tmA, kb * TC_BK, a_row);
                        }
                        // B: MN-major (B stored K x N), 64-K x 64-N boxes; or
                        // K-major (B stored N x K), one B_COLS-row x 64-K box.
                        if constexpr (B_MN) {
#pragma unroll
                            for (int j = 0; j < L::B_BOXES; ++j)
                                load(dB + j * 8192, &tmB, b_col + 64 * j, kb * TC_BK);
                        } else {
                            load(dB, &tmB, kb * TC_BK, b_col);
                        }
                        }
                        ++issued[stage];
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok && leader) {
                // Drain: wait (bounded) for the loads already issued into each
                // stage of this CTA's barriers before shared memory goes away.
                for (int s = 0; s < STAGES; ++s) {
                    if (issued[s] == 0)
                        continue;
                    const uint32_t par = static_cast<uint32_t>(issued[s] - 1) & 1u;
                    for (int j = 0; j < KSUB; ++j) {
                        const long long t0 = clock64();
                        while (!mbar_try_wait(full_sub(s, j), par) && clock64() - t0 < p.wait_budget) {
                        }
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (leader && lane == 0) {
            const uint32_t sA = sbase + L::OFF_A;
            const uint32_t sB = sbase + L::OFF_B;
            const uint32_t idesc = p.idesc;
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int t = unit; ok && t < p.num_work; t += num_units, ++local) {
                const TcWork w = tc_work(t, p);
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!tc_wait<CG == 2>(tempty_bar(acc), acc_phase ^ 1, watch)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb0 = w.kb_begin; kb0 < w.kb_end; kb0 += KSUB) {
                    const int nsub = min(KSUB, w.kb_end - kb0);
#pragma unroll
                    for (int sub = 0; sub < KSUB; ++sub) {
                    if (sub >= nsub)
                        break;
                    // this K step's operands have landed
                    if (!tc_wait(full_sub(stage, sub), phase, watch)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * L::A_STAGE + sub * L::SUB_A;
                    const uint32_t b0 = sB + stage * L::B_STAGE + sub * L::SUB_B;
#pragma unroll
                    for (int k = 0; k < TC_BK / TC_UMMA_K; ++k) {
                        // K-major operand: rows of 128 bytes, 8-row groups 1024
                        // bytes apart (SBO); a K step of 16 moves 32 bytes
                        // along the row.  MN-major operand: 64-element atoms
                        // 8 KiB apart (LBO), 8-row K groups 1024 bytes apart
                        // (SBO); a K step of 16 rows moves 2 KiB.
                        const uint64_t adesc = A_MN ? smem_desc_sw128(a0 + k * 2048, 8192, 1024)
                                                    : smem_desc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bdesc = B_MN ? smem_desc_sw128(b0 + k * 2048, 8192, 1024)
                                                    : smem_desc_sw128(b0 + k * 32, 16, 1024);
                        tc_mma_f16<CG>(d_tmem, adesc, bdesc, idesc,
                                       (kb0 != w.kb_begin) || sub != 0 || k != 0);
                    }
                    }
                    if (!ok)
                        break;
                    if constexpr (CG == 2)
                        tc_commit_pair(empty_bar(stage), 0x3);
                    else
                        tc_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                if constexpr (CG == 2)
                    tc_commit_pair(tfull_bar(acc), 0x3);
                else
                    tc_commit(tfull_bar(acc));
            }
            // Wait (bounded) until every MMA issued so far has completed, so
            // TMEM and the input stages are no longer in use.
            tc_commit_self<CG>(drain_bar);
            const long long t0 = clock64();
            while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < p.wait_budget) {
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t staging0 =
            sbase + L::OFF_STAGING + static_cast<uint32_t>((warp - TC_EPI_WARP0) * 2 * TC_STAGING_BYTES);
        const uint32_t leader_tempty0 = (CG == 2) ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
        const uint32_t leader_tempty1 = (CG == 2) ? mapa_shared(tempty_bar(1), 0) : tempty_bar(1);
        int local = 0;
        uint32_t buf = 0;
        TcParams p_raw = p;  // partial tiles are stored unscaled
        p_raw.alpha = 1.0f;
        p_raw.beta = 0.0f;
        for (int t = unit; t < p.num_work; t += num_units, ++local) {
            const TcWork w = tc_work(t, p);
            const int mb = w.mb, nb = w.nb;
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            int ok = 1;
            if (lane == 0)
                ok = tc_wait(tfull_bar(acc), acc_phase, watch) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            tc_fence_after();
            const int row0 = mb * TILE_M + static_cast<int>(rank) * TC_BM + q * 32;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            if (!SPLIT && w.partial) {
                // Tail piece: the whole TILE_M x BN FP32 partial goes to
                // workspace slot w.slot (tile-local rows and columns; the
                // reduction clips to C).
                const int trow = static_cast<int>(rank) * TC_BM + q * 32;
#pragma unroll 1
                for (int s = 0; s < BN / 32; ++s) {
                    const uint32_t stg = staging0 + buf * TC_STAGING_BYTES;
                    if (lane == 0)
                        bulk_wait_group_read<1>();
                    __syncwarp();
                    tc_strip_to_smem<float>(t_row + s * 32, stg, lane, p_raw, 0, 0);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tmW, stg, s * 32, trow, w.slot);
                        bulk_commit_group();
                    }
                    buf ^= 1;
                }
            }
            // Gap after each store, in clock cycles: the spread share of the
            // next item's tensor time (2 * BN cycles per 64-wide K step: four
            // MMAs of M = 128 rows per CTA and N = BN), per strip of this
            // warp.  None after a CTA's last item.
            long long gap = 0;
            if (!SPLIT && !w.partial && t + num_units < p.num_work) {
                const TcWork nx = tc_work(t + num_units, p);
                gap = static_cast<long long>(nx.kb_end - nx.kb_begin) * 2 * BN *
                      TMMO_STORE_SPREAD_PCT / 100 / (BN / STRIP);
            }
#pragma unroll 1
            for (int s = 0; s < BN / STRIP && (SPLIT || !w.partial); ++s) {
                const int col0 = nb * BN + s * STRIP;
                if (row0 >= p.M || col0 >= p.N)
                    break;  // the rest of this warp's strips lie wholly outside C
                const uint32_t stg = staging0 + buf * TC_STAGING_BYTES;
                // This buffer is free once at most one store group (the one
                // reading the other buffer) is still pending.
                if (lane == 0)
                    bulk_wait_group_read<1>();
                __syncwarp();
                tc_strip_to_smem<OutT>(t_row + s * STRIP, stg, lane, p,
                                       row0 + static_cast<int>(lane), col0);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (SPLIT)  // FP32 partial of split w.split (workspace)
                        tma_store_3d(&tmC, stg, col0, row0, w.split);
                    else
                        tma_store_2d(&tmC, stg, col0, row0);
                    bulk_commit_group();
                    const long long t0 = clock64();
                    while (clock64() - t0 < gap) {
                    }
                }
                buf ^= 1;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t tb = acc ? leader_tempty1 : leader_tempty0;
                if constexpr (CG == 2)
                    mbar_arrive_cluster(tb);
                else
                    mbar_arrive(tb);
            }
        }
        // Shared memory may be released once the stores have read it; the
        // grid's completion covers their writes to global memory (a
        // reduction launched as a programmatic dependent waits for it).
        if (lane == 0)
            bulk_wait_group_read<0>();
        __syncwarp();
    }

    // ---------------------------------------------------- teardown
    __syncwarp();  // reconverge each warp after its role's divergent loop
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc<CG>(tmem_base, L::TMEM_COLS);
    }
}

}  // namespace tmmo
