// A lean tensor-core kernel for products whose output tiles all fit in one
// wave of single CTAs: one CTA per 128 x BN output tile, not persistent, no
// cluster, no accumulator double-buffering, and an epilogue that stores
// straight from registers.
//
// The loop nest is the one of "Reading a matrix multiply through its tiles"
// ("Keep one output tile resident"): the FP32 accumulator of the tile lives
// in tensor memory for the whole K loop, A and B tiles stream through a
// STAGES-deep TMA ring, and C is written once at the end.  What the
// persistent kernel spends on its schedule -- the raster decode, the second
// accumulator, the epilogue's shared-memory staging and TMA stores, the
// cluster launch -- buys nothing when there is a single tile per CTA, and on
// these small products the whole launch is latency: so this kernel starts
// its first copies right after initialising its barriers, before the
// accumulator is allocated, and each thread writes its own output row
// (16-byte stores) as soon as it has read it from tensor memory.
//
// Roles (4 warps): thread 0 issues the TMA copies; warp 1 allocates the
// accumulator and its lane 0 issues tcgen05.mma (K = 16 per instruction,
// four per 64-wide K step); then all four warps read 32 accumulator rows
// each (tcgen05.ld), apply alpha and beta, round to the output type and
// store.  TMA zero fill covers the edges of A and B; the stores are guarded
// per 16-byte chunk (N * sizeof(out) is a multiple of 16, so a chunk is
// wholly inside or outside C).  Every wait is bounded, as in tc_gemm_kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "tc_launch.cuh"

namespace tmmo {
namespace {

struct SmallParams {
    int M, N, K;
    int tiles_n;
    int k_blocks;
    uint32_t idesc;
    void* C;
    float alpha, beta;
    int* status;
    long long wait_budget;
    int fault_skip_kblock;
};

template <int BN, int STAGES>
struct SmallLayout {
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KiB: 128 rows x 64 K
    static constexpr int B_BYTES = TC_BK * BN * 2;     // BN / 64 boxes of 64 K x 64 N
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int OFF_BAR = STAGES * STAGE;
    static constexpr int NUM_BARS = 2 * STAGES + 2;    // full, empty, MMA done, drain
    static constexpr int OFF_MISC = OFF_BAR + 8 * NUM_BARS;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = BYTES + 1024;    // slack for 1024-byte alignment
    static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
    static_assert(BN == 64 || BN == 128, "tile widths of 64 or 128 columns");
};

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

template <int BN, int STAGES, typename OutT, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(128, 1)
    tc_small_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const SmallParams p)
{
    using L = SmallLayout<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES);
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const int m0 = (blockIdx.x / p.tiles_n) * TC_BM;
    const int n0 = (blockIdx.x % p.tiles_n) * BN;
    const TcWatch watch{abort_flag, p.status, p.wait_budget};

    // K step kb goes to stage kb % STAGES; the producer thread issues the
    // first STAGES steps before the block-wide barrier, so the copies are in
    // flight while the accumulator is being allocated.
    int last_kb[STAGES];   // per stage, the last K step whose copies were issued (thread 0)
#pragma unroll
    for (int s = 0; s < STAGES; ++s)
        last_kb[s] = -1;
    auto issue = [&](int kb) {
        const int s = kb % STAGES;
        const uint32_t dA = sbase + s * L::STAGE;
        const uint32_t dB = dA + L::A_BYTES;
        if (p.fault_skip_kblock == kb)
            return;        // test hook: this step's copies never arrive
        mbar_arrive_expect_tx(full_bar(s), L::STAGE);
        // A as stored: one 128-row x 64-K box (K-major); A stored K x M: two
        // 64-K x 64-M boxes (MN-major).  B as stored: 64-K x 64-N boxes
        // (MN-major); B stored N x K: one BN-row x 64-K box (K-major).
        if constexpr (A_MN) {
            tma_load_2d(dA, &tmA, full_bar(s), m0, kb * TC_BK);
            tma_load_2d(dA + 8192, &tmA, full_bar(s), m0 + 64, kb * TC_BK);
        } else {
            tma_load_2d(dA, &tmA, full_bar(s), kb * TC_BK, m0);
        }
        if constexpr (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(dB + j * 8192, &tmB, full_bar(s), n0 + 64 * j, kb * TC_BK);
        } else {
            tma_load_2d(dB, &tmB, full_bar(s), kb * TC_BK, n0);
        }
        last_kb[s] = kb;
    };
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        for (int kb = 0; kb < STAGES && kb < p.k_blocks; ++kb)
            issue(kb);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (threadIdx.x == 0) {
        // ---------------------------------------------- TMA producer
        bool ok = true;
        for (int kb = STAGES; ok && kb < p.k_blocks; ++kb) {
            const int s = kb % STAGES;
            // the MMAs of step kb - STAGES have read this stage
            if (!tc_wait(empty_bar(s), static_cast<uint32_t>((kb / STAGES - 1) & 1), watch)) {
                ok = false;
                break;
            }
            issue(kb);
        }
        if (!ok) {
            // Drain (bounded): wait for the copies already issued into each
            // stage before shared memory goes away.
            for (int s = 0; s < STAGES; ++s) {
                if (last_kb[s] < 0)
                    continue;
                const uint32_t par = static_cast<uint32_t>((last_kb[s] / STAGES) & 1);
                const long long t0 = clock64();
                while (!mbar_try_wait(full_bar(s), par) && clock64() - t0 < p.wait_budget) {
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------- MMA issuer
        const uint32_t idesc = p.idesc;
        bool ok = true;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
            const int s = kb % STAGES;
            if (!tc_wait(full_bar(s), static_cast<uint32_t>((kb / STAGES) & 1), watch)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = sbase + s * L::STAGE;
            const uint32_t b0 = a0 + L::A_BYTES;
#pragma unroll
            for (int k = 0; k < TC_BK / TC_UMMA_K; ++k) {
                // K-major: 128-byte rows, 8-row groups 1024 bytes apart, 32
                // bytes per 16-wide K slice; MN-major: 64-element atoms 8 KiB
                // apart, 8-row K groups 1024 bytes apart, 2 KiB per K slice.
                const uint64_t adesc = A_MN ? smem_desc_sw128(a0 + k * 2048, 8192, 1024)
                                            : smem_desc_sw128(a0 + k * 32, 16, 1024);
                const uint64_t bdesc = B_MN ? smem_desc_sw128(b0 + k * 2048, 8192, 1024)
                                            : smem_desc_sw128(b0 + k * 32, 16, 1024);
                tc_mma_f16<1>(tmem_base, adesc, bdesc, idesc, kb != 0 || k != 0);
            }
            tc_commit(empty_bar(s));
        }
        if (ok)
            tc_commit(done_bar);
        // every MMA issued has completed before TMEM is released (bounded)
        tc_commit(drain_bar);
        const long long t0 = clock64();
        while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < p.wait_budget) {
        }
    }
    __syncwarp();

    // -------------------------------------------------- epilogue: all warps
    int ok = 1;
    if (lane == 0)
        ok = tc_wait(done_bar, 0, watch) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
        tc_fence_after();
        const int row = m0 + warp * 32 + static_cast<int>(lane);
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
        OutT* crow = static_cast<OutT*>(p.C) + static_cast<long long>(row) * p.N;
        const bool scale = (p.alpha != 1.0f) || (p.beta != 0.0f);
        // the whole row of the tile in one round trip: every strip's load
        // issued before a single wait
        uint32_t v[BN];
#pragma unroll
        for (int s = 0; s < BN / 32; ++s)
            tmem_ld_32x32b_x32(t_row + s * 32, *reinterpret_cast<uint32_t(*)[32]>(&v[s * 32]));
        tmem_wait_ld();
        constexpr int PER = 16 / sizeof(OutT);  // values per 16-byte chunk
        if (scale) {
            // v <- alpha * v + beta * C_in, C read only where beta != 0 and
            // the chunk lies inside C
#pragma unroll
            for (int c = 0; c < BN / PER; ++c) {
                const int col = n0 + c * PER;
                const bool in = row < p.M && col < p.N && p.beta != 0.0f;
                OutT e[PER];
                if (in)
                    *reinterpret_cast<uint4*>(e) = *reinterpret_cast<const uint4*>(crow + col);
#pragma unroll
                for (int i = 0; i < PER; ++i) {
                    float f = p.alpha * __uint_as_float(v[c * PER + i]);
                    if (in)
                        f = fmaf(p.beta, out_to_f32(e[i]), f);
                    v[c * PER + i] = __float_as_uint(f);
                }
            }
        }
        if (row < p.M) {
#pragma unroll
            for (int c = 0; c < BN / PER; ++c) {
                const int col = n0 + c * PER;
                if (col >= p.N)
                    break;
                if constexpr (sizeof(OutT) == 4) {
                    st_global_v4(crow + col, v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                } else {
                    OutT* tag = nullptr;
                    const uint32_t* w = &v[8 * c];
                    st_global_v4(crow + col,
                                 pack2(__uint_as_float(w[0]), __uint_as_float(w[1]), tag),
                                 pack2(__uint_as_float(w[2]), __uint_as_float(w[3]), tag),
                                 pack2(__uint_as_float(w[4]), __uint_as_float(w[5]), tag),
                                 pack2(__uint_as_float(w[6]), __uint_as_float(w[7]), tag));
                }
            }
        }
    }

    // ---------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc<1>(tmem_base, L::TMEM_COLS);
    }
}

// Stages of the copy ring: as many as 192 KiB hold (8 of 24 KiB for 64-column
// tiles, 6 of 32 KiB for 128-column ones).  A single CTA streams its K
// steps from DRAM with a full ring's worth of copies in flight, so its rate
// is about that many bytes per memory latency.
#ifndef TMMO_SMALL_RING_BYTES
#define TMMO_SMALL_RING_BYTES (192 * 1024)
#endif
template <int BN, typename OutT, bool A_MN, bool B_MN>
cudaError_t launch_small(const TcLaunch& l, cudaStream_t stream)
{
    constexpr int STAGES = TMMO_SMALL_RING_BYTES / SmallLayout<BN, 1>::STAGE;
    using L = SmallLayout<BN, STAGES>;
    auto kern = tc_small_kernel<BN, STAGES, OutT, A_MN, B_MN>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static bool ready[kMaxDevices] = {};
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 0 || dev >= kMaxDevices)
            return cudaErrorInvalidDevice;
        if (!ready[dev]) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::SMEM_ALLOC);
            if (err != cudaSuccess)
                return err;
            ready[dev] = true;
        }
    }
    // A as stored: M x K, boxes of 128 rows x 64 K; transposed: K x M, boxes
    // of 64 K x 64 M.  B as stored: K x N, boxes of 64 K x 64 N; transposed:
    // N x K, boxes of BN rows x 64 K.
    CUtensorMap ta, tb;
    const bool ok_a = A_MN ? encode_2d(&ta, l.in_dtype, l.A, l.K, l.M, TC_BK, 64)
                           : encode_2d(&ta, l.in_dtype, l.A, l.M, l.K, TC_BM, TC_BK);
    const bool ok_b = B_MN ? encode_2d(&tb, l.in_dtype, l.B, l.K, l.N, TC_BK, 64)
                           : encode_2d(&tb, l.in_dtype, l.B, l.N, l.K, BN, TC_BK);
    if (!ok_a || !ok_b)
        return cudaErrorNotSupported;
    SmallParams p{};
    p.M = l.M;
    p.N = l.N;
    p.K = l.K;
    p.tiles_n = (l.N + BN - 1) / BN;
    p.k_blocks = (l.K + TC_BK - 1) / TC_BK;
    p.idesc = tc_idesc(l.in_dtype == DT_BF16, TC_BM, BN, A_MN, B_MN);
    p.C = l.C;
    p.alpha = l.alpha;
    p.beta = l.beta;
    p.status = l.status;
    p.wait_budget = l.wait_budget;
    p.fault_skip_kblock = l.fault_skip_kblock;
    const long long tiles = static_cast<long long>((l.M + TC_BM - 1) / TC_BM) * p.tiles_n;
    if (tiles > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    note_launch();
    kern<<<static_cast<unsigned>(tiles), 128, L::SMEM_ALLOC, stream>>>(ta, tb, p);
    return cudaGetLastError();
}

template <int BN, bool A_MN, bool B_MN>
cudaError_t small_out(const TcLaunch& l, cudaStream_t s)
{
    switch (l.out_dtype) {
    case DT_F32:
        return launch_small<BN, float, A_MN, B_MN>(l, s);
    case DT_F16:
        return launch_small<BN, __half, A_MN, B_MN>(l, s);
    default:
        return launch_small<BN, __nv_bfloat16, A_MN, B_MN>(l, s);
    }
}

template <bool A_MN, bool B_MN>
cudaError_t small_layout(const TcLaunch& l, cudaStream_t s)
{
    if (tc_small_tile_n(l.M, l.N, l.num_sms) == 64)
        return small_out<64, A_MN, B_MN>(l, s);
    return small_out<128, A_MN, B_MN>(l, s);
}

}  // namespace

int tc_small_tile_n(int64_t M, int64_t N, int num_sms)
{
    // 64-column tiles while twice as many CTAs still fit in one wave: a
    // 128 x 64 K step takes half the tensor time of a 128 x 128 one.
    const int64_t tiles128 = ((M + TC_BM - 1) / TC_BM) * ((N + 127) / 128);
    return (2 * tiles128 <= num_sms) ? 64 : 128;
}

cudaError_t tc_small_launch(const TcLaunch& l, cudaStream_t stream)
{
    // operand layouts as in tc_gemm_launch: MN-major A when A is transposed,
    // MN-major B when B is as stored
    if (!l.op_a && !l.op_b)
        return small_layout<false, true>(l, stream);
    if (l.op_a && !l.op_b)
        return small_layout<true, true>(l, stream);
    if (!l.op_a && l.op_b)
        return small_layout<false, false>(l, stream);
    return small_layout<true, false>(l, stream);
}

}  // namespace tmmo
