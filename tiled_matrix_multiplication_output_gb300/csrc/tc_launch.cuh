// Host-side launch of tc_gemm_kernel: tensor-map encoding, grid sizing, and
// the per-layout dispatch over tile variants and output types.  Included by
// one translation unit per operand layout (tc_gemm_nn.cu ... tc_gemm_tt.cu)
// so the instantiations compile in parallel.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "launch.h"
#include "tc_gemm.cuh"

// Schedule and pipeline-depth choices, measured on GB300 (overridable at
// build time for tuning sweeps).
#ifndef TMMO_RASTER_GROUP
#define TMMO_RASTER_GROUP 8  // tile rows per raster group
#endif
// Each stage holds KSUB 64-wide K steps: one barrier wait and one commit
// per KSUB * 4 MMAs.  On GB300 the pair kernel runs 4-5 % faster with two K
// steps in each of 3 stages than with one in each of 6 (the same 192 KiB in
// flight): the single MMA-issuing thread is then no longer the limit.
#ifndef TMMO_PAIR_STAGES
#define TMMO_PAIR_STAGES 3   // shared-memory stages of the CTA-pair kernel
#endif
#ifndef TMMO_PAIR_KSUB
#define TMMO_PAIR_KSUB 2     // 64-wide K steps per stage of the CTA-pair kernel
#endif
#ifndef TMMO_PAIR128_STAGES
#define TMMO_PAIR128_STAGES 4  // stages of the 256 x 128 CTA-pair kernel
#endif
#ifndef TMMO_PAIR128_KSUB
#define TMMO_PAIR128_KSUB 2
#endif
#ifndef TMMO_WIDE_STAGES
#define TMMO_WIDE_STAGES 4   // stages of the 128 x 256 kernel
#endif
#ifndef TMMO_WIDE_KSUB
#define TMMO_WIDE_KSUB 1
#endif
#ifndef TMMO_SQ_STAGES
#define TMMO_SQ_STAGES 3     // stages of the 128 x 128 kernel (12 % faster than 6 x 1)
#endif
#ifndef TMMO_SQ_KSUB
#define TMMO_SQ_KSUB 2
#endif

namespace tmmo {
namespace {

constexpr int kMaxDevices = 64;

CUtensorMapDataType map_type(int dt)
{
    switch (dt) {
    case DT_F32:
        return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    case DT_F16:
        return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    default:
        return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    }
}

int dt_bytes(int dt) { return dt == DT_F32 ? 4 : 2; }

// Row-major rows x cols matrix, boxes of box_rows x box_cols, 128-byte swizzle.
bool encode_2d(CUtensorMap* map, int dt, const void* base, uint64_t rows, uint64_t cols,
               uint32_t box_rows, uint32_t box_cols)
{
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<uint64_t>(dt_bytes(dt))};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, map_type(dt), 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// FP32 split-K workspace [splits][rows][cols] as a 3-D tensor map with boxes
// of 32 rows x 32 columns x 1 split, 128-byte swizzle.
bool encode_workspace(CUtensorMap* map, float* base, uint64_t splits, uint64_t rows,
                      uint64_t cols)
{
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (!fn)
        return false;
    const cuuint64_t dims[3] = {cols, rows, splits};
    const cuuint64_t strides[2] = {cols * 4, rows * cols * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int CG, int BN, int STAGES, typename OutT, bool A_MN, bool B_MN, bool SPLIT = false,
          int KSUB = 1>
cudaError_t launch_variant(const TcLaunch& l, cudaStream_t stream)
{
    using L = TcLayout<CG, BN, STAGES, KSUB>;
    constexpr int STRIP = TcOut<OutT>::STRIP;
    static_assert(!SPLIT || sizeof(OutT) == 4, "split-K partials are FP32");
    auto kern = tc_gemm_kernel<CG, BN, STAGES, OutT, A_MN, B_MN, SPLIT, KSUB>;

    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    // Per-device, per-instantiation one-time set-up: the shared-memory opt-in
    // and, for CTA pairs, how many clusters can be resident at once.
    static int max_units[kMaxDevices] = {};
    static std::mutex mu;
    int units_cap = 0;
    {
        std::lock_guard<std::mutex> g(mu);
        if (dev < 0 || dev >= kMaxDevices)
            return cudaErrorInvalidDevice;
        if (max_units[dev] == 0) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::SMEM_ALLOC);
            if (err != cudaSuccess)
                return err;
            int cap = l.num_sms;
            if (CG == 2) {
                cudaLaunchConfig_t cfg{};
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 2;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.gridDim = dim3(2 * std::max(1, l.num_sms / 2), 1, 1);
                cfg.blockDim = dim3(TC_THREADS, 1, 1);
                cfg.dynamicSmemBytes = L::SMEM_ALLOC;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int clusters = 0;
                err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
                if (err != cudaSuccess)
                    return err;
                cap = std::max(1, clusters);
            }
            max_units[dev] = cap;
        }
        units_cap = max_units[dev];
    }

    // A as stored: M x K (K-major boxes of 128 rows x 64 K) or, transposed,
    // K x M (MN-major boxes of 64 K x 64 M).  B as stored: K x N (MN-major
    // boxes of 64 K x 64 N) or, transposed, N x K (K-major boxes of
    // BN / CG rows x 64 K).  C: boxes of 32 rows x one 128-byte row.
    CUtensorMap ta, tb, tc;
    const bool ok_a = A_MN ? encode_2d(&ta, l.in_dtype, l.A, l.K, l.M, TC_BK, 64)
                           : encode_2d(&ta, l.in_dtype, l.A, l.M, l.K, TC_BM, TC_BK);
    const bool ok_b = B_MN ? encode_2d(&tb, l.in_dtype, l.B, l.K, l.N, TC_BK, 64)
                           : encode_2d(&tb, l.in_dtype, l.B, l.N, l.K, BN / CG, TC_BK);
    const int k_blocks = (l.K + TC_BK - 1) / TC_BK;
    const int tiles_m = (l.M + TC_BM * CG - 1) / (TC_BM * CG);
    const int tiles_n = (l.N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    // Work plan: split-K splits every tile; the hybrid plan runs whole waves
    // of tiles and splits only the tiles of the last, partial wave (when that
    // helps and the workspace can hold their partials); otherwise all tiles
    // are whole.
    int dp_tiles = num_tiles, splits = 1, kb_per_split = k_blocks;
    if (SPLIT) {
        dp_tiles = 0;
        splits = std::max(1, std::min(l.k_splits, k_blocks));
        kb_per_split = (k_blocks + splits - 1) / splits;
        splits = (k_blocks + kb_per_split - 1) / kb_per_split;  // none empty
    } else if (l.hybrid) {
        hybrid_plan(num_tiles, std::min(num_tiles, units_cap), k_blocks, &dp_tiles, &splits,
                    &kb_per_split);
        const size_t need = static_cast<size_t>(num_tiles - dp_tiles) * splits * TC_BM * CG * BN * 4;
        if (dp_tiles < num_tiles && (!l.workspace || l.workspace_bytes < need)) {
            dp_tiles = num_tiles;
            splits = 1;
            kb_per_split = k_blocks;
        }
    }
    const int slots = (num_tiles - dp_tiles) * splits;
    const bool ok_c = SPLIT ? encode_workspace(&tc, l.workspace, splits, l.M, l.N)
                            : encode_2d(&tc, l.out_dtype, l.C, l.M, l.N, 32, STRIP);
    CUtensorMap tw = tc;  // tail workspace: slots of TILE_M x BN FP32 partials
    if (!SPLIT && slots > 0 && !encode_workspace(&tw, l.workspace, slots, TC_BM * CG, BN))
        return cudaErrorNotSupported;
    if (!ok_a || !ok_b || !ok_c)
        return cudaErrorNotSupported;
    if (l.plan) {
        l.plan[0] = dp_tiles;
        l.plan[1] = splits;
        l.plan[2] = num_tiles - dp_tiles;
        l.plan[3] = tiles_m;
        l.plan[4] = tiles_n;
        l.plan[5] = TMMO_RASTER_GROUP;
        l.plan[6] = TC_BM * CG;
        l.plan[7] = BN;
    }

    TcParams p{};
    p.M = l.M;
    p.N = l.N;
    p.K = l.K;
    p.tiles_m = tiles_m;
    p.tiles_n = tiles_n;
    p.num_tiles = num_tiles;
    p.k_blocks = k_blocks;
    p.dp_tiles = dp_tiles;
    p.k_splits = splits;
    p.kb_per_split = kb_per_split;
    p.num_work = dp_tiles + slots;
    p.group_m = TMMO_RASTER_GROUP;
    p.idesc = tc_idesc(l.in_dtype == DT_BF16, TC_BM * CG, BN, A_MN, B_MN);
    p.status = l.status;
    p.wait_budget = l.wait_budget;
    p.fault_skip_kblock = l.fault_skip_kblock;
    p.C = l.C;
    p.alpha = l.alpha;
    p.beta = l.beta;

    const int units = std::max(1, std::min(p.num_work, units_cap));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(units * CG, 1, 1);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_ALLOC;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    err = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tw, p);
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

template <int CG, int BN, int STAGES, bool A_MN, bool B_MN, int KSUB = 1>
cudaError_t launch_out(const TcLaunch& l, cudaStream_t s)
{
    switch (l.out_dtype) {
    case DT_F32:
        return launch_variant<CG, BN, STAGES, float, A_MN, B_MN, false, KSUB>(l, s);
    case DT_F16:
        return launch_variant<CG, BN, STAGES, __half, A_MN, B_MN, false, KSUB>(l, s);
    default:
        return launch_variant<CG, BN, STAGES, __nv_bfloat16, A_MN, B_MN, false, KSUB>(l, s);
    }
}

// Every tensor-core variant for one operand layout.
template <bool A_MN, bool B_MN>
cudaError_t launch_layout(const TcLaunch& l, cudaStream_t stream)
{
    switch (l.variant) {
    case TC_128x128:
        return launch_out<1, 128, TMMO_SQ_STAGES, A_MN, B_MN, TMMO_SQ_KSUB>(l, stream);
    case TC_128x256:
        return launch_out<1, 256, TMMO_WIDE_STAGES, A_MN, B_MN, TMMO_WIDE_KSUB>(l, stream);
    case TC_256x128:
        return launch_out<2, 128, TMMO_PAIR128_STAGES, A_MN, B_MN, TMMO_PAIR128_KSUB>(l, stream);
    case TC_256x256:
        return launch_out<2, 256, TMMO_PAIR_STAGES, A_MN, B_MN, TMMO_PAIR_KSUB>(l, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace tmmo
