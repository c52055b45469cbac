// Host side of the tensor-core GEMM: tensor-map encoding, grid sizing and
// launch of the tc_gemm_kernel instantiations.
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
#ifndef TMMO_PAIR_STAGES
#define TMMO_PAIR_STAGES 6   // shared-memory stages of the CTA-pair kernel
#endif

namespace tmmo {
namespace {

constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();  // leave no sticky error behind
    });
    return fn;
}

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
    auto fn = encode_fn();
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

template <int CG, int BN, int STAGES, typename OutT>
cudaError_t launch_variant(const TcLaunch& l, cudaStream_t stream)
{
    using L = TcLayout<CG, BN, STAGES>;
    constexpr int STRIP = TcOut<OutT>::STRIP;
    auto kern = tc_gemm_kernel<CG, BN, STAGES, OutT>;

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

    CUtensorMap ta, tb, tc;
    const int b_cols = BN / CG;
    if (!encode_2d(&ta, l.in_dtype, l.A, l.M, l.K, TC_BM, TC_BK) ||
        !encode_2d(&tb, l.in_dtype, l.B, l.K, l.N, TC_BK, 64) ||
        !encode_2d(&tc, l.out_dtype, l.C, l.M, l.N, 32, STRIP))
        return cudaErrorNotSupported;
    (void)b_cols;

    TcParams p{};
    p.M = l.M;
    p.N = l.N;
    p.K = l.K;
    p.tiles_m = (l.M + TC_BM * CG - 1) / (TC_BM * CG);
    p.tiles_n = (l.N + BN - 1) / BN;
    p.num_tiles = p.tiles_m * p.tiles_n;
    p.k_blocks = (l.K + TC_BK - 1) / TC_BK;
    p.group_m = TMMO_RASTER_GROUP;
    p.idesc = tc_idesc(l.in_dtype == DT_BF16, TC_BM * CG, BN);
    p.status = l.status;
    p.wait_budget = l.wait_budget;
    p.fault_skip_kblock = l.fault_skip_kblock;

    const int units = std::max(1, std::min(p.num_tiles, units_cap));
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
    err = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

template <int CG, int BN, int STAGES>
cudaError_t launch_out(const TcLaunch& l, cudaStream_t s)
{
    switch (l.out_dtype) {
    case DT_F32:
        return launch_variant<CG, BN, STAGES, float>(l, s);
    case DT_F16:
        return launch_variant<CG, BN, STAGES, __half>(l, s);
    default:
        return launch_variant<CG, BN, STAGES, __nv_bfloat16>(l, s);
    }
}

}  // namespace

void tc_tile_shape(int variant, int* tile_m, int* tile_n)
{
    switch (variant) {
    case TC_128x128:
        *tile_m = 128;
        *tile_n = 128;
        break;
    case TC_128x256:
        *tile_m = 128;
        *tile_n = 256;
        break;
    default:
        *tile_m = 256;
        *tile_n = 256;
        break;
    }
}

cudaError_t tc_gemm_launch(const TcLaunch& l, cudaStream_t stream)
{
    switch (l.variant) {
    case TC_128x128:
        return launch_out<1, 128, 6>(l, stream);
    case TC_128x256:
        return launch_out<1, 256, 4>(l, stream);
    case TC_256x256:
        return launch_out<2, 256, TMMO_PAIR_STAGES>(l, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace tmmo
