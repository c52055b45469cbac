// Internal launchers behind the C ABI (host side).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace tmmo {

// Counts one launch of a library kernel (process-wide, all devices); read
// through gemm_launch_count().
void note_launch();

// Internal dtype codes; they match gemm_dtype_t.
enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

// Tensor-core kernel variants; they match the gemm_kernel_t values.
enum { TC_128x128 = 3, TC_128x256 = 4, TC_256x256 = 5, TC_256x128 = 6, TC_SMALL = 7 };

// Whether a variant runs on CTA pairs (cta_group::2).
inline bool tc_is_pair(int variant) { return variant == TC_256x256 || variant == TC_256x128; }

struct SimtLaunch {
    bool tpb3;          // the 3 x 3 one-thread-per-output instance
    int in_dtype, out_dtype;
    int op_a, op_b;     // 0: as stored; 1: transposed
    float alpha, beta;
    const void* A;
    const void* B;
    void* C;
    int M, N, K;
    int num_sms;
};

cudaError_t simt_gemm_launch(const SimtLaunch& l, cudaStream_t stream);

// The latency-path kernel (tile16.cu): one 16 x 16 output tile per block,
// the tile's whole K range copied at once and split between the block's
// warps (warp-level MMA for 16-bit inputs, FFMA for FP32).  tile16_fits says whether it takes the operands
// (16-byte aligned A and B and row pitches, the K slices of a tile within
// a block's shared memory); tile16_launch returns cudaErrorNotSupported
// when it does not.
bool tile16_fits(const SimtLaunch& l);
cudaError_t tile16_launch(const SimtLaunch& l, cudaStream_t stream);

struct TcLaunch {
    int variant;        // TC_128x128, TC_128x256 or TC_256x256
    int op_a, op_b;     // 0: as stored; 1: transposed (A stored K x M, B stored N x K)
    float alpha, beta;  // C = alpha * op(A) op(B) + beta * C
    int in_dtype;       // DT_F16 or DT_BF16
    int out_dtype;      // DT_F32, DT_F16 or DT_BF16
    const void* A;
    const void* B;
    void* C;
    int M, N, K;
    int num_sms;
    int* status;        // device status word
    long long wait_budget;
    int fault_skip_kblock;
    int k_splits;       // split-K only: requested K ranges per tile
    float* workspace;   // split-K: [k_splits][M][N] FP32 partials; hybrid: tail partials
    size_t workspace_bytes;  // hybrid only: capacity of workspace
    bool hybrid;        // split the tiles of the last, partial wave along K
    int* plan;          // if set, receives the work plan (see tc_launch.cuh)
};

// Hybrid plan for `tiles` output tiles on `units` resident CTAs (or pairs)
// with `k_blocks` K steps: whole waves of tiles stay whole; the r tiles of
// the last, partial wave are each split into `splits` K ranges so that the
// r * splits pieces occupy the idle units.  Splitting is used only when it
// gives at least TMMO_MIN_TAIL_SPLITS (2) ranges of at least four K steps;
// measured on GB300 with interleaved runs (BF16, the reduction launched as a
// programmatic dependent), the split takes 4.1 % off 4096^3, 2.2 % off
// 8192^3 and 6.9 % off 2560^3 (three pieces per tile there).
inline void hybrid_plan(int tiles, int units, int k_blocks, int* dp_tiles, int* splits,
                        int* kb_per_split)
{
    *dp_tiles = tiles;
    *splits = 1;
    *kb_per_split = k_blocks;
    if (units <= 0 || tiles <= units)
        return;
    const int r = tiles % units;
    if (r == 0)
        return;
    int s = units / r;
    if (s > k_blocks / 4)
        s = k_blocks / 4;
#ifndef TMMO_MIN_TAIL_SPLITS
#define TMMO_MIN_TAIL_SPLITS 2
#endif
    if (s < TMMO_MIN_TAIL_SPLITS)
        return;
    const int per = (k_blocks + s - 1) / s;
    *dp_tiles = tiles - r;
    *splits = (k_blocks + per - 1) / per;
    *kb_per_split = per;
}

// Hybrid product on the CTA-pair kernel (operands as stored): launches the
// tensor-core kernel with the hybrid plan, then, if tiles were split, the
// reduction of their partials into C.
cudaError_t tc_hybrid_launch(const TcLaunch& l, cudaStream_t stream);

// Sums the split partials of the tail tiles described by plan[] (as filled
// by the tensor-core launch) into C, applying alpha and beta.
cudaError_t tail_reduce_launch(const TcLaunch& l, const int* plan, cudaStream_t stream);

// The single-tile kernel for products whose 128-row tiles fit in one wave
// of CTAs (tc_small.cu): one CTA per 128 x tc_small_tile_n() output tile.
cudaError_t tc_small_launch(const TcLaunch& l, cudaStream_t stream);
int tc_small_tile_n(int64_t M, int64_t N, int num_sms);

// Encodes the tensor maps and launches; returns cudaSuccess, a CUDA error, or
// cudaErrorNotSupported when the driver entry point for tensor maps is
// unavailable.
cudaError_t tc_gemm_launch(const TcLaunch& l, cudaStream_t stream);
cudaError_t tc_launch_nn(const TcLaunch& l, cudaStream_t stream);
cudaError_t tc_launch_tn(const TcLaunch& l, cudaStream_t stream);
cudaError_t tc_launch_nt(const TcLaunch& l, cudaStream_t stream);
cudaError_t tc_launch_tt(const TcLaunch& l, cudaStream_t stream);

// Split-K: the tensor-core kernel writes FP32 partial tiles for every range
// of K steps into l.workspace, then a reduction kernel sums them in split
// order into C (alpha, beta applied there).  Returns the split count used
// through *used_splits.
cudaError_t tc_splitk_launch(const TcLaunch& l, int* used_splits, cudaStream_t stream);

// K ranges split-K actually uses for `requested` ranges of a K extent: every
// range holds the same whole number of 64-wide K steps and none is empty.
int splitk_used_splits(int64_t K, int requested);

// cuTensorMapEncodeTiled from the driver (as void*), or null if unavailable.
void* tensor_map_encoder();

// Closed-form tile traffic and working set of the output-stationary loop nest
// (element counts of A, B, C; bytes; FLOPs; tiles; K steps; largest and full
// per-step working set in bytes) -- see model.cu.
void traffic_model(int64_t M, int64_t N, int64_t K, int64_t tm, int64_t tn, int64_t tk,
                   int64_t in_bytes, int64_t acc_bytes, int64_t c_bytes, int64_t out[9]);

// Predicted seconds of one product on a tensor-core variant (model.cu).
double predict_seconds(int64_t M, int64_t N, int64_t K, int variant, int num_sms, int in_bytes,
                       int out_bytes);

// Output tile of a tensor-core variant (rows x columns).
void tc_tile_shape(int variant, int* tile_m, int* tile_n);

}  // namespace tmmo
