// The C ABI declared in include/tiled_gemm.h: argument validation, kernel
// selection, the device status word, and the host-buffer entry point.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "launch.h"
#include "tc_params.h"
#include "tiled_gemm.h"

namespace tmmo {
namespace {

// One status word per device (the watchdog of the tensor-core kernel).
__device__ int g_status_word;

constexpr int kMaxDevices = 64;
constexpr long long kDefaultWaitBudget = 2000000000LL;  // ~1 s of SM clock

std::atomic<long long> g_wait_budget{kDefaultWaitBudget};
std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_fault_skip_kblock{-1};

struct DeviceInfo {
    int num_sms = 0;
    int* status = nullptr;
    bool ready = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Set-up of the current device, once: SM count and the status word address.
cudaError_t device_info(DeviceInfo* out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess)
            return err;
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_status_word);
        if (err != cudaSuccess)
            return err;
        d.status = static_cast<int*>(p);
        d.ready = true;
    }
    *out = d;
    return cudaSuccess;
}

bool valid_dtype(int dt) { return dt == GEMM_F32 || dt == GEMM_F16 || dt == GEMM_BF16; }
int dt_size(int dt) { return dt == GEMM_F32 ? 4 : 2; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side argument check shared by every entry point.
int validate(const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
             int in_dtype, int acc_dtype, int out_dtype)
{
    if (!valid_dtype(in_dtype) || !valid_dtype(acc_dtype) || !valid_dtype(out_dtype))
        return GEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0 || M > GEMM_MAX_DIM || N > GEMM_MAX_DIM || K > GEMM_MAX_DIM)
        return GEMM_ERR_INVALID_VALUE;
    if (M > 0 && N > 0) {
        if (!C)
            return GEMM_ERR_INVALID_VALUE;
        if (K > 0 && (!A || !B))
            return GEMM_ERR_INVALID_VALUE;
    }
    if (acc_dtype != GEMM_F32)
        return GEMM_ERR_UNSUPPORTED;
    return GEMM_OK;
}

// The operation of one call: C = alpha * op(A) op(B) + beta * C.
struct Problem {
    const void* A;
    const void* B;
    void* C;
    int64_t M, N, K;
    int op_a, op_b;  // 0: as stored; 1: transposed
    float alpha, beta;
    int in_dtype, acc_dtype, out_dtype;
};

// Whether a tensor-core kernel can take these operands: 16-bit inputs, FP32
// accumulation, 16-byte aligned bases and row pitches (TMA rules).  The row
// pitch of A is K elements as stored or M transposed; of B, N as stored or K
// transposed; of C, N.
bool tc_eligible(const Problem& q)
{
    if (((q.M + 127) / 128) * ((q.N + 127) / 128) >= (int64_t(1) << 31))
        return false;  // tile indices are 32-bit
    if (q.in_dtype != GEMM_F16 && q.in_dtype != GEMM_BF16)
        return false;
    if (q.K <= 0)
        return false;
    if (!aligned16(q.A) || !aligned16(q.B) || !aligned16(q.C))
        return false;
    const int64_t ib = dt_size(q.in_dtype);
    const int64_t pitch_a = q.op_a ? q.M : q.K;
    const int64_t pitch_b = q.op_b ? q.K : q.N;
    if ((pitch_a * ib) % 16 != 0 || (pitch_b * ib) % 16 != 0)
        return false;
    if ((q.N * dt_size(q.out_dtype)) % 16 != 0)
        return false;
    return true;
}

// K steps from which a product with few output tiles is split along K
// rather than run on one CTA per tile: below it, splitting K adds a second
// launch and the partials' traffic for little gain (measured on GB300, L2
// flushed, BF16: 512 x 512 x 1024 10.6 us on one CTA per tile against 12.3
// split; 256 x 256 x 2048 14.8 against 12.3).
constexpr int64_t kSplitMinKBlocks = 32;

// Whether the non-persistent single-tile kernel takes a product: its
// 128 x 64 tiles fit in one wave of CTAs and K is short of kSplitMinKBlocks
// steps.  Where even 128 x 128 tiles would need more than half the SMs, the
// persistent 128 x 128 kernel is as fast or faster (measured on GB300, L2
// flushed, BF16, us, single-tile / persistent: 2048 x 1024 x 512 10.6 /
// 10.2, 1536^3 15.9 / 14.3).
bool small_kernel_fits(int64_t M, int64_t N, int64_t K, int num_sms)
{
    if (tc_small_tile_n(M, N, num_sms) != 64)
        return false;
    const int64_t tiles = ((M + 127) / 128) * ((N + 63) / 64);
    return tiles <= num_sms && (K + 63) / 64 < kSplitMinKBlocks;
}

// Whether the latency-path kernel (tile16.cu) takes a product.  Its 16 x 16
// tiles each get a block with the tile's whole K range copied at once, so
// it is the fastest path while the blocks' copies are short: one tile per
// SM up to K = 2048, or up to three tiles per SM with at most 1024 x SMs
// tile-K values in all.  For operands the tensor-core kernels cannot take
// (FP32, or unaligned 16-bit rows) it also beats the tiled SIMT kernel up
// to eleven tiles per SM.  Measured on GB300 with L2 overwritten between
// calls, microseconds (this kernel / the previous choice / cuBLAS): 128^3
// F16 -> F32 6.1 / 8.3 (tc_small) / 6.4; 96 x 200 x 1000 BF16 -> F32
// 8.2 / 11.1 / 8.2; 128 x 128 x 2048 BF16 10.2 / 12.3 (split-K) / 9.2;
// 256 x 256 x 512 8.1 / 8.8 / 7.1; 320 x 320 x 256 8.2 / 8.6 / 6.2; not
// taken: 256 x 256 x 1024 10.1 / 9.8, 384 x 384 x 128 8.7 / 8.1, 512^3
// 12.3 / 8.7.  FP32: 128^3 6.6 / 12.8 (SIMT) / 10.0; 100 x 200 x 1000
// 12.0 / 59.1 / 19.1; 512^3 21.2 / 33.4 / 18.7; 640^3 (10.5 tiles per SM)
// 37.4-37.6 / 39.3-39.8 / 22.6; not taken: 768^3 (15 per SM) 57.6-57.9 /
// 46.9-47.1.
bool tile16_takes(const Problem& q, bool tensor_ok, int num_sms)
{
    SimtLaunch l{};
    l.in_dtype = q.in_dtype;
    l.out_dtype = q.out_dtype;
    l.op_a = q.op_a;
    l.op_b = q.op_b;
    l.A = q.A;
    l.B = q.B;
    l.C = q.C;
    if (q.M > GEMM_MAX_DIM || q.N > GEMM_MAX_DIM || q.K > GEMM_MAX_DIM)
        return false;
    l.M = static_cast<int>(q.M);
    l.N = static_cast<int>(q.N);
    l.K = static_cast<int>(q.K);
    l.num_sms = num_sms;
    if (!tile16_fits(l))
        return false;
    const int64_t tiles = ((q.M + 15) / 16) * ((q.N + 15) / 16);
    if (!tensor_ok)
        return tiles <= int64_t(11) * num_sms;
    if (tiles <= num_sms)
        return q.K <= 2048;
    return tiles <= int64_t(3) * num_sms && tiles * q.K <= int64_t(1024) * num_sms;
}

// The automatic choice.  Small products go to the latency-path kernel
// (tile16_takes); other operands the tensor-core kernels cannot take go
// to the tiled SIMT kernel; otherwise the tensor-core variant with the
// smallest predicted time: the tile traffic of the loop nest, the waves of
// tiles over the resident CTAs and each tile shape's measured throughput
// (predict_seconds in model.cu).
int auto_kernel(const Problem& q, int num_sms)
{
    const int64_t M = q.M, N = q.N, K = q.K;
    const bool tensor_ok = tc_eligible(q);
    if (tile16_takes(q, tensor_ok, num_sms))
        return GEMM_KERNEL_TILE16;
    if (!tensor_ok)
        return GEMM_KERNEL_SIMT;
    const double flops = 2.0 * double(M) * double(N) * double(K);
    if (flops < 2.0 * 64 * 64 * 64)
        return GEMM_KERNEL_SIMT;
    // One wave of single-tile CTAs and a short K: the non-persistent kernel
    // (tc_small.cu), the lowest fixed cost.  Measured on GB300 with L2
    // flushed between calls (BF16, microseconds, against the 128 x 128
    // persistent kernel): 64^3 6.8 / 7.4, 512^3 8.9 / 10.3, 256 x 256 x
    // 1024 10.8 / 12.0, 96 x 200 x 1000 10.9 / 13.0, equal within 0.4 us up
    // to 2048 x 1024 x 512.  From 32 K steps up, few tiles are split along K
    // instead (gemm_ex_ws).
    if (small_kernel_fits(M, N, K, num_sms))
        return GEMM_KERNEL_TC_SMALL;
    const int in_b = dt_size(q.in_dtype), out_b = dt_size(q.out_dtype);
    int best = GEMM_KERNEL_TC_256x256;
    double best_t = predict_seconds(M, N, K, TC_256x256, num_sms, in_b, out_b);
    for (int v : {GEMM_KERNEL_TC_256x128, GEMM_KERNEL_TC_128x256, GEMM_KERNEL_TC_128x128}) {
        const double t = predict_seconds(M, N, K, v, num_sms, in_b, out_b);
        if (t < best_t * 0.98) {  // prefer the larger tile unless clearly slower
            best_t = t;
            best = v;
        }
    }
    return best;
}

bool is_tc(int kernel)
{
    return kernel >= GEMM_KERNEL_TC_128x128 && kernel <= GEMM_KERNEL_TC_SMALL;
}

int validate_problem(const Problem& q)
{
    int rc = validate(q.A, q.B, q.C, q.M, q.N, q.K, q.in_dtype, q.acc_dtype, q.out_dtype);
    if (rc != GEMM_OK)
        return rc;
    if ((q.op_a != GEMM_OP_N && q.op_a != GEMM_OP_T) || (q.op_b != GEMM_OP_N && q.op_b != GEMM_OP_T))
        return GEMM_ERR_INVALID_VALUE;
    return GEMM_OK;
}

int run(const Problem& q, int kernel, cudaStream_t stream)
{
    int rc = validate_problem(q);
    if (rc != GEMM_OK)
        return rc;
    if (kernel < GEMM_KERNEL_AUTO || kernel > GEMM_KERNEL_TILE16)
        return GEMM_ERR_INVALID_VALUE;
    if (q.M == 0 || q.N == 0)
        return GEMM_OK;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (kernel == GEMM_KERNEL_AUTO)
        kernel = auto_kernel(q, d.num_sms);
    if (is_tc(kernel)) {
        if (!tc_eligible(q))
            return GEMM_ERR_UNSUPPORTED;
        TcLaunch l{};
        l.variant = kernel;
        l.op_a = q.op_a;
        l.op_b = q.op_b;
        l.alpha = q.alpha;
        l.beta = q.beta;
        l.in_dtype = q.in_dtype;
        l.out_dtype = q.out_dtype;
        l.A = q.A;
        l.B = q.B;
        l.C = q.C;
        l.M = static_cast<int>(q.M);
        l.N = static_cast<int>(q.N);
        l.K = static_cast<int>(q.K);
        l.num_sms = d.num_sms;
        l.status = d.status;
        l.wait_budget = g_wait_budget.load();
        l.fault_skip_kblock = g_fault_skip_kblock.load();
        cudaError_t err = (kernel == GEMM_KERNEL_TC_SMALL) ? tc_small_launch(l, stream)
                                                            : tc_gemm_launch(l, stream);
        if (err == cudaErrorNotSupported)
            return GEMM_ERR_UNSUPPORTED;
        return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    SimtLaunch l{};
    l.tpb3 = (kernel == GEMM_KERNEL_SIMT_TPB3);
    l.in_dtype = q.in_dtype;
    l.out_dtype = q.out_dtype;
    l.op_a = q.op_a;
    l.op_b = q.op_b;
    l.alpha = q.alpha;
    l.beta = q.beta;
    l.A = q.A;
    l.B = q.B;
    l.C = q.C;
    l.M = static_cast<int>(q.M);
    l.N = static_cast<int>(q.N);
    l.K = static_cast<int>(q.K);
    l.num_sms = d.num_sms;
    cudaError_t err = (kernel == GEMM_KERNEL_TILE16) ? tile16_launch(l, stream)
                                                         : simt_gemm_launch(l, stream);
    if (err == cudaErrorNotSupported)
        return GEMM_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

Problem plain(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int in_dtype,
              int acc_dtype, int out_dtype)
{
    return Problem{A, B, C, M, N, K, GEMM_OP_N, GEMM_OP_N, 1.0f, 0.0f, in_dtype, acc_dtype,
                   out_dtype};
}

}  // namespace

void note_launch()
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
}

}  // namespace tmmo

using namespace tmmo;

extern "C" int gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                    gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, void* stream)
{
    return run(plain(A, B, C, M, N, K, in_dtype, acc_dtype, acc_dtype), GEMM_KERNEL_AUTO,
               static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                       gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype,
                       void* stream)
{
    return run(plain(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype), GEMM_KERNEL_AUTO,
               static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_ex_kernel(const void* A, const void* B, void* C, int64_t M, int64_t N,
                              int64_t K, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                              gemm_dtype_t out_dtype, gemm_kernel_t kernel, void* stream)
{
    return run(plain(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype), kernel,
               static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_general(const void* A, const void* B, void* C, int64_t M, int64_t N,
                            int64_t K, gemm_op_t op_a, gemm_op_t op_b, float alpha, float beta,
                            gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype,
                            gemm_kernel_t kernel, void* stream)
{
    const Problem q{A, B, C, M, N, K, op_a, op_b, alpha, beta, in_dtype, acc_dtype, out_dtype};
    return run(q, kernel, static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_select_kernel(const void* A, const void* B, const void* C, int64_t M,
                                  int64_t N, int64_t K, gemm_dtype_t in_dtype,
                                  gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype)
{
    const Problem q = plain(A, B, const_cast<void*>(C), M, N, K, in_dtype, acc_dtype, out_dtype);
    int rc = validate_problem(q);
    if (rc != GEMM_OK)
        return -rc;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return -GEMM_ERR_CUDA;
    return auto_kernel(q, d.num_sms);
}

extern "C" size_t gemm_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int splits)
{
    if (M <= 0 || N <= 0 || K <= 0 || splits < 1)
        return 0;
    const int used = splitk_used_splits(K, splits);
    return static_cast<size_t>(used) * static_cast<size_t>(M) * static_cast<size_t>(N) * 4u;
}

extern "C" int gemm_splitk(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                           int splits, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                           gemm_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                           void* stream)
{
    const Problem q = plain(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype);
    int rc = validate_problem(q);
    if (rc != GEMM_OK)
        return rc;
    if (splits < 1)
        return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0)
        return GEMM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!tc_eligible(q))
        return run(q, GEMM_KERNEL_AUTO, s);  // no workspace needed or used
    const size_t need = gemm_splitk_workspace_size(M, N, K, splits);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return GEMM_ERR_INVALID_VALUE;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return GEMM_ERR_CUDA;
    TcLaunch l{};
    l.variant = TC_128x128;
    l.op_a = GEMM_OP_N;
    l.op_b = GEMM_OP_N;
    l.alpha = 1.0f;
    l.beta = 0.0f;
    l.in_dtype = in_dtype;
    l.out_dtype = out_dtype;
    l.A = A;
    l.B = B;
    l.C = C;
    l.M = static_cast<int>(M);
    l.N = static_cast<int>(N);
    l.K = static_cast<int>(K);
    l.num_sms = d.num_sms;
    l.status = d.status;
    l.wait_budget = g_wait_budget.load();
    l.fault_skip_kblock = g_fault_skip_kblock.load();
    l.k_splits = splits;
    l.workspace = static_cast<float*>(workspace);
    cudaError_t err = tc_splitk_launch(l, nullptr, s);
    if (err == cudaErrorNotSupported)
        return GEMM_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

namespace tmmo {
namespace {

// K ranges gemm_ex_ws splits a product with few output tiles into: when the
// 128 x 128 tiles would occupy at most a quarter of the SMs and K holds at
// least kSplitMinKBlocks 64-wide steps, K is divided so that up to one unit
// of work runs per SM, at most 8 ranges.  0 = no split.  Eight rather than
// more: measured on GB300 (BF16, L2 flushed between calls), 128 x 128 x
// 2048 took 12.3 us with 8 ranges against 12.7 us with 16, 256 x 256 x 4096
// 12.7 against 12.9 us; the extra partials cost more in the reduction than
// the shorter ranges save.
int few_tile_splits(int64_t M, int64_t N, int64_t K, int num_sms)
{
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    const int64_t k_blocks = (K + 63) / 64;
    if (tiles <= 0 || tiles * 4 > num_sms || k_blocks < kSplitMinKBlocks)
        return 0;
    const int64_t s = std::min<int64_t>(std::min<int64_t>(num_sms / tiles, k_blocks), 8);
    if (s < 2)
        return 0;
    return splitk_used_splits(K, static_cast<int>(s));
}

}  // namespace
}  // namespace tmmo

extern "C" size_t gemm_workspace_size(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0)
        return 0;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return 0;
    // Last-wave split: at most one piece per resident CTA pair, each a
    // 256 x 256 FP32 tile.  Few-tile split-K: its [splits][M][N] partials.
    const size_t tail = static_cast<size_t>(d.num_sms / 2) * 256u * 256u * 4u;
    const int s = few_tile_splits(M, N, K, d.num_sms);
    const size_t split = s > 1 ? gemm_splitk_workspace_size(M, N, K, s) : 0;
    return std::max(tail, split);
}

extern "C" int gemm_ws_split_count(int64_t M, int64_t N, int64_t K, gemm_dtype_t in_dtype,
                                   gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype)
{
    // Operand addresses do not enter the decision beyond 16-byte alignment,
    // so any aligned non-null address stands in for them here.
    const void* any = reinterpret_cast<const void*>(uintptr_t(256));
    const int rc = validate(any, any, any, M, N, K, in_dtype, acc_dtype, out_dtype);
    if (rc != GEMM_OK)
        return -rc;
    Problem q = plain(any, any, const_cast<void*>(any), M, N, K, in_dtype, acc_dtype, out_dtype);
    if (M == 0 || N == 0 || K == 0 || !tc_eligible(q))
        return 0;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return -GEMM_ERR_CUDA;
    if (!is_tc(auto_kernel(q, d.num_sms)))
        return 0;
    return few_tile_splits(M, N, K, d.num_sms);
}

extern "C" int gemm_ex_ws(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                          gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype,
                          void* workspace, size_t workspace_bytes, void* stream)
{
    const Problem q = plain(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype);
    int rc = validate_problem(q);
    if (rc != GEMM_OK)
        return rc;
    if (M == 0 || N == 0)
        return GEMM_OK;
    if (workspace && !aligned16(workspace))
        return GEMM_ERR_INVALID_VALUE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return GEMM_ERR_CUDA;
    const int kernel = auto_kernel(q, d.num_sms);
    if (workspace && is_tc(kernel)) {
        // Few output tiles and a long K: split K across the idle SMs.
        const int splits = few_tile_splits(M, N, K, d.num_sms);
        if (splits > 1 && workspace_bytes >= gemm_splitk_workspace_size(M, N, K, splits))
            return gemm_splitk(A, B, C, M, N, K, splits, in_dtype, acc_dtype, out_dtype, workspace,
                               workspace_bytes, stream);
    }
    if (kernel != GEMM_KERNEL_TC_256x256 || !workspace)
        return run(q, kernel, s);
    TcLaunch l{};
    l.variant = TC_256x256;
    l.op_a = GEMM_OP_N;
    l.op_b = GEMM_OP_N;
    l.alpha = 1.0f;
    l.beta = 0.0f;
    l.in_dtype = in_dtype;
    l.out_dtype = out_dtype;
    l.A = A;
    l.B = B;
    l.C = C;
    l.M = static_cast<int>(M);
    l.N = static_cast<int>(N);
    l.K = static_cast<int>(K);
    l.num_sms = d.num_sms;
    l.status = d.status;
    l.wait_budget = g_wait_budget.load();
    l.fault_skip_kblock = g_fault_skip_kblock.load();
    l.workspace = static_cast<float*>(workspace);
    l.workspace_bytes = workspace_bytes;
    cudaError_t err = tc_hybrid_launch(l, s);
    if (err == cudaErrorNotSupported)
        return GEMM_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

namespace tmmo {
namespace {

// Auxiliary streams and events of the pipelined host-buffer path, one set
// per device, created on first use and kept until exit.
constexpr int kMaxPanels = 8;
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, b_done = nullptr, done = nullptr;
    cudaEvent_t a_done[kMaxPanels] = {}, c_done[kMaxPanels] = {};
    std::mutex mu;
};
HostPipe g_pipe[kMaxDevices];

cudaError_t host_pipe(HostPipe** out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    HostPipe& h = g_pipe[dev];
    std::lock_guard<std::mutex> g(h.mu);
    if (!h.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if ((err = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking)) != cudaSuccess ||
            (err = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking)) != cudaSuccess ||
            (err = cudaEventCreateWithFlags(&h.start, ef)) != cudaSuccess ||
            (err = cudaEventCreateWithFlags(&h.b_done, ef)) != cudaSuccess ||
            (err = cudaEventCreateWithFlags(&h.done, ef)) != cudaSuccess)
            return err;
        for (int i = 0; i < kMaxPanels; ++i)
            if ((err = cudaEventCreateWithFlags(&h.a_done[i], ef)) != cudaSuccess ||
                (err = cudaEventCreateWithFlags(&h.c_done[i], ef)) != cudaSuccess)
                return err;
        h.ready = true;
    }
    *out = &h;
    return cudaSuccess;
}

}  // namespace
}  // namespace tmmo

namespace tmmo {
namespace {

// Rows per panel of the pipelined host-buffer path: whole 256-row tile rows,
// about an eighth of M, at least 1024.  Eight panels rather than four
// shorten the last copy-compute-copy chain: 1.65 vs 1.74 ms for 8192^3 BF16
// on GB300 (host links at about 210 GB/s each way).
#ifndef TMMO_HOST_PANELS
#define TMMO_HOST_PANELS 8
#endif
int64_t host_panel_rows(int64_t M)
{
    int64_t panel = ((M + TMMO_HOST_PANELS - 1) / TMMO_HOST_PANELS + 255) / 256 * 256;
    return panel < 1024 ? 1024 : panel;
}

// The host-buffer path.  Each product (the whole one, or one panel's) goes
// through gemm_ex_ws, so with a workspace it gets the last-wave and few-tile
// splits of the device path; without one it is plain gemm_ex.
int host_pipeline(const void* A_host, const void* B_host, void* C_host, int64_t M, int64_t N,
                  int64_t K, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                  gemm_dtype_t out_dtype, void* dA, void* dB, void* dC, void* workspace,
                  size_t workspace_bytes, void* stream)
{
    int rc = validate(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype, out_dtype);
    if (rc != GEMM_OK)
        return rc;
    rc = validate(dA, dB, dC, M, N, K, in_dtype, acc_dtype, out_dtype);
    if (rc != GEMM_OK)
        return rc;
    if (M == 0 || N == 0)
        return GEMM_OK;
    if (workspace && !aligned16(workspace))
        return GEMM_ERR_INVALID_VALUE;
    if (!workspace)
        workspace_bytes = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t in_b = static_cast<size_t>(dt_size(in_dtype));
    const size_t out_b = static_cast<size_t>(dt_size(out_dtype));
    const size_t a_row = size_t(K) * in_b, c_row = size_t(N) * out_b;
    // Row panels of A and C: B is copied once, then the copy of A's panel
    // i + 1 and of C's panel i - 1 overlap the product of panel i.  Small
    // products (or K == 0) run as one panel on the caller's stream.
    const int64_t panel = host_panel_rows(M);
    const int64_t panels = (M + panel - 1) / panel;
    if (K == 0 || panels <= 1 || panels > kMaxPanels) {
        if (K > 0) {
            if (cudaMemcpyAsync(dA, A_host, size_t(M) * a_row, cudaMemcpyHostToDevice, s) !=
                    cudaSuccess ||
                cudaMemcpyAsync(dB, B_host, size_t(K) * size_t(N) * in_b, cudaMemcpyHostToDevice,
                                s) != cudaSuccess)
                return GEMM_ERR_CUDA;
        }
        rc = gemm_ex_ws(dA, dB, dC, M, N, K, in_dtype, acc_dtype, out_dtype, workspace,
                        workspace_bytes, stream);
        if (rc != GEMM_OK)
            return rc;
        if (cudaMemcpyAsync(C_host, dC, size_t(M) * c_row, cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        return GEMM_OK;
    }
    HostPipe* h = nullptr;
    if (host_pipe(&h) != cudaSuccess)
        return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> g(h->mu);  // one pipelined call enqueues at a time per device
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // Everything starts after the work already queued on the caller's stream.
    if (!ok(cudaEventRecord(h->start, s)) || !ok(cudaStreamWaitEvent(h->in, h->start, 0)) ||
        !ok(cudaStreamWaitEvent(h->out, h->start, 0)))
        return GEMM_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(dB, B_host, size_t(K) * size_t(N) * in_b, cudaMemcpyHostToDevice,
                            h->in)) ||
        !ok(cudaEventRecord(h->b_done, h->in)) || !ok(cudaStreamWaitEvent(s, h->b_done, 0)))
        return GEMM_ERR_CUDA;
    for (int64_t i = 0; i < panels; ++i) {
        const int64_t r0 = i * panel;
        const int64_t rows = (M - r0 < panel) ? M - r0 : panel;
        const char* a_src = static_cast<const char*>(A_host) + size_t(r0) * a_row;
        char* a_dst = static_cast<char*>(dA) + size_t(r0) * a_row;
        char* c_dev = static_cast<char*>(dC) + size_t(r0) * c_row;
        char* c_dst = static_cast<char*>(C_host) + size_t(r0) * c_row;
        if (!ok(cudaMemcpyAsync(a_dst, a_src, size_t(rows) * a_row, cudaMemcpyHostToDevice, h->in)) ||
            !ok(cudaEventRecord(h->a_done[i], h->in)) ||
            !ok(cudaStreamWaitEvent(s, h->a_done[i], 0)))
            return GEMM_ERR_CUDA;
        rc = gemm_ex_ws(a_dst, dB, c_dev, rows, N, K, in_dtype, acc_dtype, out_dtype, workspace,
                        workspace_bytes, stream);
        if (rc != GEMM_OK)
            return rc;
        if (!ok(cudaEventRecord(h->c_done[i], s)) || !ok(cudaStreamWaitEvent(h->out, h->c_done[i], 0)) ||
            !ok(cudaMemcpyAsync(c_dst, c_dev, size_t(rows) * c_row, cudaMemcpyDeviceToHost, h->out)))
            return GEMM_ERR_CUDA;
    }
    // The caller's stream resumes once the last panel of C is on the host.
    if (!ok(cudaEventRecord(h->done, h->out)) || !ok(cudaStreamWaitEvent(s, h->done, 0)))
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

}  // namespace
}  // namespace tmmo

extern "C" int gemm_ex_host(const void* A_host, const void* B_host, void* C_host, int64_t M,
                            int64_t N, int64_t K, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                            gemm_dtype_t out_dtype, void* dA, void* dB, void* dC, void* stream)
{
    return host_pipeline(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype, out_dtype, dA, dB,
                         dC, nullptr, 0, stream);
}

extern "C" int gemm_ex_host_ws(const void* A_host, const void* B_host, void* C_host, int64_t M,
                               int64_t N, int64_t K, gemm_dtype_t in_dtype,
                               gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype, void* dA, void* dB,
                               void* dC, void* workspace, size_t workspace_bytes, void* stream)
{
    return host_pipeline(A_host, B_host, C_host, M, N, K, in_dtype, acc_dtype, out_dtype, dA, dB,
                         dC, workspace, workspace_bytes, stream);
}

extern "C" int64_t gemm_host_panel_rows(int64_t M)
{
    if (M <= 0 || M > GEMM_MAX_DIM)
        return 0;
    const int64_t panel = host_panel_rows(M);
    const int64_t panels = (M + panel - 1) / panel;
    return (panels <= 1 || panels > kMaxPanels) ? M : panel;
}

extern "C" int gemm_device_status(void* stream)
{
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, d.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpy(d.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return GEMM_ERR_CUDA;
        return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

extern "C" int gemm_traffic_model(int64_t M, int64_t N, int64_t K, int64_t tm, int64_t tn,
                                  int64_t tk, int64_t in_bytes, int64_t acc_bytes, int64_t c_bytes,
                                  int64_t* out)
{
    if (M < 0 || N < 0 || K < 0 || tm <= 0 || tn <= 0 || tk <= 0 || !out)
        return GEMM_ERR_INVALID_VALUE;
    traffic_model(M, N, K, tm, tn, tk, in_bytes, acc_bytes, c_bytes, out);
    return GEMM_OK;
}

extern "C" uint64_t gemm_launch_count(void)
{
    return g_launches.load(std::memory_order_relaxed);
}

extern "C" int gemm_debug_config(int64_t wait_budget_cycles, int fault_skip_kblock)
{
    g_wait_budget.store(wait_budget_cycles > 0 ? wait_budget_cycles : kDefaultWaitBudget);
    g_fault_skip_kblock.store(fault_skip_kblock >= 0 ? fault_skip_kblock : -1);
    return GEMM_OK;
}

extern "C" const char* gemm_error_string(int status)
{
    switch (status) {
    case GEMM_OK:
        return "success";
    case GEMM_ERR_INVALID_VALUE:
        return "invalid argument (null pointer, negative or too large size, unknown enum)";
    case GEMM_ERR_UNSUPPORTED:
        return "unsupported type combination or operand alignment for the chosen kernel";
    case GEMM_ERR_CUDA:
        return "CUDA runtime error or launch failure";
    case GEMM_ERR_TIMEOUT:
        return "a device-side wait ran out of its time budget; the output is incomplete";
    default:
        return "unknown status";
    }
}

// ------------------------------------------------------------------------
// Split-K without any allocation.
//
// Some callers cannot allocate device memory at the point where they need a
// product: code running under a framework that owns every allocation (its
// pool may already hold all free memory), real-time paths that must not
// call cudaMalloc (it can synchronize the device and take milliseconds),
// and memory-budgeted services that reserve all device memory up front.  For them,
// gemm_splitk_noalloc keeps its FP32 partials in the library's own
// fixed-size device array below instead of a caller workspace.
namespace tmmo {
namespace {

// The scratch of gemm_splitk_noalloc: GEMM_SPLITK_NOALLOC_MAX_BYTES on every
// device that loads the library, held until the process exits.  Host code
// must not use the symbol itself as a device address; it takes the address
// from cudaGetSymbolAddress for the current device.
static __device__ __align__(256) float g_splitk_scratch[GEMM_SPLITK_NOALLOC_MAX_BYTES / 4];

float* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// The device address of g_splitk_scratch on the current device, looked up
// once per device (the first call on a device does the lookup).
cudaError_t scratch_address(float** out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        float* p = nullptr;
        err = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_splitk_scratch);
        if (err != cudaSuccess)
            return err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace tmmo

extern "C" int gemm_splitk_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                   int64_t K, int splits, gemm_dtype_t in_dtype,
                                   gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype, void* stream)
{
    const Problem q = plain(A, B, C, M, N, K, in_dtype, acc_dtype, out_dtype);
    int rc = validate_problem(q);
    if (rc != GEMM_OK)
        return rc;
    if (splits < 1)
        return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0)
        return GEMM_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!tc_eligible(q))
        return run(q, GEMM_KERNEL_AUTO, s);  // these kernels use no scratch
    if (gemm_splitk_workspace_size(M, N, K, splits) > GEMM_SPLITK_NOALLOC_MAX_BYTES)
        return GEMM_ERR_UNSUPPORTED;  // the partials do not fit the fixed scratch
    float* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess)
        return GEMM_ERR_CUDA;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess)
        return GEMM_ERR_CUDA;
    TcLaunch l{};
    l.variant = TC_128x128;
    l.op_a = GEMM_OP_N;
    l.op_b = GEMM_OP_N;
    l.alpha = 1.0f;
    l.beta = 0.0f;
    l.in_dtype = in_dtype;
    l.out_dtype = out_dtype;
    l.A = A;
    l.B = B;
    l.C = C;
    l.M = static_cast<int>(M);
    l.N = static_cast<int>(N);
    l.K = static_cast<int>(K);
    l.num_sms = d.num_sms;
    l.status = d.status;
    l.wait_budget = g_wait_budget.load();
    l.fault_skip_kblock = g_fault_skip_kblock.load();
    l.k_splits = splits;
    l.workspace = scratch;
    cudaError_t err = tc_splitk_launch(l, nullptr, s);
    if (err == cudaErrorNotSupported)
        return GEMM_ERR_UNSUPPORTED;
    return err == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
