/*
 * tiled_gemm.h -- C ABI of the GB300 (sm_103a) output-stationary tiled GEMM.
 *
 * The operation is the matrix product of "Reading a matrix multiply through
 * its tiles" (introduction): C = A @ B with A of shape M x K, B of shape
 * K x N and C of shape M x N, C[i,j] = sum_k A[i,k] * B[k,j] ("Tiled Matrix
 * Multiplication", idiomatic kernel notes: standard A x B, not A x B^T).  It
 * is computed by the output-stationary loop nest of "Keep one output tile
 * resident": every output tile keeps an FP32 accumulator resident while A
 * and B tiles stream along K, and is written to C exactly once.
 *
 * Layout.  A, B and C are dense and row-major with leading dimensions K, N
 * and N elements ("Tiled Matrix Multiplication", "Layout optimization": row-
 * major for all tensors); gemm_general also takes A or B stored transposed.
 * There are no other strides.  C must not overlap A or B.
 *
 * Memory and ownership.  A, B and C are device pointers owned by the caller
 * (except where an entry point says "host").  The library allocates no
 * device memory per call.  Its state: one device status word per GPU, a
 * cached driver entry point, the fixed scratch array of gemm_splitk_noalloc
 * (on every GPU that loads the library) and the two copy streams that
 * gemm_ex_host creates once per device.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream).  Calls are stream-ordered and asynchronous: they return
 * after the launch, before the result is ready.
 *
 * Errors.  Every entry point returns a gemm_status_t; no C++ exception
 * crosses this boundary.  Argument errors are detected on the host before
 * anything is launched.  A device-side wait that runs out of its time budget
 * is reported later by gemm_device_status().
 */
#ifndef TILED_GEMM_H
#define TILED_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The largest M, N or K any entry point accepts: 2^31 - 256.  Sizes stay
   below 2^31 with a tile's worth of headroom, so that every index a kernel
   forms (a tile's first row plus its extent, a K offset plus one K tile)
   fits a 32-bit signed integer. */
#define GEMM_MAX_DIM ((int64_t)2147483392)

/* Storage / arithmetic types. */
typedef enum {
    GEMM_F32 = 0,  /* IEEE binary32 */
    GEMM_F16 = 1,  /* IEEE binary16 */
    GEMM_BF16 = 2  /* bfloat16 */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1, /* null pointer where data is needed, negative size or one
                                   above GEMM_MAX_DIM, unknown enum value */
    GEMM_ERR_UNSUPPORTED = 2,   /* valid but unsupported combination (types, or a forced
                                   kernel whose alignment rules the operands break) */
    GEMM_ERR_CUDA = 3,          /* a CUDA runtime call or the launch failed */
    GEMM_ERR_TIMEOUT = 4        /* a bounded device-side wait ran out (see gemm_device_status) */
} gemm_status_t;

/* Operand form for gemm_general. */
typedef enum {
    GEMM_OP_N = 0, /* the matrix as stored: A row-major M x K, B row-major K x N */
    GEMM_OP_T = 1  /* its transpose: A stored row-major K x M, B stored row-major N x K */
} gemm_op_t;

/* Kernel selection for gemm_ex_kernel and gemm_general. */
typedef enum {
    GEMM_KERNEL_AUTO = 0,      /* what gemm / gemm_ex use */
    GEMM_KERNEL_SIMT = 1,      /* shared-memory tiled FFMA kernel, 64 x 64 x 16 tiles */
    GEMM_KERNEL_SIMT_TPB3 = 2, /* the same kernel with 3 x 3 tiles, one thread per output
                                  element ("Tiled Matrix Multiplication", TPB = 3) */
    GEMM_KERNEL_TC_128x128 = 3,/* tcgen05, one CTA per 128 x 128 output tile */
    GEMM_KERNEL_TC_128x256 = 4,/* tcgen05, one CTA per 128 x 256 output tile */
    GEMM_KERNEL_TC_256x256 = 5,/* tcgen05 cta_group::2, one CTA pair per 256 x 256 tile */
    GEMM_KERNEL_TC_256x128 = 6,/* tcgen05 cta_group::2, one CTA pair per 256 x 128 tile */
    GEMM_KERNEL_TC_SMALL = 7,  /* tcgen05, one CTA per 128 x 64 or 128 x 128 tile, not
                                  persistent: the lowest fixed cost, for products whose
                                  tiles fit in one wave */
    GEMM_KERNEL_TILE16 = 8     /* one 16 x 16 tile per thread block with its whole K range
                                  copied at once and split between the block's warps
                                  (warp-level MMA for 16-bit inputs, FFMA for FP32): the
                                  lowest latency, for small products */
} gemm_kernel_t;

/*
 * gemm -- C = A @ B, written in acc_dtype.
 *
 * The result type equals the accumulator type, the convention of "Reading a
 * matrix multiply through its tiles" ("Count the repeated reads" counts C at
 * 4 bytes under FP32 accumulation).  in_dtype is the type of both A and B.
 * Supported: (in, acc) = (F32, F32), (F16, F32), (BF16, F32).
 *
 * M == 0 or N == 0 is a no-op.  K == 0 writes zeros to C (the empty sum: the
 * accumulator is initialised to zero and no K tile is added).
 *
 * Returns GEMM_OK, GEMM_ERR_INVALID_VALUE (a null A or B with K > 0 and
 * M*N > 0, a null C with M*N > 0, a negative size or one above GEMM_MAX_DIM, an unknown
 * dtype), GEMM_ERR_UNSUPPORTED (another type combination) or GEMM_ERR_CUDA.
 */
int gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
         gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, void* stream);

/*
 * gemm_ex -- as gemm, with an explicit output type.
 *
 * The helion kernel of "Writing a matmul GPU kernel" accumulates in FP32 and
 * stores into a tensor of the input dtype; out_dtype covers both that and the
 * FP32 output of gemm.  The FP32 accumulator is converted to out_dtype with
 * round-to-nearest-even (overflow to +-inf).  Supported (in, acc, out):
 * (F32, F32, F32/F16/BF16) and (F16 or BF16, F32, F32/F16/BF16).
 */
int gemm_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
            gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype,
            void* stream);

/*
 * gemm_ex_kernel -- as gemm_ex, with the kernel chosen by the caller.
 *
 * The tensor-core kernels need 16-bit inputs, 16-byte aligned A, B and C and
 * row pitches (K and N elements of the input type, N of the output type) that
 * are multiples of 16 bytes; a forced tensor-core kernel whose rules the
 * operands break returns GEMM_ERR_UNSUPPORTED.  GEMM_KERNEL_SIMT and
 * GEMM_KERNEL_SIMT_TPB3 take any shape and any element-aligned pointer.
 * GEMM_KERNEL_TILE16 takes any type, 16-byte aligned A and B whose row
 * pitches as stored are multiples of 16 bytes, and a K whose slices of one
 * 16 x 16 tile fit in a block's shared memory (K up to about 3,400 for
 * 16-bit inputs, 1,700 for FP32); otherwise it returns
 * GEMM_ERR_UNSUPPORTED.  All kernels give results within the same accuracy
 * bound; they differ in the order of the K summation.
 */
int gemm_ex_kernel(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                   gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype,
                   gemm_kernel_t kernel, void* stream);

/*
 * gemm_general -- C = alpha * op(A) @ op(B) + beta * C.
 *
 * op(A) is M x K and op(B) is K x N.  GEMM_OP_N uses an operand as stored;
 * GEMM_OP_T uses its transpose, i.e. A is stored row-major K x M or B is
 * stored row-major N x K -- the pre-transposed inputs of "Tiled Matrix
 * Multiplication" ("When would transposed loading be useful?"); the kernels
 * read them in place through the matching tile layout, nothing is
 * transposed in memory.  beta != 0 reads C (row-major M x N, out_dtype)
 * before it is overwritten -- the accumulate-into-C form of torch.addmm that
 * the helion kernel of "Writing a matmul GPU kernel" builds its tiles with;
 * beta == 0 never reads C.  alpha and beta are applied in FP32 to the FP32
 * accumulator before the conversion to out_dtype.  C must not overlap A or B.
 *
 * The tensor-core kernels need the row pitches of A and B as stored (K or M,
 * N or K elements) and of C (N) to be multiples of 16 bytes; otherwise the
 * automatic choice is the SIMT kernel.  Types, sizes, K == 0 (C = beta * C)
 * and errors as gemm_ex_kernel, plus GEMM_ERR_INVALID_VALUE for an unknown
 * gemm_op_t.
 */
int gemm_general(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                 gemm_op_t op_a, gemm_op_t op_b, float alpha, float beta, gemm_dtype_t in_dtype,
                 gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype, gemm_kernel_t kernel,
                 void* stream);

/*
 * gemm_workspace_size -- bytes of workspace gemm_ex_ws can use for these
 * sizes on the current device: one 256 x 256 FP32 tile per pair of SMs, or,
 * for the few-tile products it splits along K, their split partials when
 * those are larger.  0 for empty products or when no device is available.
 */
size_t gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * gemm_ex_ws -- gemm_ex with a workspace that evens out the last wave.
 *
 * The persistent kernel runs the output tiles in waves of one tile per CTA
 * pair.  When the tile count is not a multiple of the pairs resident on the
 * GPU, the last wave leaves pairs idle; with a workspace, the tiles of that
 * last wave are instead split along K into as many pieces as there are idle
 * pairs (when that makes at least two pieces, each at least four 64-wide K
 * steps long), their FP32 partials go to
 * `workspace` (caller-owned device memory,
 * 16-byte aligned; gemm_workspace_size bytes always suffice), and a second
 * kernel on the same stream adds each tile's pieces in K order and writes
 * it.  The result differs from gemm_ex's only in the summation order of those
 * tiles, and is identical run to run.  Without a workspace (NULL), with one
 * too small for the plan, or when the automatic choice is not the CTA-pair
 * kernel, this is gemm_ex.  Calls sharing a workspace must not overlap in
 * time.  Errors as gemm_ex, plus GEMM_ERR_INVALID_VALUE for a misaligned
 * workspace.
 *
 * Products with few output tiles and a long K take the other form of the
 * same idea (see gemm_ws_split_count): every tile is split along K, as
 * gemm_splitk does, so that the otherwise idle SMs share the K loop.
 */
int gemm_ex_ws(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
               gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * gemm_ws_split_count -- for products with few output tiles, the number of
 * K ranges gemm_ex_ws splits them into (as gemm_splitk with that many
 * splits), or 0 when it does not.  The rule: a tensor-core product whose
 * 128 x 128 output tiles occupy at most a quarter of the SMs, with K of at
 * least 512, is split so that up to one unit of work runs per SM, into at
 * most 8 ranges.  gemm_ex_ws does so only when its workspace holds
 * gemm_splitk_workspace_size(M, N, K, count) bytes, which
 * gemm_workspace_size always covers.  There is no counterpart in the pages:
 * they accumulate each tile over all of K in one place.  Returns the count,
 * 0, or a negated gemm_status_t (bad sizes or types, no device).
 */
int gemm_ws_split_count(int64_t M, int64_t N, int64_t K, gemm_dtype_t in_dtype,
                        gemm_dtype_t acc_dtype, gemm_dtype_t out_dtype);

/*
 * gemm_splitk_workspace_size -- bytes of FP32 workspace gemm_splitk needs:
 * used_splits * M * N * 4, where used_splits <= splits is the number of
 * equal ranges of 64-wide K steps K is divided into (no range is empty).
 * Returns 0 for non-positive sizes or splits < 1.
 */
size_t gemm_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int splits);

/*
 * gemm_splitk -- C = A @ B (as gemm_ex) with the K reduction split across
 * SMs, for products with few output tiles and a long K.
 *
 * "Reading a matrix multiply through its tiles" ("Keep one output tile
 * resident") accumulates each output tile over all of K before writing it
 * once; here each tile's K steps are divided into `splits` ranges that run
 * as separate units of work, each range's FP32 partial tile is written to
 * `workspace` (split-major, [split][M][N], caller-owned device memory of at
 * least gemm_splitk_workspace_size bytes, 16-byte aligned), and a second
 * kernel on the same stream adds the partials in split order (a fixed
 * order: the result is identical run to run) and writes C in out_dtype with
 * round-to-nearest-even.  The workspace contents are scratch: they need no
 * initial value and are overwritten.  Two calls that share a workspace must
 * not overlap in time.
 *
 * Operands the tensor-core kernels cannot take (see gemm_ex_kernel) are
 * computed by gemm_ex's automatic choice instead; the workspace is then not
 * used.  Returns as gemm_ex, plus GEMM_ERR_INVALID_VALUE for splits < 1 or a
 * missing, misaligned or too small workspace.
 */
int gemm_splitk(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                int splits, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                gemm_dtype_t out_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * gemm_splitk_noalloc -- gemm_splitk for callers that cannot allocate
 * device memory; it allocates nothing.  The pages have no counterpart: this
 * entry point exists for deployment, not for the method.
 *
 * Who needs it: code that runs inside a framework owning every device
 * allocation (its pool may already hold all free memory), real-time paths
 * where a cudaMalloc (which may synchronize the device) is not allowed, and
 * services that reserve all device memory up front.  Instead of a caller
 * workspace, the FP32 partials live in one fixed array inside the library,
 * GEMM_SPLITK_NOALLOC_MAX_BYTES on every GPU that loads the library, kept
 * until the process exits.
 *
 * Limits and rules:
 *  - gemm_splitk_workspace_size(M, N, K, splits) must not exceed
 *    GEMM_SPLITK_NOALLOC_MAX_BYTES; larger requests return
 *    GEMM_ERR_UNSUPPORTED and launch nothing (use fewer splits, or
 *    gemm_splitk with your own workspace).
 *  - Every call shares the one array and the array keeps the last call's
 *    partials; nothing in it needs to start at zero (each call overwrites
 *    every partial it reads).  Calls whose work overlaps on the GPU -- on
 *    different streams, or on different host threads -- race on the array
 *    and give wrong results; serialize them (one stream is enough).
 *  - The first call on each device looks up the array's device address;
 *    make that first call before any stream capture.
 * Arguments, results, fallback for operands the tensor-core kernels cannot
 * take, and other errors as gemm_splitk.
 */
#define GEMM_SPLITK_NOALLOC_MAX_BYTES ((size_t)8 << 20) /* 8 MiB of FP32 partials */
int gemm_splitk_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                        int splits, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                        gemm_dtype_t out_dtype, void* stream);

/*
 * gemm_select_kernel -- the kernel gemm_ex would launch for these arguments
 * on the current device (a gemm_kernel_t), or a negative gemm_status_t when
 * the arguments are invalid or unsupported.  Nothing is launched.
 */
int gemm_select_kernel(const void* A, const void* B, const void* C, int64_t M, int64_t N,
                       int64_t K, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                       gemm_dtype_t out_dtype);

/*
 * gemm_ex_host -- gemm_ex on HOST buffers, end to end.
 *
 * A_host (M x K), B_host (K x N) and C_host (M x N) are host buffers (pinned
 * memory gives asynchronous copies; pageable memory works but the copies
 * block).  dA, dB and dC are caller-owned device buffers of at least the same
 * sizes.  The call enqueues the host-to-device copies of A and B, the
 * product, and the device-to-host copy of C, ordered after the work already
 * on `stream` and before anything queued on it later; it returns after
 * enqueueing (synchronize the stream before reading C_host).  Products of
 * more than 1024 rows are pipelined in row panels: B is copied first, then
 * the copy of one panel of A and the copy back of another panel of C
 * overlap the product of a third, on two copy streams the library creates
 * once per device (calls from several host threads are enqueued one at a
 * time).  Errors as gemm_ex.
 */
int gemm_ex_host(const void* A_host, const void* B_host, void* C_host, int64_t M, int64_t N,
                 int64_t K, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                 gemm_dtype_t out_dtype, void* dA, void* dB, void* dC, void* stream);

/*
 * gemm_ex_host_ws -- gemm_ex_host whose products (the whole product, or each
 * row panel's) run as gemm_ex_ws with the caller's device workspace:
 * the tiles of a panel's last, partial wave are split along K across the
 * idle CTA pairs, as on the device path.  workspace may be NULL (then this
 * is gemm_ex_host); otherwise it must be 16-byte aligned, and
 * gemm_workspace_size(M, N, K) bytes always suffice.  The panels run one
 * after another on `stream` and share the workspace.  Errors as
 * gemm_ex_ws.
 */
int gemm_ex_host_ws(const void* A_host, const void* B_host, void* C_host, int64_t M, int64_t N,
                    int64_t K, gemm_dtype_t in_dtype, gemm_dtype_t acc_dtype,
                    gemm_dtype_t out_dtype, void* dA, void* dB, void* dC, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * gemm_host_panel_rows -- the rows of A and C in one panel of the pipelined
 * host-buffer path for an M-row product with K > 0 (M itself when the
 * product runs as one piece); 0 for M <= 0 or M > GEMM_MAX_DIM.
 */
int64_t gemm_host_panel_rows(int64_t M);

/*
 * gemm_device_status -- synchronize `stream`, then read and clear the status
 * word of the current device.  Returns GEMM_OK, GEMM_ERR_TIMEOUT if a
 * tensor-core kernel launched since the last call gave up a bounded wait
 * (its output is then incomplete), or GEMM_ERR_CUDA.
 */
int gemm_device_status(void* stream);

/*
 * gemm_debug_config -- test hook for the bounded-wait watchdog.
 *
 * wait_budget_cycles: SM clock cycles one device-side wait may take before
 * the kernel gives up (<= 0 restores the default, about one second).
 * fault_skip_kblock: when >= 0, the tensor-core producer skips the loads of
 * that K step, so the MMA warp's wait on it runs out and the kernel returns
 * GEMM_ERR_TIMEOUT through gemm_device_status; -1 (the default) disables it.
 * The setting is process-wide.  Returns GEMM_OK.
 */
int gemm_debug_config(int64_t wait_budget_cycles, int fault_skip_kblock);

/*
 * gemm_traffic_model -- the tile-level traffic and working-set counts of the
 * output-stationary loop nest ("Reading a matrix multiply through its
 * tiles", sections "What fits in local storage?", "Count the repeated reads"
 * and "Edge tiles still matter"), in closed form.  With no reuse of input
 * tiles across output tiles and tm x tn x tk tiles, out[0..8] receive: A
 * elements read M*K*ceil(N/tn); B elements read K*N*ceil(M/tm); C elements
 * written M*N; their bytes (A and B at in_bytes, C at c_bytes); FLOPs
 * 2*M*N*K; output tiles; tile steps along K; the largest per-step working
 * set (actual extents of the first tile); and the working set of one full
 * tm x tn x tk step (A, B tiles at in_bytes, accumulator at acc_bytes).  The
 * automatic kernel choice ranks tile shapes with these counts.  Host-only;
 * returns GEMM_ERR_INVALID_VALUE for negative sizes, non-positive tiles or a
 * null out.
 */
int gemm_traffic_model(int64_t M, int64_t N, int64_t K, int64_t tm, int64_t tn, int64_t tk,
                       int64_t in_bytes, int64_t acc_bytes, int64_t c_bytes, int64_t* out);

/*
 * gemm_launch_count -- how many kernels the library has launched in this
 * process so far (all devices and streams; a plain product is one launch,
 * split-K and gemm_ex_ws with split tiles are two).  For accounting only.
 */
uint64_t gemm_launch_count(void);

/* gemm_error_string -- a static description of a gemm_status_t. */
const char* gemm_error_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* TILED_GEMM_H */
