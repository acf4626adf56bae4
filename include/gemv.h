/*
 * gemv.h — C ABI of libgemv.so, the GB300 (sm_103a) decode GEMV.
 *
 * The operation ("Decode GEMV at half of HBM bandwidth", inferenceinterviews.com,
 * "A strong answer" and its split-K listing): for every batch row b and output
 * row n,
 *
 *     y[b][n] = sum_{k < K} float(W[n][k]) * float(x[b][k])
 *
 * with BF16 weights and activations, products and sums in FP32 (batch 1 on the
 * CUDA cores; batches 2..16 on the BF16 tensor cores with FP32 accumulation,
 * where B multiply-adds per weight element would otherwise make the CUDA cores,
 * not HBM, the limit: "What interviewers probe next"). At batch 1 this
 * is a byte stream: the time is the weight bytes over the HBM bandwidth the
 * kernel sustains ("How to approach it"), so the library is built to keep enough
 * 16-byte loads in flight on every SM ("A strong answer", Little's law) and to
 * size its grid to whole waves of the GPU's SMs (cause 1 and "The reversal
 * condition": split K only when the rows alone do not fill the GPU).
 *
 * Layouts (all row-major, all device memory owned by the caller):
 *   W : N rows of ldw BF16 values; only columns k < K are read. The padding
 *       columns [K, ldw) are never part of a sum (their contents may be NaN).
 *   x : B rows of K BF16 values, row stride K (row b starts at x + b*K).
 *   y : B rows of N FP32 values, row stride N. y is overwritten (not
 *       accumulated): every element is written exactly once per call.
 *
 * Preconditions checked before anything is launched (GEMV_ERR_INVALID /
 * GEMV_ERR_ALIGN on violation):
 *   1 <= N <= 2^31-1, 1 <= K <= 2^31-1, 1 <= B <= 16, K <= ldw, ldw % 8 == 0;
 *   W 16-byte aligned; x 2-byte aligned; y 4-byte aligned; no pointer NULL.
 * Not checked: y must not overlap W or x; W must hold N*ldw elements, x B*K,
 * y B*N.
 *
 * Results are deterministic: the same call on the same inputs returns the same
 * bits on every run. Partial sums (over lanes, warps and K-splits) are combined
 * in a fixed order and never with atomics ("What interviewers probe next":
 * reproducibility needs a fixed reduction order). Any FP32 summation order is
 * within the accuracy bound |y - exact| <= 1e-5 * sum_k |W[n][k] * x[b][k]|.
 *
 * Streams: every call is asynchronous on the given stream (a cudaStream_t passed
 * as void*; NULL means the legacy default stream) and never synchronizes, except
 * the three *_host_io calls, which copy host buffers in and out and wait for
 * their stream.
 * Launch failures return GEMV_ERR_CUDA; gemv_last_cuda_error() then returns the
 * cudaError_t. Faults inside a kernel surface at the caller's next
 * synchronization, as for any CUDA kernel. The kernels read W before they wait
 * for the preceding grid on the stream (programmatic dependent launch), so W
 * must not be written by a kernel that immediately precedes a call on the same
 * stream and triggers its dependents early; x and y are touched only after the
 * wait. Calls are thread-safe; the library keeps only per-device launch
 * settings, created on first use. Setting the environment variable GEMV_PDL=0
 * before the first call turns programmatic dependent launch off (each kernel
 * then starts only after the preceding one has finished), for comparison.
 */
#ifndef GEMV_H
#define GEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    GEMV_OK = 0,
    GEMV_ERR_INVALID = -1,      /* a size, count or pointer is out of range      */
    GEMV_ERR_ALIGN = -2,        /* W not 16-B aligned, ldw % 8 != 0, x or y misaligned */
    GEMV_ERR_CUDA = -3,         /* a CUDA runtime call failed (see gemv_last_cuda_error) */
    GEMV_ERR_NOMEM = -4,        /* host allocation for a plan failed             */
    GEMV_ERR_CAPTURE = -5,      /* graph capture or instantiation failed         */
    GEMV_ERR_UNSUPPORTED = -6   /* no sm_103a device, or a plan used before capture */
};

#define GEMV_MAX_BATCH 16
#define GEMV_MAX_SEGMENTS 8

/*
 * y = W·x for one weight matrix ("Decode GEMV at half of HBM bandwidth",
 * "A strong answer": the split-K GEMV). W is [N, ldw] BF16, x is [B, K] BF16,
 * y is [B, N] FP32; see the layout rules above. Returns GEMV_OK or an error
 * code; on an error nothing was launched (validation) or the launch failed.
 */
int gemv_bf16(const void *W, const void *x, float *y,
              int64_t N, int64_t K, int B, int64_t ldw, void *stream);

/*
 * Options of the *_ex calls. flags is 0 or a set of GEMV_FLAG_* bits; a NULL
 * options pointer means flags = 0.
 *
 * GEMV_FLAG_RMSNORM: RMSNorm prologue on x ("GPU performance chains", "Fused
 * RMSNorm traffic": at decode the bytes of a separate norm kernel are trivial
 * and its launch is the cost, so it is fused into the projection that reads
 * x). Each output row b is scaled by
 *     r_b = (mean_{k<K} x[b][k]^2 + rms_eps)^(-1/2),
 * computed in FP32 from the x the kernel stages anyway, i.e.
 *     y[b][n] = r_b * sum_k W[n][k] * x[b][k].
 * The norm's elementwise weight is expected folded into W's columns (W'[n][k]
 * = W[n][k] * gamma[k], done once when the weights are loaded), which makes
 * this equal to W · RMSNorm(x). rms_eps must be finite and >= 0; with
 * rms_eps = 0 an all-zero x row gives non-finite outputs.
 */
#define GEMV_FLAG_RMSNORM 1

/*
 * GEMV_FLAG_STREAMK: batch 1 only (x row of at most 24,576 columns). Run the
 * stream-K kernel ("GPU performance chains", "Wave quantization"; "Decode GEMV
 * at half of HBM bandwidth", cause 1): a grid of exactly one wave; rows that
 * fill whole rounds of its warps go one per warp, the rest are cut into
 * (row, 2,048-column) units shared out in equal, contiguous ranges; a row cut
 * between warps is finished by the last of its warps to arrive, which adds
 * their partial sums in warp order (results are bitwise reproducible; they may
 * differ in the last bits from the default kernel, which cuts K differently).
 * It needs a workspace of 8 bytes per warp of the grid plus 4 bytes per output
 * row. Direct calls use a workspace the library owns per device: it is
 * allocated (cudaMalloc, then zeroed; the call waits for the device) the first
 * time a call needs more than it has, which must not happen while a stream is
 * capturing (GEMV_ERR_CAPTURE), and it is freed by gemv_workspace_release.
 * All direct stream-K calls on one device share it, so they must not run
 * concurrently: issue them on one stream. A plan owns its own workspace.
 * Combined with a batch of more than 1 or a longer x row: GEMV_ERR_UNSUPPORTED.
 */
#define GEMV_FLAG_STREAMK 2

/*
 * GEMV_FLAG_CUDA_CORES: BF16 weights only. Run the CUDA-core kernel (lanes
 * along K, FP32 multiply-adds, B accumulators per row) at every batch size,
 * instead of the BF16 tensor-core kernel the library uses for B >= 2. At
 * B >= 4 on large matrices the CUDA-core kernel is bound by its arithmetic,
 * not by HBM. Not combinable with GEMV_FLAG_STREAMK (GEMV_ERR_INVALID);
 * INT4 and FP8 calls reject it (GEMV_ERR_UNSUPPORTED).
 */
#define GEMV_FLAG_CUDA_CORES 4

typedef struct {
    int flags;
    float rms_eps;
} gemv_options;

/* gemv_bf16 with options (see gemv_options). */
int gemv_bf16_ex(const void *W, const void *x, float *y,
                 int64_t N, int64_t K, int B, int64_t ldw,
                 const gemv_options *opt, void *stream);

/*
 * gemv_bf16_ex for a caller whose activations live in host memory: copies x
 * from x_host (B*K BF16, pinned memory recommended) to the device buffer x_dev,
 * runs the GEMV, brings y to y_host (B*N floats) and waits for the stream, so
 * y_host holds the result on return. When y is at most 256 KB and y_host is
 * pinned memory mapped into the device's address space (cudaHostAlloc / pinned
 * tensors under unified addressing, or cudaHostRegister with the mapped flag)
 * the kernel stores y straight into it and y_dev is not used; otherwise the
 * GEMV writes y_dev and a device-to-host copy follows. The wait polls the stream for up to a
 * millisecond before it blocks. The device buffers are the caller's (x_dev B*K
 * BF16, 16-byte aligned; y_dev B*N floats); the library allocates nothing (but
 * the stream-K workspace, see GEMV_FLAG_STREAMK). This is the whole
 * host-to-host path of one decode-step projection, timed end to end by the
 * benchmark. Returns GEMV_ERR_CAPTURE on a capturing stream (the call waits for
 * its stream).
 */
int gemv_bf16_host_io(const void *W, const void *x_host, float *y_host,
                      void *x_dev, float *y_dev,
                      int64_t N, int64_t K, int B, int64_t ldw,
                      const gemv_options *opt, void *stream);

/*
 * One weight matrix of a fused launch: y_i = W_i · x, W_i [N_i, ldw_i], y_i
 * [B, N_i] (row stride N_i).
 */
typedef struct {
    const void *W;
    float *y;
    int64_t N;
    int64_t ldw;
} gemv_segment;

/*
 * Several projections that share x, in ONE launch ("Decode GEMV at half of HBM
 * bandwidth", "A strong answer", cause 3: fuse Q, K and V into one 6,144-row
 * projection, and gate with up, so that launch gaps do not rival the few
 * microseconds a small matrix takes to stream). segs holds 1..GEMV_MAX_SEGMENTS
 * host-side descriptors (read during the call only); each segment obeys the
 * same rules as gemv_bf16 with the common x, K and B. The sum of N_i must not
 * exceed 2^31-1. Each y_i is computed exactly as a separate gemv_bf16 on the
 * concatenated rows would compute it.
 */
int gemv_bf16_multi(const gemv_segment *segs, int nsegs, const void *x,
                    int64_t K, int B, void *stream);

/* gemv_bf16_multi with options; the options apply to every segment (one x). */
int gemv_bf16_multi_ex(const gemv_segment *segs, int nsegs, const void *x,
                       int64_t K, int B, const gemv_options *opt, void *stream);

/*
 * gemv_bf16_multi_ex for a caller whose activations live in host memory (the
 * end-to-end path of a fused projection, "How to optimize an ML kernel that
 * underutilizes the GPU", Step 5: compare the end-to-end time with the
 * kernel's): copies x from x_host (B*K BF16, pinned memory recommended) to the
 * device buffer x_dev (B*K BF16), runs the fused launch over segs (their y are
 * device buffers, as for gemv_bf16_multi_ex), copies each segment's y to the
 * host buffer y_host[i] (B*N_i floats) and waits for the stream, so the host
 * buffers hold the results on return. The wait polls the stream for up to a
 * millisecond before it blocks. Allocates nothing. Returns GEMV_ERR_CAPTURE on
 * a capturing stream (the call waits for its stream).
 */
int gemv_bf16_multi_host_io(const gemv_segment *segs, int nsegs, const void *x_host, void *x_dev,
                            float *const *y_host, int64_t K, int B, const gemv_options *opt,
                            void *stream);

/*
 * One projection of a decode step. Projections with the same fuse_group > 0,
 * the same x, K, B, flags, rms_eps and weight kind, that are adjacent in the
 * list, become one fused launch (at most GEMV_MAX_SEGMENTS per launch);
 * fuse_group 0 means "alone". flags and rms_eps are those of gemv_options.
 * weight_kind selects the weight format, with the layouts and preconditions
 * of the single-matrix calls:
 *   GEMV_WEIGHT_BF16 (0): W BF16 [N, ldw] (gemv_bf16_ex); S and lds unused.
 *   GEMV_WEIGHT_INT4 (1): W the codes [N, ldw bytes], S the BF16 group scales
 *                         [N, lds] (gemv_w4_bf16, ldw = ldq).
 *   GEMV_WEIGHT_FP8  (2): W the E4M3 codes [N, ldw bytes], S the FP32 row
 *                         scales [N] (gemv_fp8_bf16, ldw = ldq); lds unused.
 * Quantised kinds take no GEMV_FLAG_STREAMK or GEMV_FLAG_CUDA_CORES.
 */
#define GEMV_WEIGHT_BF16 0
#define GEMV_WEIGHT_INT4 1
#define GEMV_WEIGHT_FP8 2

typedef struct {
    const void *W;
    const void *x;
    float *y;
    int64_t N;
    int64_t K;
    int64_t ldw;
    int B;
    int fuse_group;
    int flags;
    float rms_eps;
    int weight_kind;
    const void *S;
    int64_t lds;
} gemv_proj;

typedef struct gemv_plan gemv_plan;   /* opaque; owned by the library */

/*
 * Build a decode-step plan over nproj projections, launched in list order
 * ("GPU performance chains", "Launch gaps in a decode step": many small gaps
 * between kernels call for CUDA graphs). The projection list is copied; every
 * pointer in it must stay valid while the plan is used. Validates every
 * projection as gemv_bf16 would. On success *out owns a plan to be released
 * with gemv_plan_destroy. Allocates host memory only.
 */
int gemv_plan_create(const gemv_proj *projs, int nproj, gemv_plan **out);

/*
 * Record the plan's launches on `stream` (which must not be the legacy NULL
 * stream and must not already be capturing) into a CUDA graph and instantiate
 * it. Nothing executes. Calling it again replaces the previous graph.
 */
int gemv_plan_capture(gemv_plan *plan, void *stream);

/*
 * Run the whole captured step as one graph launch on `stream`. Inputs are read
 * at the addresses given at create time, so callers update x in place between
 * launches. Returns GEMV_ERR_UNSUPPORTED if the plan was never captured.
 */
int gemv_plan_launch(gemv_plan *plan, void *stream);

/*
 * A decode step from host to host ("GPU performance chains", "Launch gaps in
 * a decode step": the step's time is what the caller waits for, gaps and
 * copies included): copies x_bytes from x_host to x_dev, launches the captured
 * plan, copies y_bytes from y_dev to y_host and waits for the stream, so
 * y_host holds the step's outputs on return. The caller lays the plan's
 * activation vectors out in one device buffer (x_dev) and its outputs in
 * another (y_dev), so that each direction is one copy; x_bytes or y_bytes may
 * be 0 (no copy, pointers then unused). Pinned host buffers are recommended.
 * The wait polls the stream for up to a millisecond before it blocks.
 * Returns GEMV_ERR_UNSUPPORTED if the plan was never captured,
 * GEMV_ERR_CAPTURE on a capturing stream. Allocates nothing.
 */
int gemv_plan_launch_host_io(gemv_plan *plan, const void *x_host, void *x_dev, int64_t x_bytes,
                             const void *y_dev, void *y_host, int64_t y_bytes, void *stream);

/* Number of kernel launches one gemv_plan_launch performs (after fusion). */
int gemv_plan_num_launches(const gemv_plan *plan);

/*
 * 1 if the plan's launches are independent, 0 if not (or plan is NULL).
 * gemv_plan_create compares the device byte ranges every projection reads (x,
 * W, the scales) and writes (y): when no launch writes memory that another
 * launch of the plan reads or writes, and no launch uses the stream-K option
 * (whose launches share the plan's workspace), the launches do not wait for
 * the preceding grid before they touch x and y, so each one's start overlaps
 * its predecessor's end ("GPU performance chains", "Launch gaps in a decode
 * step"). The graph as a whole still starts after the work before it on the
 * stream and ends before the work after it. A plan with any such overlap keeps
 * every wait. In an independent plan of two or more launches, the batch-1
 * launches are also planned to run alongside their neighbours rather than to
 * fill the GPU alone: each asks for one streaming warp per SM, so K is split
 * only for very few rows, and the INT4 and FP8 kernels take their standard
 * instance. Results stay within the same tolerance (partial sums combine in a
 * fixed order either way; the bits may differ from a direct call of the same
 * projection, which may split K). Setting GEMV_FORCE_VARIANT=planwait=1
 * before gemv_plan_create keeps the waits (and the single-launch planning) in
 * any plan, for comparison.
 */
int gemv_plan_independent(const gemv_plan *plan);

/* Release a plan and its graph. NULL is ignored. Not while a launch runs. */
void gemv_plan_destroy(gemv_plan *plan);

/*
 * How a shape is launched, for tests and the benchmark. Pure host arithmetic;
 * makes no CUDA call. sm_count is the GPU's SM count (152 on a GB300).
 */
typedef struct {
    int64_t rows_per_cta;    /* output rows one CTA produces                      */
    int64_t row_tiles;       /* ceil(N / rows_per_cta), per fused launch summed   */
    int64_t grid;            /* CTAs launched = row_tiles * splits (rounded up to
                                whole clusters of mcast CTAs when mcast > 1)      */
    int64_t kslice;          /* columns per K-split (all but the last)            */
    int64_t kchunk;          /* columns of x staged in shared memory at a time    */
    int32_t warps_per_cta;
    int32_t warps_per_row;   /* warps of one CTA that share a row group along K   */
    int32_t splits;          /* CTAs along K (one thread-block cluster)           */
    int32_t rows_per_warp;   /* rows one warp streams together (16: tensor-core tile) */
    int32_t unroll;          /* loads per lane per row in flight before any is used */
    int32_t smem_bytes;      /* dynamic shared memory per CTA                     */
    int32_t path;            /* 0: CUDA-core FP32 FMA (batch 1), 1: BF16 tensor-core MMA,
                                2: INT4 weights on the BF16 tensor cores,
                                3: stream-K, batch 1 (CUDA cores, one-wave grid),
                                4: FP8 weights on the BF16 tensor cores,
                                5: BF16, 9..16 rows of x (8 on matrices of at least
                                16,384 rows): tcgen05 MMAs with the accumulator in
                                tensor memory, W and x streamed through a
                                shared-memory ring by tensor copies (calls with one
                                or more weight matrices in this GPU's memory and x
                                16-byte aligned there, K a multiple of 8, no
                                RMSNorm prologue; 128-row tiles, warps_per_cta 8) */
    int32_t xstride;         /* shared-memory elements per staged x row           */
    int32_t nbuf;            /* x buffers: 2 when the K-range is staged in chunks */
    /* stream-K (path 3) only; zero otherwise: */
    int64_t units;           /* (row, 2,048-column) units of the split part       */
    int64_t warps;           /* warps that take split-part units (equal ranges)   */
    int32_t chunks;          /* units per row                                     */
    int32_t ctas_per_sm;     /* resident CTAs per SM the one-wave grid assumes    */
    int32_t dp_rounds;       /* rounds of whole rows, one per warp of the grid,
                                taken before the split part                       */
    int32_t mcast;           /* path 0, batch 1, no K split, x in one chunk: CTAs
                                of a cluster along the rows that share one
                                multicast copy of x (CTA rank 0 copies x once
                                into all of their shared memory with the
                                Tensor Memory Accelerator); 1: each CTA copies
                                its own. A call whose x is not 16-byte aligned
                                falls back to 1                                   */
    int32_t xbox;            /* path 1, B > 8, x in one chunk, K a multiple of
                                32: x is copied by the Tensor Memory Accelerator
                                as tensor boxes of 8 MMA blocks (256 columns) of
                                all B rows, in pieces each counted on its own
                                mbarrier (1: narrow boxes, landing block-major;
                                2: wide boxes, landing row-major); 0: one bulk
                                copy per x row (K a multiple of 8) or 16-byte
                                copies from every thread. A call whose x is not
                                16-byte aligned memory of this GPU, or that has
                                the RMSNorm prologue, falls back to 0 (and
                                smem_bytes to that of the row layout)             */
    int32_t xpieces;         /* xbox > 0: pieces per warp group along K           */
    int32_t xboxes_per_piece;/* xbox > 0: boxes per piece                         */
    int32_t persistent;      /* path 5: 1 when the grid (fewer CTAs than row
                                tiles) takes the tiles in turn, each CTA an equal
                                share, over the whole K (splits == 1)             */
    int32_t l2_prefetch;     /* paths 0 and 2: batches of W (unroll loads per
                                lane each) that every warp asks the L2 for ahead
                                of the batch in its registers, by the Tensor
                                Memory Accelerator's bulk prefetch; path 5 (one
                                wave): ring stages of W prefetched beyond the
                                ring; 0: none. A call with W outside this GPU's
                                memory falls back to 0, and the launches of a
                                plan (gemv_plan_create) take 0 unless the
                                GEMV_FORCE_VARIANT sweep knob sets l2pf           */
} gemv_launch_info;

int gemv_query_launch(int64_t N, int64_t K, int B, int sm_count,
                      gemv_launch_info *out);

/* gemv_query_launch for a call with option flags (GEMV_FLAG_STREAMK selects
 * path 3, GEMV_ERR_UNSUPPORTED where that kernel does not apply;
 * GEMV_FLAG_CUDA_CORES selects path 0 at every batch size). */
int gemv_query_launch_ex(int64_t N, int64_t K, int B, int sm_count, int flags,
                         gemv_launch_info *out);

/* Free the stream-K workspace the library holds for the current device. No
 * stream-K call on that device may be in flight. Returns GEMV_OK. */
int gemv_workspace_release(void);

/*
 * Status bits the kernels recorded on the current device since the last reset:
 * GEMV_STATUS_WAIT_TIMEOUT means a kernel gave up waiting for a copy of x into
 * shared memory (an mbarrier wait has an iteration limit instead of spinning
 * forever); the CTAs that gave up store NaN in place of their outputs, so a
 * timed-out launch never returns plausible numbers. The calls themselves still
 * return GEMV_OK (the wait happens on the device, after the call): a caller
 * that must know reads the bits after synchronizing. Writes the bits to
 * *bits and clears them when reset != 0. Synchronous with respect to the
 * device's work (like cudaMemcpyFromSymbol). Returns GEMV_OK, GEMV_ERR_INVALID
 * for a NULL pointer, or GEMV_ERR_CUDA.
 */
#define GEMV_STATUS_WAIT_TIMEOUT 1u
int gemv_device_status(unsigned int *bits, int reset);

/*
 * Test support, not part of the method. In a library built with
 * -DGEMV_DEBUG_WRITECOUNT every kernel store to an output element also adds 1
 * to counts[element - y_base], or to counts[n] for a store outside
 * [y_base, y_base + n), for every launch prepared (or plan created) after the
 * call; counts = NULL turns it off. counts: n + 1 int32 on the device, zeroed
 * by the caller. It checks that each output is written exactly once and
 * nothing else is. Other builds return GEMV_ERR_UNSUPPORTED and never count.
 * Not thread-safe.
 */
int gemv_debug_write_count(int32_t *counts, const float *y_base, int64_t n);

/*
 * gemv_bf16_ex with GEMV_FLAG_STREAMK for callers that must not allocate
 * device memory: the same stream-K kernel (batch 1, same results bit for bit),
 * with its partial sums and per-row counters in a fixed scratch area compiled
 * into the library (80 KB of device memory per device, zero when the library
 * is loaded, left at zero by every launch) instead of the workspace the
 * library would allocate. The pages have no counterpart to this call; it
 * exists for callers in which a cudaMalloc is not allowed or not wanted: a
 * serving loop that has fixed its memory footprint at start-up, code that runs
 * under another allocator's control (an out-of-memory handler, a caching
 * allocator's own callbacks), or work that must not wait for the device
 * synchronization an allocation implies.
 *   - Same arguments as gemv_bf16_ex with B = 1 (opt may set
 *     GEMV_FLAG_RMSNORM; GEMV_FLAG_STREAMK is implied). y[n] for n < N.
 *   - Capacity: the split part of the launch (the rows left over after whole
 *     rounds of one row per warp; on a 152-SM GB300 N mod 4,864 when K is a
 *     multiple of 2,048, else N mod 3,648, and N itself when N is smaller)
 *     must need at most 4,096 row counters, and the grid at most 8,192 warps.
 *     A larger shape returns GEMV_ERR_UNSUPPORTED before any launch, as do a
 *     batch above 1 and an x row longer than 24,576 columns.
 *   - The first call on a device looks up the scratch's device address (with
 *     that device current) and sets the library's kernels up on the device;
 *     make that first call before any stream capture.
 *   - All calls on one device share the one scratch area: calls whose
 *     launches overlap (on different streams, or from several threads without
 *     ordering) race on it and give undefined results. Issue them on one
 *     stream, or order them. Its scratch is separate from the workspace of
 *     GEMV_FLAG_STREAMK calls and of plans, so those may overlap with it.
 */
int gemv_bf16_streamk_noalloc(const void *W, const void *x, float *y,
                              int64_t N, int64_t K, int64_t ldw,
                              const gemv_options *opt, void *stream);

/*
 * y = W·x with group-quantised INT4 weights ("Decode GEMV at half of HBM
 * bandwidth", "What interviewers probe next": with INT4 weights the bytes fall
 * four times; the codes are unpacked in registers while the next loads are in
 * flight). Element (n, k) of W is (u - 8) * S[n][k / 128], u the 4-bit code:
 *   Wq : N rows of ldq bytes (ldq >= K/2, ldq % 16 == 0, Wq 16-byte aligned).
 *        Row n, little-endian 32-bit word w (bytes 4w..4w+3) holds the codes of
 *        k = 8w..8w+7: k = 8w + 2j in bits 4j..4j+3 and k = 8w + 2j + 1 in bits
 *        16+4j..16+4j+3 (j = 0..3), i.e. even k in the low half-word and odd k
 *        in the high half-word.
 *   S  : N rows of lds BF16 scales (lds >= K/128), S[n][g] for k in
 *        [128 g, 128 g + 128).
 *   x, y, B and the options as for gemv_bf16_ex; K must be a multiple of 128.
 * The contraction runs on the BF16 tensor cores with FP32 accumulation for
 * every B (dequantised codes are exact in BF16; each 128-column group is summed
 * and then scaled). Accuracy bound and tolerance as for gemv_bf16, with
 * |W[n][k]| = |u - 8| * S[n][k/128].
 */
int gemv_w4_bf16(const void *Wq, const void *S, const void *x, float *y,
                 int64_t N, int64_t K, int B, int64_t ldq, int64_t lds,
                 const gemv_options *opt, void *stream);

/* gemv_query_launch for the INT4-weight GEMV (K a multiple of 128). */
int gemv_w4_query_launch(int64_t N, int64_t K, int B, int sm_count,
                         gemv_launch_info *out);

/*
 * y = W·x with FP8 weights ("Decode GEMV at half of HBM bandwidth", "What
 * interviewers probe next": INT4, then FP8 weights). Element (n, k) of W is
 * e4m3(Wq[n][k]) * S[n]:
 *   Wq : N rows of ldq bytes (ldq >= K, ldq % 16 == 0, Wq 16-byte aligned),
 *        one E4M3 code per weight: sign in bit 7, exponent bits 3..6 with bias
 *        7, mantissa bits 0..2, subnormals at exponent 0. The two NaN codes
 *        (0x7F, 0xFF) must not occur in columns k < K (the kernel reads them
 *        as 480); columns k >= K are never read.
 *   S  : N FP32 scales, one per output row (4-byte aligned).
 *   x, y, B and the options as for gemv_bf16_ex; K must be a multiple of 64.
 * The codes are widened to BF16 exactly in registers and contracted on the
 * BF16 tensor cores with FP32 accumulation for every B; each row's sum is
 * multiplied by S[n] once at the end. Accuracy bound and tolerance as for
 * gemv_bf16, with |W[n][k]| = |e4m3(Wq[n][k])| * S[n].
 */
int gemv_fp8_bf16(const void *Wq, const float *S, const void *x, float *y,
                  int64_t N, int64_t K, int B, int64_t ldq,
                  const gemv_options *opt, void *stream);

/* gemv_query_launch for the FP8-weight GEMV (K a multiple of 64). */
int gemv_fp8_query_launch(int64_t N, int64_t K, int B, int sm_count,
                          gemv_launch_info *out);

/*
 * Read-only bandwidth probe: streams `bytes` (a multiple of 16, >= 16) from the
 * 16-byte aligned device buffer `src` with the same 16-byte non-allocating
 * loads as the GEMV and writes one checksum word per CTA to `sink` (at least
 * gemv_probe_sink_words() floats). It measures the read-only HBM ceiling the
 * GEMV is held to ("How to optimize an ML kernel that underutilizes the GPU",
 * Step 5: compare achieved bandwidth with peak).
 */
int gemv_probe_stream_read(const void *src, int64_t bytes, float *sink, void *stream);
int gemv_probe_sink_words(void);

/* Human-readable name of a status code. Never NULL. */
const char *gemv_status_string(int status);

/* The cudaError_t behind the calling thread's most recent GEMV_ERR_CUDA (0 if none). */
int gemv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMV_H */
