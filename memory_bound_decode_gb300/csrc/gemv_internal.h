// Internal declarations shared by the kernel translation units and the C-ABI
// front end. Not installed; the public interface is include/gemv.h.
#pragma once

#include <cstdint>
#include <cuda.h>   // CUtensorMap (the type only; the library calls no driver API directly)
#include <cuda_runtime.h>

namespace gemv {

constexpr int kWarps = 8;                 // warps per CTA
constexpr int kThreads = kWarps * 32;     // threads per CTA
constexpr int kMaxSegs = 8;               // segments of one fused launch
constexpr int kMaxBatch = 16;
constexpr int kMaxSplits = 8;             // CTAs along K: one portable cluster

// One weight matrix of a launch. Row tiles of all segments are numbered
// consecutively; tile_begin is the first tile of this segment.
struct Seg {
    const uint16_t* W;     // BF16 weights, or packed INT4 codes (then ldw is in bytes)
    float* y;
    int64_t N;
    int64_t ldw;
    int64_t tile_begin;
    const uint16_t* S;     // INT4 weights: BF16 group scales [N, lds]; unused otherwise
    int64_t lds;
    const float* rs;       // FP8 weights: FP32 row scales [N]; unused otherwise
};

// Test support: where a build with GEMV_DEBUG_WRITECOUNT counts output
// stores (counts[element - base], counts[n] for a store outside [base, base + n)).
// Null counts: no counting. Other builds never read it.
struct WriteCount {
    int32_t* counts;
    const float* base;
    int64_t n;
};

// Everything one launch needs; passed by value as a __grid_constant__.
struct Params {
    Seg seg[kMaxSegs];
    const uint16_t* x;
    int64_t K;
    int64_t kslice;   // columns per K-split (multiple of the warp batch width)
    int64_t kchunk;   // columns of x staged in shared memory at a time
    int32_t nseg;
    int32_t splits;   // CTAs per row tile along K (== cluster size when > 1)
    int32_t kw;       // warps of one CTA that share a row group along K (1, 2, 4, 8)
    int32_t xstride;  // shared-memory elements per staged x row (>= kchunk)
    int32_t batch;    // B
    int32_t nbuf;     // x buffers (2 when the K-range takes more than one chunk)
    int32_t flags;    // kFlagRmsNorm, kFlagNoWait
    float rms_eps;    // epsilon of the RMSNorm prologue
    int32_t mcast;    // CUDA-core kernel, batch 1, one K chunk, no K split: CTAs of a cluster along
                      // the rows that share one multicast copy of x (1: every CTA stages its own)
    int32_t xper;     // BF16 tensor-core kernel, x as tensor boxes: pieces per warp group along K
    int32_t xbpp;     // ... and boxes of 8 blocks (256 columns) per piece
    int32_t xwide;    // ... 1: boxes of 256 columns x B rows, 0: of 32 columns x B rows (stage_x_boxes)
    int32_t l2pf;     // CUDA-core and INT4 kernels: batches of W each warp asks the L2 for ahead of
                      // the batch in its registers (bulk prefetch); tcgen05 kernel (one wave): ring
                      // stages of W prefetched beyond the ring (tensor prefetch); W in this GPU's
                      // memory; 0: none
    WriteCount wc;
    CUtensorMap xmap; // ... and the 3-D view of x the boxes are copied through (stage_x_boxes);
                      // path 5: x as [B][K] in boxes of 64 columns x 16 rows
    CUtensorMap wmap[kMaxSegs];   // path 5: each segment's W as [N][ldw] in boxes of 64 columns x 128 rows
};

// The BF16 tensor-core kernel's x, copied as tensor boxes, lands in up to
// kMaxXPieces pieces, each counted on its own mbarrier (see stage_x_boxes).
constexpr int kMaxXPieces = 8;
// Bytes at the start of the multicast instance's dynamic shared memory before
// x: its mbarrier (16 to keep x 16-byte aligned). Planned for every CUDA-core
// launch; the other instances leave them unused.
constexpr int kFmaSmemHead = 16;
// The same for the BF16 tensor-core and FP8 kernels: the mbarriers of their
// copies of x (x starts 128-byte aligned, as a tensor copy needs).
constexpr int kBulkSmemHead = 128;
// Multicast x for batch 1 when the launch has no K split and x is at least
// this many 16-byte vectors, i.e. K >= 8,192 (measured: down_proj, x = 28 KB,
// 18.25 -> 17.94 us with clusters of 2; with x = 8 KB the launches with and
// without it were within noise, so they keep the plain grid).
constexpr int kMcastCtas = 2;
constexpr int kMcastMinVectors = 1024;

// Scale each output row b by (mean_k x[b][k]^2 + rms_eps)^(-1/2) (RMSNorm
// prologue; the norm's elementwise weight is folded into W).
constexpr int32_t kFlagRmsNorm = 1;
// Skip the wait for the preceding grid (programmatic dependent launch): set
// only on the launches of a plan none of whose launches writes memory that
// another of its launches reads or writes, so that neighbouring launches may
// run at the same time (the graph as a whole still starts after, and ends
// before, the stream work around it).
constexpr int32_t kFlagNoWait = 2;

// Shared floats after the partial sums: per-warp sums of squares of x
// [kWarps][kMaxBatch], the CTA's sums [kMaxBatch], the row scales [kMaxBatch]
// and, for a cluster along K, every rank's sums [kMaxSplits][kMaxBatch].
constexpr int kMiscFloats = kWarps * kMaxBatch + 2 * kMaxBatch + kMaxSplits * kMaxBatch;

// Kernel families.
enum Path : int32_t {
    kPathFma = 0,       // CUDA-core FP32 multiply-adds, one warp streams RPW whole rows
    kPathMma = 1,       // BF16 tensor-core mma.sync, one warp streams a 16-row tile
    kPathW4 = 2,        // INT4 weights dequantised to BF16 in registers, tensor-core mma.sync
    kPathStreamK = 3,   // batch 1, one wave of CTAs, warps take balanced ranges of (row, K-unit)
    kPathFp8 = 4,       // FP8 (E4M3) weights widened to BF16 in registers, tensor-core mma.sync
    kPathTc = 5,        // BF16, 2..16 rows of x: W streamed by tensor copies into a shared-memory
                        // ring, tcgen05.mma with the accumulator in tensor memory
};

// The tcgen05 kernel (path 5): a CTA owns 128 weight rows (the MMA's M) and one
// K-range, streamed in stages of 128 columns (two 64-column tensor boxes of W,
// two of x, 128-byte swizzle) through a ring of kTcStages stages; x rows are
// padded to 16 (the MMA's N; rows past B are zero-filled by the copies).
constexpr int kTcRows = 128;
constexpr int kTcN = 16;
constexpr int kTcStageCols = 128;                // stage width unless the tccols knob says otherwise
constexpr int kTcStages = 2;                     // ring depth unless the tcstages knob says otherwise
constexpr int kTcWBox = kTcRows * 64 * 2;        // bytes of one W box (64 columns)
constexpr int kTcXBox = kTcN * 64 * 2;           // bytes of one x box
constexpr int32_t kTcMaxDynSmem = 227 * 1024;

// Weight formats the planner knows.
enum WeightKind : int32_t {
    kWeightBf16 = 0,
    kWeightInt4 = 1,   // 128-column groups, BF16 scales
    kWeightFp8 = 2,    // E4M3 codes, FP32 row scales
    kWeightBf16CudaCores = 3,   // BF16 on the CUDA-core kernel at every batch size
};
constexpr int kW4Group = 128;
constexpr int kW4Unroll = 4;      // 128-column groups in flight per lane (2 x 16 B each)
constexpr int kW4DeepUnroll = 8;  // the deep instance (up to 8 rows of x, one x chunk): 2 CTAs per SM
constexpr int kF8Slot = 64;       // FP8: columns of one slot (4 lanes x 16 codes); K is a multiple
constexpr int kF8Unroll = 4;      // slots in flight per lane (2 x 16 B each)
constexpr int kF8DeepUnroll = 8;  // the deep instance (up to 8 rows of x): 2 CTAs per SM

// Compile-time shape of the CUDA-core kernel instance for batch B.
struct Variant {
    int rows_per_warp;   // rows one warp streams at once
    int unroll;          // 16-byte loads per lane per row issued before any is used
};

constexpr Variant fma_variant(int B) { return B <= 1 ? Variant{1, 8} : Variant{1, 8}; }

// The tensor-core kernel: 16-row tile per warp, n8 blocks of the batch, and
// k32 blocks (two 16-byte loads per lane each) in flight per batch.
constexpr int kMmaRows = 16;
constexpr int kMmaUnroll = 8;
constexpr int mma_nblocks(int B) { return B <= 8 ? 1 : 2; }

// Which family serves batch B.
constexpr Path path_for(int B) { return B == 1 ? kPathFma : kPathMma; }

// Host-side launch decision (see planner.cpp).
struct Launch {
    int64_t rows_per_cta;
    int64_t row_tiles;
    int64_t grid;
    int64_t kslice;
    int64_t kchunk;
    int32_t kw;
    int32_t splits;
    int32_t rows_per_warp;   // rows of one warp's group (RPW, or 16 for the tensor-core path)
    int32_t unroll;
    int32_t smem_bytes;
    int32_t path;
    int32_t xstride;
    int32_t nbuf;
    int32_t mcast;     // CTAs sharing one multicast copy of x (cluster along the rows); 1: none
    int32_t xbulk;     // FP8 path: x copied by bulk copies (one chunk, aligned rows)
    int32_t xbox;      // BF16 tensor-core path: x copied as tensor boxes (one chunk, K % 32 == 0):
                       // 1 narrow boxes (32 columns), 2 wide boxes (256 columns)
    int32_t xper;      // ... pieces per warp group along K
    int32_t xbpp;      // ... boxes of 8 blocks per piece
    int32_t smem_rows; // shared memory of the same launch with x staged row by row (no boxes)
    int32_t stage_cols;// path 5: columns per ring stage (64 or 128); the ring depth is in `unroll`
    int32_t tc_persist;// path 5: the persistent form (a fixed grid taking row tiles in turn, no K split)
    int32_t tc_slots;  // ... CTAs resident at once (the grid takes equal shares of the tiles within them)
    int32_t l2pf;      // W prefetched into L2 ahead (Params::l2pf)
};

// Sweep knob of the planner (GEMV_FORCE_VARIANT planwait=1): every launch of
// a plan waits for the preceding grid even when the plan's launches are
// independent.
bool plan_force_wait();

// Returns 0 and fills `out`, or a negative GEMV_ERR_* code.
// overlap: the launch belongs to an independent plan of several launches
// (see gemv_plan_create), whose neighbours run alongside it.
// allow_tc: the call can take the tcgen05 kernel (one weight matrix, aligned
// operands, no RMSNorm prologue); the rules (or the tc knob) decide whether it does.
// tc_clusters: clusters of 1, 2, 4 and 8 CTAs of the tcgen05 kernel the
// device keeps resident at once (null: not known, no limit assumed).
int plan_launch(int64_t N, int64_t K, int B, int sm_count, Launch* out, int weight_kind = kWeightBf16,
                bool overlap = false, bool allow_tc = false, const int32_t* tc_clusters = nullptr);

// Shared memory of a tcgen05 launch with batch B and a ring of `stages` of
// `stage_cols` columns (the ring, the combine areas, the barriers and 1 KB to
// align the ring to 1,024 bytes), and whether that kernel instance exists.
int64_t tc_smem_bytes(int B, int stages, int stage_cols);
bool tc_has_instance(int stages, int stage_cols);
// Shared memory of the persistent tcgen05 launch with that ring (the ring, its
// barriers, 1 KB of alignment); -1 where no such instance exists.
int64_t tcp_smem_bytes(int stages, int stage_cols);
// Clusters of S CTAs of the tcgen05 kernel the current device keeps resident at
// once (cudaOccupancyMaxActiveClusters); -1 if unknown.
int tc_max_active_clusters(int S);

// Stream-K launch (batch 1): the grid is one wave of GW warps. Rows (of all
// segments, numbered consecutively) that fill whole rounds of GW are taken
// one per warp: row r * GW + w in round r < dp_rounds. The rest, cut into
// units of kSkUnitCols columns and numbered row-major, are split evenly: warp
// w takes units [w * units / warps, (w + 1) * units / warps). A row whose units
// belong to more than one warp is finished by the last of them to arrive
// (per-row counter), which adds the warps' partial sums in warp order.
constexpr int kSkUnroll = 8;                          // 16-byte loads per lane per unit
constexpr int kSkUnitCols = 32 * 8 * kSkUnroll;       // 2,048 columns per unit
constexpr int kSkMaxCtasPerSm = 4;
constexpr int64_t kSkMaxXBytes = 48 * 1024;           // whole x row staged per CTA

struct SkParams {
    Seg seg[kMaxSegs];    // tile_begin holds the segment's first global row
    const uint16_t* x;
    int64_t K;
    int64_t units;        // units of the split part: (rows - dp_rounds * grid warps) * chunks
    int64_t warps;        // warps that take split-part units (<= units, <= grid * kWarps)
    float* part;          // [warps][2] partial sums (a warp's first and last split row)
    int32_t* ticket;      // [split-part rows] arrival counters, zero between launches
    int32_t chunks;       // units per row
    int32_t dp_rounds;    // rounds of whole rows, one per warp of the grid
    int32_t nseg;
    int32_t xstride;      // staged x elements (whole vectors up to K)
    int32_t flags;        // kFlagRmsNorm
    float rms_eps;
    WriteCount wc;
};

struct SkLaunch {
    int64_t grid;         // CTAs (one wave)
    int64_t warps;        // split-part warps
    int64_t units;        // split-part units
    int32_t dp_rounds;
    int32_t chunks;
    int32_t smem_bytes;
    int32_t ctas_per_sm;
    int32_t xstride;
    int64_t part_floats;  // workspace the launch needs
    int64_t tickets;
};

// Capacity of the fixed scratch of gemv_bf16_streamk_noalloc (gemv_noalloc.cu):
// partial sums for 8,192 warps (a one-wave grid of up to 256 SMs x 4 CTAs x 8
// warps) and counters for 4,096 split-part rows. 80 KB of device memory.
constexpr int64_t kNoallocPartFloats = 2 * 8192;
constexpr int64_t kNoallocTickets = 4096;
// Device addresses of that scratch for the current device.
cudaError_t noalloc_scratch(float** part, int32_t** ticket);

// Returns 0 and fills `out`, or a negative GEMV_ERR_* code (GEMV_ERR_UNSUPPORTED
// when the shape does not fit the stream-K kernel: B > 1 or x too large).
int plan_streamk(int64_t rows, int64_t K, int B, int sm_count, SkLaunch* out);
// Whether the planner prefers the stream-K kernel for this batch-1 shape.
bool prefer_streamk(int64_t rows, int64_t K, int B, int sm_count);

// Largest dynamic shared memory any plan requests (set as the kernel attribute).
constexpr int32_t kMaxDynSmem = 112 * 1024;

// Kernel launchers, defined in the kernel translation units.
cudaError_t launch_gemv(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t launch_streamk(const SkParams& p, const SkLaunch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_streamk();
cudaError_t prepare_kernels(int device);   // per-device function attributes
// Status bits the CUDA-core kernels' translation unit recorded on the current
// device (kStatusWaitTimeout...), cleared when `reset`.
cudaError_t read_fma_status(unsigned int* bits, bool reset);
cudaError_t read_mma_status_nb1(unsigned int* bits, bool reset);
cudaError_t read_mma_status_nb2(unsigned int* bits, bool reset);
cudaError_t read_fp8_status(unsigned int* bits, bool reset);
cudaError_t read_tc_status(unsigned int* bits, bool reset);
cudaError_t launch_probe_read(const void* src, int64_t bytes, float* sink, int grid,
                              cudaStream_t s);

}  // namespace gemv
