// C-ABI front end of libgemv.so: argument checks, per-device set-up, fused
// launches and the CUDA-graph decode-step plan. Every operation on data runs
// in the kernels; this file only validates, plans and launches.
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/gemv.h"
#include "gemv_internal.h"

using gemv::Launch;
using gemv::Params;

namespace gemv {
// Whether the sweep knob GEMV_FORCE_VARIANT l2pf=<n> is set (planner.cpp):
// plans then keep the planner's L2 prefetch depth instead of turning it off.
bool l2pf_forced();
}  // namespace gemv

namespace {

thread_local int g_last_cuda_error = 0;

// Output-store counting for tests (gemv_debug_write_count); copied into every
// launch prepared while set. Only a build with GEMV_DEBUG_WRITECOUNT sets it.
gemv::WriteCount g_write_count = {nullptr, nullptr, 0};

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return GEMV_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

// Device memory of the stream-K kernel: partial sums and per-row counters
// (zero between launches).
struct Workspace {
    float* part = nullptr;
    int32_t* ticket = nullptr;
    int64_t part_cap = 0;
    int64_t ticket_cap = 0;
};

struct DeviceState {
    bool ready = false;
    int status = GEMV_OK;
    int sm_count = 0;
    int32_t tc_clusters[4] = {-1, -1, -1, -1};   // resident clusters of 1, 2, 4, 8 tcgen05 CTAs
    Workspace ws;   // shared by direct stream-K calls on this device
};

std::mutex g_dev_mutex;
DeviceState g_dev[kMaxDevices];

// Per-device set-up on first use: check for an sm_103 device, read the SM
// count and raise the kernels' dynamic shared-memory limit.
int device_state(int* sm_count) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e);
        if (major != 10 || minor != 3) {
            st.status = GEMV_ERR_UNSUPPORTED;
        } else if ((e = gemv::prepare_kernels(dev)) != cudaSuccess) {
            return cuda_fail(e);
        } else {
            st.status = GEMV_OK;
            for (int i = 0; i < 4; ++i) st.tc_clusters[i] = gemv::tc_max_active_clusters(1 << i);
        }
        st.sm_count = sms;
        st.ready = true;
    }
    *sm_count = st.sm_count;
    return st.status;
}

// The current device's resident-cluster counts for the tcgen05 kernel (set
// once by device_state, read-only afterwards); null if the device is unknown.
const int32_t* current_tc_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    const DeviceState& st = g_dev[dev];
    return st.ready ? st.tc_clusters : nullptr;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("GEMV_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}

// Largest y that gemv_bf16_host_io stores straight into mapped host memory.
constexpr size_t kMappedYMaxBytes = 256 * 1024;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// cuTensorMapEncodeTiled, looked up once through the runtime (the library
// links no driver library of its own); null where the driver lacks it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<EncodeTiledFn>(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// The 3-D view of x [B][K] that the tensor-core kernel copies tensor boxes
// through. Narrow (K a multiple of 32): 32 columns x B rows x K / 32 blocks
// (row stride 2K bytes, block stride 64 bytes), boxes of 32 x B x 8 bpp. Wide
// (K a multiple of 256): 256 columns x B rows x K / 256, boxes of
// 256 x B x bpp. Zero fill past the end. False if the driver rejects it.
bool encode_x_boxes(CUtensorMap* map, const void* x, int64_t K, int B, int bpp, bool wide) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const int64_t w = wide ? 256 : 32;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(w), static_cast<cuuint64_t>(B),
                                static_cast<cuuint64_t>(K / w)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(w) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(w), static_cast<cuuint32_t>(B),
                               static_cast<cuuint32_t>(wide ? bpp : 8 * bpp)};
    const cuuint32_t elem[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tcgen05 kernel's 2-D views: W [N][ldw] in boxes of 64 columns x 128 rows
// and x [B][K] in boxes of 64 columns x 16 rows, both with the 128-byte
// swizzle its shared-memory descriptors expect; columns past K and rows past N
// (W) or B (x) are zero-filled. False if the driver rejects the view.
bool encode_tc_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int64_t ld, int box_rows) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint32_t elem[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t stride[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, stride, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether p points into device memory of the current device: the x multicast
// and the tensor copies of x read from there only (a pointer into mapped host
// or managed memory takes the per-CTA staging instead).
bool on_current_device(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

int check_common(const void* x, int64_t K, int B) {
    if (!x) return GEMV_ERR_INVALID;
    if (K < 1 || K > 0x7fffffffLL || B < 1 || B > GEMV_MAX_BATCH) return GEMV_ERR_INVALID;
    if (!aligned(x, 2)) return GEMV_ERR_ALIGN;
    return GEMV_OK;
}

int check_matrix(const void* W, const float* y, int64_t N, int64_t K, int64_t ldw) {
    if (!W || !y) return GEMV_ERR_INVALID;
    if (N < 1 || N > 0x7fffffffLL || ldw < K) return GEMV_ERR_INVALID;
    if (ldw % 8 != 0 || !aligned(W, 16) || !aligned(y, 4)) return GEMV_ERR_ALIGN;
    return GEMV_OK;
}

int check_options(const gemv_options* opt, int* flags, float* eps) {
    *flags = 0;
    *eps = 0.f;
    if (!opt) return GEMV_OK;
    if (opt->flags & ~(GEMV_FLAG_RMSNORM | GEMV_FLAG_STREAMK | GEMV_FLAG_CUDA_CORES)) return GEMV_ERR_INVALID;
    if ((opt->flags & GEMV_FLAG_STREAMK) && (opt->flags & GEMV_FLAG_CUDA_CORES)) return GEMV_ERR_INVALID;
    if (opt->flags & GEMV_FLAG_RMSNORM) {
        if (!std::isfinite(opt->rms_eps) || opt->rms_eps < 0.f) return GEMV_ERR_INVALID;
        *eps = opt->rms_eps;
    }
    *flags = opt->flags;
    return GEMV_OK;
}

// One prepared launch: parameters plus grid shape (one of the two kinds).
struct Prepared {
    Params p;
    Launch l;
    int B;
    bool sk = false;
    gemv::SkParams skp;
    gemv::SkLaunch skl;
};

void ws_free(Workspace& ws) {
    if (ws.part) cudaFree(ws.part);
    if (ws.ticket) cudaFree(ws.ticket);
    ws = Workspace{};
}

// Make ws hold at least part_floats partial sums and `tickets` zeroed counters.
// Growing waits for the device (the old buffers may still be in use) and is
// refused while `s` is capturing.
int ws_reserve(Workspace& ws, int64_t part_floats, int64_t tickets, cudaStream_t s) {
    if (ws.part_cap >= part_floats && ws.ticket_cap >= tickets) return GEMV_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cs != cudaStreamCaptureStatusNone) return GEMV_ERR_CAPTURE;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
    const int64_t np = part_floats > ws.part_cap ? part_floats : ws.part_cap;
    const int64_t nt = tickets > ws.ticket_cap ? tickets : ws.ticket_cap;
    ws_free(ws);
    if (cudaMalloc(&ws.part, static_cast<size_t>(np) * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&ws.ticket, static_cast<size_t>(nt) * sizeof(int32_t)) != cudaSuccess) {
        cudaGetLastError();
        ws_free(ws);
        return GEMV_ERR_NOMEM;
    }
    if ((e = cudaMemset(ws.ticket, 0, static_cast<size_t>(nt) * sizeof(int32_t))) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess) {
        ws_free(ws);
        return cuda_fail(e);
    }
    ws.part_cap = np;
    ws.ticket_cap = nt;
    return GEMV_OK;
}

// Stream-K launch over the segments (batch 1; see gemv_streamk_kernel.cuh).
int prepare_streamk(const gemv_segment* segs, int nsegs, int64_t total, const void* x, int64_t K, int flags,
                    float eps, int sm_count, Prepared* out) {
    gemv::SkLaunch l;
    int rc = gemv::plan_streamk(total, K, 1, sm_count, &l);
    if (rc != GEMV_OK) return rc;
    gemv::SkParams p;
    std::memset(&p, 0, sizeof p);
    int64_t row = 0;
    for (int i = 0; i < nsegs; ++i) {
        p.seg[i].W = static_cast<const uint16_t*>(segs[i].W);
        p.seg[i].y = segs[i].y;
        p.seg[i].N = segs[i].N;
        p.seg[i].ldw = segs[i].ldw;
        p.seg[i].tile_begin = row;
        row += segs[i].N;
    }
    p.x = static_cast<const uint16_t*>(x);
    p.K = K;
    p.units = l.units;
    p.warps = l.warps;
    p.chunks = l.chunks;
    p.dp_rounds = l.dp_rounds;
    p.nseg = nsegs;
    p.xstride = l.xstride;
    p.flags = (flags & GEMV_FLAG_RMSNORM) ? gemv::kFlagRmsNorm : 0;
    p.rms_eps = eps;
    p.wc = g_write_count;
    out->sk = true;
    out->skp = p;
    out->skl = l;
    out->B = 1;
    return GEMV_OK;
}

// Validate a group of segments sharing x, K, B and plan one launch over them.
int prepare(const gemv_segment* segs, int nsegs, const void* x, int64_t K, int B, int flags, float eps,
            int sm_count, Prepared* out, bool overlap = false) {
    if (!segs || nsegs < 1 || nsegs > GEMV_MAX_SEGMENTS) return GEMV_ERR_INVALID;
    int rc = check_common(x, K, B);
    if (rc != GEMV_OK) return rc;
    int64_t total = 0;
    for (int i = 0; i < nsegs; ++i) {
        if ((rc = check_matrix(segs[i].W, segs[i].y, segs[i].N, K, segs[i].ldw)) != GEMV_OK) return rc;
        total += segs[i].N;
        if (total > 0x7fffffffLL) return GEMV_ERR_INVALID;
    }
    if (flags & GEMV_FLAG_STREAMK) {
        if (B != 1) return GEMV_ERR_UNSUPPORTED;
        return prepare_streamk(segs, nsegs, total, x, K, flags, eps, sm_count, out);
    }
    if (B == 1 && gemv::prefer_streamk(total, K, B, sm_count) &&
        prepare_streamk(segs, nsegs, total, x, K, flags, eps, sm_count, out) == GEMV_OK)
        return GEMV_OK;
    Launch l;
    const int kind = (flags & GEMV_FLAG_CUDA_CORES) ? gemv::kWeightBf16CudaCores : gemv::kWeightBf16;
    // The tcgen05 kernel takes calls without the RMSNorm prologue, with W and x
    // in this GPU's memory (its tensor copies read from there only) and x rows
    // of whole 16-byte vectors.
    bool allow_tc = B >= 2 && kind == gemv::kWeightBf16 && !(flags & GEMV_FLAG_RMSNORM) && K % 8 == 0 &&
                    aligned(x, 16) && on_current_device(x);
    for (int i = 0; allow_tc && i < nsegs; ++i) allow_tc = on_current_device(segs[i].W);
    if ((rc = gemv::plan_launch(total, K, B, sm_count, &l, kind, overlap, allow_tc, current_tc_clusters())) !=
        GEMV_OK)
        return rc;

    Params p;
    std::memset(&p, 0, sizeof p);
    if (l.path == gemv::kPathTc) {
        bool ok = encode_tc_map(&p.xmap, x, K, B, K, gemv::kTcN);
        for (int i = 0; ok && i < nsegs; ++i)
            ok = encode_tc_map(&p.wmap[i], segs[i].W, K, segs[i].N, segs[i].ldw, gemv::kTcRows);
        if (!ok && (rc = gemv::plan_launch(total, K, B, sm_count, &l, kind, overlap, false)) != GEMV_OK) return rc;
    }
    int64_t tiles = 0;
    for (int i = 0; i < nsegs; ++i) {
        p.seg[i].W = static_cast<const uint16_t*>(segs[i].W);
        p.seg[i].y = segs[i].y;
        p.seg[i].N = segs[i].N;
        p.seg[i].ldw = segs[i].ldw;
        p.seg[i].tile_begin = tiles;
        tiles += (segs[i].N + l.rows_per_cta - 1) / l.rows_per_cta;
    }
    l.row_tiles = tiles;
    // The bulk copy reads x from a 16-byte boundary, and only from this GPU's memory.
    if (l.mcast > 1 && (!aligned(x, 16) || !on_current_device(x))) l.mcast = 1;
    // The tensor copies of x read from a 16-byte boundary, and only from this
    // GPU's memory; the RMSNorm statistic reads x staged row by row.
    if (l.xbox && ((flags & GEMV_FLAG_RMSNORM) || !aligned(x, 16) || !on_current_device(x) ||
                   !encode_x_boxes(&p.xmap, x, K, B, l.xbpp, l.xbox == 2))) {
        l.xbox = 0;
        l.smem_bytes = l.smem_rows;
    }
    // The bulk copies of x read from a 16-byte boundary, and only from this GPU's memory.
    if (l.xbulk && (!aligned(x, 16) || !on_current_device(x))) l.xbulk = 0;
    l.grid = l.mcast > 1 ? (tiles + l.mcast - 1) / l.mcast * l.mcast : tiles * l.splits;
    if (l.path == gemv::kPathTc && l.tc_persist) {   // equal shares of the tiles within the resident CTAs
        const int64_t each = (tiles + l.tc_slots - 1) / l.tc_slots;
        l.grid = (tiles + each - 1) / each;
    }
    if (l.grid > 0x7fffffffLL) return GEMV_ERR_UNSUPPORTED;
    p.x = static_cast<const uint16_t*>(x);
    p.K = K;
    p.kslice = l.kslice;
    p.kchunk = l.kchunk;
    p.nseg = nsegs;
    p.splits = l.splits;
    p.kw = l.kw;
    p.xstride = l.xstride;
    p.batch = B;
    p.nbuf = l.nbuf;
    p.flags = (flags & GEMV_FLAG_RMSNORM) ? gemv::kFlagRmsNorm : 0;
    p.rms_eps = eps;
    p.mcast = l.mcast > 1 ? l.mcast : 1;
    p.xper = l.xbox ? l.xper : 0;
    p.xbpp = l.xbox ? l.xbpp : 0;
    p.xwide = l.xbox == 2 ? 1 : 0;
    // The bulk prefetch of W reads only from this GPU's memory.
    for (int i = 0; l.l2pf && i < nsegs; ++i)
        if (!on_current_device(segs[i].W)) l.l2pf = 0;
    p.l2pf = l.l2pf;
    p.wc = g_write_count;
    out->p = p;
    out->l = l;
    out->B = B;
    return GEMV_OK;
}

// One quantised weight matrix of a launch.
struct QSeg {
    const void* Wq;    // codes
    const void* S;     // INT4: BF16 group scales [N, lds]; FP8: FP32 row scales [N]
    float* y;
    int64_t N;
    int64_t ldq;       // row stride of the codes in bytes
    int64_t lds;       // INT4 only
};

// Plan one launch over INT4 (kind gemv::kWeightInt4) or FP8 (gemv::kWeightFp8)
// segments sharing x, K and B.
int prepare_quant(int kind, const QSeg* segs, int nsegs, const void* x, int64_t K, int B, int flags, float eps,
                  int sm_count, Prepared* out, bool overlap = false) {
    if (nsegs < 1 || nsegs > GEMV_MAX_SEGMENTS) return GEMV_ERR_INVALID;
    int64_t total = 0;
    for (int i = 0; i < nsegs; ++i) {
        total += segs[i].N;
        if (total > 0x7fffffffLL) return GEMV_ERR_INVALID;
    }
    Launch l;
    int rc = gemv::plan_launch(total, K, B, sm_count, &l, kind, overlap);
    if (rc != GEMV_OK) return rc;
    Params p;
    std::memset(&p, 0, sizeof p);
    int64_t tiles = 0;
    for (int i = 0; i < nsegs; ++i) {
        p.seg[i].W = static_cast<const uint16_t*>(segs[i].Wq);
        p.seg[i].y = segs[i].y;
        p.seg[i].N = segs[i].N;
        p.seg[i].ldw = segs[i].ldq;
        p.seg[i].tile_begin = tiles;
        if (kind == gemv::kWeightInt4) {
            p.seg[i].S = static_cast<const uint16_t*>(segs[i].S);
            p.seg[i].lds = segs[i].lds;
        } else {
            p.seg[i].rs = static_cast<const float*>(segs[i].S);
        }
        tiles += (segs[i].N + l.rows_per_cta - 1) / l.rows_per_cta;
    }
    l.row_tiles = tiles;
    l.grid = tiles * l.splits;
    if (l.grid > 0x7fffffffLL) return GEMV_ERR_UNSUPPORTED;
    // The bulk copies of x read from a 16-byte boundary, and only from this GPU's memory.
    if (l.xbulk && (!aligned(x, 16) || !on_current_device(x))) l.xbulk = 0;
    p.x = static_cast<const uint16_t*>(x);
    p.K = K;
    p.kslice = l.kslice;
    p.kchunk = l.kchunk;
    p.nseg = nsegs;
    p.splits = l.splits;
    p.kw = l.kw;
    p.xstride = l.xstride;
    p.batch = B;
    p.nbuf = l.nbuf;
    p.flags = (flags & GEMV_FLAG_RMSNORM) ? gemv::kFlagRmsNorm : 0;
    p.rms_eps = eps;
    p.mcast = 1;
    // The bulk prefetch of W reads only from this GPU's memory.
    for (int i = 0; l.l2pf && i < nsegs; ++i)
        if (!on_current_device(segs[i].Wq)) l.l2pf = 0;
    p.l2pf = l.l2pf;
    p.wc = g_write_count;
    out->p = p;
    out->l = l;
    out->B = B;
    return GEMV_OK;
}

int check_fp8(const void* Wq, const float* S, const void* x, const float* y, int64_t N, int64_t K, int B,
              int64_t ldq) {
    if (!Wq || !S || !x || !y) return GEMV_ERR_INVALID;
    if (N < 1 || N > 0x7fffffffLL || K < gemv::kF8Slot || K > 0x7fffffffLL || K % gemv::kF8Slot != 0)
        return GEMV_ERR_INVALID;
    if (B < 1 || B > GEMV_MAX_BATCH || ldq < K) return GEMV_ERR_INVALID;
    if (ldq % 16 != 0 || !aligned(Wq, 16) || !aligned(S, 4) || !aligned(x, 2) || !aligned(y, 4))
        return GEMV_ERR_ALIGN;
    return GEMV_OK;
}

int check_w4(const void* Wq, const void* S, const void* x, const float* y, int64_t N, int64_t K, int B,
             int64_t ldq, int64_t lds) {
    if (!Wq || !S || !x || !y) return GEMV_ERR_INVALID;
    if (N < 1 || N > 0x7fffffffLL || K < gemv::kW4Group || K > 0x7fffffffLL || K % gemv::kW4Group != 0)
        return GEMV_ERR_INVALID;
    if (B < 1 || B > GEMV_MAX_BATCH) return GEMV_ERR_INVALID;
    if (ldq < K / 2 || lds < K / gemv::kW4Group) return GEMV_ERR_INVALID;
    if (ldq % 16 != 0 || !aligned(Wq, 16) || !aligned(S, 2) || !aligned(x, 2) || !aligned(y, 4))
        return GEMV_ERR_ALIGN;
    return GEMV_OK;
}

// Launch a prepared GEMV; a stream-K launch takes its workspace from `ws`
// (the plan's), or from the device's when ws is null.
int run(const Prepared& pr, cudaStream_t s, Workspace* ws = nullptr) {
    cudaError_t e;
    if (pr.sk) {
        gemv::SkParams p = pr.skp;
        if (ws) {
            if (ws->part_cap < pr.skl.part_floats || ws->ticket_cap < pr.skl.tickets) return GEMV_ERR_INVALID;
            p.part = ws->part;
            p.ticket = ws->ticket;
        } else {
            int dev = 0;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
            std::lock_guard<std::mutex> lock(g_dev_mutex);
            Workspace& dws = g_dev[dev].ws;
            int rc = ws_reserve(dws, pr.skl.part_floats, pr.skl.tickets, s);
            if (rc != GEMV_OK) return rc;
            p.part = dws.part;
            p.ticket = dws.ticket;
        }
        e = gemv::launch_streamk(p, pr.skl, s, pdl_enabled());
    } else {
        e = gemv::launch_gemv(pr.B, pr.p, pr.l, s, pdl_enabled());
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return GEMV_OK;
}

}  // namespace

namespace {

void fill_info(const Launch& l, gemv_launch_info* out) {
    out->rows_per_cta = l.rows_per_cta;
    out->row_tiles = l.row_tiles;
    out->grid = l.grid;
    out->kslice = l.kslice;
    out->kchunk = l.kchunk;
    out->warps_per_cta = gemv::kWarps;
    out->warps_per_row = l.kw;
    out->splits = l.splits;
    out->rows_per_warp = l.rows_per_warp;
    out->unroll = l.unroll;
    out->smem_bytes = l.smem_bytes;
    out->path = l.path;
    out->xstride = l.xstride;
    out->nbuf = l.nbuf;
    out->mcast = l.mcast;
    out->xbox = l.xbox;
    out->xpieces = l.xbox ? l.xper : 0;
    out->xboxes_per_piece = l.xbox ? l.xbpp : 0;
    out->persistent = (l.path == gemv::kPathTc && l.tc_persist) ? 1 : 0;
    out->l2_prefetch = l.l2pf;
}

}  // namespace

namespace {

// Wait for the end of a host-to-host call: poll for up to a millisecond (a
// decode projection takes tens of microseconds and a blocking wait adds a
// wake-up), then block.
int wait_host_io(cudaStream_t s) {
    const auto t0 = std::chrono::steady_clock::now();
    cudaError_t e;
    for (;;) {
        e = cudaStreamQuery(s);
        if (e == cudaSuccess) return GEMV_OK;
        if (e != cudaErrorNotReady) return cuda_fail(e);
        if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(1)) break;
    }
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e);
    return GEMV_OK;
}

// The host-to-host calls wait for their stream, which a capturing stream
// cannot do.
int not_capturing(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e);
    return cs == cudaStreamCaptureStatusNone ? GEMV_OK : GEMV_ERR_CAPTURE;
}

}  // namespace

struct gemv_plan {
    std::vector<Prepared> launches;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    Workspace ws;   // stream-K launches of this plan (run one after another)
    bool independent = false;   // launches skip the wait for the preceding grid
};

namespace {

// Byte range [lo, hi) of device memory one projection reads or writes.
struct Extent {
    uintptr_t lo, hi;
    size_t launch;
};

bool overlap(const Extent& a, const Extent& b) { return a.lo < b.hi && b.lo < a.hi; }

// Whether no launch of the plan writes memory that another of its launches
// reads or writes: then none depends on another, and each may start its work
// without waiting for the preceding grid ("GPU performance chains", "Launch
// gaps in a decode step": the gap between dependent kernels is the cost; an
// independent kernel has none to pay). launch_of[q] is the launch projection
// q belongs to. (Stream-K launches also share the plan's workspace; the
// caller checks for them.)
bool plan_is_independent(const gemv_proj* projs, int nproj, const std::vector<size_t>& launch_of) {
    std::vector<Extent> reads, writes;
    auto ext = [](const void* p, int64_t bytes, size_t l) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        return Extent{a, a + static_cast<uintptr_t>(bytes), l};
    };
    for (int i = 0; i < nproj; ++i) {
        const gemv_proj& q = projs[i];
        const size_t l = launch_of[static_cast<size_t>(i)];
        reads.push_back(ext(q.x, static_cast<int64_t>(q.B) * q.K * 2, l));
        const int64_t wbytes = q.weight_kind == GEMV_WEIGHT_BF16 ? q.N * q.ldw * 2 : q.N * q.ldw;
        reads.push_back(ext(q.W, wbytes, l));
        if (q.weight_kind == GEMV_WEIGHT_INT4) reads.push_back(ext(q.S, q.N * q.lds * 2, l));
        if (q.weight_kind == GEMV_WEIGHT_FP8) reads.push_back(ext(q.S, q.N * 4, l));
        writes.push_back(ext(q.y, static_cast<int64_t>(q.B) * q.N * 4, l));
    }
    for (const Extent& w : writes) {
        for (const Extent& r : reads)
            if (r.launch != w.launch && overlap(w, r)) return false;
        for (const Extent& v : writes)
            if (v.launch != w.launch && overlap(w, v)) return false;
    }
    return true;
}

}  // namespace

extern "C" {

int gemv_bf16_ex(const void* W, const void* x, float* y, int64_t N, int64_t K, int B, int64_t ldw,
                 const gemv_options* opt, void* stream) {
    gemv_segment seg{W, y, N, ldw};
    int flags = 0;
    float eps = 0.f;
    int rc = check_common(x, K, B);
    if (rc != GEMV_OK) return rc;
    if ((rc = check_matrix(W, y, N, K, ldw)) != GEMV_OK) return rc;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    int sm_count = 0;
    if ((rc = device_state(&sm_count)) != GEMV_OK) return rc;
    Prepared pr;
    if ((rc = prepare(&seg, 1, x, K, B, flags, eps, sm_count, &pr)) != GEMV_OK) return rc;
    return run(pr, static_cast<cudaStream_t>(stream));
}

int gemv_bf16_host_io(const void* W, const void* x_host, float* y_host, void* x_dev, float* y_dev,
                      int64_t N, int64_t K, int B, int64_t ldw, const gemv_options* opt, void* stream) {
    if (!x_host || !y_host) return GEMV_ERR_INVALID;
    int rc = check_common(x_dev, K, B);
    if (rc != GEMV_OK) return rc;
    if ((rc = check_matrix(W, y_dev, N, K, ldw)) != GEMV_OK) return rc;
    int flags = 0;
    float eps = 0.f;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = not_capturing(s)) != GEMV_OK) return rc;
    const size_t xbytes = static_cast<size_t>(B) * static_cast<size_t>(K) * 2;
    const size_t ybytes = static_cast<size_t>(B) * static_cast<size_t>(N) * 4;
    // A device-mapped y_host (pinned memory) takes the kernel's stores directly
    // when y is small; a large y goes back in one bulk copy (the kernel's
    // scattered 32-byte stores cross the host link less efficiently).
    float* y_mapped = nullptr;
    void* dp = nullptr;
    if (ybytes <= kMappedYMaxBytes && cudaHostGetDevicePointer(&dp, y_host, 0) == cudaSuccess && aligned(dp, 4)) {
        y_mapped = static_cast<float*>(dp);
    } else {
        cudaGetLastError();   // not mapped: the copy path below
    }
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, xbytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((rc = gemv_bf16_ex(W, x_dev, y_mapped ? y_mapped : y_dev, N, K, B, ldw, opt, stream)) != GEMV_OK) return rc;
    if (!y_mapped &&
        (e = cudaMemcpyAsync(y_host, y_dev, ybytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e);
    return wait_host_io(s);
}

int gemv_bf16_multi_host_io(const gemv_segment* segs, int nsegs, const void* x_host, void* x_dev,
                            float* const* y_host, int64_t K, int B, const gemv_options* opt, void* stream) {
    if (!segs || nsegs < 1 || nsegs > GEMV_MAX_SEGMENTS || !x_host || !y_host) return GEMV_ERR_INVALID;
    for (int i = 0; i < nsegs; ++i)
        if (!y_host[i]) return GEMV_ERR_INVALID;
    int rc = check_common(x_dev, K, B);
    if (rc != GEMV_OK) return rc;
    for (int i = 0; i < nsegs; ++i)
        if ((rc = check_matrix(segs[i].W, segs[i].y, segs[i].N, K, segs[i].ldw)) != GEMV_OK) return rc;
    int flags = 0;
    float eps = 0.f;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((rc = not_capturing(s)) != GEMV_OK) return rc;
    const size_t xbytes = static_cast<size_t>(B) * static_cast<size_t>(K) * 2;
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, xbytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((rc = gemv_bf16_multi_ex(segs, nsegs, x_dev, K, B, opt, stream)) != GEMV_OK) return rc;
    for (int i = 0; i < nsegs; ++i) {
        const size_t ybytes = static_cast<size_t>(B) * static_cast<size_t>(segs[i].N) * 4;
        if ((e = cudaMemcpyAsync(y_host[i], segs[i].y, ybytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_fail(e);
    }
    return wait_host_io(s);
}

int gemv_bf16(const void* W, const void* x, float* y, int64_t N, int64_t K, int B, int64_t ldw,
              void* stream) {
    return gemv_bf16_ex(W, x, y, N, K, B, ldw, nullptr, stream);
}

int gemv_bf16_multi_ex(const gemv_segment* segs, int nsegs, const void* x, int64_t K, int B,
                       const gemv_options* opt, void* stream) {
    if (!segs || nsegs < 1 || nsegs > GEMV_MAX_SEGMENTS) return GEMV_ERR_INVALID;
    int rc = check_common(x, K, B);
    if (rc != GEMV_OK) return rc;
    for (int i = 0; i < nsegs; ++i)
        if ((rc = check_matrix(segs[i].W, segs[i].y, segs[i].N, K, segs[i].ldw)) != GEMV_OK) return rc;
    int flags = 0;
    float eps = 0.f;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    int sm_count = 0;
    if ((rc = device_state(&sm_count)) != GEMV_OK) return rc;
    Prepared pr;
    if ((rc = prepare(segs, nsegs, x, K, B, flags, eps, sm_count, &pr)) != GEMV_OK) return rc;
    return run(pr, static_cast<cudaStream_t>(stream));
}

int gemv_bf16_multi(const gemv_segment* segs, int nsegs, const void* x, int64_t K, int B,
                    void* stream) {
    return gemv_bf16_multi_ex(segs, nsegs, x, K, B, nullptr, stream);
}

int gemv_plan_create(const gemv_proj* projs, int nproj, gemv_plan** out) {
    if (!out) return GEMV_ERR_INVALID;
    *out = nullptr;
    if (!projs || nproj < 1) return GEMV_ERR_INVALID;
    // Check every projection before touching the device.
    for (int i = 0; i < nproj; ++i) {
        const gemv_proj& q = projs[i];
        int rc = check_common(q.x, q.K, q.B);
        if (rc != GEMV_OK) return rc;
        if (q.weight_kind == GEMV_WEIGHT_BF16) {
            rc = check_matrix(q.W, q.y, q.N, q.K, q.ldw);
        } else if (q.weight_kind == GEMV_WEIGHT_INT4) {
            rc = check_w4(q.W, q.S, q.x, q.y, q.N, q.K, q.B, q.ldw, q.lds);
        } else if (q.weight_kind == GEMV_WEIGHT_FP8) {
            rc = check_fp8(q.W, static_cast<const float*>(q.S), q.x, q.y, q.N, q.K, q.B, q.ldw);
        } else {
            rc = GEMV_ERR_INVALID;
        }
        if (rc != GEMV_OK) return rc;
        if (q.fuse_group < 0) return GEMV_ERR_INVALID;
        gemv_options o{q.flags, q.rms_eps};
        int f = 0;
        float e = 0.f;
        if ((rc = check_options(&o, &f, &e)) != GEMV_OK) return rc;
        if (q.weight_kind != GEMV_WEIGHT_BF16 && (f & (GEMV_FLAG_STREAMK | GEMV_FLAG_CUDA_CORES)))
            return GEMV_ERR_UNSUPPORTED;
    }
    int sm_count = 0;
    int rc = device_state(&sm_count);
    if (rc != GEMV_OK) return rc;

    gemv_plan* plan = new (std::nothrow) gemv_plan;
    if (!plan) return GEMV_ERR_NOMEM;
    try {
        // Launches: runs of adjacent projections of one fuse group with the
        // same x, K, B, options and weight kind (at most GEMV_MAX_SEGMENTS).
        std::vector<std::pair<int, int>> groups;
        std::vector<size_t> launch_of(static_cast<size_t>(nproj));
        for (int i = 0; i < nproj;) {
            const gemv_proj& a = projs[i];
            int j = i + 1;
            if (a.fuse_group > 0) {
                while (j < nproj && j - i < GEMV_MAX_SEGMENTS && projs[j].fuse_group == a.fuse_group &&
                       projs[j].x == a.x && projs[j].K == a.K && projs[j].B == a.B &&
                       projs[j].flags == a.flags && projs[j].rms_eps == a.rms_eps &&
                       projs[j].weight_kind == a.weight_kind)
                    ++j;
            }
            for (int q = i; q < j; ++q) launch_of[static_cast<size_t>(q)] = groups.size();
            groups.emplace_back(i, j);
            i = j;
        }
        bool independent = !gemv::plan_force_wait() && plan_is_independent(projs, nproj, launch_of);
        for (int q = 0; q < nproj && independent; ++q)
            if (projs[q].flags & GEMV_FLAG_STREAMK) independent = false;

        // Plan every launch; with overlap, as a member of an independent plan
        // of several launches (gemv::plan_launch).
        auto build = [&](bool overlap) -> int {
            plan->launches.clear();
            for (const auto& grp : groups) {
                const int i = grp.first, j = grp.second;
                const gemv_proj& a = projs[i];
                Prepared pr;
                const float eps = (a.flags & GEMV_FLAG_RMSNORM) ? a.rms_eps : 0.f;
                int r;
                if (a.weight_kind == GEMV_WEIGHT_BF16) {
                    gemv_segment segs[GEMV_MAX_SEGMENTS];
                    for (int q = i; q < j; ++q)
                        segs[q - i] = gemv_segment{projs[q].W, projs[q].y, projs[q].N, projs[q].ldw};
                    r = prepare(segs, j - i, a.x, a.K, a.B, a.flags, eps, sm_count, &pr, overlap);
                } else {
                    QSeg segs[GEMV_MAX_SEGMENTS];
                    for (int q = i; q < j; ++q)
                        segs[q - i] = QSeg{projs[q].W, projs[q].S, projs[q].y, projs[q].N, projs[q].ldw, projs[q].lds};
                    r = prepare_quant(a.weight_kind == GEMV_WEIGHT_INT4 ? gemv::kWeightInt4 : gemv::kWeightFp8, segs,
                                      j - i, a.x, a.K, a.B, a.flags, eps, sm_count, &pr, overlap);
                }
                if (r != GEMV_OK) return r;
                // The L2 prefetch rule was measured on chains of the same call; among
                // a plan's differing neighbours it cost time (the decode step with
                // every wait kept: 2.298 -> 2.325 ms), so plans leave it off unless
                // the sweep knob sets it.
                if (!gemv::l2pf_forced()) {
                    pr.p.l2pf = 0;
                    pr.l.l2pf = 0;
                }
                plan->launches.push_back(pr);
            }
            return GEMV_OK;
        };
        const bool overlap = independent && groups.size() >= 2;
        rc = build(overlap);
        // A launch the planner sent to the stream-K kernel (its sweep knob)
        // shares the plan's workspace: then every launch waits, planned alone.
        bool any_sk = false;
        for (const Prepared& pr : plan->launches) any_sk = any_sk || pr.sk;
        if (rc == GEMV_OK && any_sk) {
            independent = false;
            if (overlap) rc = build(false);
        }
        if (rc != GEMV_OK) {
            delete plan;
            return rc;
        }
        plan->independent = independent;
    } catch (const std::bad_alloc&) {
        delete plan;
        return GEMV_ERR_NOMEM;
    }
    if (plan->independent)
        for (Prepared& pr : plan->launches) pr.p.flags |= gemv::kFlagNoWait;
    int64_t need_part = 0, need_tickets = 0;
    for (const Prepared& pr : plan->launches) {
        if (!pr.sk) continue;
        if (pr.skl.part_floats > need_part) need_part = pr.skl.part_floats;
        if (pr.skl.tickets > need_tickets) need_tickets = pr.skl.tickets;
    }
    if (need_part > 0 && (rc = ws_reserve(plan->ws, need_part, need_tickets, nullptr)) != GEMV_OK) {
        delete plan;
        return rc;
    }
    *out = plan;
    return GEMV_OK;
}

int gemv_plan_capture(gemv_plan* plan, void* stream) {
    if (!plan || !stream) return GEMV_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e);
    if (cs != cudaStreamCaptureStatusNone) return GEMV_ERR_CAPTURE;

    if ((e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal)) != cudaSuccess) return cuda_fail(e);
    int rc = GEMV_OK;
    for (const Prepared& pr : plan->launches) {
        if ((rc = run(pr, s, &plan->ws)) != GEMV_OK) break;
    }
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(s, &g);
    if (rc != GEMV_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        g_last_cuda_error = static_cast<int>(e);
        return GEMV_ERR_CAPTURE;
    }
    cudaGraphExec_t ex = nullptr;
    if ((e = cudaGraphInstantiate(&ex, g, 0)) != cudaSuccess) {
        cudaGraphDestroy(g);
        g_last_cuda_error = static_cast<int>(e);
        return GEMV_ERR_CAPTURE;
    }
    if (plan->exec) cudaGraphExecDestroy(plan->exec);
    if (plan->graph) cudaGraphDestroy(plan->graph);
    plan->graph = g;
    plan->exec = ex;
    return GEMV_OK;
}

int gemv_plan_launch(gemv_plan* plan, void* stream) {
    if (!plan) return GEMV_ERR_INVALID;
    if (!plan->exec) return GEMV_ERR_UNSUPPORTED;
    cudaError_t e = cudaGraphLaunch(plan->exec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return GEMV_OK;
}

int gemv_plan_launch_host_io(gemv_plan* plan, const void* x_host, void* x_dev, int64_t x_bytes,
                             const void* y_dev, void* y_host, int64_t y_bytes, void* stream) {
    if (!plan || x_bytes < 0 || y_bytes < 0) return GEMV_ERR_INVALID;
    if (x_bytes > 0 && (!x_host || !x_dev)) return GEMV_ERR_INVALID;
    if (y_bytes > 0 && (!y_host || !y_dev)) return GEMV_ERR_INVALID;
    if (!plan->exec) return GEMV_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = not_capturing(s);
    if (rc != GEMV_OK) return rc;
    cudaError_t e;
    if (x_bytes > 0 &&
        (e = cudaMemcpyAsync(x_dev, x_host, static_cast<size_t>(x_bytes), cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaGraphLaunch(plan->exec, s)) != cudaSuccess) return cuda_fail(e);
    if (y_bytes > 0 &&
        (e = cudaMemcpyAsync(y_host, y_dev, static_cast<size_t>(y_bytes), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail(e);
    return wait_host_io(s);
}

int gemv_plan_num_launches(const gemv_plan* plan) {
    return plan ? static_cast<int>(plan->launches.size()) : 0;
}

int gemv_plan_independent(const gemv_plan* plan) { return plan && plan->independent ? 1 : 0; }

void gemv_plan_destroy(gemv_plan* plan) {
    if (!plan) return;
    if (plan->exec) cudaGraphExecDestroy(plan->exec);
    if (plan->graph) cudaGraphDestroy(plan->graph);
    ws_free(plan->ws);
    delete plan;
}

int gemv_debug_write_count(int32_t* counts, const float* y_base, int64_t n) {
#ifdef GEMV_DEBUG_WRITECOUNT
    if (counts && (!y_base || n < 1)) return GEMV_ERR_INVALID;
    g_write_count = counts ? gemv::WriteCount{counts, y_base, n} : gemv::WriteCount{nullptr, nullptr, 0};
    return GEMV_OK;
#else
    (void)counts;
    (void)y_base;
    (void)n;
    return GEMV_ERR_UNSUPPORTED;
#endif
}

int gemv_workspace_release(void) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return GEMV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    ws_free(g_dev[dev].ws);
    return GEMV_OK;
}

int gemv_bf16_streamk_noalloc(const void* W, const void* x, float* y, int64_t N, int64_t K, int64_t ldw,
                              const gemv_options* opt, void* stream) {
    // Per-device addresses of the fixed scratch, looked up once per device
    // with that device current.
    static std::mutex scratch_mutex;
    static float* scratch_part[kMaxDevices] = {};
    static int32_t* scratch_ticket[kMaxDevices] = {};

    int rc = check_common(x, K, 1);
    if (rc != GEMV_OK) return rc;
    if ((rc = check_matrix(W, y, N, K, ldw)) != GEMV_OK) return rc;
    int flags = 0;
    float eps = 0.f;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    int sm_count = 0;
    if ((rc = device_state(&sm_count)) != GEMV_OK) return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    float* part = nullptr;
    int32_t* ticket = nullptr;
    {
        std::lock_guard<std::mutex> lock(scratch_mutex);
        if (!scratch_part[dev]) {
            if ((e = gemv::noalloc_scratch(&scratch_part[dev], &scratch_ticket[dev])) != cudaSuccess) {
                scratch_part[dev] = nullptr;
                scratch_ticket[dev] = nullptr;
                return cuda_fail(e);
            }
        }
        part = scratch_part[dev];
        ticket = scratch_ticket[dev];
    }
    gemv_segment seg{W, y, N, ldw};
    Prepared pr;
    if ((rc = prepare_streamk(&seg, 1, N, x, K, flags | GEMV_FLAG_STREAMK, eps, sm_count, &pr)) != GEMV_OK)
        return rc;
    if (pr.skl.part_floats > gemv::kNoallocPartFloats || pr.skl.tickets > gemv::kNoallocTickets)
        return GEMV_ERR_UNSUPPORTED;
    gemv::SkParams p = pr.skp;
    p.part = part;
    p.ticket = ticket;
    if ((e = gemv::launch_streamk(p, pr.skl, static_cast<cudaStream_t>(stream), pdl_enabled())) != cudaSuccess)
        return cuda_fail(e);
    return GEMV_OK;
}

int gemv_query_launch_ex(int64_t N, int64_t K, int B, int sm_count, int flags, gemv_launch_info* out) {
    if (!out) return GEMV_ERR_INVALID;
    if (flags & ~(GEMV_FLAG_RMSNORM | GEMV_FLAG_STREAMK | GEMV_FLAG_CUDA_CORES)) return GEMV_ERR_INVALID;
    if ((flags & GEMV_FLAG_STREAMK) && (flags & GEMV_FLAG_CUDA_CORES)) return GEMV_ERR_INVALID;
    if (flags & GEMV_FLAG_CUDA_CORES) {
        std::memset(out, 0, sizeof *out);
        Launch l;
        int rc = gemv::plan_launch(N, K, B, sm_count, &l, gemv::kWeightBf16CudaCores);
        if (rc != GEMV_OK) return rc;
        fill_info(l, out);
        return GEMV_OK;
    }
    const bool sk = (flags & GEMV_FLAG_STREAMK) ||
                    (B == 1 && gemv::prefer_streamk(N, K, B, sm_count));
    if (!sk) return gemv_query_launch(N, K, B, sm_count, out);
    gemv::SkLaunch l;
    int rc = gemv::plan_streamk(N, K, B, sm_count, &l);
    if (rc != GEMV_OK) {
        if (flags & GEMV_FLAG_STREAMK) return rc;
        return gemv_query_launch(N, K, B, sm_count, out);
    }
    std::memset(out, 0, sizeof *out);
    out->grid = l.grid;
    out->kslice = gemv::kSkUnitCols;
    out->kchunk = K;
    out->warps_per_cta = gemv::kWarps;
    out->warps_per_row = 1;
    out->splits = 1;
    out->rows_per_warp = 1;
    out->unroll = gemv::kSkUnroll;
    out->smem_bytes = l.smem_bytes;
    out->path = gemv::kPathStreamK;
    out->xstride = l.xstride;
    out->nbuf = 1;
    out->units = l.units;
    out->warps = l.warps;
    out->chunks = l.chunks;
    out->ctas_per_sm = l.ctas_per_sm;
    out->dp_rounds = l.dp_rounds;
    return GEMV_OK;
}

int gemv_query_launch(int64_t N, int64_t K, int B, int sm_count, gemv_launch_info* out) {
    if (!out) return GEMV_ERR_INVALID;
    std::memset(out, 0, sizeof *out);
    Launch l;
    // As a call with one weight matrix and aligned operands in this GPU's memory
    // (with the current GPU's resident-cluster counts where there is one).
    int dev_sms = 0;
    const bool have_device = device_state(&dev_sms) == GEMV_OK;
    if (!have_device) cudaGetLastError();
    int rc = gemv::plan_launch(N, K, B, sm_count, &l, gemv::kWeightBf16, false, B >= 2 && K % 8 == 0,
                               have_device ? current_tc_clusters() : nullptr);
    if (rc != GEMV_OK) return rc;
    fill_info(l, out);
    return GEMV_OK;
}

int gemv_w4_bf16(const void* Wq, const void* S, const void* x, float* y, int64_t N, int64_t K, int B,
                 int64_t ldq, int64_t lds, const gemv_options* opt, void* stream) {
    int rc = check_w4(Wq, S, x, y, N, K, B, ldq, lds);
    if (rc != GEMV_OK) return rc;
    int flags = 0;
    float eps = 0.f;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    if (flags & (GEMV_FLAG_STREAMK | GEMV_FLAG_CUDA_CORES)) return GEMV_ERR_UNSUPPORTED;
    int sm_count = 0;
    if ((rc = device_state(&sm_count)) != GEMV_OK) return rc;
    Prepared pr;
    const QSeg seg{Wq, S, y, N, ldq, lds};
    if ((rc = prepare_quant(gemv::kWeightInt4, &seg, 1, x, K, B, flags, eps, sm_count, &pr)) != GEMV_OK) return rc;
    return run(pr, static_cast<cudaStream_t>(stream));
}

int gemv_fp8_bf16(const void* Wq, const float* S, const void* x, float* y, int64_t N, int64_t K, int B,
                  int64_t ldq, const gemv_options* opt, void* stream) {
    int rc = check_fp8(Wq, S, x, y, N, K, B, ldq);
    if (rc != GEMV_OK) return rc;
    int flags = 0;
    float eps = 0.f;
    if ((rc = check_options(opt, &flags, &eps)) != GEMV_OK) return rc;
    if (flags & (GEMV_FLAG_STREAMK | GEMV_FLAG_CUDA_CORES)) return GEMV_ERR_UNSUPPORTED;
    int sm_count = 0;
    if ((rc = device_state(&sm_count)) != GEMV_OK) return rc;
    Prepared pr;
    const QSeg seg{Wq, S, y, N, ldq, 0};
    if ((rc = prepare_quant(gemv::kWeightFp8, &seg, 1, x, K, B, flags, eps, sm_count, &pr)) != GEMV_OK) return rc;
    return run(pr, static_cast<cudaStream_t>(stream));
}

int gemv_fp8_query_launch(int64_t N, int64_t K, int B, int sm_count, gemv_launch_info* out) {
    if (!out) return GEMV_ERR_INVALID;
    if (K < gemv::kF8Slot || K % gemv::kF8Slot != 0) return GEMV_ERR_INVALID;
    std::memset(out, 0, sizeof *out);
    Launch l;
    int rc = gemv::plan_launch(N, K, B, sm_count, &l, gemv::kWeightFp8);
    if (rc != GEMV_OK) return rc;
    fill_info(l, out);
    return GEMV_OK;
}

int gemv_w4_query_launch(int64_t N, int64_t K, int B, int sm_count, gemv_launch_info* out) {
    if (!out) return GEMV_ERR_INVALID;
    if (K < gemv::kW4Group || K % gemv::kW4Group != 0) return GEMV_ERR_INVALID;
    std::memset(out, 0, sizeof *out);
    Launch l;
    int rc = gemv::plan_launch(N, K, B, sm_count, &l, gemv::kWeightInt4);
    if (rc != GEMV_OK) return rc;
    fill_info(l, out);
    return GEMV_OK;
}

int gemv_probe_sink_words(void) { return 4096; }

int gemv_probe_stream_read(const void* src, int64_t bytes, float* sink, void* stream) {
    if (!src || !sink || bytes < 16 || bytes % 16 != 0) return GEMV_ERR_INVALID;
    if (!aligned(src, 16) || !aligned(sink, 4)) return GEMV_ERR_ALIGN;
    int sm_count = 0;
    int rc = device_state(&sm_count);
    if (rc != GEMV_OK) return rc;
    int grid = sm_count * 8;
    if (grid > gemv_probe_sink_words()) grid = gemv_probe_sink_words();
    cudaError_t e = gemv::launch_probe_read(src, bytes, sink, grid, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return GEMV_OK;
}

const char* gemv_status_string(int status) {
    switch (status) {
    case GEMV_OK: return "GEMV_OK";
    case GEMV_ERR_INVALID: return "GEMV_ERR_INVALID: a size, count or pointer is out of range";
    case GEMV_ERR_ALIGN: return "GEMV_ERR_ALIGN: W must be 16-byte aligned, ldw a multiple of 8, x 2-byte and y 4-byte aligned";
    case GEMV_ERR_CUDA: return "GEMV_ERR_CUDA: a CUDA runtime call failed (see gemv_last_cuda_error)";
    case GEMV_ERR_NOMEM: return "GEMV_ERR_NOMEM: host allocation failed";
    case GEMV_ERR_CAPTURE: return "GEMV_ERR_CAPTURE: graph capture or instantiation failed";
    case GEMV_ERR_UNSUPPORTED: return "GEMV_ERR_UNSUPPORTED: needs an sm_103 GPU, a captured plan, or a smaller problem";
    default: return "unknown gemv status";
    }
}

int gemv_last_cuda_error(void) { return g_last_cuda_error; }

int gemv_device_status(unsigned int* bits, int reset) {
    if (!bits) return GEMV_ERR_INVALID;
    *bits = 0;
    // Each kernel translation unit keeps its own status word.
    unsigned int b1 = 0, b2 = 0, b3 = 0, b4 = 0, b5 = 0;
    cudaError_t e = gemv::read_fma_status(&b1, reset != 0);
    if (e == cudaSuccess) e = gemv::read_mma_status_nb1(&b2, reset != 0);
    if (e == cudaSuccess) e = gemv::read_mma_status_nb2(&b3, reset != 0);
    if (e == cudaSuccess) e = gemv::read_fp8_status(&b4, reset != 0);
    if (e == cudaSuccess) e = gemv::read_tc_status(&b5, reset != 0);
    if (e != cudaSuccess) return cuda_fail(e);
    *bits = b1 | b2 | b3 | b4 | b5;
    return GEMV_OK;
}

}  // extern "C"
