// Launch planner: which kernel family, how many rows a CTA takes, how far K is
// split, how much of x is staged at a time. Pure host arithmetic, no CUDA call.
//
// Rules (restating "Decode GEMV at half of HBM bandwidth", "A strong answer",
// cause 1 and "The reversal condition", and "GPU performance chains",
// "Wave quantization"):
//   * The GPU streams at full bandwidth only when every SM holds enough loads
//     in flight; a grid whose warps do not cover the SMs caps bandwidth whatever
//     else is right. The planner therefore asks for enough streaming warps to
//     put kTargetInflightPerSm bytes of loads in flight on every SM.
//   * Rows come first. K is split only when the rows alone do not give enough
//     warps, and never below one full batch of loads per warp: splitting costs
//     partial sums and a combine, pure waste once the grid covers the GPU.
//   * Batch 1 splits K first among the warps of one CTA (combined in shared
//     memory), then among the CTAs of a cluster. The tensor-core path splits
//     over a cluster of up to 4 CTAs first: that keeps many rows per CTA, so the
//     x slice each CTA stages (B rows of it) stays small next to the weight bytes
//     it streams; then among the warps of a CTA; then over up to 8 CTAs.
//
// Sweep knobs (environment, read on every plan; unset in normal use), so that
// the measured alternatives to these rules can be reproduced:
//   GEMV_FORCE_SPLIT=<kw>x<S>   warps along K (1, 2, 4, 8) and CTAs along K
//                               (1, 2, 4, 8) instead of the rules' choice;
//   GEMV_FORCE_VARIANT=<list>   comma-separated: mcast=<1|2|4|8> (CTAs sharing
//                               one multicast copy of x, where the multicast
//                               instance applies), unroll=<4|8> (INT4 / FP8:
//                               the standard or the deep instance, where the
//                               deep one applies), streamk=<0|1> (batch-1 BF16
//                               calls: the stream-K kernel or not), planwait=1
//                               (every launch of a plan waits for the
//                               preceding grid, even in an independent plan),
//                               xbox=<0|1|2> (BF16 tensor-core path, more than
//                               8 rows of x: x staged by bulk copies per row,
//                               as narrow or as wide tensor boxes, where boxes
//                               apply), xpieces=<1..8> (the most mbarrier-counted
//                               pieces of those boxes per CTA), tc=<0|1> (BF16,
//                               2..16 rows of x: the tcgen05 kernel or not, where
//                               the call allows it; GEMV_FORCE_SPLIT's CTA count
//                               applies to it, its warp count must be 1),
//                               tcstages=<2..10> and tccols=<64|128> (its ring
//                               depth and stage width, where an instance exists),
//                               l2pf=<0..4> (CUDA-core, INT4 and one-wave
//                               tcgen05 kernels: W batches or ring stages
//                               prefetched into L2 ahead).
// A value the planner cannot use makes every plan fail with GEMV_ERR_INVALID,
// so that a mistyped sweep stops instead of timing the default.
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/gemv.h"
#include "gemv_internal.h"

namespace gemv {

namespace {

struct Overrides {
    int kw = 0, splits = 0;    // 0: the rules decide
    int mcast = 0;             // 0: the rules decide
    int unroll = 0;            // 0: the rules decide
    int streamk = -1;          // -1: the rules decide
    int planwait = 0;          // 1: plans keep every wait for the preceding grid
    int xbox = -1;             // -1: the rules decide
    int xpieces = 0;           // 0: kMaxXPieces
    int tc = -1;               // -1: the rules decide
    int tcstages = 0;          // 0: kTcStages
    int tccols = 0;            // 0: kTcStageCols
    int l2pf = -1;             // -1: the rules decide
    bool bad = false;
};

bool pow2_upto8(long v) { return v == 1 || v == 2 || v == 4 || v == 8; }

Overrides read_overrides() {
    Overrides o;
    if (const char* s = std::getenv("GEMV_FORCE_SPLIT")) {
        char* end = nullptr;
        const long kw = std::strtol(s, &end, 10);
        if (end && *end == 'x') {
            const char* t = end + 1;
            const long sp = std::strtol(t, &end, 10);
            if (end != t && *end == '\0' && pow2_upto8(kw) && pow2_upto8(sp)) {
                o.kw = static_cast<int>(kw);
                o.splits = static_cast<int>(sp);
            } else {
                o.bad = true;
            }
        } else if (*s != '\0') {
            o.bad = true;
        }
    }
    if (const char* s = std::getenv("GEMV_FORCE_VARIANT")) {
        const char* p = s;
        while (*p) {
            const char* comma = std::strchr(p, ',');
            const size_t len = comma ? static_cast<size_t>(comma - p) : std::strlen(p);
            const char* eq = static_cast<const char*>(std::memchr(p, '=', len));
            if (!eq) {
                o.bad = true;
                break;
            }
            const size_t klen = static_cast<size_t>(eq - p);
            char* end = nullptr;
            const long v = std::strtol(eq + 1, &end, 10);
            const bool num = end == p + len && end != eq + 1;
            if (num && klen == 5 && std::strncmp(p, "mcast", 5) == 0 && pow2_upto8(v)) {
                o.mcast = static_cast<int>(v);
            } else if (num && klen == 6 && std::strncmp(p, "unroll", 6) == 0 && (v == 4 || v == 8)) {
                o.unroll = static_cast<int>(v);
            } else if (num && klen == 7 && std::strncmp(p, "streamk", 7) == 0 && (v == 0 || v == 1)) {
                o.streamk = static_cast<int>(v);
            } else if (num && klen == 8 && std::strncmp(p, "planwait", 8) == 0 && (v == 0 || v == 1)) {
                o.planwait = static_cast<int>(v);
            } else if (num && klen == 4 && std::strncmp(p, "xbox", 4) == 0 && v >= 0 && v <= 2) {
                o.xbox = static_cast<int>(v);
            } else if (num && klen == 7 && std::strncmp(p, "xpieces", 7) == 0 && v >= 1 && v <= kMaxXPieces) {
                o.xpieces = static_cast<int>(v);
            } else if (num && klen == 2 && std::strncmp(p, "tc", 2) == 0 && (v == 0 || v == 1)) {
                o.tc = static_cast<int>(v);
            } else if (num && klen == 8 && std::strncmp(p, "tcstages", 8) == 0 && v >= 2 && v <= 10) {
                o.tcstages = static_cast<int>(v);
            } else if (num && klen == 6 && std::strncmp(p, "tccols", 6) == 0 && (v == 64 || v == 128)) {
                o.tccols = static_cast<int>(v);
            } else if (num && klen == 4 && std::strncmp(p, "l2pf", 4) == 0 && v >= 0 && v <= 4) {
                o.l2pf = static_cast<int>(v);
            } else {
                o.bad = true;
                break;
            }
            p = comma ? comma + 1 : p + len;
        }
    }
    return o;
}

constexpr int64_t kTargetInflightPerSm = 64 * 1024;
constexpr int64_t kXBudgetBytes = 80 * 1024;   // staged x per CTA, all buffers
constexpr int64_t kSliceGrain = 256;           // K-slices and chunks are multiples of this
constexpr int kMmaXPad = 32;                   // per-row padding of x: conflict-free fragment reads
constexpr int kW4XPad = 8;                     // INT4: rows 16 bytes apart mod 128 (with the swizzle)

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t m) { return cdiv(a, m) * m; }

}  // namespace

namespace {
int plan_with(int64_t N, int64_t K, int B, int sm_count, Launch* out, int weight_kind, int q_unroll,
              const Overrides& ov, bool overlap);

// The tcgen05 kernel: one 128-row tile per CTA, one or two CTAs per SM by the
// ring's shared memory, only where the row tiles fit one wave; the K-range is
// split over a cluster of a power of two, up to 8 CTAs, so that the grid
// fills the SMs (slices of whole 128-column stages). Clusters of 3 and 6 CTAs
// measured far slower (6144 x 4096 at B = 16: 17.3-18.8 us against 11.4 with
// 4).
int plan_tc(int64_t N, int64_t K, int B, int sm_count, Launch* out, const Overrides& ov,
            const int32_t* tc_clusters) {
    const int stages = ov.tcstages > 0 ? ov.tcstages : kTcStages;
    const int cols = ov.tccols > 0 ? ov.tccols : kTcStageCols;
    if (!tc_has_instance(stages, cols)) return GEMV_ERR_UNSUPPORTED;
    const int64_t smem = tc_smem_bytes(B, stages, cols);
    constexpr int64_t kSmemPerSm = 228 * 1024, kReservedPerCta = 1024;
    int64_t per_sm = kSmemPerSm / (smem + kReservedPerCta);
    if (per_sm > 2) per_sm = 2;
    const int64_t tiles = cdiv(N, kTcRows);
    if (per_sm < 1 || ov.kw > 1) return GEMV_ERR_UNSUPPORTED;
    if (tiles > per_sm * sm_count) {
        // More tiles than one wave: the persistent form, a grid that gives
        // every CTA the same number of tiles within the CTAs resident at once
        // (by its shared memory, at most 3 per SM).
        const int64_t psmem = tcp_smem_bytes(stages, cols);
        if (psmem < 0 || ov.splits > 1) return GEMV_ERR_UNSUPPORTED;
        int64_t pper = kSmemPerSm / (psmem + kReservedPerCta);
        if (pper > 3) pper = 3;
        const int64_t slots = pper * sm_count;
        const int64_t each = cdiv(tiles, slots);
        out->rows_per_cta = kTcRows;
        out->row_tiles = tiles;
        out->grid = cdiv(tiles, each);
        out->kslice = round_up(K, kTcStageCols);
        out->kchunk = out->kslice;
        out->kw = 1;
        out->splits = 1;
        out->rows_per_warp = kTcRows;
        out->unroll = stages;
        out->stage_cols = cols;
        out->smem_bytes = static_cast<int32_t>(psmem);
        out->path = kPathTc;
        out->xstride = 0;
        out->nbuf = 1;
        out->mcast = 1;
        out->xbulk = 0;
        out->xbox = 0;
        out->xper = 0;
        out->xbpp = 0;
        out->smem_rows = out->smem_bytes;
        out->tc_persist = 1;
        out->tc_slots = static_cast<int32_t>(slots);
        out->l2pf = 0;
        return GEMV_OK;
    }
    // A cluster must fit in one GPC: with clusters of 4 or 8 CTAs fewer CTAs
    // are resident at once than SMs x CTAs per SM (measured, B = 16: 9728 x 14336
    // with 4 CTAs per cluster 60.3 us, with 2 47.9; 4864 x 14336 with 8 33.6, with
    // 4 29.0), so the split also keeps the tiles' clusters resident at once.
    auto fits = [&](int64_t s) {
        const int li = s == 1 ? 0 : s == 2 ? 1 : s == 4 ? 2 : 3;
        return tc_clusters == nullptr || tc_clusters[li] < 0 || tiles <= tc_clusters[li];
    };
    int64_t S = ov.splits;
    if (S == 0) {
        S = 1;
        while (S < kMaxSplits && tiles * S * 2 <= per_sm * sm_count && fits(S * 2)) S *= 2;
    }
    const int64_t kslice = round_up(cdiv(K, S), kTcStageCols);
    S = cdiv(K, kslice);
    out->rows_per_cta = kTcRows;
    out->row_tiles = tiles;
    out->grid = tiles * S;
    out->kslice = kslice;
    out->kchunk = kslice;
    out->kw = 1;
    out->splits = static_cast<int32_t>(S);
    out->rows_per_warp = kTcRows;
    out->unroll = stages;
    out->stage_cols = cols;
    out->tc_persist = 0;
    out->tc_slots = 0;
    out->l2pf = ov.l2pf >= 0 ? ov.l2pf : 0;
    out->smem_bytes = static_cast<int32_t>(smem);
    out->path = kPathTc;
    out->xstride = 0;
    out->nbuf = 1;
    out->mcast = 1;
    out->xbulk = 0;
    out->xbox = 0;
    out->xper = 0;
    out->xbpp = 0;
    out->smem_rows = out->smem_bytes;
    return out->smem_bytes <= kTcMaxDynSmem ? GEMV_OK : GEMV_ERR_UNSUPPORTED;
}
}  // namespace

int plan_launch(int64_t N, int64_t K, int B, int sm_count, Launch* out, int weight_kind, bool overlap,
                bool allow_tc, const int32_t* tc_clusters) {
    const Overrides ov = read_overrides();
    if (ov.bad) return GEMV_ERR_INVALID;
    if (!out || N < 1 || K < 1 || B < 1 || B > kMaxBatch || sm_count < 1) return GEMV_ERR_INVALID;
    // BF16 with more than 8 rows of x (2..16 with the tc=1 knob): the tcgen05
    // kernel where the call allows it and its grid of one wave fills the SMs.
    // Measured (us, graph-replayed chains, register-fed tensor-core kernel /
    // tcgen05 with a ring of 2 stages): B = 16 on 4096 x 14336 22.2 / 21.2,
    // 4096 x 4096 8.5 / 8.3, 6144 x 4096 12.2 / 11.4, 28672 x 4096 54.9 / 39.0;
    // 1024 x 4096 (64 CTAs) 4.4 / 5.6; 4096 x 14336 at B = 8 19.9 / 20.9 and at
    // B = 2 19.1 / 20.4.
    // At 8 rows the tcgen05 kernel also wins on the widest matrices (µs, register-
    // fed / tcgen05: 28672 x 4096 40.7 / 37.7, 19456 x 14336 101.0 / 83.0, the LM
    // head shape 165.9 / 154.5), while on the narrower ones its fixed cost per
    // launch still loses (4096 x 14336 19.9 / 20.9, 14336 x 4096 21.1 / 21.2).
    const bool tc_rule = B > 8 || (B == 8 && N >= 16384);
    if (allow_tc && weight_kind == kWeightBf16 && B >= 2 && ov.tc != 0 && (tc_rule || ov.tc == 1) &&
        plan_tc(N, K, B, sm_count, out, ov, tc_clusters) == GEMV_OK && (ov.tc == 1 || out->grid >= sm_count))
        return GEMV_OK;
    // A batch-1 launch of an independent plan runs alongside its neighbours
    // (no wait for the preceding grid): it needs only one streaming warp per
    // SM of its own, so K is split only for very few rows, and the quantised
    // kernels keep their standard instance (3 CTAs per SM instead of 2), which
    // leaves room for the neighbours' CTAs. Measured on the decode step with
    // INT4 weights: 0.997 ms with the single-launch rules, 0.755 with no K
    // split in the deep instance, 0.696 with no K split in the standard one.
    overlap = overlap && B == 1;
    // INT4 and FP8 with up to 8 rows: the deep instance (8 slots in flight per
    // lane; 2 CTAs per SM by registers, one x chunk) when its grid fits in one
    // wave of it and spreads over the SMs at least as evenly as the standard
    // plan's: with CTAs of equal work the busiest SM sets the time, so the
    // share of CTA places in use, grid / (SMs * ceil(grid / SMs)), is compared
    // (measured per decode shape).
    const bool w4 = weight_kind == kWeightInt4, f8 = weight_kind == kWeightFp8;
    int rc = plan_with(N, K, B, sm_count, out, weight_kind, w4 ? kW4Unroll : kF8Unroll, ov, overlap);
    if (rc != GEMV_OK || !(w4 || f8) || B > 8 || ov.unroll == 4 || (overlap && ov.unroll != 8)) return rc;
    Launch deep;
    if (plan_with(N, K, B, sm_count, &deep, weight_kind, w4 ? kW4DeepUnroll : kF8DeepUnroll, ov, overlap) !=
            GEMV_OK ||
        deep.nbuf != 1)
        return rc;
    if (ov.unroll == 8) {
        *out = deep;
        return GEMV_OK;
    }
    auto balance = [&](int64_t grid) {
        const int64_t per_sm = cdiv(grid, sm_count);
        return static_cast<double>(grid) / static_cast<double>(per_sm * sm_count);
    };
    if (deep.grid <= 2LL * sm_count && balance(deep.grid) >= balance(out->grid)) *out = deep;
    return GEMV_OK;
}

namespace {

int plan_with(int64_t N, int64_t K, int B, int sm_count, Launch* out, int weight_kind, int q_unroll,
              const Overrides& ov, bool overlap) {
    if (!out || N < 1 || K < 1 || B < 1 || B > kMaxBatch || sm_count < 1) return GEMV_ERR_INVALID;
    if (weight_kind != kWeightBf16 && weight_kind != kWeightInt4 && weight_kind != kWeightFp8 &&
        weight_kind != kWeightBf16CudaCores)
        return GEMV_ERR_INVALID;
    const Path path = weight_kind == kWeightInt4           ? kPathW4
                      : weight_kind == kWeightFp8          ? kPathFp8
                      : weight_kind == kWeightBf16CudaCores ? kPathFma
                                                           : path_for(B);
    int group_rows, unroll, xpad;
    int64_t batch_cols, warp_inflight;
    bool cluster_first;
    if (path == kPathFma) {
        const Variant v = fma_variant(B);
        group_rows = v.rows_per_warp;
        unroll = v.unroll;
        batch_cols = 256LL * v.unroll;     // 32 lanes x 8 columns per load
        warp_inflight = 32LL * 16 * v.unroll * v.rows_per_warp;
        cluster_first = false;
        xpad = 0;
    } else if (path == kPathMma) {
        group_rows = kMmaRows;
        unroll = kMmaUnroll;
        batch_cols = 32LL * kMmaUnroll;    // 4 lanes x 8 columns per load and row
        warp_inflight = 32LL * 16 * kMmaUnroll * 2;
        cluster_first = true;
        xpad = kMmaXPad;
    } else if (path == kPathW4) {
        group_rows = kMmaRows;
        unroll = q_unroll;
        batch_cols = static_cast<int64_t>(kW4Group) * q_unroll;   // one group per slot
        warp_inflight = 32LL * 16 * q_unroll * 2;
        cluster_first = true;
        xpad = kW4XPad;
    } else {
        group_rows = kMmaRows;
        unroll = q_unroll;
        batch_cols = static_cast<int64_t>(kF8Slot) * q_unroll;
        warp_inflight = 32LL * 16 * q_unroll * 2;
        cluster_first = true;
        xpad = kMmaXPad;
    }
    const int64_t target_warps =
        overlap ? sm_count : static_cast<int64_t>(sm_count) * kTargetInflightPerSm / warp_inflight;
    auto warps_for = [&](int kw, int splits) {
        const int64_t rows_per_cta = static_cast<int64_t>(kWarps / kw) * group_rows;
        return cdiv(N, rows_per_cta) * kWarps * splits;
    };
    auto room = [&](int kw, int splits) {   // can K take one more halving?
        return K / (static_cast<int64_t>(kw) * splits * 2) >= batch_cols;
    };

    int kw = 1, splits = 1;
    if (path == kPathFp8 && B == 1) {
        // FP8, one activation row (measured per decode shape): at least two
        // warps along K, more warps along K while the grid lacks warps, CTAs
        // along K only when even that leaves the GPU short of half of them.
        if (room(kw, splits)) kw = 2;
        while (kw < kWarps && warps_for(kw, splits) < target_warps && room(kw, splits)) kw *= 2;
        while (splits < kMaxSplits && warps_for(kw, splits) < target_warps / 2 && room(kw, splits)) splits *= 2;
    } else if (path == kPathFp8) {
        // FP8, several rows: CTAs along K first (at most 4 for more than 8
        // rows, whose staged x is twice as large), then warps along K up to half
        // the target; from 8 rows on at least two CTAs, which halves the x each stages.
        const int max_s = B > 8 ? 4 : kMaxSplits;
        while (splits < max_s && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
        while (kw < kWarps && warps_for(kw, splits) < target_warps / 2 && room(kw, splits)) kw *= 2;
        if (B >= 8 && splits == 1 && room(kw, splits)) splits = 2;
    } else if (path == kPathW4 && B == 1) {
        // INT4, one activation row: up to four warps along K first (combined in
        // shared memory), then CTAs along K (measured best on the decode shapes:
        // o_proj and the QKV shape take no cluster at all, down_proj two CTAs).
        while (kw < 4 && warps_for(kw, splits) < target_warps && room(kw, splits)) kw *= 2;
        while (splits < 4 && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
        while (kw < kWarps && warps_for(kw, splits) < target_warps && room(kw, splits)) kw *= 2;
        while (splits < kMaxSplits && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
    } else if (path == kPathW4) {
        // INT4, several rows: warps along K would each re-read the CTA's B rows
        // of x from shared memory for fewer weight rows, so only CTAs along K;
        // from 8 rows on, at least two, which halves each CTA's staged x.
        while (splits < kMaxSplits && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
        if (B >= 8 && splits == 1 && room(kw, splits)) splits = 2;
    } else if (cluster_first) {
        while (splits < 4 && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
        while (kw < kWarps && warps_for(kw, splits) < target_warps && room(kw, splits)) kw *= 2;
        while (splits < kMaxSplits && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
    } else {
        while (kw < kWarps && warps_for(kw, splits) < target_warps && room(kw, splits)) kw *= 2;
        while (splits < kMaxSplits && warps_for(kw, splits) < target_warps && room(kw, splits)) splits *= 2;
    }

    // BF16 tensor-core path with one warp along K (nothing left to trade
    // below): split K further, up to a full cluster of 8 CTAs, while the CTA's
    // x slice would not fit in one staged chunk. Chunked x costs a barrier and
    // a copy round per chunk; measured, B = 16 on N x 14,336 (us, chunked /
    // one chunk): N = 4,864 49.6 / 36.1, N = 9,728 67.5 / 60.9, N = 19,456
    // 130.2 / 107.7. Where x already fits, more splits only cost (B = 2 on
    // 4,864 x 14,336: 24.4 us with 4 CTAs along K, 30.6 with 8), so they stay.
    if (path == kPathMma && ov.kw == 0 && !overlap && kw == 1) {
        auto xbytes = [&](int s_) { return static_cast<int64_t>(B) * (cdiv(K, s_) + xpad) * 2; };
        int s2 = splits;
        while (s2 < kMaxSplits && xbytes(s2) > kXBudgetBytes && room(kw, s2)) s2 *= 2;
        if (xbytes(s2) <= kXBudgetBytes) splits = s2;   // only where x then fits one chunk
    }

    // On the BF16 and INT4 tensor-core paths, trade warps along K for CTAs
    // along K while the CTA's x slice does not fit in one staged chunk (same
    // warps, fewer x bytes per CTA, no chunk barriers). The FP8 kernel measured
    // faster with the chunks.
    if (ov.kw > 0) {
        kw = ov.kw;
        splits = ov.splits;
    } else if (cluster_first && path != kPathFp8) {
        while (splits < kMaxSplits && kw > 1 &&
               static_cast<int64_t>(B) * (cdiv(K, splits) + xpad) * 2 > kXBudgetBytes) {
            splits *= 2;
            kw /= 2;
        }
    }

    // Slices are whole multiples of the grain; recount so that no slice is empty.
    int64_t kslice = round_up(cdiv(K, splits), kSliceGrain);
    splits = static_cast<int>(cdiv(K, kslice));
    if (splits == 1) kslice = round_up(K, kSliceGrain);

    // x: one chunk if it fits, else double-buffered chunks.
    int64_t kchunk = kslice;
    int nbuf = 1;
    if (static_cast<int64_t>(B) * (kslice + xpad) * 2 > kXBudgetBytes) {
        nbuf = 2;
        kchunk = (kXBudgetBytes / 2 / (2LL * B) - xpad) / kSliceGrain * kSliceGrain;
        if (kchunk < kSliceGrain) kchunk = kSliceGrain;
    }
    const int64_t xstride = kchunk + xpad;

    const int64_t rows_per_cta = static_cast<int64_t>(kWarps / kw) * group_rows;
    const int64_t row_tiles = cdiv(N, rows_per_cta);
    // Batch 1 on the CUDA cores without a K split and with x in one chunk: CTAs
    // in clusters of kMcastCtas along the rows share one multicast copy of x
    // (the grid is rounded up to whole clusters; the extra CTAs' rows are past
    // N and their results dropped).
    const bool mcast_ok = path == kPathFma && B == 1 && splits == 1 && nbuf == 1;
    int mcast = (mcast_ok && K / 8 >= kMcastMinVectors && row_tiles >= kMcastCtas) ? kMcastCtas : 1;
    if (ov.mcast > 0) mcast = (mcast_ok && K >= 8 && row_tiles >= ov.mcast) ? ov.mcast : 1;
    const int64_t grid = mcast > 1 ? round_up(row_tiles, mcast) : row_tiles * splits;
    if (grid > 0x7fffffffLL) return GEMV_ERR_UNSUPPORTED;
    const int64_t smem = (path == kPathFma ? kFmaSmemHead : (path == kPathMma || path == kPathFp8) ? kBulkSmemHead : 0) +
                         nbuf * static_cast<int64_t>(B) * xstride * 2 +
                         rows_per_cta * (B + 1) * kw * 4 + (rows_per_cta * B + kMaxSplits) * 4 + kMiscFloats * 4;
    if (smem > kMaxDynSmem) return GEMV_ERR_UNSUPPORTED;

    out->rows_per_cta = rows_per_cta;
    out->row_tiles = row_tiles;
    out->grid = grid;
    out->kslice = kslice;
    out->kchunk = kchunk;
    out->kw = kw;
    out->splits = splits;
    out->rows_per_warp = group_rows;
    out->unroll = unroll;
    out->smem_bytes = static_cast<int32_t>(smem);
    out->path = path;
    out->xstride = static_cast<int32_t>(xstride);
    out->nbuf = nbuf;
    out->mcast = mcast;
    // BF16 tensor-core and FP8 paths with x in one chunk of whole 16-byte
    // vectors: bulk copies of x (the front end checks the pointer itself).
    out->xbulk = ((path == kPathMma || path == kPathFp8) && nbuf == 1 && K % 8 == 0) ? 1 : 0;
    out->xbox = 0;
    out->xper = 0;
    out->xbpp = 0;
    out->smem_rows = static_cast<int32_t>(smem);
    out->stage_cols = 0;
    out->tc_persist = 0;
    out->tc_slots = 0;
    // L2 prefetch one batch ahead (Params::l2pf) for batch 1 on the CUDA cores
    // in a single launch whose grid is at most two waves of 4 CTAs per SM.
    // Measured (us per call, graph-replayed chains, without / with): QKV
    // 9.65 / 9.48, o_proj 5.68 / 5.56, down_proj 18.14 / 17.88, k_proj 2.66 /
    // 2.64; two or four batches ahead gained no more (down_proj 18.35, 20.33);
    // a grid of many waves lost (gate/up, 3,584 CTAs: 33.26 / 35.32), and so
    // did the INT4 kernel (down_proj 11.13 / 11.23).
    constexpr int64_t kPrefetchMaxCtasPerSm = 8;
    const int pf_rule = (path == kPathFma && B == 1 && !overlap && grid <= kPrefetchMaxCtasPerSm * sm_count) ? 1 : 0;
    out->l2pf = (path == kPathFma || path == kPathW4) ? (ov.l2pf >= 0 ? ov.l2pf : pf_rule) : 0;
    // BF16 tensor-core path with more than 8 rows of x (the largest slices) in
    // a grid of one wave (every CTA waits for its x at the same moment, with
    // the HBM idle), x in one chunk and K a multiple of 32 (whole blocks, so
    // the 3-D view of x stays inside every row): x as tensor boxes of 8
    // blocks, in up to kMaxXPieces pieces (stage_x_boxes), where the box
    // layout needs no more CTAs' worth of shared memory per SM than the padded
    // rows. Wide boxes (256 columns) need K a multiple of 256 and warp groups
    // that start on a box. The front end checks the pointer and builds the
    // tensor map. Measured (us, row bulk copies / boxes, graph-replayed
    // chains) at B = 16: 4096 x 14336 22.4-22.7 / 22.0-22.4, 6144 x 4096
    // 12.6 / 12.1-12.2, 4096 x 4096 8.7 / 8.3-8.5; grids of several waves
    // lost (28672 x 4096 55.8 / 56.5, 128256 x 4096 197.2 / 200.5: there the
    // later CTAs' copies overlap other CTAs' streams, and the boxes' shorter
    // requests cost), and so did 8 rows and fewer (within 3% either way).
    constexpr int64_t kMmaCtasByRegs = 2;   // up to 128 registers per thread at 256 threads
    if (path == kPathMma && nbuf == 1 && K % 32 == 0 && B > 8 && ov.xbox != 0 &&
        (grid <= kMmaCtasByRegs * sm_count || ov.xbox > 0)) {
        const int64_t nblk = kslice / 32;
        const int64_t span = cdiv(nblk, kw);
        const int64_t boxes = cdiv(span, 8);                    // per warp group
        const int cap = (ov.xpieces > 0 ? ov.xpieces : kMaxXPieces) / kw;
        const int64_t per = boxes < cap ? boxes : (cap > 0 ? cap : 1);
        const int64_t bpp = cdiv(boxes, per);
        const int64_t region = static_cast<int64_t>(kw) * per * bpp * 8 * B * 32 * 2;
        const int64_t smem_box = kBulkSmemHead + region + rows_per_cta * (B + 1) * kw * 4 +
                                 (rows_per_cta * B + kMaxSplits) * 4 + kMiscFloats * 4;
        // CTAs per SM: by shared memory, and at most 2 by registers.
        constexpr int64_t kSmemPerSm = 228 * 1024, kReservedPerCta = 1024;
        auto ctas = [&](int64_t b) {
            const int64_t c = kSmemPerSm / (b + kReservedPerCta);
            return c < kMmaCtasByRegs ? c : kMmaCtasByRegs;
        };
        const bool fits = smem_box <= kMaxDynSmem && 8 * bpp <= 256 && ctas(smem_box) >= ctas(smem);
        // (every K-slice as long as the first where groups split it, so that the
        // kernel's group starts, taken from its own slice, stay on a box)
        const bool wide_ok = K % 256 == 0 && span % 8 == 0 && (kw == 1 || K % kslice == 0);
        if (fits && (ov.xbox != 2 || wide_ok)) {
            out->xbox = ov.xbox == 2 ? 2 : 1;
            out->xper = static_cast<int32_t>(per);
            out->xbpp = static_cast<int32_t>(bpp);
            out->smem_bytes = static_cast<int32_t>(smem_box);
        }
    }
    return GEMV_OK;
}

}  // namespace

// Stream-K (batch 1): one wave of CTAs, as many as fit on an SM by shared
// memory (the whole x row) and registers (kSkMaxCtasPerSm for whole units,
// one fewer for ragged K), and never more warps than units, so that every warp
// takes at least one unit.
int plan_streamk(int64_t rows, int64_t K, int B, int sm_count, SkLaunch* out) {
    if (!out || rows < 1 || K < 1 || B < 1 || B > kMaxBatch || sm_count < 1) return GEMV_ERR_INVALID;
    if (B != 1) return GEMV_ERR_UNSUPPORTED;
    const int64_t nv = cdiv(K, 8);
    const int64_t xbytes = 16 * nv;
    if (xbytes > kSkMaxXBytes) return GEMV_ERR_UNSUPPORTED;
    const int64_t chunks = cdiv(K, kSkUnitCols);
    if (rows > 0x7fffffffLL) return GEMV_ERR_UNSUPPORTED;
    const int64_t units = rows * chunks;
    if (units > 0x7fffffffLL) return GEMV_ERR_UNSUPPORTED;   // 32-bit unit numbers in the kernel
    const int64_t smem = xbytes + kMiscFloats * 4;
    constexpr int64_t kSmemPerSm = 228 * 1024, kSmemReservedPerCta = 1024;
    int64_t per_sm = kSmemPerSm / (smem + kSmemReservedPerCta);
    // The ragged-K instance (predicated last unit) holds one CTA fewer by registers.
    const int64_t reg_cap = (K % kSkUnitCols == 0) ? kSkMaxCtasPerSm : kSkMaxCtasPerSm - 1;
    if (per_sm > reg_cap) per_sm = reg_cap;
    const int64_t grid_warps = static_cast<int64_t>(sm_count) * per_sm * kWarps;
    // Whole rounds of rows one per warp; the rest split evenly. With fewer rows
    // than warps, every row is split; a grid with more warps than units is cut
    // to the units (every warp takes at least one).
    const int64_t rounds = rows / grid_warps;
    const int64_t rest_units = (rows - rounds * grid_warps) * chunks;
    int64_t grid = cdiv(grid_warps, kWarps);
    int64_t warps = grid_warps < rest_units ? grid_warps : rest_units;
    if (rounds == 0) grid = cdiv(warps, kWarps);
    out->grid = grid;
    out->warps = warps;
    out->units = rest_units;
    out->dp_rounds = static_cast<int32_t>(rounds);
    out->chunks = static_cast<int32_t>(chunks);
    out->smem_bytes = static_cast<int32_t>(smem);
    out->ctas_per_sm = static_cast<int32_t>(per_sm);
    out->xstride = static_cast<int32_t>(8 * nv);
    out->part_floats = 2 * (warps > 0 ? warps : 1);
    out->tickets = rows - rounds * grid_warps > 0 ? rows - rounds * grid_warps : 1;
    return GEMV_OK;
}

bool plan_force_wait() {
    const Overrides ov = read_overrides();
    return !ov.bad && ov.planwait == 1;
}

bool l2pf_forced() {
    const Overrides ov = read_overrides();
    return !ov.bad && ov.l2pf >= 0;
}

// The default grid measured faster than the stream-K grid on every decode
// shape (batch 1, 2,000 calls each), so the rules never pick it; the sweep
// knob streamk=1 does, for batch-1 shapes the stream-K kernel takes.
bool prefer_streamk(int64_t rows, int64_t K, int B, int sm_count) {
    const Overrides ov = read_overrides();
    if (ov.bad || ov.streamk != 1 || B != 1) return false;
    SkLaunch l;
    return plan_streamk(rows, K, B, sm_count, &l) == GEMV_OK;
}

}  // namespace gemv
