// Launch planner: how many rows a CTA takes, how far K is split, how much of x
// is staged at a time. Pure host arithmetic, no CUDA call.
//
// Rules (restating "Decode GEMV at half of HBM bandwidth", "A strong answer",
// cause 1 and "The reversal condition", and "GPU performance chains",
// "Wave quantization"):
//   * The GPU streams at full bandwidth only when every SM holds enough loads
//     in flight; a grid whose warps do not cover the SMs caps bandwidth whatever
//     else is right. The planner therefore asks for at least kTargetWarpsPerSm
//     streaming warps per SM.
//   * Rows come first: one warp streams RPW whole rows. K is split only when the
//     rows alone do not give enough warps, and never below one full batch of
//     loads per warp (splitting costs partial sums and a combine, pure waste
//     once the grid already covers the GPU).
//   * K is split first among the warps of one CTA (combined in shared memory),
//     then among the CTAs of one cluster (combined in distributed shared
//     memory), at most kMaxSplits.
#include <cstdint>

#include "../../include/gemv.h"
#include "gemv_internal.h"

namespace gemv {

namespace {

constexpr int kTargetWarpsPerSm = 16;
constexpr int64_t kXBudgetBytes = 40 * 1024;   // staged x per CTA

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t m) { return cdiv(a, m) * m; }

}  // namespace

int32_t smem_bytes_for(int B, int64_t kchunk, int64_t rows_per_cta, int kw) {
    const int64_t xbytes = round_up(static_cast<int64_t>(B) * kchunk * 2, 16);
    const int64_t red = static_cast<int64_t>(rows_per_cta) * B * kw * 4;
    const int64_t cpart = static_cast<int64_t>(rows_per_cta) * B * 4;
    return static_cast<int32_t>(xbytes + red + cpart);
}

int plan_launch(int64_t N, int64_t K, int B, int sm_count, Launch* out) {
    if (!out || N < 1 || K < 1 || B < 1 || B > kMaxBatch || sm_count < 1) return GEMV_ERR_INVALID;
    const Variant v = variant_for(B);
    const int64_t target_warps = static_cast<int64_t>(sm_count) * kTargetWarpsPerSm;
    const int64_t batch_cols = static_cast<int64_t>(kStepCols) * v.unroll;   // one warp, one batch

    auto warps_for = [&](int kw, int splits) {
        const int64_t rows_per_cta = static_cast<int64_t>(kWarps / kw) * v.rows_per_warp;
        return cdiv(N, rows_per_cta) * kWarps * splits;
    };

    int kw = 1;
    while (kw < kWarps && warps_for(kw, 1) < target_warps && K / (2 * kw) >= batch_cols) kw *= 2;

    int splits = 1;
    while (splits < kMaxSplits && warps_for(kw, splits) < target_warps &&
           K / (static_cast<int64_t>(kw) * 2 * splits) >= batch_cols)
        splits *= 2;

    // Slices are whole warp-steps; recount so that no slice is empty.
    int64_t kslice = round_up(cdiv(K, splits), kStepCols);
    splits = static_cast<int>(cdiv(K, kslice));
    if (splits == 1) kslice = round_up(K, kStepCols);

    int64_t chunk_cap = (kXBudgetBytes / (2 * B)) / kStepCols * kStepCols;
    if (chunk_cap < kStepCols) chunk_cap = kStepCols;
    const int64_t kchunk = kslice < chunk_cap ? kslice : chunk_cap;

    const int64_t rows_per_cta = static_cast<int64_t>(kWarps / kw) * v.rows_per_warp;
    const int64_t row_tiles = cdiv(N, rows_per_cta);
    const int64_t grid = row_tiles * splits;
    if (grid > 0x7fffffffLL) return GEMV_ERR_UNSUPPORTED;

    out->rows_per_cta = rows_per_cta;
    out->row_tiles = row_tiles;
    out->grid = grid;
    out->kslice = kslice;
    out->kchunk = kchunk;
    out->kw = kw;
    out->splits = splits;
    out->rows_per_warp = v.rows_per_warp;
    out->unroll = v.unroll;
    out->smem_bytes = smem_bytes_for(B, kchunk, rows_per_cta, kw);
    if (out->smem_bytes > kMaxDynSmem) return GEMV_ERR_UNSUPPORTED;
    return GEMV_OK;
}

}  // namespace gemv
