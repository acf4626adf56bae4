// Stream-K decode GEMV for sm_103a, batch 1: y[n] = sum_k W[n][k] * x[k], BF16
// in, FP32 multiply-adds, with a grid of exactly one wave.
//
// "GPU performance chains" ("Wave quantization") and "Decode GEMV at half of
// HBM bandwidth" (cause 1) describe the loss this kernel removes: a grid of
// whole-row CTAs leaves the last wave partly empty whenever the tile count is
// not a multiple of the resident CTAs. Here the grid is one wave of GW warps.
// The rows that fill whole rounds of GW are taken one per warp, round-robin
// (row r * GW + w in round r), so that the rows in flight at any time are
// neighbours in memory. The remaining rows are cut into units of 2,048
// columns (one batch of 8 loads of 16 bytes per lane), numbered row-major, and
// warp w takes the contiguous units [w * units / warps, (w + 1) * units /
// warps): every warp gets the same number of units, give or take one.
//
// A row that lies wholly inside one warp's range is reduced and stored as in
// the row-per-warp kernel. A row cut between warps is finished without any
// waiting: each of its warps writes its partial sum to a workspace slot (its
// first or its last row) and counts itself on the row's counter; the warp
// that counts last adds the partials in warp order (so the value does not
// depend on which warp came last), stores y and resets the counter to zero for
// the next launch. No warp ever spins on another. The count is one acq_rel
// atomic (release of the partial written before it, acquire of the others'
// for the last), and a warp issues its next row's first loads before it
// stores or counts a finished row.
//
// x is staged whole in shared memory once per CTA (the grid is persistent, so
// once per resident CTA); the first W batch goes out before the
// programmatic-dependent-launch wait, the workspace is touched only after it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_common.cuh"
#include "gemv_kernel.cuh"

namespace gemv {

// First unit of warp w under the balanced partition of `units` over `warps`.
__device__ __forceinline__ int32_t sk_begin(int32_t w, int32_t units, int32_t warps) {
    return static_cast<int32_t>(static_cast<int64_t>(w) * units / warps);
}

// The warp whose range holds unit u: the largest w with sk_begin(w) <= u.
__device__ __forceinline__ int32_t sk_owner(int32_t u, int32_t units, int32_t warps) {
    return static_cast<int32_t>(((static_cast<int64_t>(u) + 1) * warps - 1) / units);
}

struct SkRow {
    const uint16_t* W;   // row base
    float* y;            // output element
};

__device__ __forceinline__ SkRow sk_row(const SkParams& p, int32_t row) {
    int si = 0;
#pragma unroll 1
    for (int i = 1; i < p.nseg; ++i)
        if (row >= p.seg[i].tile_begin) si = i;
    const int64_t local = row - p.seg[si].tile_begin;
    return SkRow{p.seg[si].W + local * p.seg[si].ldw, p.seg[si].y + local};
}

// RAGGED: K is not a multiple of the unit width, so the last unit of every row
// is partial (predicated loads); otherwise every unit is whole and the lean
// instance fits kSkMaxCtasPerSm CTAs per SM.
template <int UJ, bool RAGGED>
__global__ void __launch_bounds__(kThreads, RAGGED ? kSkMaxCtasPerSm - 1 : kSkMaxCtasPerSm)
gemv_streamk_kernel(const __grid_constant__ SkParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    pdl_launch_dependents();

    const int lane = threadIdx.x & 31;
    const int32_t w = static_cast<int32_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int32_t GW = static_cast<int32_t>(gridDim.x) * kWarps;   // warps of the grid
    const int32_t R = p.dp_rounds;                                  // whole-row rounds
    const int32_t row0 = R * GW;                                    // first row of the split part
    const int32_t U = static_cast<int32_t>(p.units), NW = static_cast<int32_t>(p.warps);
    const int32_t C = p.chunks;
    const int32_t u0 = (w < NW) ? sk_begin(w, U, NW) : 0;
    const int32_t u1 = (w < NW) ? sk_begin(w + 1, U, NW) : 0;
    const int32_t n_first = u0 / C;   // first split-part row of this warp's range (relative to row0)

    const int64_t K = p.K;
    const int nfull = static_cast<int>(K >> 3);                   // whole 8-column vectors
    const int nv = nfull + ((K & 7) ? 1 : 0);
    const int tail_m = static_cast<int>(K & 7);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);
    float* misc = reinterpret_cast<float*>(smem_raw + static_cast<size_t>(p.xstride) * 2);
    const bool norm = (p.flags & kFlagRmsNorm) != 0;

    uint4 wv[UJ][1];
    bool ok[UJ];

    // Loads of unit c of a row: columns 2048 c ... 2048 c + 2047.
    auto issue = [&](const uint16_t* wrow, int c) {
        const int v0 = c * 32 * UJ + lane;
        const uint16_t* const wp[1] = {wrow + 8 * v0};
        if (!RAGGED || (c + 1) * 32 * UJ <= nfull) {
            issue_batch<1, UJ, false>(wv, ok, wp, v0, UJ, nv, nfull, 0);
        } else {
            issue_batch<1, UJ, true>(wv, ok, wp, v0, UJ, nv, nfull, tail_m);
        }
    };

    // This warp's tasks, in order: whole rows r * GW + w for r < R, then the
    // rows of its split-part range [u0, u1). A task is (row, first unit, end unit).
    int32_t r = 0;          // whole-row rounds taken
    int32_t u = u0;         // next split-part unit
    int32_t n = 0;          // current task's row (global)
    int cb = 0, ce = 0;     // its unit range
    bool split = false;     // from the split part
    auto next_task = [&]() -> bool {
        if (r < R) {
            n = r * GW + w;
            cb = 0;
            ce = C;
            split = false;
            ++r;
            return true;
        }
        if (u < u1) {
            const int32_t nl = u / C;
            n = row0 + nl;
            cb = u - nl * C;
            ce = (u1 - nl * C < C) ? u1 - nl * C : C;
            split = true;
            u = nl * C + ce;
            return true;
        }
        return false;
    };

    bool have = next_task();
    SkRow row = {};
    if (have) row = sk_row(p, n);
    // The first unit's loads go out before the wait when it is a whole one.
    const bool pre = have && (!RAGGED || (cb + 1) * 32 * UJ <= nfull);
    if (pre) {
        const int v0 = cb * 32 * UJ + lane;
        const uint16_t* const wp[1] = {row.W + 8 * v0};
        issue_batch<1, UJ, false>(wv, ok, wp, v0, UJ, nv, nfull, 0);
    }
    pdl_wait_prerequisites();
    stage_x(xs, p.xstride, p.x, 1, K, 0, nv);
    cp_async_wait<0>();
    __syncthreads();
    float rs = 1.f;
    if (norm) {
        xsq_accumulate(xs, p.xstride, 1, nv, misc, true);
        __syncthreads();
        rs = 1.0f / sqrtf(misc[kWarps * kMaxBatch] / static_cast<float>(K) + p.rms_eps);
    }

    bool inflight = pre;   // the loads of the task's first unit are already issued
#pragma unroll 1
    while (have) {
        float acc[1][1] = {{0.f}};
#pragma unroll 1
        for (int c = cb; c < ce; ++c) {
            if (!inflight) issue(row.W, c);
            inflight = false;
            const uint16_t* xl = xs + 8 * (c * 32 * UJ + lane);
            if (!RAGGED || (c + 1) * 32 * UJ <= nfull)
                consume_batch<1, 1, UJ, false>(acc, wv, ok, xl, p.xstride);
            else
                consume_batch<1, 1, UJ, true>(acc, wv, ok, xl, p.xstride);
        }
        float* const yout = row.y;
        const int32_t nd = n;
        const int cbd = cb, ced = ce;
        const bool sd = split;
        // The next task's first loads go out before this row is stored.
        have = next_task();
        if (have) {
            row = sk_row(p, n);
            issue(row.W, cb);
            inflight = true;
        }
        float s = acc[0][0];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane != 0) continue;

        if (cbd == 0 && ced == C) {   // the whole row is this warp's
            store_y(yout, norm ? s * rs : s, p.wc);
            continue;
        }
        // A split-part row cut between warps wa .. wb (row index nl relative to
        // row0). Slot 2q holds warp q's partial of its first row, slot 2q + 1 of
        // its last row when that is another row; of the warps of a row only wa
        // can have it as its last row but not its first.
        (void)sd;
        const int32_t nl = nd - row0;
        const int32_t wa = sk_owner(nl * C, U, NW);
        const int32_t wb = sk_owner(nl * C + C - 1, U, NW);
        p.part[2 * w + (nl == n_first ? 0 : 1)] = s;
        // Release this warp's partial and count it in one acq_rel atomic; the
        // warp that counts last acquires every other warp's partial.
        int32_t t;
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(t) : "l"(&p.ticket[nl]) : "memory");
        if (t == wb - wa) {
            const int side_a = (sk_begin(wa, U, NW) < nl * C) ? 1 : 0;
            float v = __ldcg(&p.part[2 * wa + side_a]);
            for (int32_t q = wa + 1; q <= wb; ++q) v += __ldcg(&p.part[2 * q]);
            store_y(yout, norm ? v * rs : v, p.wc);
            p.ticket[nl] = 0;
        }
    }
}

}  // namespace gemv
