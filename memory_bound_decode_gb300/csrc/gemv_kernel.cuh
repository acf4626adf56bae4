// CUDA-core decode GEMV for sm_103a: y[b][n] = sum_k W[n][k] * x[b][k], BF16 in,
// FP32 multiply-adds. Serves batch 1, where the GEMV does one FLOP per byte and
// the CUDA cores have several times the arithmetic the byte stream needs.
//
// Design (restating "Decode GEMV at half of HBM bandwidth", "A strong answer",
// and "GPU performance chains", "A coalesced warp load", for Blackwell):
//   * Lanes run along K. One warp-wide load reads 32 x 16 B = 512 contiguous
//     bytes of one weight row, whole 32-byte sectors only.
//   * Each lane issues UJ independent 16-byte ld.global.nc.L1::no_allocate loads
//     per row before it consumes any, so a resident warp keeps
//     32 * UJ * RPW * 16 bytes in flight (Little's law sets how many are needed).
//   * x (the CTA's K-range, in chunks) is staged once per CTA in shared memory
//     with asynchronous 16-byte copies (all in flight at once; the next chunk
//     is copied while the current one is used) and reused by every row of the
//     CTA; W is never staged: it has no reuse.
//   * The first batch of W loads is issued before the CTA waits on the
//     preceding grid (programmatic dependent launch) and before x is staged, so
//     neither the previous kernel's tail nor the x copy leaves the HBM idle.
//   * Split-K has two levels, both combined in a fixed order (bitwise
//     reproducible, "What interviewers probe next"): `kw` warps of one CTA share
//     a row group (combined through shared memory), and `splits` CTAs of one
//     thread-block cluster share a row tile (combined through distributed shared
//     memory, rank 0 first). No atomics, no global workspace.
//   * Accumulation is blocked: each batch of 8*UJ products goes into a fresh
//     FP32 partial that is then added to the running sum, which bounds the
//     longest rounding chain by 8*UJ + (batches) + 5 + kw + splits additions.
//   * Columns k >= K inside the last 16-byte vector are masked by selecting
//     zero bits in W (and zero-filled x), never by multiplying padding by zero.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_common.cuh"

namespace gemv {

// Issue one batch of W loads: UJ warp-steps (32 vectors each) per row, each
// lane's vectors 256 columns apart, all before any is used. PRED handles the
// first and the last batches of a range (steps past the range, the partial
// warp-step and the partial 16-byte vector at column K); full batches skip it.
template <int RPW, int UJ, bool PRED>
__device__ __forceinline__ void issue_batch(uint4 (&wv)[UJ][RPW], bool (&ok)[UJ],
                                            const uint16_t* const (&wp)[RPW], int v0,
                                            int steps_left, int nv, int nfull, int tail_m) {
#pragma unroll
    for (int u = 0; u < UJ; ++u) {
        const int v = v0 + 32 * u;
        ok[u] = PRED ? (u < steps_left && v < nv) : true;
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (ok[u]) w = ld_stream16(wp[r] + 256 * u);
            if (PRED && ok[u] && v == nfull && tail_m != 0) w = keep_first(w, tail_m);
            wv[u][r] = w;
        }
    }
}

// Two FP32 values in one 64-bit register pair, for the packed multiply-add.
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo_bits, uint32_t hi_bits) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
    return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
// d = a * b + d on both halves (fma.rn.f32x2: one instruction, two FP32
// multiply-adds, each rounded as an fmaf).
__device__ __forceinline__ void fma_f32x2(uint64_t& d, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// Multiply-add one batch into the running sums. The batch is summed into a
// fresh partial first (blocked summation), then added to acc.
//
// Batches of two or more rows of x use the packed FP32 multiply-add: the
// BF16 pair of one 32-bit word (columns 2q and 2q + 1) widens into one
// register pair, and one fma.rn.f32x2 adds both products into a pair of
// partial sums (even columns, odd columns), halving the multiply-add
// instructions. The two partials are added at the end of the batch, so the
// rounding chain is shorter than the scalar one. Batch 1 keeps the scalar
// form (its stream is HBM-bound; its results stay bit for bit as they were).
template <int B, int RPW, int UJ, bool PRED>
__device__ __forceinline__ void consume_batch(float (&acc)[RPW][B], const uint4 (&wv)[UJ][RPW],
                                              const bool (&ok)[UJ], const uint16_t* xl, int xstride) {
    if constexpr (B >= 2) {
        uint64_t t2[RPW][B];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) t2[r][b] = 0ull;   // (+0.0f, +0.0f)
#pragma unroll
        for (int u = 0; u < UJ; ++u) {
            if (PRED && !ok[u]) continue;
            uint64_t wp[RPW][4];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                const uint32_t w[4] = {wv[u][r].x, wv[u][r].y, wv[u][r].z, wv[u][r].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) wp[r][q] = pack_f32x2(w[q] << 16, w[q] & 0xffff0000u);
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const uint4 xr = *reinterpret_cast<const uint4*>(xl + b * xstride + 256 * u);
                const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint64_t xp = pack_f32x2(xw[q] << 16, xw[q] & 0xffff0000u);
#pragma unroll
                    for (int r = 0; r < RPW; ++r) fma_f32x2(t2[r][b], wp[r][q], xp);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const float2 h = unpack_f32x2(t2[r][b]);
                acc[r][b] += h.x + h.y;
            }
    } else {
        float t[RPW][B];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) t[r][b] = 0.f;
#pragma unroll
        for (int u = 0; u < UJ; ++u) {
            if (PRED && !ok[u]) continue;
            float wf[RPW][8];
#pragma unroll
            for (int r = 0; r < RPW; ++r) unpack8(wv[u][r], wf[r]);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const uint4 xr = *reinterpret_cast<const uint4*>(xl + b * xstride + 256 * u);
                float xf[8];
                unpack8(xr, xf);
#pragma unroll
                for (int r = 0; r < RPW; ++r)
#pragma unroll
                    for (int e = 0; e < 8; ++e) t[r][b] = fmaf(wf[r][e], xf[e], t[r][b]);
            }
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) acc[r][b] += t[r][b];
    }
}

// This warp's contiguous range of warp-steps (32 vectors each) within a chunk.
struct FmaRange {
    int s_begin;
    int my_steps;
};

__device__ __forceinline__ FmaRange fma_range(const Chunk& c, int kw, int kq) {
    const int nsteps = (c.nv + 31) >> 5;
    const int span = (nsteps + kw - 1) / kw;
    FmaRange r;
    r.s_begin = kq * span;
    const int s_end = (r.s_begin + span < nsteps) ? r.s_begin + span : nsteps;
    r.my_steps = s_end > r.s_begin ? s_end - r.s_begin : 0;
    return r;
}

// CHUNKED: the CTA's K-range is staged in several double-buffered chunks;
// otherwise it is one chunk and the chunk loop runs once (a separate, leaner
// instance, since the common large projections need no chunking).
// Launch bounds: the batch-16 chunked instance is held to 2 CTAs per SM (128
// registers); the others are left to the compiler.
// MCAST: the batch-1 single-chunk instance that receives x by cluster
// multicast (launched with a cluster along the rows, p.mcast CTAs). It is a
// separate instance: the others carry none of its bulk-copy and mbarrier code
// and launch without a cluster.
template <int B, int RPW, int UJ, bool CHUNKED, bool MCAST = false>
__global__ void __launch_bounds__(kThreads, (B == 16 && CHUNKED) ? 2 : 0)
gemv_bf16_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];

    // Let the next grid on the stream start as SMs free up; it only reads W
    // before it waits on this grid.
    pdl_launch_dependents();

    // x multicast (batch 1, one chunk, no K split): initialise this CTA's
    // mbarrier and announce it to the cluster before anything else.
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem_raw);
    constexpr bool mcast = MCAST && B == 1 && !CHUNKED;
    if constexpr (mcast) {
        if (threadIdx.x == 0) {
            mbar_init(mbar, 1);
            fence_mbar_init_cluster();
        }
        cluster_arrive_relaxed();
    }

    const int S = p.splits;
    if (S > 1) cluster_arrive_relaxed();   // see combine_and_store
    const int64_t tile = blockIdx.x / S;
    const int split = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const SegView sg = segment_of(p, tile);

    const int kw = p.kw;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = warp / kw;        // row group of this warp
    const int kq = warp - g * kw;   // position of this warp along K within the group
    const int rows_per_cta = (kWarps / kw) * RPW;
    const int64_t row0 = sg.tile_local * rows_per_cta + static_cast<int64_t>(g) * RPW;

    const uint16_t* wrow[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        int64_t n = row0 + r;
        n = n < sg.N ? n : sg.N - 1;    // rows past N stream a valid row; results dropped
        wrow[r] = sg.W + n * sg.ldw;
    }

    const int xstride = p.xstride;
    const int xbuf = B * xstride;      // elements per x buffer
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw + (mcast ? kFmaSmemHead : 0));
    float* red = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(xs) + static_cast<size_t>(p.nbuf) * xbuf * 2);
    float* cpart = red + rows_per_cta * (B + 1) * kw;
    float* misc = cpart + rows_per_cta * B + kMaxSplits;   // cpart: cluster slots, see combine_and_store
    const bool norm = (p.flags & kFlagRmsNorm) != 0;

    const int64_t K = p.K;
    const int64_t k0 = static_cast<int64_t>(split) * p.kslice;
    const int64_t k1 = (k0 + p.kslice < K) ? k0 + p.kslice : K;

    float acc[RPW][B];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) acc[r][b] = 0.f;

    uint4 wv[UJ][RPW];
    bool ok[UJ];
    const uint16_t* wp[RPW];
    bool x_ok = true;   // false when the wait for the multicast copy of x ran out

    // Chunk 0: weight loads go out first; then wait for the preceding grid (x
    // may be its output) and start copying x.
    Chunk ch = chunk_at(k0, k1, p.kchunk, K);
    FmaRange rg = fma_range(ch, kw, kq);
    int v0 = rg.s_begin * 32 + lane;
#pragma unroll
    for (int r = 0; r < RPW; ++r) wp[r] = wrow[r] + ch.c0 + 8 * static_cast<int64_t>(v0);
    issue_batch<RPW, UJ, true>(wv, ok, wp, v0, rg.my_steps, ch.nv, ch.nfull, ch.tail_m);
    // L2 prefetch, p.l2pf batches ahead of the registers: lane 0 asks for the
    // bytes of this warp's rows in warp-steps [pf, upto) of its range, so that
    // the HBM keeps streaming while the warp waits (for the preceding grid, for
    // x, for its registers) without holding registers for the bytes. Called
    // just after the batch at warp-step j was issued (wp and v0 still at j;
    // lane 0's are the warp's first vector).
    const int ahead = p.l2pf * UJ;
    int pf = UJ;   // warp-steps of the range loaded or prefetched so far
    auto prefetch_to = [&](int j, int upto) {
        if (upto > rg.my_steps) upto = rg.my_steps;
        if (upto <= pf) return;
        if (lane == 0) {
            const int va = v0 + 32 * (pf - j);
            int vb = v0 + 32 * (upto - j);
            if (vb > ch.nv) vb = ch.nv;
            if (vb > va) {
#pragma unroll
                for (int r = 0; r < RPW; ++r)
                    l2_prefetch(wp[r] + 256 * (pf - j), 16u * static_cast<uint32_t>(vb - va));
            }
        }
        pf = upto;
    };
    if (ahead) prefetch_to(0, UJ + ahead);
    if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
    if constexpr (mcast) {
        // Every CTA of the cluster has initialised its mbarrier; rank 0 copies
        // the whole vectors of x into all of them (pieces of at most 32 KB);
        // each CTA writes the partial vector at column K itself (zero-filled).
        cluster_wait();
        const uint32_t bytes = 16u * static_cast<uint32_t>(ch.nfull);
        if (threadIdx.x == 0) mbar_arrive_expect_tx(mbar, bytes);
        if (threadIdx.x == 0 && cluster_rank() == 0) {
            const uint16_t mask = static_cast<uint16_t>((1u << p.mcast) - 1u);
            for (uint32_t off = 0; off < bytes; off += 32768u) {
                const uint32_t n = bytes - off < 32768u ? bytes - off : 32768u;
                bulk_copy_multicast(reinterpret_cast<unsigned char*>(xs) + off,
                                    reinterpret_cast<const unsigned char*>(p.x) + off, n, mbar, mask);
            }
        }
        if (ch.tail_m != 0 && threadIdx.x == 32) {
            const int64_t col = 8 * static_cast<int64_t>(ch.nfull);
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t lo = (col + 2 * q < K) ? __ldg(p.x + col + 2 * q) : 0u;
                const uint32_t hi = (col + 2 * q + 1 < K) ? __ldg(p.x + col + 2 * q + 1) : 0u;
                w[q] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(xs + col) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        x_ok = mbar_wait_bounded(mbar, 0);
        // Second phase of the cluster barrier: arrive now, wait just before
        // exit, so that no CTA of the cluster leaves while its peers still run.
        cluster_arrive_relaxed();
    } else {
        stage_x(xs, xstride, p.x, B, K, ch.c0, ch.nv);
    }

#pragma unroll 1
    for (int c = 0;; ++c) {
        const uint16_t* xcur = xs + (c & 1) * xbuf;
        const int64_t next_c0 = ch.c0 + p.kchunk;
        const bool more = CHUNKED && next_c0 < k1;
        Chunk nch{};
        if (more) {   // copy the next chunk of x while this one is used
            nch = chunk_at(next_c0, k1, p.kchunk, K);
            stage_x(xs + ((c + 1) & 1) * xbuf, xstride, p.x, B, K, nch.c0, nch.nv);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        const uint16_t* xl = xcur + 8 * v0;
        consume_batch<B, RPW, UJ, true>(acc, wv, ok, xl, xstride);
        int j = UJ;
        auto advance = [&]() {
#pragma unroll
            for (int r = 0; r < RPW; ++r) wp[r] += 256 * UJ;
            v0 += 32 * UJ;
            xl += 256 * UJ;
        };
        advance();
#pragma unroll 1
        for (; j + UJ <= rg.my_steps && (v0 - lane) + 32 * UJ <= ch.nfull; j += UJ) {
            issue_batch<RPW, UJ, false>(wv, ok, wp, v0, UJ, ch.nv, ch.nfull, 0);
            if (ahead) prefetch_to(j, j + UJ + ahead);
            consume_batch<B, RPW, UJ, false>(acc, wv, ok, xl, xstride);
            advance();
        }
#pragma unroll 1
        for (; j < rg.my_steps; j += UJ) {
            issue_batch<RPW, UJ, true>(wv, ok, wp, v0, rg.my_steps - j, ch.nv, ch.nfull, ch.tail_m);
            if (ahead) prefetch_to(j, j + UJ + ahead);
            consume_batch<B, RPW, UJ, true>(acc, wv, ok, xl, xstride);
            advance();
        }
        if (norm) xsq_accumulate(xcur, xstride, B, ch.nv, misc, c == 0);
        if (!more) break;

        // The next chunk's first weight batch goes out before the barrier that
        // frees this chunk's x buffer.
        ch = nch;
        rg = fma_range(ch, kw, kq);
        v0 = rg.s_begin * 32 + lane;
#pragma unroll
        for (int r = 0; r < RPW; ++r) wp[r] = wrow[r] + ch.c0 + 8 * static_cast<int64_t>(v0);
        issue_batch<RPW, UJ, true>(wv, ok, wp, v0, rg.my_steps, ch.nv, ch.nfull, ch.tail_m);
        pf = UJ;
        if (ahead) prefetch_to(0, UJ + ahead);
        __syncthreads();
    }

    // Lane reduction: the same xor butterfly for every row, so the result does
    // not depend on where a row sits in the grid. A launch whose copy of x did
    // not arrive in time stores NaN (and has set the status bit) rather than
    // sums over an incomplete x.
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = x_ok ? acc[r][b] : __uint_as_float(0x7fc00000u);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[r][b] = v;
        }

    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) red[red_index(kq, rows_per_cta, g * RPW + r, B, b)] = acc[r][b];
    }
    combine_and_store(red, cpart, misc, rows_per_cta, B, kw, S, split, sg.tile_local * rows_per_cta, sg.N, sg.y,
                      norm, K, p.rms_eps, p.wc);
    if constexpr (mcast) {
        // After a timed-out wait the copy may still be in flight into this
        // CTA's shared memory: wait for it once more (bounded) before leaving.
        if (!x_ok) mbar_wait_bounded(mbar, 0);
        cluster_wait();
    }
}

template <int B>
cudaError_t launch_fma(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    constexpr Variant v = fma_variant(B);
    if (l.nbuf > 1) return launch_kernel(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll, true>, p, l, s, pdl);
    if constexpr (B == 1) {
        if (p.mcast > 1)
            return launch_kernel(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll, false, true>, p, l, s, pdl);
    }
    return launch_kernel(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll, false>, p, l, s, pdl);
}

template <int B>
cudaError_t prepare_fma() {
    constexpr Variant v = fma_variant(B);
    cudaError_t e = cudaFuncSetAttribute(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    if constexpr (B == 1) {
        e = cudaFuncSetAttribute(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
        if (e != cudaSuccess) return e;
    }
    return cudaFuncSetAttribute(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

}  // namespace gemv
