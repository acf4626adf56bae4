// Decode GEMV with group-quantised INT4 weights, BF16 activations, FP32
// accumulation, for sm_103a: y[b][n] = sum_k ((u[n][k] - 8) * S[n][k/128]) * x[b][k].
//
// "Decode GEMV at half of HBM bandwidth", "What interviewers probe next": with
// INT4 weights the bytes fall four times and the kernel has to unpack in
// registers while the next loads are outstanding. Unpacking four bits into an
// FP32 multiply-add costs more issue slots per weight byte than the CUDA cores
// have at HBM speed, so every batch size (1..16) runs the contraction on the
// BF16 tensor cores; the dequantisation is a shift, one three-input logic
// operation and one BF16 subtraction per pair of codes.
//
// Weight layout (see include/gemv.h): per row, 32-bit words of eight codes,
// even k in the low half-word, odd k in the high half-word, so that
//     ((w >> 4j) & 0x000F000F) | 0x43004300
// is a BF16 pair (128 + u[k], 128 + u[k+1]) for k = 8w' + 2j, and subtracting
// the BF16 pair (136, 136) leaves (u - 8) for both, exactly.
//
// Mapping. A warp owns a 16-row tile; lane (g, t) = (lane / 4, lane % 4) loads,
// per 128-column group, 16 bytes (32 codes, columns 32t .. 32t+31 of the group)
// of row g and of row g + 8, and the two rows' scales. The 4 lanes of a row
// team cover the whole group, so the 8 MMAs of a slot (m16n8k16 each: two per
// 32-bit word) sum exactly one group, which is then scaled by the row's
// S[n][group] and added to the running FP32 tile. As in the BF16 tensor-core
// kernel, a fixed permutation of k pairs each lane's dequantised codes with the
// x values in the same columns (one 16-byte shared-memory read of x per word;
// x rows are swizzled so the four lanes of a row team hit distinct banks),
// x is staged per CTA with asynchronous copies, the first batch of loads goes
// out before the programmatic-dependent-launch wait, and partial sums combine
// in a fixed order over warps and cluster CTAs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_common.cuh"
#include "gemv_mma_kernel.cuh"

namespace gemv {

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
    uint16_t v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Four BF16 pairs (u - 8) from one word of eight codes: out[j] holds the codes
// of columns 8w + 2j (low half) and 8w + 2j + 1 (high half). The mask and the
// exponent bits go in one three-input logic operation ((a & b) | c, truth table
// 0xEA); written as two C++ operators after a shift they cost two.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t (&out)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t biased;   // 128 + u, both halves
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(biased) : "r"(w >> (4 * j)), "r"(0x000F000Fu), "r"(0x43004300u));
        uint32_t q;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(biased), "r"(0x43084308u));  // - 136
        out[j] = q;
    }
}

// This warp's contiguous range of 128-column groups within a chunk.
struct W4Range {
    int j_begin;
    int my_groups;
};

__device__ __forceinline__ W4Range w4_range(int ngroups, int kw, int kq) {
    const int span = (ngroups + kw - 1) / kw;
    W4Range r;
    r.j_begin = kq * span;
    const int j_end = (r.j_begin + span < ngroups) ? r.j_begin + span : ngroups;
    r.my_groups = j_end > r.j_begin ? j_end - r.j_begin : 0;
    return r;
}

// Launch bounds: 3 CTAs per SM for the standard one-block instance, 2 for
// the others (the occupancy the planner assumes for each).
template <int NB, int UJ, bool CHUNKED>
__global__ void __launch_bounds__(kThreads, NB == 2 ? 2 : (UJ == kW4Unroll && !CHUNKED) ? 3 : 0)
gemv_w4_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];

    pdl_launch_dependents();

    const int S = p.splits;
    if (S > 1) cluster_arrive_relaxed();   // see combine_and_store
    const int64_t tile = blockIdx.x / S;
    const int split = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const SegView sg = segment_of(p, tile);
    const uint16_t* __restrict__ Sseg = sg.S;
    const int64_t lds = sg.lds;
    const uint8_t* __restrict__ Wq = reinterpret_cast<const uint8_t*>(sg.W);

    const int B = p.batch;
    const int kw = p.kw;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gw = warp / kw;
    const int kq = warp - gw * kw;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int rows_per_cta = (kWarps / kw) * kMmaRows;
    const int64_t tile_row0 = sg.tile_local * rows_per_cta + static_cast<int64_t>(gw) * kMmaRows;
    int64_t n0 = tile_row0 + g, n1 = tile_row0 + g + 8;
    n0 = n0 < sg.N ? n0 : sg.N - 1;   // rows past N stream a valid row; results dropped
    n1 = n1 < sg.N ? n1 : sg.N - 1;
    // This lane's 16-byte slice (columns 32t .. 32t+31 of a group) of rows n0 and
    // n1 at column 0; ldw is the row stride in bytes here.
    const uint8_t* q0p = Wq + n0 * sg.ldw + 16 * t;
    const uint8_t* q1p = Wq + n1 * sg.ldw + 16 * t;
    const uint16_t* s0p = Sseg + n0 * lds;
    const uint16_t* s1p = Sseg + n1 * lds;

    const int xstride = p.xstride;
    const int xbuf = B * xstride;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);
    float* red = reinterpret_cast<float*>(smem_raw + static_cast<size_t>(p.nbuf) * xbuf * 2);
    float* cpart = red + rows_per_cta * (B + 1) * kw;
    float* misc = cpart + rows_per_cta * B + kMaxSplits;   // cpart: cluster slots, see combine_and_store
    const bool norm = (p.flags & kFlagRmsNorm) != 0;

    // Byte offset, within one staged x buffer, of the 8 columns that word m of
    // this lane's slice multiplies in group 0: batch row b, vector 4t + m at its
    // swizzled place xswz(16 j + 4t + m) = 16 j + 4t + (m ^ (t & 2)). Group j
    // adds 256 bytes.
    uint32_t xo[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int b = (nb * 8 + g < B) ? nb * 8 + g : B - 1;
#pragma unroll
        for (int m = 0; m < 4; ++m) xo[nb][m] = 2u * static_cast<uint32_t>(b * xstride + 8 * (4 * t + (m ^ (t & 2))));
    }

    const int64_t K = p.K;
    const int64_t k0 = static_cast<int64_t>(split) * p.kslice;
    const int64_t k1 = (k0 + p.kslice < K) ? k0 + p.kslice : K;

    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nb][i] = 0.f;

    uint4 qa[UJ], qb[UJ];
    uint16_t sa[UJ], sb[UJ];
    int rg_begin = 0;   // first group of this warp's range in the current chunk
    // L2 prefetch, p.l2pf batches ahead of the registers: with each batch the
    // lanes with t == 0 (whose slices start their rows' groups) ask for their
    // two rows' bytes of groups [pf, jr + UJ + ahead) of the warp's range (64
    // bytes per group and row, contiguous), so that the HBM keeps streaming
    // while the warp waits, without registers held for the bytes.
    const int ahead = p.l2pf * UJ;
    int pf = 0;   // groups of the range loaded or prefetched so far

    // Issue the slots of groups jr .. jr+UJ-1 of this warp's range (chunk at c0).
    // A full batch addresses its slots by immediate offsets; the last, partial
    // batch repeats its last group in the unused slots, which are not consumed.
    auto issue = [&](int64_t c0, int jr, int my) {
        const int rem = my - jr;
        if (rem <= 0) return;
        const int64_t col0 = c0 + 128LL * (rg_begin + jr);
        const uint8_t* a0 = q0p + (col0 >> 1);
        const uint8_t* a1 = q1p + (col0 >> 1);
        const uint16_t* z0 = s0p + (col0 >> 7);
        const uint16_t* z1 = s1p + (col0 >> 7);
        if (ahead) {
            const int upto = rem < UJ + ahead ? my : jr + UJ + ahead;
            const int from = pf > jr + UJ ? pf : jr + UJ;
            if (t == 0 && upto > from) {
                const uint32_t bytes = 64u * static_cast<uint32_t>(upto - from);
                l2_prefetch(a0 + 64 * (from - jr), bytes);
                l2_prefetch(a1 + 64 * (from - jr), bytes);
            }
            pf = upto > from ? upto : from;
        }
        if (rem >= UJ) {
#pragma unroll
            for (int u = 0; u < UJ; ++u) {
                qa[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a0 + 64 * u));
                qb[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a1 + 64 * u));
                sa[u] = ld_stream_u16(z0 + u);
                sb[u] = ld_stream_u16(z1 + u);
            }
        } else {
#pragma unroll
            for (int u = 0; u < UJ; ++u) {
                const int uu = u < rem ? u : rem - 1;
                qa[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a0 + 64 * uu));
                qb[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a1 + 64 * uu));
                sa[u] = ld_stream_u16(z0 + uu);
                sb[u] = ld_stream_u16(z1 + uu);
            }
        }
    };

    // Contract slot u (one 128-column group of rows n0, n1) with x at xg (the
    // staged x of this batch's first group) and add it, scaled, to acc.
    auto consume = [&](int u, const unsigned char* xg) {
        float d[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) d[nb][i] = 0.f;
        const uint32_t wa[4] = {qa[u].x, qa[u].y, qa[u].z, qa[u].w};
        const uint32_t wb[4] = {qb[u].x, qb[u].y, qb[u].z, qb[u].w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t A[4], Bq[4];
            dequant_word(wa[m], A);
            dequant_word(wb[m], Bq);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const uint4 xr = *reinterpret_cast<const uint4*>(xg + xo[nb][m] + 256 * u);
                mma_bf16_16816(d[nb], A[0], Bq[0], A[1], Bq[1], xr.x, xr.y);
                mma_bf16_16816(d[nb], A[2], Bq[2], A[3], Bq[3], xr.z, xr.w);
            }
        }
        const float s_a = __uint_as_float(static_cast<uint32_t>(sa[u]) << 16);
        const float s_b = __uint_as_float(static_cast<uint32_t>(sb[u]) << 16);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] = fmaf(d[nb][0], s_a, acc[nb][0]);
            acc[nb][1] = fmaf(d[nb][1], s_a, acc[nb][1]);
            acc[nb][2] = fmaf(d[nb][2], s_b, acc[nb][2]);
            acc[nb][3] = fmaf(d[nb][3], s_b, acc[nb][3]);
        }
    };

    Chunk ch = chunk_at(k0, k1, p.kchunk, K);
    int ngroups = (ch.nv + 15) >> 4;
    W4Range rg = w4_range(ngroups, kw, kq);
    rg_begin = rg.j_begin;
    issue(ch.c0, 0, rg.my_groups);
    if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
    stage_x<true>(xs, xstride, p.x, B, K, ch.c0, ch.nv);

#pragma unroll 1
    for (int c = 0;; ++c) {
        const unsigned char* xsb = reinterpret_cast<const unsigned char*>(xs + (c & 1) * xbuf);
        const int64_t next_c0 = ch.c0 + p.kchunk;
        const bool more = CHUNKED && next_c0 < k1;
        Chunk nch{};
        if (more) {
            nch = chunk_at(next_c0, k1, p.kchunk, K);
            stage_x<true>(xs + ((c + 1) & 1) * xbuf, xstride, p.x, B, K, nch.c0, nch.nv);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        const int my = rg.my_groups;
#pragma unroll 1
        for (int j0 = 0; j0 < my; j0 += UJ) {
            if (j0 > 0) issue(ch.c0, j0, my);
            const unsigned char* xg = xsb + 256 * (rg_begin + j0);
            const int rem = my - j0;
            if (rem >= UJ) {
#pragma unroll
                for (int u = 0; u < UJ; ++u) consume(u, xg);
            } else {
#pragma unroll
                for (int u = 0; u < UJ; ++u)
                    if (u < rem) consume(u, xg);
            }
        }
        if (norm) xsq_accumulate(reinterpret_cast<const uint16_t*>(xsb), xstride, B, ch.nv, misc, c == 0);
        if (!more) break;

        ch = nch;
        ngroups = (ch.nv + 15) >> 4;
        rg = w4_range(ngroups, kw, kq);
        rg_begin = rg.j_begin;
        pf = 0;
        issue(ch.c0, 0, rg.my_groups);
        __syncthreads();
    }

    const int rl0 = gw * kMmaRows + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = nb * 8 + 2 * t + (i & 1);
            const int rl = rl0 + ((i & 2) ? 8 : 0);
            if (b < B) red[red_index(kq, rows_per_cta, rl, B, b)] = acc[nb][i];
        }
    }
    combine_and_store(red, cpart, misc, rows_per_cta, B, kw, S, split, sg.tile_local * rows_per_cta, sg.N, sg.y,
                      norm, K, p.rms_eps, p.wc);
}

template <int NB>
cudaError_t launch_w4(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    if (l.unroll == kW4DeepUnroll) {   // the deep instance: up to 8 rows, one x chunk
        if (NB != 1 || l.nbuf != 1) return cudaErrorInvalidValue;
        return launch_kernel(gemv_w4_kernel<1, kW4DeepUnroll, false>, p, l, s, pdl);
    }
    if (l.unroll != kW4Unroll) return cudaErrorInvalidValue;
    if (l.nbuf > 1) return launch_kernel(gemv_w4_kernel<NB, kW4Unroll, true>, p, l, s, pdl);
    return launch_kernel(gemv_w4_kernel<NB, kW4Unroll, false>, p, l, s, pdl);
}

template <int NB>
cudaError_t prepare_w4() {
    cudaError_t e = cudaFuncSetAttribute(gemv_w4_kernel<NB, kW4Unroll, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    if (NB == 1 && (e = cudaFuncSetAttribute(gemv_w4_kernel<1, kW4DeepUnroll, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem)) !=
                       cudaSuccess)
        return e;
    return cudaFuncSetAttribute(gemv_w4_kernel<NB, kW4Unroll, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

}  // namespace gemv
