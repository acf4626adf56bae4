// Skinny-batch decode GEMV on the BF16 tensor cores (mma.sync m16n8k16, FP32
// accumulate) for sm_103a: y[b][n] = sum_k W[n][k] * x[b][k] with 2 <= B <= 16.
//
// Why tensor cores here: at batch B every weight element feeds B multiply-adds.
// On the CUDA cores that, plus the BF16 widening and the shared-memory x reads,
// costs more issue slots than the byte stream leaves for B >= 4, so the kernel
// would run at the ALU roof, not the HBM roof ("Decode GEMV at half of HBM
// bandwidth", "What interviewers probe next": at batch 16 the operation is a
// skinny GEMM and tensor cores become worth using for the arithmetic). The
// contraction over k is done by the tensor cores; W still streams straight
// from HBM into registers with 16-byte loads and is never staged.
//
// Layout. A warp owns a 16-row tile of W. Lane (g, t) = (lane / 4, lane % 4)
// loads, per 32-column block j, the 16-byte vectors W[row g][32j + 8t .. +7]
// and W[row g + 8][same columns]; the 4 lanes of a row read 64 contiguous
// bytes, whole sectors, and UJ blocks per batch are in flight per lane before
// any is used. Those two vectors ARE the A fragments of two m16n8k16 MMAs
// under a fixed permutation of k: the MMA's k-slots {2t, 2t+1, 2t+8, 2t+9}
// map to physical columns {8t, 8t+1, 8t+2, 8t+3} in the first MMA and
// {8t+4, .., 8t+7} in the second. The B fragments (x, k x batch) use the same
// permutation, so one 16-byte shared-memory read of x[b][32j + 8t .. +7]
// feeds both MMAs; any permutation of k applied to both operands leaves the
// dot products unchanged. Batch rows b >= B enter as zeros.
//
// Accumulation: the 2*UJ MMAs of a batch accumulate into two fresh FP32 tiles
// (even and odd blocks), which are then added to the running tile (blocked
// summation), and the usual
// fixed-order combine over warps and cluster CTAs follows. x staging, the
// programmatic dependent launch and the split-K cluster are those of the
// CUDA-core kernel.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_common.cuh"

namespace gemv {

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// This warp's contiguous range of 32-column blocks within a chunk.
struct MmaRange {
    int j_begin;
    int my_blocks;
    int span;   // blocks per warp group along K
};

__device__ __forceinline__ MmaRange mma_range(const Chunk& c, int kw, int kq) {
    const int nblk = (c.nv + 3) >> 2;
    const int span = (nblk + kw - 1) / kw;
    MmaRange r;
    r.span = span;
    r.j_begin = kq * span;
    const int j_end = (r.j_begin + span < nblk) ? r.j_begin + span : nblk;
    r.my_blocks = j_end > r.j_begin ? j_end - r.j_begin : 0;
    return r;
}

// Issue one batch: UJ 32-column blocks, two 16-byte W loads (rows g and g+8)
// per block per lane. `v` is the lane's vector index for block u = 0.
template <int UJ, bool PRED>
__device__ __forceinline__ void mma_issue(uint4 (&w0)[UJ], uint4 (&w1)[UJ], bool (&ok)[UJ],
                                          const uint16_t* p0, const uint16_t* p1, int v,
                                          int blocks_left, const Chunk& c) {
#pragma unroll
    for (int u = 0; u < UJ; ++u) {
        const int vu = v + 4 * u;
        ok[u] = PRED ? (u < blocks_left && vu < c.nv) : true;
        uint4 a = make_uint4(0u, 0u, 0u, 0u);
        uint4 b = make_uint4(0u, 0u, 0u, 0u);
        if (ok[u]) {
            a = ld_stream16(p0 + 32 * u);
            b = ld_stream16(p1 + 32 * u);
            if (PRED && vu == c.nfull && c.tail_m != 0) {
                a = keep_first(a, c.tail_m);
                b = keep_first(b, c.tail_m);
            }
        }
        w0[u] = a;
        w1[u] = b;
    }
}

// x fragment of vector vu (block vu / 4, lane column 8 (vu % 4)) for batch
// rows g and g + 8: rows `xstride` elements apart; blocks 32 elements apart
// (rows of x staged whole) or, BOXL (x as tensor boxes), boxes of 8 blocks
// 256 B elements apart and blocks within a box `bstride` apart.
template <int NB, bool PRED, bool BOXL>
__device__ __forceinline__ void load_xfrag(uint4 (&xr)[NB], bool ok, const uint16_t* xrow0, int xstride,
                                           int vu, int g, int B, int bstride) {
    const int off = BOXL ? (vu >> 5) * (256 * B) + ((vu >> 2) & 7) * bstride + 8 * (vu & 3) : 8 * vu;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        xr[nb] = make_uint4(0u, 0u, 0u, 0u);
        if ((nb * 8 + g < B) && (!PRED || ok))
            xr[nb] = *reinterpret_cast<const uint4*>(xrow0 + nb * 8 * xstride + off);
    }
}

// Tensor-core multiply-adds of one batch. The x fragments of block u+1 are
// read from shared memory while block u's MMAs run, and even and odd blocks
// accumulate into separate tiles, so neither the shared-memory latency nor
// the MMA latency is exposed block after block.
template <int NB, int UJ, bool PRED, bool BOXL>
__device__ __forceinline__ void mma_consume(float (&acc)[NB][4], const uint4 (&w0)[UJ], const uint4 (&w1)[UJ],
                                            const bool (&ok)[UJ], const uint16_t* xrow0, int xstride,
                                            int v, int g, int B, int bstride) {
    float t[2][NB][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) t[h][nb][i] = 0.f;
    uint4 xr[NB];
    load_xfrag<NB, PRED, BOXL>(xr, ok[0], xrow0, xstride, v, g, B, bstride);
#pragma unroll
    for (int u = 0; u < UJ; ++u) {
        uint4 xn[NB];
        if (u + 1 < UJ)
            load_xfrag<NB, PRED, BOXL>(xn, ok[u + 1 < UJ ? u + 1 : u], xrow0, xstride, v + 4 * (u + 1), g, B,
                                       bstride);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            mma_bf16_16816(t[u & 1][nb], w0[u].x, w1[u].x, w0[u].y, w1[u].y, xr[nb].x, xr[nb].y);
            mma_bf16_16816(t[u & 1][nb], w0[u].z, w1[u].z, w0[u].w, w1[u].w, xr[nb].z, xr[nb].w);
        }
        if (u + 1 < UJ) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) xr[nb] = xn[nb];
        }
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nb][i] += t[0][nb][i] + t[1][nb][i];
}

// How x reaches shared memory (one chunk; x 16-byte aligned, in this GPU's
// memory, for the two copy-engine forms).
constexpr int kXCopy = 0;   // 16-byte asynchronous copies from every thread
constexpr int kXBulk = 1;   // one bulk copy per x row (K a multiple of 8), one mbarrier
constexpr int kXBox = 2;    // tensor boxes in pieces, one mbarrier each (stage_x_boxes; K a multiple of 32)

// CHUNKED: as for the CUDA-core kernel, a separate instance for K-ranges
// staged in several chunks (always with kXCopy).
// XM = kXBulk / kXBox: x is copied by the Tensor Memory Accelerator, issued by
// one thread. The per-thread copies of kXCopy queue behind the first batch of
// W loads the warps have just issued; the copy engine's do not, so x arrives
// while that batch is still landing. With kXBox (more than 8 rows of x, whose
// slice is the largest) a warp starts as soon as the piece its first batch
// reads has landed.
template <int NB, int UJ, bool CHUNKED, int XM = kXCopy>
__global__ void __launch_bounds__(kThreads)
gemv_bf16_mma_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr bool XBULK = XM == kXBulk, XBOX = XM == kXBox;

    pdl_launch_dependents();

    // The copy engine's mbarriers sit in the bytes before x; every thread
    // must see them initialised before it waits on one.
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem_raw);
    if constexpr (XBULK) {
        if (threadIdx.x == 0) {
            mbar_init(mbar, 1);
            fence_mbar_init_cluster();
        }
        __syncthreads();
    }
    if constexpr (XBOX) {
        xpieces_init(mbar);
        __syncthreads();
    }

    const int S = p.splits;
    if (S > 1) cluster_arrive_relaxed();   // see combine_and_store
    const int64_t tile = blockIdx.x / S;
    const int split = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const SegView sg = segment_of(p, tile);

    const int B = p.batch;
    const int kw = p.kw;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gw = warp / kw;        // 16-row tile of this warp within the CTA
    const int kq = warp - gw * kw;   // position of this warp along K within the tile
    const int g = lane >> 2;
    const int t = lane & 3;
    const int rows_per_cta = (kWarps / kw) * kMmaRows;
    const int64_t tile_row0 = sg.tile_local * rows_per_cta + static_cast<int64_t>(gw) * kMmaRows;
    int64_t n0 = tile_row0 + g, n1 = tile_row0 + g + 8;
    n0 = n0 < sg.N ? n0 : sg.N - 1;   // rows past N stream a valid row; results dropped
    n1 = n1 < sg.N ? n1 : sg.N - 1;
    const uint16_t* w0row = sg.W + n0 * sg.ldw;
    const uint16_t* w1row = sg.W + n1 * sg.ldw;

    const int xstride = p.xstride;
    const int xbuf = B * xstride;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw + kBulkSmemHead);
    const int xregion = XBOX ? kw * p.xper * p.xbpp * 8 * B * 32 : p.nbuf * xbuf;   // x elements staged
    float* red = reinterpret_cast<float*>(smem_raw + kBulkSmemHead + static_cast<size_t>(xregion) * 2);
    float* cpart = red + rows_per_cta * (B + 1) * kw;
    float* misc = cpart + rows_per_cta * B + kMaxSplits;   // cpart: cluster slots, see combine_and_store
    const bool norm = (p.flags & kFlagRmsNorm) != 0;

    const int64_t K = p.K;
    const int64_t k0 = static_cast<int64_t>(split) * p.kslice;
    const int64_t k1 = (k0 + p.kslice < K) ? k0 + p.kslice : K;

    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nb][i] = 0.f;

    uint4 w0[UJ], w1[UJ];
    bool ok[UJ];

    Chunk ch = chunk_at(k0, k1, p.kchunk, K);
    MmaRange rg = mma_range(ch, kw, kq);
    int v = 4 * rg.j_begin + t;   // this lane's vector index in the chunk
    const uint16_t* p0 = w0row + ch.c0 + 8 * static_cast<int64_t>(v);
    const uint16_t* p1 = w1row + ch.c0 + 8 * static_cast<int64_t>(v);
    mma_issue<UJ, true>(w0, w1, ok, p0, p1, v, rg.my_blocks, ch);
    if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
    bool x_ok = true;   // false when a wait for a copy of x ran out (or x could not be copied)
    // kXBox: this warp group's x, its first piece barrier, the next piece to
    // wait for and the blocks per piece.
    const uint16_t* xgroup = xs;
    uint64_t* gbars = mbar;
    int xnext = 0;
    int piece_blocks = 1;
    if constexpr (XBOX) {
        const int group_elems = p.xper * p.xbpp * 8 * B * 32;
        xgroup = xs + static_cast<int64_t>(kq) * group_elems;
        gbars = mbar + kq * p.xper;
        piece_blocks = 8 * p.xbpp;
        if ((smem_addr(xs) & 127) == 0) {   // a tensor copy needs a 128-byte aligned destination
            stage_x_boxes(mbar, &p.xmap, kw, rg.span, p.xper, p.xbpp, xs, B, ch.c0 / 32, p.xwide != 0);
        } else {
            x_ok = false;
            xnext = p.xper;   // nothing was issued: wait for nothing
            if (threadIdx.x == 0) atomicOr(&g_device_status, kStatusWaitTimeout);
        }
    } else if constexpr (XBULK) {
        bulk_stage_x(mbar, xs, xstride, p.x, B, K, ch.c0, ch.nv);   // K % 8 == 0: whole vectors
        x_ok = mbar_wait_bounded(mbar, 0);
    } else {
        stage_x_rows(xs, xstride, p.x, B, K, ch.c0, ch.nv);
    }

    // x row stride in shared memory, and (kXBox) the stride of blocks within a box.
    const int xrs = XBOX ? (p.xwide ? 256 : 32) : xstride;
    const int xbs = p.xwide ? 32 : B * 32;
#pragma unroll 1
    for (int c = 0;; ++c) {
        const uint16_t* xrow0 = XBOX ? xgroup + g * xrs : xs + (c & 1) * xbuf + g * xstride;
        int xv = XBOX ? t : v;   // the lane's x vector index: in the group's boxes or the chunk
        const int64_t next_c0 = ch.c0 + p.kchunk;
        const bool more = CHUNKED && next_c0 < k1;
        Chunk nch{};
        if (more) {
            nch = chunk_at(next_c0, k1, p.kchunk, K);
            stage_x_rows(xs + ((c + 1) & 1) * xbuf, xstride, p.x, B, K, nch.c0, nch.nv);
            cp_async_wait<1>();
        } else if constexpr (XM == kXCopy) {
            cp_async_wait<0>();
        }
        if constexpr (XM == kXCopy) __syncthreads();   // otherwise the mbarrier waits make x visible

        if constexpr (XBOX) x_ok = xpieces_wait(gbars, xnext, 0) && x_ok;
        mma_consume<NB, UJ, true, XBOX>(acc, w0, w1, ok, xrow0, xrs, xv, g, B, xbs);
        int j = UJ;
        auto advance = [&]() {
            p0 += 32 * UJ;
            p1 += 32 * UJ;
            v += 4 * UJ;
            xv += 4 * UJ;
        };
        advance();
#pragma unroll 1
        for (; j + UJ <= rg.my_blocks && (v - t) + 4 * UJ <= ch.nfull; j += UJ) {
            mma_issue<UJ, false>(w0, w1, ok, p0, p1, v, UJ, ch);
            if constexpr (XBOX) x_ok = xpieces_wait(gbars, xnext, j / piece_blocks) && x_ok;
            mma_consume<NB, UJ, false, XBOX>(acc, w0, w1, ok, xrow0, xrs, xv, g, B, xbs);
            advance();
        }
#pragma unroll 1
        for (; j < rg.my_blocks; j += UJ) {
            mma_issue<UJ, true>(w0, w1, ok, p0, p1, v, rg.my_blocks - j, ch);
            if constexpr (XBOX) x_ok = xpieces_wait(gbars, xnext, j / piece_blocks) && x_ok;
            mma_consume<NB, UJ, true, XBOX>(acc, w0, w1, ok, xrow0, xrs, xv, g, B, xbs);
            advance();
        }
        if (norm) xsq_accumulate(xs + (c & 1) * xbuf, xstride, B, ch.nv, misc, c == 0);   // never with kXBox
        if (!more) break;

        ch = nch;
        rg = mma_range(ch, kw, kq);
        v = 4 * rg.j_begin + t;
        p0 = w0row + ch.c0 + 8 * static_cast<int64_t>(v);
        p1 = w1row + ch.c0 + 8 * static_cast<int64_t>(v);
        mma_issue<UJ, true>(w0, w1, ok, p0, p1, v, rg.my_blocks, ch);
        __syncthreads();
    }

    // acc[nb] holds D[row g][b], D[row g][b+1], D[row g+8][b], D[row g+8][b+1]
    // with b = 8*nb + 2t. A CTA whose copy of x did not arrive in time stores
    // NaN (and has set the status bit) rather than sums over an incomplete x.
    const int rl0 = gw * kMmaRows + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = nb * 8 + 2 * t + (i & 1);
            const int rl = rl0 + ((i & 2) ? 8 : 0);
            if (b < B) red[red_index(kq, rows_per_cta, rl, B, b)] = x_ok ? acc[nb][i] : __uint_as_float(0x7fc00000u);
        }
    }
    combine_and_store(red, cpart, misc, rows_per_cta, B, kw, S, split, sg.tile_local * rows_per_cta, sg.N, sg.y,
                      norm, K, p.rms_eps, p.wc);
    // Pieces no warp of this CTA read (ranges shorter than the planned ones),
    // and, after a timed-out wait, copies still in flight: every issued copy
    // has landed before the CTA leaves (bounded waits).
    if constexpr (XBOX) {
        if ((smem_addr(xs) & 127) == 0) xpieces_wait_all(mbar, kw * p.xper);
    }
    if constexpr (XBULK) {
        if (!x_ok) mbar_wait_bounded(mbar, 0);
    }
}

// The tensor-box instance exists for more than 8 rows of x (NB = 2) only.
template <int NB>
cudaError_t launch_mma(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    if (l.nbuf > 1) return launch_kernel(gemv_bf16_mma_kernel<NB, kMmaUnroll, true>, p, l, s, pdl);
    if constexpr (NB == 2) {
        if (l.xbox) return launch_kernel(gemv_bf16_mma_kernel<NB, kMmaUnroll, false, kXBox>, p, l, s, pdl);
    }
    if (l.xbox) return cudaErrorInvalidValue;
    if (l.xbulk) return launch_kernel(gemv_bf16_mma_kernel<NB, kMmaUnroll, false, kXBulk>, p, l, s, pdl);
    return launch_kernel(gemv_bf16_mma_kernel<NB, kMmaUnroll, false>, p, l, s, pdl);
}

template <int NB>
cudaError_t prepare_mma() {
    cudaError_t e = cudaFuncSetAttribute(gemv_bf16_mma_kernel<NB, kMmaUnroll, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(gemv_bf16_mma_kernel<NB, kMmaUnroll, false, kXBulk>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem)) != cudaSuccess)
        return e;
    if constexpr (NB == 2) {
        if ((e = cudaFuncSetAttribute(gemv_bf16_mma_kernel<NB, kMmaUnroll, false, kXBox>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem)) != cudaSuccess)
            return e;
    }
    return cudaFuncSetAttribute(gemv_bf16_mma_kernel<NB, kMmaUnroll, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

// Status bits this translation unit's kernels recorded (bulk-copy waits that
// ran out), cleared when `reset`.
inline cudaError_t read_mma_status(unsigned int* bits, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess || !reset || *bits == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace gemv
