// Device helpers shared by the decode-GEMV kernels: streaming loads, BF16
// unpacking, programmatic dependent launch, cluster / distributed shared memory,
// asynchronous x staging and the fixed-order combine of partial sums.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_internal.h"

namespace gemv {

// 16-byte weight load: read-only path, not allocated in L1 (W is read once).
__device__ __forceinline__ uint4 ld_stream16(const uint16_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// BF16 -> FP32 is exact: the BF16 bits are the high half of the FP32 pattern.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Keep the first m (1..7) BF16 elements of an 8-element vector, zero the rest
// (bits are selected, so a NaN in the padding never enters a product).
__device__ __forceinline__ uint4 keep_first(uint4 v, int m) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t keep = (2 * q < m ? 0x0000ffffu : 0u) | (2 * q + 1 < m ? 0xffff0000u : 0u);
        w[q] &= keep;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Split cluster barrier: every CTA of a cluster along K arrives at kernel
// entry and waits just before its first store into another CTA's shared
// memory, so that no CTA writes there before the owner has started.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Generic address of the same shared-memory location in CTA `rank` of this
// cluster. Stores through it are ordinary stores; the cluster barrier that
// follows them (release / acquire) makes them visible to that CTA.
__device__ __forceinline__ float* dsmem_at(float* local, uint32_t rank) {
    uint64_t r;
    asm("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(local), "r"(rank));
    return reinterpret_cast<float*>(r);
}

// i / B for 0 <= i < 2^16 and 2 <= B <= 16 with magic = 0xFFFFFFFF / B + 1
// (ceil(2^32 / B), or 2^32 / B exactly when B is a power of two): the
// rounding up adds less than i * B / 2^32 < 1/B to i / B, too little to
// reach the next integer.
__device__ __forceinline__ int div_by_batch(int i, int B, uint32_t magic) {
    return B == 1 ? i : static_cast<int>(__umulhi(static_cast<uint32_t>(i), magic));
}

// ---- x multicast (batch 1, one K chunk): one bulk copy per cluster ------------
//
// Every CTA of a launch without a K split stages the same x. With a cluster of
// C CTAs along the rows, the CTA of rank 0 copies x once from global memory
// into the shared memory of all C CTAs (cp.async.bulk with .multicast::cluster,
// the Tensor Memory Accelerator's 1-D copy); each CTA's mbarrier counts the
// bytes that arrive in its own shared memory. The L2 then serves x once per
// cluster instead of once per CTA, which matters at kernel start, when every
// CTA asks for x at the same moment.

// Device status word of this translation unit: bit 0 is set when an mbarrier
// wait ran out of iterations (the copy it waited for never completed). Read and
// cleared by the host through gemv_device_status.
static __device__ unsigned int g_device_status;
constexpr unsigned int kStatusWaitTimeout = 1u;
#ifdef GEMV_DEBUG_DROP_X
constexpr int kMbarWaitLimit = 1 << 14;      // the test build whose waits are meant to run out
#else
constexpr int kMbarWaitLimit = 1 << 20;      // try_wait rounds before giving up
#endif

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make this CTA's mbarrier initialisation visible to the cluster (the copy
// engine of another CTA's bulk copy completes transactions on it).
__device__ __forceinline__ void fence_mbar_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive on the barrier and add `bytes` to the transactions it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Wait for phase `parity` of the barrier to complete, for at most
// kMbarWaitLimit rounds of try_wait (each returns when the phase completes or
// after a time limit of the hardware's choosing). Returns false, and sets the
// status bit, if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_addr(bar);
#pragma unroll 1
    for (int it = 0; it < kMbarWaitLimit; ++it) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred P1;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 P1, [%1], %2;\n\t"
                     "selp.b32 %0, 1, 0, P1;\n\t}"
                     : "=r"(done) : "r"(a), "r"(parity) : "memory");
        if (done) return true;
    }
    atomicOr(&g_device_status, kStatusWaitTimeout);
    return false;
}

// Copy `bytes` (a multiple of 16, 16-byte aligned source) from global memory
// to the same shared-memory offset `dst` in every CTA of `mask`, completing
// `bytes` transactions on the mbarrier at the same offset `bar` in each.
__device__ __forceinline__ void bulk_copy_multicast(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                    uint16_t mask) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "h"(mask) : "memory");
}

// Ask the L2 for `bytes` (a multiple of 16) of global memory from `src`
// (16-byte aligned, this GPU's memory) without waiting for them or holding a
// register: the TMA's bulk prefetch. The later loads of those bytes then hit L2.
__device__ __forceinline__ void l2_prefetch(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// Copy `bytes` (a multiple of 16, both addresses 16-byte aligned) from global
// memory into this CTA's shared memory at `dst`, completing `bytes`
// transactions on the mbarrier `bar` (the Tensor Memory Accelerator's 1-D copy).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// x by bulk copies (one thread, one copy per x row, in pieces of at most
// 32 KB), counted on the mbarrier `bar`: rows b < B of x[b][c0 .. c0 + 8 nv)
// into xs (row stride xstride elements). Needs x 16-byte aligned, K a multiple
// of 8, c0 a multiple of 8 and xstride a multiple of 8, so that every piece
// starts and ends on a 16-byte boundary on both sides. Thread 0 arms the
// barrier with the byte count and issues the copies; every thread then waits
// with mbar_wait_bounded (the barrier was initialised, and made visible to the
// CTA, before).
__device__ __forceinline__ void bulk_stage_x(uint64_t* bar, uint16_t* xs, int xstride, const uint16_t* x, int B,
                                             int64_t K, int64_t c0, int nv) {
    if (threadIdx.x != 0) return;
    const uint32_t row_bytes = 16u * static_cast<uint32_t>(nv);
    mbar_arrive_expect_tx(bar, row_bytes * static_cast<uint32_t>(B));
    for (int b = 0; b < B; ++b) {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(x + static_cast<int64_t>(b) * K + c0);
        unsigned char* dst = reinterpret_cast<unsigned char*>(xs + static_cast<int64_t>(b) * xstride);
        for (uint32_t off = 0; off < row_bytes; off += 32768u) {
            const uint32_t n = row_bytes - off < 32768u ? row_bytes - off : 32768u;
            bulk_copy(dst + off, src + off, n, bar);
        }
    }
}

// ---- x as tensor boxes, in pieces with one mbarrier each -----------------------
//
// The tensor-core kernel stages x with the Tensor Memory Accelerator's tensor
// copies (cp.async.bulk.tensor) through a 3-D view of x, so that one copy
// moves a whole piece (all B rows of several 256-column boxes), where one copy
// per row and piece would cost the issuing thread tens of nanoseconds each.
// Each piece is counted on its own mbarrier, so a warp waits only for the
// piece its next batch reads: the first piece lands in a fraction of the time
// the whole slice takes, and the rest land while the warps stream W.
//   narrow: 32 columns (one MMA block) x B rows x K / 32 blocks; a box lands
//     block-major, [block][row][32 columns]: rows of one block are 64 bytes
//     apart, so the two rows a quarter-warp reads for its x fragments fall in
//     different banks;
//   wide: 256 columns x B rows x K / 256; a box lands [row][256 columns]
//     (rows 512 bytes apart: those two rows share banks), in fewer and longer
//     requests.
// Geometry: warp group kq of the kw groups along K takes the blocks
// [kq * span, (kq + 1) * span) of the CTA's slice; its range is cut into `per`
// pieces of `bpp` boxes of 8 blocks (one batch of UJ = 8 blocks per box), so a
// batch never reads two pieces. Piece r of group kq is counted on mbarrier
// kq * per + r and lands at xs + (kq * per + r) * bpp * 8 * B * 32. Boxes past
// the end of the tensor are zero-filled by the copy engine.

__device__ __forceinline__ void xpieces_init(uint64_t* bars) {
    if (threadIdx.x == 0) {
        for (int q = 0; q < kMaxXPieces; ++q) mbar_init(bars + q, 1);
        fence_mbar_init_cluster();
    }
}

// 3-D tensor copy of one box at coordinates (0, 0, blk) into shared memory,
// completing its bytes on the mbarrier `bar`. `map` is the kernel parameter
// holding the tensor map (param space, so no proxy fence is needed).
__device__ __forceinline__ void tensor_copy_3d(void* dst, const void* map, int blk, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];"
                 :: "r"(smem_addr(dst)), "l"(map), "r"(0), "r"(0), "r"(blk), "r"(smem_addr(bar)) : "memory");
}

// Thread 0 arms every piece's mbarrier with its bytes and issues its copy,
// piece 0 of every group first. blk0: the slice's first block (column / 32);
// wide boxes are addressed in units of 8 blocks (blk0 and span multiples of 8).
__device__ __forceinline__ void stage_x_boxes(uint64_t* bars, const void* map, int kw, int span, int per, int bpp,
                                              uint16_t* xs, int B, int64_t blk0, bool wide) {
    if (threadIdx.x != 0) return;
    const int piece_elems = bpp * 8 * B * 32;
    const uint32_t piece_bytes = 2u * static_cast<uint32_t>(piece_elems);
    for (int r = 0; r < per; ++r) {
        for (int kq = 0; kq < kw; ++kq) {
            uint64_t* bar = bars + kq * per + r;
            mbar_arrive_expect_tx(bar, piece_bytes);
            const int64_t blk = blk0 + kq * span + r * 8 * bpp;
            tensor_copy_3d(xs + static_cast<int64_t>(kq * per + r) * piece_elems, map,
                           static_cast<int>(wide ? blk / 8 : blk), bar);
        }
    }
}

// Wait (bounded) for pieces next .. r of this warp's group (`gbars` = its
// first barrier); false if a wait ran out.
__device__ __forceinline__ bool xpieces_wait(uint64_t* gbars, int& next, int r) {
    bool ok = true;
    for (; next <= r; ++next) ok = mbar_wait_bounded(gbars + next, 0) && ok;
    return ok;
}

// Wait (bounded) for the first n barriers.
__device__ __forceinline__ bool xpieces_wait_all(uint64_t* bars, int n) {
    bool ok = true;
    for (int q = 0; q < n; ++q) ok = mbar_wait_bounded(bars + q, 0) && ok;
    return ok;
}

// 16-byte asynchronous global->shared copy of `nbytes` (2..16) bytes; the rest
// of the 16 bytes is zero-filled. Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, int nbytes) {
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(gmem_src), "r"(nbytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most `pending` of this thread's committed copy groups are in flight.
template <int pending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" :: "n"(pending) : "memory");
}

// Copy x[b][c0 .. c0 + 8*nv) for b < B into shared memory (row stride
// xstride; with SWZ, vector i of a row at position xswz(i)), zero-filling
// columns >= K. Aligned 16-byte pieces go out as
// asynchronous copies, all in flight at once and holding no registers;
// misaligned ones (rows of x start at 2-byte offsets when K % 8 != 0) are
// loaded element by element. Commits one copy group.
// Position of x vector i in a swizzled row: bit 1 flips with bit 3, so the
// four 64-byte-apart vectors that the lanes of an INT4 row team read at once
// fall on distinct banks (with rows 16 bytes apart mod 128).
__device__ __forceinline__ int xswz(int i) { return i ^ (((i >> 3) & 1) << 1); }

template <bool SWZ = false>
__device__ __forceinline__ void stage_x(uint16_t* xs, int xstride, const uint16_t* __restrict__ x,
                                        int B, int64_t K, int64_t c0, int nv) {
    const int items = B * nv;
#pragma unroll 4
    for (int it = threadIdx.x; it < items; it += kThreads) {
        const int b = (B == 1) ? 0 : it / nv;
        const int i = it - b * nv;
        const int64_t col = c0 + 8 * static_cast<int64_t>(i);
        const uint16_t* src = x + static_cast<int64_t>(b) * K + col;
        uint16_t* dst = xs + static_cast<int64_t>(b) * xstride + 8 * (SWZ ? xswz(i) : i);
        if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
            cp_async16(dst, src, (col + 8 <= K) ? 16 : static_cast<int>(K - col) * 2);
        } else {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t lo = (col + 2 * q < K) ? __ldg(src + 2 * q) : 0u;
                uint32_t hi = (col + 2 * q + 1 < K) ? __ldg(src + 2 * q + 1) : 0u;
                w[q] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    cp_async_commit();
}

// stage_x for B >= 2 rows without a division per piece: pieces (b, i),
// numbered b * nv + i, are taken with stride kThreads as in stage_x, but the
// position advances by (db, di) per step with one carry, so every thread of
// the CTA stays busy whatever nv is. Same copies, same zero fill, one copy
// group.
__device__ __forceinline__ void stage_x_rows(uint16_t* xs, int xstride, const uint16_t* __restrict__ x,
                                             int B, int64_t K, int64_t c0, int nv) {
    if (nv > 0) {
        int b = static_cast<int>(threadIdx.x) / nv;
        int i = static_cast<int>(threadIdx.x) - b * nv;
        const int db = kThreads / nv;
        const int di = kThreads - db * nv;
#pragma unroll 1
        for (; b < B; i += di, b += db) {
            if (i >= nv) {
                i -= nv;
                ++b;
                if (b >= B) break;
            }
            const int64_t col = c0 + 8 * static_cast<int64_t>(i);
            const uint16_t* s = x + static_cast<int64_t>(b) * K + col;
            uint16_t* d = xs + static_cast<int64_t>(b) * xstride + 8 * i;
            if ((reinterpret_cast<uintptr_t>(s) & 15u) == 0) {
                cp_async16(d, s, (col + 8 <= K) ? 16 : static_cast<int>(K - col) * 2);
            } else {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t lo = (col + 2 * q < K) ? __ldg(s + 2 * q) : 0u;
                    uint32_t hi = (col + 2 * q + 1 < K) ? __ldg(s + 2 * q + 1) : 0u;
                    w[q] = lo | (hi << 16);
                }
                *reinterpret_cast<uint4*>(d) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    cp_async_commit();
}

// Geometry of one staged chunk of K, [c0, c1), in 8-column vectors.
struct Chunk {
    int64_t c0;
    int nfull;    // whole vectors
    int nv;       // vectors including a partial one at column K
    int tail_m;   // valid columns of the partial vector (0 if none)
};

__device__ __forceinline__ Chunk chunk_at(int64_t c0, int64_t k1, int64_t kchunk, int64_t K) {
    Chunk c;
    const int64_t c1 = (c0 + kchunk < k1) ? c0 + kchunk : k1;
    c.c0 = c0;
    c.nfull = static_cast<int>((c1 - c0) >> 3);
    const bool tailv = (c1 == K) && ((K & 7) != 0);
    c.nv = c.nfull + (tailv ? 1 : 0);
    c.tail_m = tailv ? static_cast<int>(K - (c0 + 8 * static_cast<int64_t>(c.nfull))) : 0;
    return c;
}

// Sum of squares of the staged x rows (the RMSNorm statistic), from the chunk
// in xbuf: every thread takes vectors tid, tid + kThreads, ...; lanes combine by
// xor butterfly, warps in index order. The CTA total for row b goes to
// misc[kWarps * kMaxBatch + b] (first chunk: assigned, later chunks: added).
// Called by every thread of the CTA; zero-filled columns >= K add nothing.
__device__ __forceinline__ void xsq_accumulate(const uint16_t* xbuf, int xstride, int B, int nv,
                                               float* misc, bool first) {
    float* wsum = misc;
    float* xsq = misc + kWarps * kMaxBatch;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int b = 0; b < B; ++b) {
        float s = 0.f;
        for (int i = threadIdx.x; i < nv; i += kThreads) {
            float f[8];
            unpack8(*reinterpret_cast<const uint4*>(xbuf + b * xstride + 8 * i), f);
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(f[e], f[e], s);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) wsum[warp * kMaxBatch + b] = s;
    }
    __syncthreads();
    if (threadIdx.x < B) {
        float t = wsum[threadIdx.x];
        for (int w = 1; w < kWarps; ++w) t += wsum[w * kMaxBatch + threadIdx.x];
        xsq[threadIdx.x] = first ? t : xsq[threadIdx.x] + t;
    }
}

// Store one output element. A build with GEMV_DEBUG_WRITECOUNT also counts the
// store in the caller's array (test support: every element must be written
// exactly once); other builds only store.
__device__ __forceinline__ void store_y(float* dst, float v, const WriteCount& wc) {
    *dst = v;
#ifdef GEMV_DEBUG_WRITECOUNT
    if (wc.counts) {
        const int64_t i = dst - wc.base;
        atomicAdd(wc.counts + ((i >= 0 && i < wc.n) ? i : wc.n), 1);
    }
#else
    (void)wc;
#endif
}

// Where warp kq of a row group puts its partial sum of (row_local, b): rows
// of B + 1 floats, so that the lanes of a warp writing neighbouring rows do
// not fall on the same shared-memory bank.
__device__ __forceinline__ int red_index(int kq, int rows_per_cta, int row_local, int B, int b) {
    return (kq * rows_per_cta + row_local) * (B + 1) + b;
}

// After every warp has written its partial sums with red_index: sum them over
// kq in order, then (with a cluster along K) over the CTAs of the cluster in
// rank order, scale by the RMSNorm factor of the batch row when asked (its sum
// of squares combined over the cluster in rank order as well), and store each
// output once.
//
// Cluster combine (S > 1), a reduce-scatter through distributed shared memory:
// rank r owns outputs [r * chunk, (r + 1) * chunk). Every rank pushes its
// partial of each output into slot [rank][output - owner * chunk] of the
// owner's cpart (and its sums of squares into every rank's slot [rank][b] of
// the RMSNorm exchange area), one cluster barrier publishes the stores, and
// each owner adds its S slots in rank order. No CTA reads another CTA's shared
// memory, so none has to wait for its peers before it exits. cpart holds
// S * chunk <= rows_per_cta * B + kMaxSplits floats. Kernels with S > 1 call
// cluster_arrive_relaxed() at entry.
__device__ __forceinline__ void combine_and_store(const float* red, float* cpart, float* misc, int rows_per_cta,
                                                  int B, int kw, int S, int split, int64_t n_base, int64_t N,
                                                  float* __restrict__ y, bool norm, int64_t K, float eps,
                                                  const WriteCount& wc) {
    float* xsq = misc + kWarps * kMaxBatch;
    float* rsc = xsq + kMaxBatch;
    float* xrecv = rsc + kMaxBatch;   // [kMaxSplits][kMaxBatch]
    const uint32_t magic = B > 1 ? 0xFFFFFFFFu / static_cast<uint32_t>(B) + 1u : 0u;
    const int nout = rows_per_cta * B;   // index i = row_local * B + b
    __syncthreads();
    if (S == 1) {
        if (norm) {
            if (threadIdx.x < B) rsc[threadIdx.x] = 1.0f / sqrtf(xsq[threadIdx.x] / static_cast<float>(K) + eps);
            __syncthreads();
        }
        for (int i = threadIdx.x; i < nout; i += kThreads) {
            const int rl = div_by_batch(i, B, magic), b = i - rl * B;
            float s = red[red_index(0, rows_per_cta, rl, B, b)];
#pragma unroll 1
            for (int q = 1; q < kw; ++q) s += red[red_index(q, rows_per_cta, rl, B, b)];
            const int64_t n = n_base + rl;
            if (n < N) store_y(y + static_cast<int64_t>(b) * N + n, norm ? s * rsc[b] : s, wc);
        }
        return;
    }

    const int chunk = (nout + S - 1) / S;
    cluster_wait();   // pairs with the arrival at kernel entry: every owner has started
#pragma unroll 1
    for (int owner = 0; owner < S; ++owner) {
        float* dst = dsmem_at(cpart + split * chunk, static_cast<uint32_t>(owner));
        const int i0 = owner * chunk;
        const int i1 = (i0 + chunk < nout) ? i0 + chunk : nout;
        for (int i = i0 + static_cast<int>(threadIdx.x); i < i1; i += kThreads) {
            const int rl = div_by_batch(i, B, magic), b = i - rl * B;
            float s = red[red_index(0, rows_per_cta, rl, B, b)];
#pragma unroll 1
            for (int q = 1; q < kw; ++q) s += red[red_index(q, rows_per_cta, rl, B, b)];
            dst[i - i0] = s;
        }
    }
    if (norm && threadIdx.x < B) {
#pragma unroll 1
        for (int q = 0; q < S; ++q)
            dsmem_at(xrecv + split * kMaxBatch + threadIdx.x, static_cast<uint32_t>(q))[0] = xsq[threadIdx.x];
    }
    cluster_sync_all();   // every rank's partials are in their owners' shared memory
    if (norm) {
        if (threadIdx.x < B) {
            float t = xrecv[threadIdx.x];
            for (int q = 1; q < S; ++q) t += xrecv[q * kMaxBatch + threadIdx.x];
            rsc[threadIdx.x] = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
        }
        __syncthreads();
    }
    const int i0 = split * chunk;
    const int i1 = (i0 + chunk < nout) ? i0 + chunk : nout;
    for (int i = i0 + static_cast<int>(threadIdx.x); i < i1; i += kThreads) {
        const int j = i - i0;
        float s = cpart[j];
#pragma unroll 1
        for (int q = 1; q < S; ++q) s += cpart[q * chunk + j];
        const int rl = div_by_batch(i, B, magic), b = i - rl * B;
        const int64_t n = n_base + rl;
        if (n < N) store_y(y + static_cast<int64_t>(b) * N + n, norm ? s * rsc[b] : s, wc);
    }
}

// Segment of a (possibly fused) launch that owns row tile `tile`.
struct SegView {
    int si;              // segment index
    const uint16_t* W;
    float* y;
    int64_t N;
    int64_t ldw;
    int64_t tile_local;
    const uint16_t* S;   // INT4 weights: group scales
    int64_t lds;
    const float* rs;     // FP8 weights: row scales
};

__device__ __forceinline__ SegView segment_of(const Params& p, int64_t tile) {
    int si = 0;
#pragma unroll 1
    for (int i = 1; i < p.nseg; ++i)
        if (tile >= p.seg[i].tile_begin) si = i;
    SegView s;
    s.si = si;
    s.W = p.seg[si].W;
    s.y = p.seg[si].y;
    s.N = p.seg[si].N;
    s.ldw = p.seg[si].ldw;
    s.tile_local = tile - p.seg[si].tile_begin;
    s.S = p.seg[si].S;
    s.lds = p.seg[si].lds;
    s.rs = p.seg[si].rs;
    return s;
}

// Launch a kernel with the plan's grid, cluster (when K is split over CTAs,
// or CTAs share a multicast copy of x) and programmatic dependent launch.
template <typename KernelT>
cudaError_t launch_kernel(KernelT kernel, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem_bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    const int cluster = l.splits > 1 ? l.splits : (l.mcast > 1 ? l.mcast : 1);
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace gemv
