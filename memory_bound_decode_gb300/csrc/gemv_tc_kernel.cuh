// Skinny-batch decode GEMV on the fifth-generation tensor cores (tcgen05) for
// sm_103a: y[b][n] = sum_k W[n][k] * x[b][k] with 2 <= B <= 16, BF16 operands,
// FP32 accumulation in tensor memory.
//
// Why this form ("Decode GEMV at half of HBM bandwidth", "What interviewers
// probe next": at batch 16 the operation is a skinny GEMM): the register-fed
// kernel keeps one batch of W loads per warp in flight and must wait for the
// CTA's slice of x before it can consume that batch and issue the next, so the
// HBM idles while x is copied. Here W never enters registers: the Tensor
// Memory Accelerator streams it, with x, into a ring of shared-memory stages,
// and the ring is deep enough (kTcStages x 32 KB per SM) that the first stages
// of W are in flight before the wait for the preceding grid and keep landing
// while x arrives.
//
// A CTA's tile belongs to one weight matrix of the launch (up to 8 share x,
// each with its own tensor map). Roles in a CTA of 8 warps:
//   thread 0      issues the tensor copies of each stage (W: two boxes of 64
//                 columns x 128 rows; x: two boxes of 64 columns x 16 rows;
//                 128-byte swizzle), counted on the stage's "full" mbarrier,
//                 after waiting on its "empty" mbarrier for the slot's reuse;
//   warp 1        allocates 32 columns of tensor memory; its lane 0 issues, per
//                 stage, 8 tcgen05.mma (M = 128, N = 16, K = 16, both operands
//                 K-major in shared memory) and commits them to the stage's
//                 "empty" barrier, and after the last stage to "done";
//   warps 4..7    read the 128 x 16 FP32 accumulator (tcgen05.ld, warp w the
//                 lanes 32 (w - 4) ..) into the partial-sum area;
//   all           the fixed-order split-K combine over the cluster
//                 (combine_and_store) and the stores of y.
// Every wait is bounded; a CTA that gives up stores NaN and sets the status
// bit, waits (bounded) for the copies it issued, and frees its tensor memory.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_common.cuh"

namespace gemv {

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle (8-row groups 1,024 bytes apart; the leading offset is unused for a
// swizzled K-major layout), version 1.
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of kind::f16: D FP32, A and B BF16, both K-major,
// N = 16, M = 128.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((static_cast<uint32_t>(kTcN) >> 3) << 17) |
                              ((static_cast<uint32_t>(kTcRows) >> 4) << 24);

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t a, uint64_t b, bool accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(tmem), "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate ? 1u : 0u) : "memory");
}

// The barrier's phase completes once every tcgen05 operation this thread
// issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tensor_copy_2d(uint32_t dst, const void* map, int x, int y, uint64_t* bar) {
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar)) : "memory");
}

// Ask the L2 for the box at (x, y) of `map` (no shared memory, no barrier):
// the later copy of the same box then reads it from L2.
__device__ __forceinline__ void tensor_prefetch_2d(const void* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(map), "r"(x), "r"(y) : "memory");
}

// 32 lanes x 16 columns of FP32 from tensor memory (lane i of the warp gets
// lane taddr.lane + i), then the wait for the load.
__device__ __forceinline__ void tc_load16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                   "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bytes of one ring stage of SC columns: W (SC / 64 boxes of 64 columns x
// 128 rows) and x (SC / 64 boxes of 64 columns x 16 rows).
__host__ __device__ constexpr uint32_t tc_wstage(int sc) { return static_cast<uint32_t>(sc / 64) * kTcWBox; }
__host__ __device__ constexpr uint32_t tc_xstage(int sc) { return static_cast<uint32_t>(sc / 64) * kTcXBox; }

// Byte offsets of the dynamic shared memory (after aligning its start to
// 1,024 bytes): the W ring, the x ring, the combine areas, the barriers.
struct TcLayout {
    uint32_t x_ring, red, cpart, misc, bars, tslot, total;
};

__host__ __device__ constexpr uint32_t tc_align(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline TcLayout tc_layout(int B, int ns, int sc) {
    TcLayout L{};
    L.x_ring = static_cast<uint32_t>(ns) * tc_wstage(sc);
    L.red = L.x_ring + static_cast<uint32_t>(ns) * tc_xstage(sc);
    L.cpart = L.red + static_cast<uint32_t>(kTcRows * (B + 1)) * 4u;
    L.misc = L.cpart + static_cast<uint32_t>(kTcRows * B + kMaxSplits) * 4u;
    L.bars = tc_align(L.misc + static_cast<uint32_t>(kMiscFloats) * 4u, 16u);
    L.tslot = L.bars + static_cast<uint32_t>(2 * ns + 1) * 8u;
    L.total = L.tslot + 16u + 1024u;   // + the alignment of the start
    return L;
}

template <int NS, int SC>
__global__ void __launch_bounds__(kThreads, NS * SC <= 256 ? 2 : 1)
gemv_tc_kernel(const __grid_constant__ Params p) {
    constexpr uint32_t WST = tc_wstage(SC), XST = tc_xstage(SC);
    extern __shared__ __align__(1024) unsigned char smem_raw[];

    pdl_launch_dependents();

    const int B = p.batch;
    const TcLayout L = tc_layout(B, NS, SC);
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t ring = smem_addr(sm);
    float* red = reinterpret_cast<float*>(sm + L.red);
    float* cpart = reinterpret_cast<float*>(sm + L.cpart);
    float* misc = reinterpret_cast<float*>(sm + L.misc);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.bars);
    uint64_t* empty = full + NS;
    uint64_t* done = empty + NS;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L.tslot);
    int* fail = reinterpret_cast<int*>(sm + L.tslot + 4);

    const int S = p.splits;
    if (S > 1) cluster_arrive_relaxed();   // see combine_and_store
    const int64_t tile = blockIdx.x / S;
    const int split = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;"
                     :: "r"(smem_addr(tslot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * NS + 1; ++i) mbar_init(full + i, 1);
        *fail = 0;
        fence_mbar_init_cluster();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    const int64_t K = p.K;
    const int64_t k0 = static_cast<int64_t>(split) * p.kslice;
    const int64_t k1 = (k0 + p.kslice < K) ? k0 + p.kslice : K;
    const int nst = static_cast<int>((k1 - k0 + SC - 1) / SC);
    const SegView sg = segment_of(p, tile);
    const int row0 = static_cast<int>(sg.tile_local * kTcRows);   // within the segment's W
    const void* wmap = &p.wmap[sg.si];
    const uint32_t stage_bytes = WST + XST;

    if (threadIdx.x == 0) {
        // Producer. The first stages' W goes out before the wait for the
        // preceding grid (W is not its output); their x right after it.
        int arms[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) arms[i] = 0;
        auto issue_w = [&](int s) {
            const int slot = s % NS;
            const int col = static_cast<int>(k0) + s * SC;
            const uint32_t w = ring + static_cast<uint32_t>(slot) * WST;
#pragma unroll
            for (int b = 0; b < SC / 64; ++b)
                tensor_copy_2d(w + static_cast<uint32_t>(b) * kTcWBox, wmap, col + 64 * b, row0, full + slot);
        };
        auto issue_x = [&](int s) {
#ifdef GEMV_DEBUG_DROP_X
            return;   // the test build: x never arrives, the stage's wait runs out
#endif
            const int slot = s % NS;
            const int col = static_cast<int>(k0) + s * SC;
            const uint32_t x = ring + L.x_ring + static_cast<uint32_t>(slot) * XST;
#pragma unroll
            for (int b = 0; b < SC / 64; ++b)
                tensor_copy_2d(x + static_cast<uint32_t>(b) * kTcXBox, &p.xmap, col + 64 * b, 0, full + slot);
        };
        // L2 prefetch of W, p.l2pf stages beyond the ring: more bytes in flight
        // than the ring's shared memory holds.
        auto prefetch_w = [&](int s) {
            if (s >= nst) return;
            const int col = static_cast<int>(k0) + s * SC;
#pragma unroll
            for (int b = 0; b < SC / 64; ++b) tensor_prefetch_2d(wmap, col + 64 * b, row0);
        };
        const int npro = nst < NS ? nst : NS;
        for (int s = 0; s < npro; ++s) {
            mbar_arrive_expect_tx(full + s, stage_bytes);
            ++arms[s];
            issue_w(s);
        }
        for (int s = npro; s < npro + p.l2pf; ++s) prefetch_w(s);
        if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
        for (int s = 0; s < npro; ++s) issue_x(s);
        for (int s = npro; s < nst; ++s) {
            const int slot = s % NS;
            if (!mbar_wait_bounded(empty + slot, static_cast<uint32_t>((s / NS - 1) & 1))) {
                atomicOr(fail, 1);
                break;
            }
            mbar_arrive_expect_tx(full + slot, stage_bytes);
            ++arms[slot];
            issue_w(s);
            issue_x(s);
            if (p.l2pf) prefetch_w(s + p.l2pf);
        }
        // Every copy issued has landed before the CTA may leave (bounded; on the
        // normal path the MMA issuer has already seen each of these phases).
#pragma unroll
        for (int i = 0; i < NS; ++i)
            if (arms[i] > 0 && !mbar_wait_bounded(full + i, static_cast<uint32_t>((arms[i] - 1) & 1))) atomicOr(fail, 1);
    } else {
        // Every thread that stores y has waited for the preceding grid.
        if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
    }

    if (threadIdx.x == 32) {
        // MMA issuer: SC / 16 MMAs of K = 16 per stage (32 bytes along K
        // within a 128-byte swizzled row; each further box 16 KB (W) / 2 KB (x) on).
        int s = 0;
        for (; s < nst; ++s) {
            const int slot = s % NS;
            if (!mbar_wait_bounded(full + slot, static_cast<uint32_t>((s / NS) & 1))) {
                atomicOr(fail, 1);
                break;
            }
            tc_fence_after();
            const uint32_t w = ring + static_cast<uint32_t>(slot) * WST;
            const uint32_t x = ring + L.x_ring + static_cast<uint32_t>(slot) * XST;
#pragma unroll
            for (int k = 0; k < SC / 16; ++k) {
                const uint32_t kb = static_cast<uint32_t>(k >> 2), kk = static_cast<uint32_t>(k & 3) * 32u;
                tc_mma(tmem, tc_smem_desc(w + kb * kTcWBox + kk), tc_smem_desc(x + kb * kTcXBox + kk), (s | k) != 0);
            }
            tc_commit(empty + slot);
        }
        tc_commit(done);
    }

    if (warp >= 4) {
        const bool ok = mbar_wait_bounded(done, 0);
        __syncwarp();   // the tensor-memory load is warp-wide
        tc_fence_after();
        float v[16];
        tc_load16(tmem + (static_cast<uint32_t>(32 * (warp - 4)) << 16), v);
        const int rl = 32 * (warp - 4) + lane;
#pragma unroll
        for (int b = 0; b < 16; ++b)
            if (b < B) red[red_index(0, kTcRows, rl, B, b)] = v[b];
        if (!ok) atomicOr(fail, 1);
    }
    tc_fence_before();
    __syncthreads();
    // A CTA that gave up on a wait stores NaN (and sets the status bit).
    if (*fail) {
        if (threadIdx.x == 0) atomicOr(&g_device_status, kStatusWaitTimeout);
        for (int i = threadIdx.x; i < kTcRows * (B + 1); i += kThreads) red[i] = __uint_as_float(0x7fc00000u);
    }
    combine_and_store(red, cpart, misc, kTcRows, B, 1, S, split, sg.tile_local * kTcRows, sg.N, sg.y, false, K,
                      p.rms_eps, p.wc);
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" :: "r"(tmem) : "memory");
    }
}

// ---- persistent form: grids of more than one wave ---------------------------
//
// Where the row tiles exceed one wave, a fixed grid of G CTAs takes tiles in
// turn (CTA c: tiles c, c + G, ...), each over the whole K (no split, no
// combine): G is chosen so that every CTA gets the same number of tiles (up to
// one fewer for the last few), where a grid of one CTA per tile would leave a
// partial last wave. The ring keeps streaming across a CTA's tiles; the
// accumulator alternates between two 16-column halves of tensor memory, so
// the MMAs of tile i + 1 run while the epilogue warps read tile i (they
// release each half on its "tfree" barrier) and store its outputs directly.

__host__ __device__ inline uint32_t tcp_bars_offset(int ns, int sc) {
    return static_cast<uint32_t>(ns) * (tc_wstage(sc) + tc_xstage(sc));
}

__host__ __device__ inline uint32_t tcp_total(int ns, int sc) {
    return tcp_bars_offset(ns, sc) + static_cast<uint32_t>(2 * ns + 5) * 8u + 16u + 1024u;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

template <int NS, int SC>
__global__ void __launch_bounds__(kThreads, NS * SC <= 256 ? 3 : 2)
gemv_tcp_kernel(const __grid_constant__ Params p) {
    constexpr uint32_t WST = tc_wstage(SC), XST = tc_xstage(SC);
    extern __shared__ __align__(1024) unsigned char smem_raw[];

    pdl_launch_dependents();

    const int B = p.batch;
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t ring = smem_addr(sm);
    const uint32_t x_ring = static_cast<uint32_t>(NS) * WST;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + tcp_bars_offset(NS, SC));
    uint64_t* empty = full + NS;
    uint64_t* done = empty + NS;     // [2]
    uint64_t* tfree = done + 2;      // [2]
    uint64_t* drain = tfree + 2;     // every MMA issued has completed (before tensor memory is freed)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* fail = reinterpret_cast<volatile int*>(drain + 1) + 1;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;"
                     :: "r"(smem_addr(tslot)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * NS + 2; ++i) mbar_init(full + i, 1);
        mbar_init(tfree, 4 * 32);
        mbar_init(tfree + 1, 4 * 32);
        mbar_init(drain, 1);
        *fail = 0;
        fence_mbar_init_cluster();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    const int64_t K = p.K;
    const int nst = static_cast<int>((K + SC - 1) / SC);
    const int64_t tiles = p.seg[p.nseg - 1].tile_begin + (p.seg[p.nseg - 1].N + kTcRows - 1) / kTcRows;
    const int64_t G = gridDim.x;
    const int mine = static_cast<int>(blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / G + 1 : 0);
    const uint32_t stage_bytes = WST + XST;

    if (threadIdx.x == 0) {
        // Producer: stage g of the CTA's sequence is stage g % nst of its tile
        // g / nst; the first NS stages' W before the wait for the preceding grid.
        int arms[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) arms[i] = 0;
        auto issue = [&](int g, bool w, bool x) {
            const int slot = g % NS;
            const int64_t t = blockIdx.x + static_cast<int64_t>(g / nst) * G;
            const int col = (g % nst) * SC;
            if (w) {
                const SegView sg = segment_of(p, t);
                const uint32_t dst = ring + static_cast<uint32_t>(slot) * WST;
#pragma unroll
                for (int b = 0; b < SC / 64; ++b)
                    tensor_copy_2d(dst + static_cast<uint32_t>(b) * kTcWBox, &p.wmap[sg.si], col + 64 * b,
                                   static_cast<int>(sg.tile_local * kTcRows), full + slot);
            }
#ifdef GEMV_DEBUG_DROP_X
            x = false;   // the test build: x never arrives, the stage's wait runs out
#endif
            if (x) {
                const uint32_t dst = ring + x_ring + static_cast<uint32_t>(slot) * XST;
#pragma unroll
                for (int b = 0; b < SC / 64; ++b)
                    tensor_copy_2d(dst + static_cast<uint32_t>(b) * kTcXBox, &p.xmap, col + 64 * b, 0, full + slot);
            }
        };
        const int total = mine * nst;
        const int npro = total < NS ? total : NS;
        for (int g = 0; g < npro; ++g) {
            mbar_arrive_expect_tx(full + g, stage_bytes);
            ++arms[g];
            issue(g, true, false);
        }
        if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
        for (int g = 0; g < npro; ++g) issue(g, false, true);
        for (int g = npro; g < total; ++g) {
            const int slot = g % NS;
            if (*fail || !mbar_wait_bounded(empty + slot, static_cast<uint32_t>((g / NS - 1) & 1))) {
                *fail = 1;
                break;
            }
            mbar_arrive_expect_tx(full + slot, stage_bytes);
            ++arms[slot];
            issue(g, true, true);
        }
#pragma unroll
        for (int i = 0; i < NS; ++i)
            if (arms[i] > 0 && !mbar_wait_bounded(full + i, static_cast<uint32_t>((arms[i] - 1) & 1))) *fail = 1;
    } else {
        // Every thread that stores y has waited for the preceding grid.
        if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
    }

    if (threadIdx.x == 32) {
        // MMA issuer: tile i accumulates into tensor-memory half i % 2, once
        // the epilogue has released it (tile i - 2).
        int g = 0;
        for (int i = 0; i < mine && !*fail; ++i) {
            const int buf = i & 1;
            if (i >= 2 && !mbar_wait_bounded(tfree + buf, static_cast<uint32_t>((i / 2 - 1) & 1))) {
                *fail = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(buf * kTcN);
            for (int s = 0; s < nst; ++s, ++g) {
                const int slot = g % NS;
                if (*fail || !mbar_wait_bounded(full + slot, static_cast<uint32_t>((g / NS) & 1))) {
                    *fail = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t w = ring + static_cast<uint32_t>(slot) * WST;
                const uint32_t x = ring + x_ring + static_cast<uint32_t>(slot) * XST;
#pragma unroll
                for (int k = 0; k < SC / 16; ++k) {
                    const uint32_t kb = static_cast<uint32_t>(k >> 2), kk = static_cast<uint32_t>(k & 3) * 32u;
                    tc_mma(d, tc_smem_desc(w + kb * kTcWBox + kk), tc_smem_desc(x + kb * kTcXBox + kk),
                           (s | k) != 0);
                }
                tc_commit(empty + slot);
            }
            tc_commit(done + buf);
        }
        // Epilogue warps waiting for a tile that will not come: an ordinary
        // arrival (release: they see the failure flag) completes the phase they
        // may be waiting on, so their bounded waits end early.
        if (*fail) {
            mbar_arrive(done);
            mbar_arrive(done + 1);
        }
        // Every MMA issued has completed before the tensor memory is freed.
        tc_commit(drain);
        if (!mbar_wait_bounded(drain, 0)) *fail = 1;
    }

    if (warp >= 4) {
        // Epilogue: tile i's 128 x 16 accumulator from tensor-memory half i % 2
        // into y, rows along the warp's lanes (coalesced per batch row).
        // After a failure every remaining tile of the CTA is stored as NaN
        // (no tensor memory read, no further wait).
        const int q = warp - 4;
        for (int i = 0; i < mine; ++i) {
            const int buf = i & 1;
            bool ok = *fail == 0 && mbar_wait_bounded(done + buf, static_cast<uint32_t>((i / 2) & 1));
            ok = __all_sync(0xffffffffu, ok && *fail == 0);   // warp-uniform: the load below is warp-wide
            float v[16];
#pragma unroll
            for (int b = 0; b < 16; ++b) v[b] = 0.f;
            if (ok) {
                tc_fence_after();
                tc_load16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * kTcN), v);
                tc_fence_before();
            }
            mbar_arrive(tfree + buf);
            if (!ok) *fail = 1;
            const bool bad = !ok;
            const int64_t t = blockIdx.x + static_cast<int64_t>(i) * G;
            const SegView sg = segment_of(p, t);
            const int64_t n = sg.tile_local * kTcRows + 32 * q + lane;
            if (n < sg.N) {
#pragma unroll
                for (int b = 0; b < 16; ++b)
                    if (b < B) store_y(sg.y + static_cast<int64_t>(b) * sg.N + n, bad ? __uint_as_float(0x7fc00000u) : v[b], p.wc);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*fail && threadIdx.x == 0) atomicOr(&g_device_status, kStatusWaitTimeout);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" :: "r"(tmem) : "memory");
    }
}

// Instances by ring depth and stage width (Launch::unroll, Launch::stage_cols):
// rings of up to 256 columns leave room for two CTAs per SM, deeper ones take one.
#define GEMV_TC_INSTANCES(X) X(2, 128) X(3, 128) X(4, 128) X(5, 128) X(2, 64) X(3, 64) X(4, 64) X(8, 64) X(10, 64)

// Persistent-form instances (ring depth, stage width).
#define GEMV_TCP_INSTANCES(X) X(2, 128) X(3, 128) X(4, 128)

inline cudaError_t launch_tc(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    if (l.tc_persist) {
#define GEMV_TCP_LAUNCH(ns, sc) \
    if (l.unroll == ns && l.stage_cols == sc) return launch_kernel(gemv_tcp_kernel<ns, sc>, p, l, s, pdl);
        GEMV_TCP_INSTANCES(GEMV_TCP_LAUNCH)
#undef GEMV_TCP_LAUNCH
        return cudaErrorInvalidValue;
    }
#define GEMV_TC_LAUNCH(ns, sc) \
    if (l.unroll == ns && l.stage_cols == sc) return launch_kernel(gemv_tc_kernel<ns, sc>, p, l, s, pdl);
    GEMV_TC_INSTANCES(GEMV_TC_LAUNCH)
#undef GEMV_TC_LAUNCH
    return cudaErrorInvalidValue;
}

inline cudaError_t prepare_tc() {
    cudaError_t e = cudaSuccess;
#define GEMV_TC_PREPARE(ns, sc)                                                                            \
    if (e == cudaSuccess)                                                                                   \
        e = cudaFuncSetAttribute(gemv_tc_kernel<ns, sc>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 kTcMaxDynSmem);
    GEMV_TC_INSTANCES(GEMV_TC_PREPARE)
#undef GEMV_TC_PREPARE
#define GEMV_TCP_PREPARE(ns, sc)                                                                           \
    if (e == cudaSuccess)                                                                                   \
        e = cudaFuncSetAttribute(gemv_tcp_kernel<ns, sc>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 kTcMaxDynSmem);
    GEMV_TCP_INSTANCES(GEMV_TCP_PREPARE)
#undef GEMV_TCP_PREPARE
    return e;
}

// Whether an instance of this depth and width exists (read off the lists above).
#define GEMV_TC_IS(n, c) (ns == (n) && sc == (c)) ||
__host__ __device__ constexpr bool tcp_instance(int ns, int sc) { return GEMV_TCP_INSTANCES(GEMV_TC_IS) false; }
__host__ __device__ constexpr bool tc_instance(int ns, int sc) { return GEMV_TC_INSTANCES(GEMV_TC_IS) false; }
#undef GEMV_TC_IS

inline cudaError_t read_tc_status_tu(unsigned int* bits, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess || !reset || *bits == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace gemv
