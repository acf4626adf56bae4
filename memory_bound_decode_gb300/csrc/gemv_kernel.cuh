// Decode GEMV kernel for sm_103a: y[b][n] = sum_k W[n][k] * x[b][k], BF16 in,
// FP32 accumulate.
//
// Design (restating "Decode GEMV at half of HBM bandwidth", "A strong answer",
// and "GPU performance chains", "A coalesced warp load", for Blackwell):
//   * Lanes run along K. One warp-wide load reads 32 x 16 B = 512 contiguous
//     bytes of one weight row, whole 32-byte sectors only.
//   * Each lane issues UJ independent 16-byte ld.global.nc.L1::no_allocate loads
//     per row before it consumes any, so a resident warp keeps
//     32 * UJ * RPW * 16 bytes in flight (Little's law sets how many are needed).
//   * x (the CTA's K-range, in chunks) is staged once per CTA in shared memory
//     with asynchronous 16-byte copies (all in flight at once) and reused by
//     every row of the CTA; W is never staged: it has no reuse.
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

#include "gemv_internal.h"

namespace gemv {

__device__ __forceinline__ uint4 ld_stream16(const uint16_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Keep the first m (1..7) BF16 elements of an 8-element vector, zero the rest.
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

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Load a float from the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t r;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
    return v;
}

// 16-byte asynchronous global->shared copy of `nbytes` (2..16) bytes; the rest
// of the 16 bytes is zero-filled. Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, int nbytes) {
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(gmem_src), "r"(nbytes) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Copy x[b][c0 .. c0 + 8*nv) for every batch row into shared memory (row
// stride xstride), zero-filling columns >= K. Aligned 16-byte pieces go out as
// asynchronous copies, all in flight at once and holding no registers;
// misaligned ones (rows of x start at 2-byte offsets when K % 8 != 0) are
// loaded element by element. The caller waits with cp_async_wait_all() and a
// barrier.
template <int B>
__device__ __forceinline__ void stage_x(uint16_t* xs, int xstride, const uint16_t* __restrict__ x,
                                        int64_t K, int64_t c0, int nv) {
    const int items = B * nv;
#pragma unroll 4
    for (int it = threadIdx.x; it < items; it += kThreads) {
        const int b = (B == 1) ? 0 : it / nv;
        const int i = it - b * nv;
        const int64_t col = c0 + 8 * static_cast<int64_t>(i);
        const uint16_t* src = x + static_cast<int64_t>(b) * K + col;
        uint16_t* dst = xs + static_cast<int64_t>(b) * xstride + 8 * i;
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
}

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

// Multiply-add one batch into the running sums. The batch is summed into a
// fresh partial first (blocked summation), then added to acc.
template <int B, int RPW, int UJ, bool PRED>
__device__ __forceinline__ void consume_batch(float (&acc)[RPW][B], const uint4 (&wv)[UJ][RPW],
                                              const bool (&ok)[UJ], const uint16_t* xl, int xstride) {
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

template <int B, int RPW, int UJ>
__global__ void __launch_bounds__(kThreads)
gemv_bf16_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];

    // Let the next grid on the stream start as SMs free up; it only reads W
    // before it waits on this grid.
    pdl_launch_dependents();

    const int S = p.splits;
    const int64_t tile = blockIdx.x / S;
    const int split = (S > 1) ? static_cast<int>(cluster_rank()) : 0;

    int si = 0;
#pragma unroll 1
    for (int i = 1; i < p.nseg; ++i)
        if (tile >= p.seg[i].tile_begin) si = i;
    const uint16_t* __restrict__ Wseg = p.seg[si].W;
    float* __restrict__ yseg = p.seg[si].y;
    const int64_t N = p.seg[si].N;
    const int64_t ldw = p.seg[si].ldw;
    const int64_t tile_local = tile - p.seg[si].tile_begin;

    const int kw = p.kw;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = warp / kw;        // row group of this warp
    const int kq = warp - g * kw;   // position of this warp along K within the group
    const int rows_per_cta = (kWarps / kw) * RPW;
    const int64_t row0 = tile_local * rows_per_cta + static_cast<int64_t>(g) * RPW;

    const uint16_t* wrow[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        int64_t n = row0 + r;
        n = n < N ? n : N - 1;    // rows past N stream a valid row; results dropped
        wrow[r] = Wseg + n * ldw;
    }

    const int xstride = p.xstride;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);
    float* red = reinterpret_cast<float*>(smem_raw + static_cast<size_t>(B) * xstride * 2);
    float* cpart = red + rows_per_cta * B * kw;

    const int64_t K = p.K;
    const int64_t k0 = static_cast<int64_t>(split) * p.kslice;
    const int64_t k1 = (k0 + p.kslice < K) ? k0 + p.kslice : K;

    float acc[RPW][B];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) acc[r][b] = 0.f;

    bool first_chunk = true;
#pragma unroll 1
    for (int64_t c0 = k0; c0 < k1; c0 += p.kchunk) {
        const int64_t c1 = (c0 + p.kchunk < k1) ? c0 + p.kchunk : k1;
        const int nfull = static_cast<int>((c1 - c0) >> 3);          // whole 8-column vectors
        const bool tailv = (c1 == K) && ((K & 7) != 0);              // one partial vector at the end
        const int nv = nfull + (tailv ? 1 : 0);
        const int tail_m = tailv ? static_cast<int>(K - (c0 + 8 * static_cast<int64_t>(nfull))) : 0;
        const int nsteps = (nv + 31) >> 5;                           // warp-steps of 32 vectors
        const int span = (nsteps + kw - 1) / kw;                     // contiguous steps per warp
        const int s_begin = kq * span;
        const int s_end = (s_begin + span < nsteps) ? s_begin + span : nsteps;
        const int my_steps = s_end > s_begin ? s_end - s_begin : 0;

        int v0 = s_begin * 32 + lane;   // this lane's first vector in the chunk
        const uint16_t* wp[RPW];
#pragma unroll
        for (int r = 0; r < RPW; ++r) wp[r] = wrow[r] + c0 + 8 * static_cast<int64_t>(v0);
        const uint16_t* xl = xs + 8 * v0;

        uint4 wv[UJ][RPW];
        bool ok[UJ];

        // Weight loads go out first; then wait for the preceding grid (x may be
        // its output) and stage this chunk of x.
        issue_batch<RPW, UJ, true>(wv, ok, wp, v0, my_steps, nv, nfull, tail_m);
        if (first_chunk) {
            pdl_wait_prerequisites();
            first_chunk = false;
        } else {
            __syncthreads();   // every warp is done reading the previous chunk
        }
        stage_x<B>(xs, xstride, p.x, K, c0, nv);
        cp_async_wait_all();
        __syncthreads();
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
        for (; j + UJ <= my_steps && (v0 - lane) + 32 * UJ <= nfull; j += UJ) {
            issue_batch<RPW, UJ, false>(wv, ok, wp, v0, UJ, nv, nfull, 0);
            consume_batch<B, RPW, UJ, false>(acc, wv, ok, xl, xstride);
            advance();
        }
#pragma unroll 1
        for (; j < my_steps; j += UJ) {
            issue_batch<RPW, UJ, true>(wv, ok, wp, v0, my_steps - j, nv, nfull, tail_m);
            consume_batch<B, RPW, UJ, true>(acc, wv, ok, xl, xstride);
            advance();
        }
    }

    // Lane reduction: the same xor butterfly for every row, so the result does
    // not depend on where a row sits in the grid.
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[r][b];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[r][b] = v;
        }

    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int b = 0; b < B; ++b) red[((g * RPW + r) * B + b) * kw + kq] = acc[r][b];
    }
    __syncthreads();

    const int nout = rows_per_cta * B;   // outputs of this CTA, index i = row_local * B + b
    const int64_t n_base = tile_local * rows_per_cta;
    for (int i = threadIdx.x; i < nout; i += kThreads) {
        float s = red[i * kw];
        for (int q = 1; q < kw; ++q) s += red[i * kw + q];
        if (S == 1) {
            const int64_t n = n_base + i / B;
            if (n < N) yseg[static_cast<int64_t>(i % B) * N + n] = s;
        } else {
            cpart[i] = s;
        }
    }

    if (S > 1) {
        cluster_sync_all();   // every CTA of the cluster has its partials in shared memory
        for (int i = threadIdx.x; i < nout; i += kThreads) {
            if (i % S != split) continue;   // outputs are shared out over the ranks
            float s = ld_dsmem(&cpart[i], 0);
            for (int q = 1; q < S; ++q) s += ld_dsmem(&cpart[i], static_cast<uint32_t>(q));
            const int64_t n = n_base + i / B;
            if (n < N) yseg[static_cast<int64_t>(i % B) * N + n] = s;
        }
        cluster_sync_all();   // no CTA leaves while another still reads its shared memory
    }
}

template <int B>
cudaError_t launch_batch(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    constexpr Variant v = variant_for(B);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem_bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (l.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(l.splits);
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
    return cudaLaunchKernelEx(&cfg, gemv_bf16_kernel<B, v.rows_per_warp, v.unroll>, p);
}

template <int B>
cudaError_t prepare_batch() {
    constexpr Variant v = variant_for(B);
    return cudaFuncSetAttribute(gemv_bf16_kernel<B, v.rows_per_warp, v.unroll>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

}  // namespace gemv
