// Decode GEMV with FP8 (E4M3) weights and one FP32 scale per output row, BF16
// activations, FP32 accumulation, for sm_103a:
//     y[b][n] = S[n] * sum_k e4m3(Wq[n][k]) * x[b][k].
//
// "Decode GEMV at half of HBM bandwidth", "What interviewers probe next": after
// INT4, FP8 weights halve the bytes of BF16 ones, and the kernel has to widen
// them in registers while the next loads are outstanding. As in the INT4
// kernel the contraction runs on the BF16 tensor cores at every batch size
// (mma.sync m16n8k16, FP32 accumulate), fed straight from the loaded codes.
//
// Widening E4M3 to BF16, exactly. Per pair of codes (one 16-bit half each):
//   * a byte permute with sign replication puts each code in the low byte of
//     its half and copies its sign bit over the high byte;
//   * shifting left by 4 and keeping bit 15 and bits 4..10 (mask 0x87F0) gives
//     the BF16 pattern with the sign in place, the 4 exponent bits at the
//     bottom of BF16's 8-bit exponent field and the 3 mantissa bits at the top
//     of its mantissa. That BF16 number is the E4M3 value times 2^-120, for
//     normal codes and for subnormal ones alike (both formats place the
//     subnormals where the exponent field is zero);
//   * a BF16 multiply by 2^120 restores the value (a power of two: exact).
// The two E4M3 NaN codes come out as 480; weights are finite by contract.
//
// Mapping. A warp owns a 16-row tile; lane (g, t) = (lane / 4, lane % 4) loads,
// per 64-column slot, 16 bytes (16 codes, columns 16t .. 16t+15 of the slot) of
// row g and of row g + 8, so the 4 lanes of a row team cover the slot. One
// 32-bit word (4 codes) of each row feeds one MMA: its two code pairs fill the
// lane's k-slots (2t, 2t+1) and (2t+8, 2t+9), and the x operand takes the same
// physical columns (one 16-byte shared-memory read of x per two words). Each
// batch of UJ slots is summed into a fresh FP32 tile before it is added to the
// running sums (blocked accumulation); the row scale multiplies the final
// sums. x is staged per CTA with bulk or asynchronous copies (rows padded so
// the eight batch rows of a warp's read fall on different banks), the first batch of
// loads goes out before the programmatic-dependent-launch wait, and partial
// sums combine in a fixed order over warps and cluster CTAs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_common.cuh"
#include "gemv_mma_kernel.cuh"

namespace gemv {

// Two BF16 pairs from one word of four E4M3 codes: out[0] holds the codes of
// the word's columns 0 and 1 (low, high half), out[1] those of columns 2 and 3.
__device__ __forceinline__ void fp8_widen_word(uint32_t w, uint32_t (&out)[2]) {
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(lo) : "r"(w));   // sext(c0) | sext(c1) << 16
    asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(hi) : "r"(w));   // sext(c2) | sext(c3) << 16
    const uint32_t tl = (lo << 4) & 0x87F087F0u;
    const uint32_t th = (hi << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out[0]) : "r"(tl), "r"(0x7B807B80u));   // * 2^120
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out[1]) : "r"(th), "r"(0x7B807B80u));
}

// This warp's contiguous range of 64-column slots within a chunk.
struct F8Range {
    int j_begin;
    int my_slots;
};

__device__ __forceinline__ F8Range f8_range(int nslots, int kw, int kq) {
    const int span = (nslots + kw - 1) / kw;
    F8Range r;
    r.j_begin = kq * span;
    const int j_end = (r.j_begin + span < nslots) ? r.j_begin + span : nslots;
    r.my_slots = j_end > r.j_begin ? j_end - r.j_begin : 0;
    return r;
}

// XB (one chunk, x 16-byte aligned in this GPU's memory): x is copied into
// shared memory by bulk copies counted on an mbarrier (bulk_stage_x), which do
// not queue behind the code loads the warps have just issued, instead of
// 16-byte asynchronous copies from every thread.
template <int NB, int UJ, bool CHUNKED, bool XB = false>
__global__ void __launch_bounds__(kThreads)
gemv_fp8_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];

    pdl_launch_dependents();

    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem_raw);   // the 16 bytes before x
    if constexpr (XB) {
        if (threadIdx.x == 0) {
            mbar_init(mbar, 1);
            fence_mbar_init_cluster();
        }
        __syncthreads();
    }

    const int S = p.splits;
    if (S > 1) cluster_arrive_relaxed();   // see combine_and_store
    const int64_t tile = blockIdx.x / S;
    const int split = (S > 1) ? static_cast<int>(cluster_rank()) : 0;
    const SegView sg = segment_of(p, tile);
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
    // This lane's 16 codes (columns 16t .. 16t+15 of a slot) of rows n0 and n1
    // at column 0; ldw is the row stride in bytes here.
    const uint8_t* q0p = Wq + n0 * sg.ldw + 16 * t;
    const uint8_t* q1p = Wq + n1 * sg.ldw + 16 * t;
    // Row scales: weights, not outputs of an earlier kernel, so read before the wait.
    const float rs0 = __ldg(sg.rs + n0);
    const float rs1 = __ldg(sg.rs + n1);

    const int xstride = p.xstride;
    const int xbuf = B * xstride;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw + kBulkSmemHead);
    float* red = reinterpret_cast<float*>(smem_raw + kBulkSmemHead + static_cast<size_t>(p.nbuf) * xbuf * 2);
    float* cpart = red + rows_per_cta * (B + 1) * kw;
    float* misc = cpart + rows_per_cta * B + kMaxSplits;   // cpart: cluster slots, see combine_and_store
    const bool norm = (p.flags & kFlagRmsNorm) != 0;

    // Byte offset, within one staged x buffer, of the 8 columns that words
    // 2h and 2h + 1 of this lane's slice multiply in slot 0 (batch row b,
    // columns 16t + 8h ..); slot j adds 128 bytes.
    uint32_t xo[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int b = (nb * 8 + g < B) ? nb * 8 + g : B - 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) xo[nb][h] = 2u * static_cast<uint32_t>(b * xstride + 16 * t + 8 * h);
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
    int rg_begin = 0;   // first slot of this warp's range in the current chunk

    // Issue the slots jr .. jr+UJ-1 of this warp's range (chunk at c0). A full
    // batch addresses its slots by immediate offsets; the last, partial batch
    // repeats its last slot in the unused ones, which are not consumed.
    auto issue = [&](int64_t c0, int jr, int my) {
        const int rem = my - jr;
        if (rem <= 0) return;
        const int64_t col0 = c0 + 64LL * (rg_begin + jr);
        const uint8_t* a0 = q0p + col0;
        const uint8_t* a1 = q1p + col0;
        if (rem >= UJ) {
#pragma unroll
            for (int u = 0; u < UJ; ++u) {
                qa[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a0 + 64 * u));
                qb[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a1 + 64 * u));
            }
        } else {
#pragma unroll
            for (int u = 0; u < UJ; ++u) {
                const int uu = u < rem ? u : rem - 1;
                qa[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a0 + 64 * uu));
                qb[u] = ld_stream16(reinterpret_cast<const uint16_t*>(a1 + 64 * uu));
            }
        }
    };

    // Contract slot u (64 columns of rows n0, n1) with x at xg (the staged x of
    // this batch's first slot) into the batch tile d.
    auto consume = [&](int u, const unsigned char* xg, float (&d)[NB][4]) {
        const uint32_t wa[4] = {qa[u].x, qa[u].y, qa[u].z, qa[u].w};
        const uint32_t wb[4] = {qb[u].x, qb[u].y, qb[u].z, qb[u].w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t A0[2], B0[2], A1[2], B1[2];
            fp8_widen_word(wa[2 * h], A0);
            fp8_widen_word(wb[2 * h], B0);
            fp8_widen_word(wa[2 * h + 1], A1);
            fp8_widen_word(wb[2 * h + 1], B1);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const uint4 xr = *reinterpret_cast<const uint4*>(xg + xo[nb][h] + 128 * u);
                mma_bf16_16816(d[nb], A0[0], B0[0], A0[1], B0[1], xr.x, xr.y);
                mma_bf16_16816(d[nb], A1[0], B1[0], A1[1], B1[1], xr.z, xr.w);
            }
        }
    };

    Chunk ch = chunk_at(k0, k1, p.kchunk, K);
    int nslots = ch.nv >> 3;   // K is a multiple of 64: whole slots only
    F8Range rg = f8_range(nslots, kw, kq);
    rg_begin = rg.j_begin;
    issue(ch.c0, 0, rg.my_slots);
    if (!(p.flags & kFlagNoWait)) pdl_wait_prerequisites();
    bool x_ok = true;   // false when the wait for the bulk copy of x ran out
    if constexpr (XB) {
        bulk_stage_x(mbar, xs, xstride, p.x, B, K, ch.c0, ch.nv);   // K % 64 == 0: whole vectors
        x_ok = mbar_wait_bounded(mbar, 0);
    } else {
        stage_x(xs, xstride, p.x, B, K, ch.c0, ch.nv);
    }

#pragma unroll 1
    for (int c = 0;; ++c) {
        const unsigned char* xsb = reinterpret_cast<const unsigned char*>(xs + (c & 1) * xbuf);
        const int64_t next_c0 = ch.c0 + p.kchunk;
        const bool more = CHUNKED && next_c0 < k1;
        Chunk nch{};
        if (more) {
            nch = chunk_at(next_c0, k1, p.kchunk, K);
            stage_x(xs + ((c + 1) & 1) * xbuf, xstride, p.x, B, K, nch.c0, nch.nv);
            cp_async_wait<1>();
        } else if constexpr (!XB) {
            cp_async_wait<0>();
        }
        if constexpr (!XB) __syncthreads();   // with XB the mbarrier wait made x visible

        const int my = rg.my_slots;
#pragma unroll 1
        for (int j0 = 0; j0 < my; j0 += UJ) {
            if (j0 > 0) issue(ch.c0, j0, my);
            const unsigned char* xg = xsb + 128 * (rg_begin + j0);
            const int rem = my - j0;
            float d[NB][4];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int i = 0; i < 4; ++i) d[nb][i] = 0.f;
            if (rem >= UJ) {
#pragma unroll
                for (int u = 0; u < UJ; ++u) consume(u, xg, d);
            } else {
#pragma unroll
                for (int u = 0; u < UJ; ++u)
                    if (u < rem) consume(u, xg, d);
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nb][i] += d[nb][i];
        }
        if (norm) xsq_accumulate(reinterpret_cast<const uint16_t*>(xsb), xstride, B, ch.nv, misc, c == 0);
        if (!more) break;

        ch = nch;
        nslots = ch.nv >> 3;
        rg = f8_range(nslots, kw, kq);
        rg_begin = rg.j_begin;
        issue(ch.c0, 0, rg.my_slots);
        __syncthreads();
    }

    const int rl0 = gw * kMmaRows + g;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = nb * 8 + 2 * t + (i & 1);
            const int rl = rl0 + ((i & 2) ? 8 : 0);
            // A CTA whose copy of x did not arrive in time stores NaN (and
            // has set the status bit) rather than sums over an incomplete x.
            if (b < B)
                red[red_index(kq, rows_per_cta, rl, B, b)] =
                    x_ok ? acc[nb][i] * ((i & 2) ? rs1 : rs0) : __uint_as_float(0x7fc00000u);
        }
    }
    combine_and_store(red, cpart, misc, rows_per_cta, B, kw, S, split, sg.tile_local * rows_per_cta, sg.N, sg.y,
                      norm, K, p.rms_eps, p.wc);
    if constexpr (XB) {
        if (!x_ok) mbar_wait_bounded(mbar, 0);   // the copy may still be in flight: wait once more
    }
}

template <int NB, int UJ>
cudaError_t launch_fp8_uj(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    if (l.nbuf > 1) return launch_kernel(gemv_fp8_kernel<NB, UJ, true>, p, l, s, pdl);
    if (l.xbulk) return launch_kernel(gemv_fp8_kernel<NB, UJ, false, true>, p, l, s, pdl);
    return launch_kernel(gemv_fp8_kernel<NB, UJ, false>, p, l, s, pdl);
}

template <int NB, int UJ>
cudaError_t prepare_fp8_uj() {
    cudaError_t e = cudaFuncSetAttribute(gemv_fp8_kernel<NB, UJ, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(gemv_fp8_kernel<NB, UJ, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kMaxDynSmem)) != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(gemv_fp8_kernel<NB, UJ, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

// Status bits this translation unit's kernels recorded, cleared when `reset`.
inline cudaError_t read_fp8_status_tu(unsigned int* bits, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess || !reset || *bits == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace gemv
