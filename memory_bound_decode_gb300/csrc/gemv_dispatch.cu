// Batch-size dispatch and the read-only bandwidth probe.
#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_internal.h"

namespace gemv {

cudaError_t launch_fma_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_fma_all();
cudaError_t launch_mma_nb1(const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t launch_mma_nb2(const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_mma_nb1();
cudaError_t prepare_mma_nb2();
cudaError_t launch_w4_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_w4_all();
cudaError_t launch_fp8_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_fp8_all();
cudaError_t launch_tc_batch(const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_tc_all();

cudaError_t launch_gemv(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    if (B < 1 || B > kMaxBatch) return cudaErrorInvalidValue;
    if (l.path == kPathFma) return launch_fma_batch(B, p, l, s, pdl);
    if (l.path == kPathW4) return launch_w4_batch(B, p, l, s, pdl);
    if (l.path == kPathFp8) return launch_fp8_batch(B, p, l, s, pdl);
    if (l.path == kPathTc) return launch_tc_batch(p, l, s, pdl);
    return mma_nblocks(B) == 1 ? launch_mma_nb1(p, l, s, pdl) : launch_mma_nb2(p, l, s, pdl);
}

cudaError_t prepare_kernels(int /*device: attributes apply to the current device*/) {
    cudaError_t e;
    if ((e = prepare_fma_all()) != cudaSuccess) return e;
    if ((e = prepare_mma_nb1()) != cudaSuccess) return e;
    if ((e = prepare_w4_all()) != cudaSuccess) return e;
    if ((e = prepare_fp8_all()) != cudaSuccess) return e;
    if ((e = prepare_streamk()) != cudaSuccess) return e;
    if ((e = prepare_tc_all()) != cudaSuccess) return e;
    return prepare_mma_nb2();
}

// Streams `nvec` 16-byte vectors with the GEMV's load form, 8 independent loads
// per thread in flight, and leaves one checksum per CTA so that nothing is
// optimised away. Measures the read-only HBM ceiling.
__global__ void __launch_bounds__(256) probe_read_kernel(const uint4* __restrict__ src, int64_t nvec,
                                                         float* __restrict__ sink) {
    constexpr int U = 8;
    uint32_t h = 0;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + (U - 1) * stride < nvec; i += U * stride) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint4* q = src + i + u * stride;
            asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                : "=r"(v[u].x), "=r"(v[u].y), "=r"(v[u].z), "=r"(v[u].w)
                : "l"(q));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) h ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < nvec; i += stride) {
        const uint4 v = __ldg(src + i);
        h ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) h ^= __shfl_xor_sync(0xffffffffu, h, off);
    __shared__ uint32_t part[8];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = h;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t ^= part[w];
        sink[blockIdx.x] = __uint_as_float(t & 0x007fffffu);   // a finite float
    }
}

cudaError_t launch_probe_read(const void* src, int64_t bytes, float* sink, int grid, cudaStream_t s) {
    probe_read_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(src), bytes / 16, sink);
    return cudaGetLastError();
}

}  // namespace gemv
