// CUDA-core kernel instances: batch 1 and 2 here, 3..8 and 9..16 in their own
// translation units (compiled in parallel); the batch dispatch.
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_fma_b3_8(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t launch_fma_b9_16(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl);
cudaError_t prepare_fma_b3_8();
cudaError_t prepare_fma_b9_16();

cudaError_t launch_fma_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 1: return launch_fma<1>(p, l, s, pdl);
    case 2: return launch_fma<2>(p, l, s, pdl);
    default: return B <= 8 ? launch_fma_b3_8(B, p, l, s, pdl) : launch_fma_b9_16(B, p, l, s, pdl);
    }
}

cudaError_t prepare_fma_all() {
    cudaError_t e = prepare_fma<1>();
    if (e != cudaSuccess) return e;
    if ((e = prepare_fma<2>()) != cudaSuccess) return e;
    if ((e = prepare_fma_b3_8()) != cudaSuccess) return e;
    return prepare_fma_b9_16();
}

cudaError_t read_fma_status(unsigned int* bits, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess || !reset || *bits == 0) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace gemv
