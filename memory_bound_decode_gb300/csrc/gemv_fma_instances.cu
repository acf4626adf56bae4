// CUDA-core kernel instances (batch 1 and 2).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_fma_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 1: return launch_fma<1>(p, l, s, pdl);
    case 2: return launch_fma<2>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_fma_all() {
    cudaError_t e = prepare_fma<1>();
    if (e != cudaSuccess) return e;
    return prepare_fma<2>();
}

}  // namespace gemv
