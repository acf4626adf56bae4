// CUDA-core kernel instances for batches 9..16 (the GEMV_FLAG_CUDA_CORES path).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_fma_b9_16(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 9: return launch_fma<9>(p, l, s, pdl);
    case 10: return launch_fma<10>(p, l, s, pdl);
    case 11: return launch_fma<11>(p, l, s, pdl);
    case 12: return launch_fma<12>(p, l, s, pdl);
    case 13: return launch_fma<13>(p, l, s, pdl);
    case 14: return launch_fma<14>(p, l, s, pdl);
    case 15: return launch_fma<15>(p, l, s, pdl);
    case 16: return launch_fma<16>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_fma_b9_16() {
    cudaError_t e = cudaSuccess;
    if ((e = prepare_fma<9>()) != cudaSuccess) return e;
    if ((e = prepare_fma<10>()) != cudaSuccess) return e;
    if ((e = prepare_fma<11>()) != cudaSuccess) return e;
    if ((e = prepare_fma<12>()) != cudaSuccess) return e;
    if ((e = prepare_fma<13>()) != cudaSuccess) return e;
    if ((e = prepare_fma<14>()) != cudaSuccess) return e;
    if ((e = prepare_fma<15>()) != cudaSuccess) return e;
    if ((e = prepare_fma<16>()) != cudaSuccess) return e;
    return e;
}

}  // namespace gemv
