// CUDA-core kernel instances for batches 3..8 (the GEMV_FLAG_CUDA_CORES path).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_fma_b3_8(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 3: return launch_fma<3>(p, l, s, pdl);
    case 4: return launch_fma<4>(p, l, s, pdl);
    case 5: return launch_fma<5>(p, l, s, pdl);
    case 6: return launch_fma<6>(p, l, s, pdl);
    case 7: return launch_fma<7>(p, l, s, pdl);
    case 8: return launch_fma<8>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_fma_b3_8() {
    cudaError_t e = cudaSuccess;
    if ((e = prepare_fma<3>()) != cudaSuccess) return e;
    if ((e = prepare_fma<4>()) != cudaSuccess) return e;
    if ((e = prepare_fma<5>()) != cudaSuccess) return e;
    if ((e = prepare_fma<6>()) != cudaSuccess) return e;
    if ((e = prepare_fma<7>()) != cudaSuccess) return e;
    if ((e = prepare_fma<8>()) != cudaSuccess) return e;
    return e;
}

}  // namespace gemv
