// Kernel instances for batch sizes 5..8 (one translation unit per range so
// the instances compile in parallel).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_gemv_b5_8(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 5: return launch_batch<5>(p, l, s, pdl);
    case 6: return launch_batch<6>(p, l, s, pdl);
    case 7: return launch_batch<7>(p, l, s, pdl);
    case 8: return launch_batch<8>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_b5_8() {
    cudaError_t e = cudaSuccess;
    if ((e = prepare_batch<5>()) != cudaSuccess) return e;
    if ((e = prepare_batch<6>()) != cudaSuccess) return e;
    if ((e = prepare_batch<7>()) != cudaSuccess) return e;
    if ((e = prepare_batch<8>()) != cudaSuccess) return e;
    return e;
}

}  // namespace gemv
