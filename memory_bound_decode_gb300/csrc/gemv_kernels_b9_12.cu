// Kernel instances for batch sizes 9..12 (one translation unit per range so
// the instances compile in parallel).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_gemv_b9_12(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 9: return launch_batch<9>(p, l, s, pdl);
    case 10: return launch_batch<10>(p, l, s, pdl);
    case 11: return launch_batch<11>(p, l, s, pdl);
    case 12: return launch_batch<12>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_b9_12() {
    cudaError_t e = cudaSuccess;
    if ((e = prepare_batch<9>()) != cudaSuccess) return e;
    if ((e = prepare_batch<10>()) != cudaSuccess) return e;
    if ((e = prepare_batch<11>()) != cudaSuccess) return e;
    if ((e = prepare_batch<12>()) != cudaSuccess) return e;
    return e;
}

}  // namespace gemv
