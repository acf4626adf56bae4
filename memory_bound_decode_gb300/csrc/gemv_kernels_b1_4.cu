// Kernel instances for batch sizes 1..4 (one translation unit per range so
// the instances compile in parallel).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_gemv_b1_4(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 1: return launch_batch<1>(p, l, s, pdl);
    case 2: return launch_batch<2>(p, l, s, pdl);
    case 3: return launch_batch<3>(p, l, s, pdl);
    case 4: return launch_batch<4>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_b1_4() {
    cudaError_t e = cudaSuccess;
    if ((e = prepare_batch<1>()) != cudaSuccess) return e;
    if ((e = prepare_batch<2>()) != cudaSuccess) return e;
    if ((e = prepare_batch<3>()) != cudaSuccess) return e;
    if ((e = prepare_batch<4>()) != cudaSuccess) return e;
    return e;
}

}  // namespace gemv
