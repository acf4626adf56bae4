// Kernel instances for batch sizes 13..16 (one translation unit per range so
// the instances compile in parallel).
#include "gemv_kernel.cuh"

namespace gemv {

cudaError_t launch_gemv_b13_16(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    switch (B) {
    case 13: return launch_batch<13>(p, l, s, pdl);
    case 14: return launch_batch<14>(p, l, s, pdl);
    case 15: return launch_batch<15>(p, l, s, pdl);
    case 16: return launch_batch<16>(p, l, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t prepare_b13_16() {
    cudaError_t e = cudaSuccess;
    if ((e = prepare_batch<13>()) != cudaSuccess) return e;
    if ((e = prepare_batch<14>()) != cudaSuccess) return e;
    if ((e = prepare_batch<15>()) != cudaSuccess) return e;
    if ((e = prepare_batch<16>()) != cudaSuccess) return e;
    return e;
}

}  // namespace gemv
