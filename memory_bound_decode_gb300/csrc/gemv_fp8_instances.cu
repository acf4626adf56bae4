// FP8-weight kernel instances (batches of up to 8 and up to 16 rows).
#include "gemv_fp8_kernel.cuh"

namespace gemv {

// The deep instance (kF8DeepUnroll) serves up to 8 rows only.
cudaError_t launch_fp8_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    if (mma_nblocks(B) == 1) {
        if (l.unroll == kF8DeepUnroll) return launch_fp8_uj<1, kF8DeepUnroll>(p, l, s, pdl);
        if (l.unroll == kF8Unroll) return launch_fp8_uj<1, kF8Unroll>(p, l, s, pdl);
        return cudaErrorInvalidValue;
    }
    if (l.unroll != kF8Unroll) return cudaErrorInvalidValue;
    return launch_fp8_uj<2, kF8Unroll>(p, l, s, pdl);
}

cudaError_t read_fp8_status(unsigned int* bits, bool reset) { return read_fp8_status_tu(bits, reset); }

cudaError_t prepare_fp8_all() {
    cudaError_t e = prepare_fp8_uj<1, kF8Unroll>();
    if (e != cudaSuccess) return e;
    if ((e = prepare_fp8_uj<1, kF8DeepUnroll>()) != cudaSuccess) return e;
    return prepare_fp8_uj<2, kF8Unroll>();
}

}  // namespace gemv
