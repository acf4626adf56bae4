// INT4-weight kernel instances (batches of up to 8 and up to 16 rows).
#include "gemv_w4_kernel.cuh"

namespace gemv {

cudaError_t launch_w4_batch(int B, const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    return mma_nblocks(B) == 1 ? launch_w4<1>(p, l, s, pdl) : launch_w4<2>(p, l, s, pdl);
}

cudaError_t prepare_w4_all() {
    cudaError_t e = prepare_w4<1>();
    if (e != cudaSuccess) return e;
    return prepare_w4<2>();
}

}  // namespace gemv
