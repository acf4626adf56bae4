// Tensor-core kernel instance for batches of up to 16 rows.
#include "gemv_mma_kernel.cuh"

namespace gemv {

cudaError_t launch_mma_nb2(const Params& p, const Launch& l, cudaStream_t s, bool pdl) {
    return launch_mma<2>(p, l, s, pdl);
}

cudaError_t prepare_mma_nb2() { return prepare_mma<2>(); }

cudaError_t read_mma_status_nb2(unsigned int* bits, bool reset) { return read_mma_status(bits, reset); }

}  // namespace gemv
