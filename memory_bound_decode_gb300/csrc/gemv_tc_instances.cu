// The tcgen05 kernel instance (2..16 rows of x, BF16 weights).
#include "gemv_tc_kernel.cuh"

namespace gemv {

cudaError_t launch_tc_batch(const Params& p, const Launch& l, cudaStream_t s, bool pdl) { return launch_tc(p, l, s, pdl); }

cudaError_t prepare_tc_all() { return prepare_tc(); }

cudaError_t read_tc_status(unsigned int* bits, bool reset) { return read_tc_status_tu(bits, reset); }

int64_t tc_smem_bytes(int B, int stages, int stage_cols) { return tc_layout(B, stages, stage_cols).total; }

bool tc_has_instance(int stages, int stage_cols) { return tc_instance(stages, stage_cols); }

int64_t tcp_smem_bytes(int stages, int stage_cols) {
    return tcp_instance(stages, stage_cols) ? static_cast<int64_t>(tcp_total(stages, stage_cols)) : -1;
}

}  // namespace gemv
