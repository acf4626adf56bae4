// The tcgen05 kernel instance (2..16 rows of x, BF16 weights).
#include "gemv_tc_kernel.cuh"

namespace gemv {

cudaError_t launch_tc_batch(const Params& p, const Launch& l, cudaStream_t s, bool pdl) { return launch_tc(p, l, s, pdl); }

cudaError_t prepare_tc_all() { return prepare_tc(); }

cudaError_t read_tc_status(unsigned int* bits, bool reset) { return read_tc_status_tu(bits, reset); }

int64_t tc_smem_bytes(int B, int stages, int stage_cols) { return tc_layout(B, stages, stage_cols).total; }

bool tc_has_instance(int stages, int stage_cols) { return tc_instance(stages, stage_cols); }

// A kernel of the tcgen05 kernel's block size, registers within its bound and
// no body: the occupancy query below asks about it, because for the tcgen05
// kernel itself the runtime reported half the clusters that measurably run at
// once (15 of 8 CTAs where 36 do).
__global__ void __launch_bounds__(kThreads, 2) tc_residency_kernel() {}

// Clusters of S CTAs of the tcgen05 kernel's block size and shared memory
// (batch 16, the default ring) the current device keeps resident at once; -1
// if it cannot say.
int tc_max_active_clusters(int S) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = tc_layout(kMaxBatch, kTcStages, kTcStageCols).total;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(S);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(tc_residency_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxDynSmem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, tc_residency_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return n;
}

int64_t tcp_smem_bytes(int stages, int stage_cols) {
    return tcp_instance(stages, stage_cols) ? static_cast<int64_t>(tcp_total(stages, stage_cols)) : -1;
}

}  // namespace gemv
