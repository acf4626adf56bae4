// Instance and launcher of the stream-K batch-1 kernel.
#include "gemv_streamk_kernel.cuh"

namespace gemv {

cudaError_t launch_streamk(const SkParams& p, const SkLaunch& l, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem_bytes);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if (p.K % kSkUnitCols != 0) return cudaLaunchKernelEx(&cfg, gemv_streamk_kernel<kSkUnroll, true>, p);
    return cudaLaunchKernelEx(&cfg, gemv_streamk_kernel<kSkUnroll, false>, p);
}

cudaError_t prepare_streamk() {
    const int smem = static_cast<int>(kSkMaxXBytes + kMiscFloats * 4);
    cudaError_t e = cudaFuncSetAttribute(gemv_streamk_kernel<kSkUnroll, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemv_streamk_kernel<kSkUnroll, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace gemv
