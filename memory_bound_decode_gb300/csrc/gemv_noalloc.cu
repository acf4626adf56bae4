// Fixed scratch of gemv_bf16_streamk_noalloc: the stream-K kernel's partial
// sums and per-row counters in file-scope device arrays, so that the call
// never allocates. Device globals start at zero when the module is loaded,
// which is the state the counters must be in before the first launch; every
// launch leaves them at zero again.
#include <cstdint>
#include <cuda_runtime.h>

#include "gemv_internal.h"

namespace gemv {

static __device__ __align__(256) float g_noalloc_part[kNoallocPartFloats];
static __device__ __align__(256) int32_t g_noalloc_ticket[kNoallocTickets];

cudaError_t noalloc_scratch(float** part, int32_t** ticket) {
    void* a = nullptr;
    void* b = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_noalloc_part);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetSymbolAddress(&b, g_noalloc_ticket)) != cudaSuccess) return e;
    *part = static_cast<float*>(a);
    *ticket = static_cast<int32_t*>(b);
    return cudaSuccess;
}

}  // namespace gemv
