// gdn_check.cu -- GDN_CHECK_FINITE: a scan of an output for NaN and Inf that
// raises a flag word in the workspace's status block (word 1) instead of
// trapping, so the host learns of it through gdn_last_device_status.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ __forceinline__ bool finite_el(float x) { return isfinite(x); }
__device__ __forceinline__ bool finite_el(__nv_bfloat16 x) { return isfinite(__bfloat162float(x)); }

template <typename T>
__global__ void check_finite_kernel(const T* p, size_t n, uint32_t* flag)
{
    bool bad = false;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        bad |= !finite_el(p[i]);
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(flag, 1u);
}

}  // namespace

cudaError_t launch_check_finite(const void* p, size_t n, int io, void* ws, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    uint32_t* flag = reinterpret_cast<uint32_t*>(ws) + 1;
    const size_t want = (n + 255) / 256;
    const int blocks = (int)(want < 8 * 152 ? want : 8 * 152);
    if (io == GDN_BF16)
        check_finite_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(p), n, flag);
    else
        check_finite_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const float*>(p), n, flag);
    return cudaGetLastError();
}

}  // namespace gdn
