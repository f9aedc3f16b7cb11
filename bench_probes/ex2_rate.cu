// ex2_rate.cu -- throughput of the special-function unit's exp2 (ex2.approx.f32)
// on the current device.  A measurement aid, not part of the method: the
// chunked forward evaluates its decay factors with this instruction, and the
// rate bounds how fast those exponentials can go.  Built as its own library
// (libgdn_probe.so) so that libgdn's boundary holds only the method.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// eight independent chains per thread; x <- 2^(-x) keeps every value in [0.5, 1]
__global__ void ex2_kernel(float* out, int iters)
{
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; k++) x[k] = 0.25f + 0.01f * k + 1e-6f * threadIdx.x;
    for (int i = 0; i < iters; i++) {
#pragma unroll
        for (int k = 0; k < 8; k++) x[k] = ex2(-x[k]);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; k++) s += x[k];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

// Measures exp2 evaluations per second over the whole device (every SM, four
// 256-thread CTAs each, eight chains per thread): one warm-up launch, then the
// median of five timed launches (CUDA events).  Returns 0 on success, -1 if a
// CUDA call failed.
extern "C" int gdn_probe_ex2_rate(double* ex2_per_s)
{
    int dev = 0, sms = 0;
    if (!ex2_per_s || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    const int blocks = 4 * sms, threads = 256, iters = 1 << 14;
    float* out = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int rc = -1;
    float ms[5];
    if (cudaMalloc(&out, sizeof(float) * blocks * threads) != cudaSuccess) return -1;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) goto done;
    ex2_kernel<<<blocks, threads>>>(out, iters);
    if (cudaDeviceSynchronize() != cudaSuccess) goto done;
    for (int r = 0; r < 5; r++) {
        cudaEventRecord(e0);
        ex2_kernel<<<blocks, threads>>>(out, iters);
        cudaEventRecord(e1);
        if (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms[r], e0, e1) != cudaSuccess)
            goto done;
    }
    for (int i = 1; i < 5; i++)   // sort the five times
        for (int j = i; j > 0 && ms[j] < ms[j - 1]; j--) {
            const float t = ms[j]; ms[j] = ms[j - 1]; ms[j - 1] = t;
        }
    *ex2_per_s = (double)blocks * threads * iters * 8 / (ms[2] * 1e-3);
    rc = 0;
done:
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(out);
    return rc;
}
