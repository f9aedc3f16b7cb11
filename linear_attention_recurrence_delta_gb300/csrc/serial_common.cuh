// serial_common.cuh -- device helpers shared by the token-serial kernels:
// I/O conversions, the padded row-vector layout, cp.async and packed fp32x2
// arithmetic (sm_100 family).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace rec {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename IO>
__device__ __forceinline__ IO from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// A staged per-token row vector (alpha, b or c over the d_k state rows) keeps
// rows 16q..16q+15 at offsets 20q..20q+15 (a padded length of 5/4 of the rows):
// a thread that owns 16 consecutive rows reads them as four 16-byte loads, and
// the row groups of a warp land in disjoint banks.
__device__ __forceinline__ int prow(int i) { return i + ((i >> 4) << 2); }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// 2^x on the special-function unit (relative error about 2^-22)
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// alpha = exp(g A): the library expf for fp32 I/O; for bf16 I/O the SFU exp2
// of g (A log2 e), whose ~1e-6 relative error is far below bf16 rounding
template <typename IO>
__device__ __forceinline__ float decay(float g, float A, float A_log2e)
{
    if (sizeof(IO) == 4) return expf(g * A);
    return ex2_approx(g * A_log2e);
}

// logistic function, for g and beta given as logits (GDN_GATE_LOGITS)
__device__ __forceinline__ float sigmoidf(float z) { return 1.f / (1.f + expf(-z)); }
__device__ __forceinline__ float gate(float x, int logits) { return logits ? sigmoidf(x) : x; }

__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// 16 consecutive staged rows (padded layout) as 8 packed pairs
__device__ __forceinline__ void ld_rows16(const float* p, float2 (&r)[8])
{
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const float4 x = *reinterpret_cast<const float4*>(p + 4 * q);
        r[2 * q] = f2(x.x, x.y);
        r[2 * q + 1] = f2(x.z, x.w);
    }
}

// sum_k x[k] . y[k] over 8 packed pairs, four independent partial sums
__device__ __forceinline__ float dot8x2(const float2 (&x)[8], const float2 (&y)[8])
{
    float2 s0 = mul2(x[0], y[0]), s1 = mul2(x[1], y[1]), s2 = mul2(x[2], y[2]), s3 = mul2(x[3], y[3]);
    s0 = fma2(x[4], y[4], s0);
    s1 = fma2(x[5], y[5], s1);
    s2 = fma2(x[6], y[6], s2);
    s3 = fma2(x[7], y[7], s3);
    s0 = add2(add2(s0, s1), add2(s2, s3));
    return s0.x + s0.y;
}

}  // namespace rec
}  // namespace gdn
