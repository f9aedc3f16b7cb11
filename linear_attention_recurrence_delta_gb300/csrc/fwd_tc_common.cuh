// fwd_tc_common.cuh -- pieces shared by the chunked tcgen05 forward kernels:
// swizzled-tile row access, bf16 hi/lo splitting, decay scaling, bounded
// waits and the TMA descriptor for the [B, T, H, d] bf16 tensors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <string.h>

#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace fwdtc {

using namespace tc;

constexpr int kC = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kSafeLog2 = 100.f;   // bound on |A| log2(e) * (sum of 4 g) for the 8-block split

// Per-launch parameters (tensor maps live in the kernel parameter space).
struct TcParams {
    CUtensorMap tm_v, tm_b, tm_c;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    const float* A_log;
    const float* h0;
    __nv_bfloat16* o;
    float* o32;              // if not null: o is written here in fp32 instead (time-split intermediate runs)
    float* hT;
    uint32_t* status;
    int B, H, T, dk, dv, nchunks;
    int logits;   // g, beta arrive before their sigmoid
    int starve_chunk;        // failure-path test hook: the loads of this chunk are never issued (-1: none)
    uint64_t wait_ns;        // limit of every bounded wait
    float* st;               // saving forward: the states entering the chunks
    unsigned char* sv;       // saving forward: the solve's results per chunk
    uint32_t sv_stride;      // saving forward: bytes per chunk of sv
    int seg, seg_len;        // saving forward over a time split: segments per sequence (else 1), chunks each
};

// Limit of a bounded wait: a chunk's loads or products take microseconds, so two
// seconds only expire when something that should arrive never will.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kTestWaitNs = 200000000ull;   // under the failure-path test hook

// g or beta as the rule uses it: the logistic function of a logit (SFU exponential;
// this path takes bf16 inputs), or the value itself
__device__ __forceinline__ float gate_in(float x, int logits) { return logits ? 1.f / (1.f + __expf(-x)) : x; }

__device__ __forceinline__ float bf2f(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

// 8 bf16 of row `row`, chunk q (elements 8q..8q+7) of a swizzled [.][64] tile
__device__ __forceinline__ void ld_row8(const unsigned char* tile, int row, int q, float (&v)[8])
{
    const uint4 u = *reinterpret_cast<const uint4*>(tile + sw128(row, 8 * q));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void st_row8(unsigned char* tile, int row, int q, const float (&v)[8])
{
    uint4 u;
    u.x = pack_bf16(v[0], v[1]);
    u.y = pack_bf16(v[2], v[3]);
    u.z = pack_bf16(v[4], v[5]);
    u.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(tile + sw128(row, 8 * q)) = u;
}

// 8 values of row `row`, chunk q, stored as fp16 (for operands bounded by
// the inputs' magnitude, where fp16's finer rounding beats bf16)
__device__ __forceinline__ void st_row8_f16(unsigned char* tile, int row, int q, const float (&v)[8])
{
    uint4 u;
    u.x = pack_f16(v[0], v[1]);
    u.y = pack_f16(v[2], v[3]);
    u.z = pack_f16(v[4], v[5]);
    u.w = pack_f16(v[6], v[7]);
    *reinterpret_cast<uint4*>(tile + sw128(row, 8 * q)) = u;
}

// store hi = bf16(v) and lo = bf16(v - hi): together ~16 significant bits
__device__ __forceinline__ void st_row8_split(unsigned char* thi, unsigned char* tlo, int row, int q,
                                              const float (&v)[8])
{
    uint32_t hp[4], lp[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        hp[k] = pack_bf16(v[2 * k], v[2 * k + 1]);
        const float h0 = __uint_as_float(hp[k] << 16), h1 = __uint_as_float(hp[k] & 0xFFFF0000u);
        lp[k] = pack_bf16(v[2 * k] - h0, v[2 * k + 1] - h1);
    }
    const uint32_t off = sw128(row, 8 * q);
    *reinterpret_cast<uint4*>(thi + off) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
    *reinterpret_cast<uint4*>(tlo + off) = make_uint4(lp[0], lp[1], lp[2], lp[3]);
}

// 8 consecutive floats from shared memory (16-byte aligned)
__device__ __forceinline__ void ld_f8(const float* p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// 2^x on the SFU (ex2.approx, flush-to-zero; relative error ~2^-22)
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x[k] * exp2(A2[8q+k] * dG) for the 8 channels of chunk q
__device__ __forceinline__ void scale8(const float (&x)[8], const float* A2, int q, float dG, float (&y)[8])
{
#pragma unroll
    for (int k = 0; k < 8; k++) y[k] = x[k] * exp2f(A2[8 * q + k] * dG);
}

// Bounded wait; after the first expiry every later wait returns at once, the
// status word records the timeout and the kernel winds down.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* abort_flag,
                                              uint32_t* status, uint64_t limit_ns)
{
    if (*(volatile uint32_t*)abort_flag) return false;
    if (mbar_wait(bar, parity, nullptr, limit_ns)) return true;
    *(volatile uint32_t*)abort_flag = 1;
    atomicExch(status, kDevTimeout);
    return false;
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = (EncodeTiledFn)ptr;
    }
    return fn;
}

// [B, T, H, d] bf16 -> 4-D map, box = 64 (d) x 1 (H) x 64 (T) x 1 (B), 128B swizzle
inline bool make_map(CUtensorMap* m, const void* base, int B, int T, int H, int d)
{
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2, (cuuint64_t)T * H * d * 2};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


}  // namespace fwdtc
}  // namespace gdn
