// chunk_common.cuh -- pieces shared by the chunk-parallel kernels of the chunked
// backward (gdn_chunk_bwd.cu): general tcgen05 products over shared-memory tiles
// in either major order, and 16-column tile rows in bf16, fp16 and hi/lo pairs.
//
// Tiles are [rows][64] 16-bit elements with 128-byte swizzling (tc_ptx.cuh).  A
// tile read "K-major" has its rows along M (or N) and K contiguous; read
// "MN-major" it has its rows along K and M (or N) contiguous, so the same bytes
// serve as a matrix or as its transpose.
#pragma once

#include <cuda_fp16.h>

#include "fwd_tc_common.cuh"

namespace gdn {
namespace chunk {

using namespace tc;
using namespace fwdtc;

// D[d] (+)= A x B over `ksteps` K-steps of 16.
//   K-major operand: step ks reads base + (ks / 4) * kblk + (ks % 4) * 32 (64-wide K blocks kblk bytes apart).
//   MN-major operand: step ks reads base + ks * 2048 (16 K-rows of 128 bytes); lbo = bytes between the
//   64-wide M (or N) blocks.
__device__ __forceinline__ void mma_tiles(uint32_t d, uint32_t a, bool a_mn, uint32_t a_lbo, uint32_t a_kblk,
                                          uint32_t b, bool b_mn, uint32_t b_lbo, uint32_t b_kblk, int ksteps,
                                          uint32_t idesc, bool acc)
{
    for (int ks = 0; ks < ksteps; ks++) {
        const uint32_t ao = a_mn ? (uint32_t)ks * 2048u : (uint32_t)(ks >> 2) * a_kblk + (uint32_t)(ks & 3) * 32u;
        const uint32_t bo = b_mn ? (uint32_t)ks * 2048u : (uint32_t)(ks >> 2) * b_kblk + (uint32_t)(ks & 3) * 32u;
        mma_bf16(d, sdesc(a + ao, a_mn ? a_lbo : 16u, 1024u), sdesc(b + bo, b_mn ? b_lbo : 16u, 1024u), idesc,
                 (acc || ks > 0) ? 1u : 0u);
    }
}

// 16 values into row `row`, columns 16 g .. 16 g + 15 of a tile
__device__ __forceinline__ void st16_bf16(unsigned char* t, int row, int g, const float (&v)[16])
{
    float a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; k++) { a[k] = v[k]; b[k] = v[8 + k]; }
    st_row8(t, row, 2 * g, a);
    st_row8(t, row, 2 * g + 1, b);
}

__device__ __forceinline__ void st16_f16(unsigned char* t, int row, int g, const float (&v)[16])
{
    float a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; k++) { a[k] = v[k]; b[k] = v[8 + k]; }
    st_row8_f16(t, row, 2 * g, a);
    st_row8_f16(t, row, 2 * g + 1, b);
}

// fp16 hi = f16(v) and lo = f16(v - hi): together ~22 significant bits
__device__ __forceinline__ void st16_f16_split(unsigned char* thi, unsigned char* tlo, int row, int g,
                                               const float (&v)[16])
{
    float h[16], l[16];
#pragma unroll
    for (int k = 0; k < 16; k++) {
        h[k] = __half2float(__float2half_rn(v[k]));
        l[k] = v[k] - h[k];
    }
    st16_f16(thi, row, g, h);
    st16_f16(tlo, row, g, l);
}

__device__ __forceinline__ void st16_split(unsigned char* thi, unsigned char* tlo, int row, int g,
                                           const float (&v)[16])
{
    float a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; k++) { a[k] = v[k]; b[k] = v[8 + k]; }
    st_row8_split(thi, tlo, row, 2 * g, a);
    st_row8_split(thi, tlo, row, 2 * g + 1, b);
}

__device__ __forceinline__ void zero16(unsigned char* t, int row, int g)
{
    *reinterpret_cast<uint4*>(t + sw128(row, 16 * g)) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(t + sw128(row, 16 * g + 8)) = make_uint4(0, 0, 0, 0);
}

// 16 bf16 of row `row`, columns 16 g .. 16 g + 15 of a swizzled tile, as fp32
__device__ __forceinline__ void ld16_bf16(const unsigned char* t, int row, int g, float (&v)[16])
{
    float a[8], b[8];
    ld_row8(t, row, 2 * g, a);
    ld_row8(t, row, 2 * g + 1, b);
#pragma unroll
    for (int k = 0; k < 8; k++) { v[k] = a[k]; v[8 + k] = b[k]; }
}

// Row of the 16-block level's column operand for row block I (1..3) and token s < 16 I: the three blocks'
// column operands are stacked, 16, 32 and 48 rows.
__host__ __device__ __forceinline__ int seg_base(int I) { return I == 1 ? 0 : (I == 2 ? 16 : 48); }

}  // namespace chunk
}  // namespace gdn
