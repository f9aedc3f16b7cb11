// chunk_common.cuh -- pieces shared by the chunk-parallel kernels of the chunked
// backward (gdn_chunk_bwd.cu): general tcgen05 products over shared-memory tiles
// in either major order, 16-column tile rows, and the per-chunk decay tables.
//
// Tiles are [rows][64] 16-bit elements with 128-byte swizzling (tc_ptx.cuh).  A
// tile read "K-major" has its rows along M (or N) and K contiguous; read
// "MN-major" it has its rows along K and M (or N) contiguous, so the same bytes
// serve as a matrix or as its transpose.
#pragma once

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

// one element (row, col) of a tile, 16-bit store
__device__ __forceinline__ void st1_bf16(unsigned char* t, int row, int col, float x)
{
    *reinterpret_cast<__nv_bfloat16*>(t + sw128(row, col)) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ void st1_split(unsigned char* thi, unsigned char* tlo, int row, int col, float x)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const uint32_t off = sw128(row, col);
    *reinterpret_cast<__nv_bfloat16*>(thi + off) = h;
    *reinterpret_cast<__nv_bfloat16*>(tlo + off) = __float2bfloat16_rn(x - __bfloat162float(h));
}

// The chunk's decay tables.  With G_t the inclusive sum of g within the chunk, A2 = A log2(e) and the anchor
// token r(k8) = 8 k8 + 3 of each 8-block, every decay factor the kernels use is an anchor
// alpha_t = 2^(A2 (G_t - G_r(t))) (or its inverse) times one of these per-(8-block, channel) constants, all <= 1:
//   KA1[k8]    = 2^(A2 (G_r(k8) - G_{16 I - 1})),  I = k8 / 2 >= 1   (row factor of the 16-block level)
//   K0[k8]     = 2^(A2 G_r(k8))                                     (exp(A G_t) = alpha_t K0)
//   KB1[I][k8] = 2^(A2 (G_{16 I - 1} - G_r(k8))),  k8 < 2 I          (column factor towards row block I)
//   KBH[k8]    = 2^(A2 (G_63 - G_r(k8)))                            (exp(A (G_63 - G_t)) = KBH / alpha_t)
//   KAP[J]     = 2^(A2 (G_{16 J + 11} - G_{16 J + 3}))              (upper vs lower 8-half of 16-block J)
//   EC         = 2^(A2 G_63)                                        (the chunk's decay)
struct Tables {
    float KA1[8][64];
    float K0[8][64];
    float KB1[3][8][64];
    float KBH[8][64];
    float KAP[4][64];
    float EC[64];
};

// entry e (0 .. 8 * 64 - 1) of every [8][64] table, and the [4][64] and [64] ones for the first 4 * 64 entries
__device__ __forceinline__ void table_entries(Tables& K, const float* G, const float* A2, int e)
{
    const int k8 = e >> 6, i = e & 63, I = k8 >> 1;
    const float a2 = A2[i], Gr = G[8 * k8 + 3];
    K.KA1[k8][i] = I >= 1 ? fast_exp2(a2 * (Gr - G[16 * I - 1])) : 0.f;
    K.K0[k8][i] = fast_exp2(a2 * Gr);
#pragma unroll
    for (int J = 1; J <= 3; J++) K.KB1[J - 1][k8][i] = k8 < 2 * J ? fast_exp2(a2 * (G[16 * J - 1] - Gr)) : 0.f;
    K.KBH[k8][i] = fast_exp2(a2 * (G[63] - Gr));
    if (k8 < 4) K.KAP[k8][i] = fast_exp2(a2 * (G[16 * k8 + 11] - G[16 * k8 + 3]));
    if (k8 == 0) K.EC[i] = fast_exp2(a2 * G[63]);
}

// Row of the 16-block level's column operand for row block I (1..3) and token s < 16 I: the three blocks'
// column operands are stacked, 16, 32 and 48 rows.
__host__ __device__ __forceinline__ int seg_base(int I) { return I == 1 ? 0 : (I == 2 ? 16 : 48); }

}  // namespace chunk
}  // namespace gdn
