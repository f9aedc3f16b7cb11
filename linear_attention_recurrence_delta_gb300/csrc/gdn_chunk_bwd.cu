// gdn_chunk_bwd.cu -- the chunked backward of the gated delta rule on tcgen05
// tensor cores (bf16 I/O, d_k, d_v <= 64): three chunk-level passes instead of a
// token-serial walk.
//
// "GDN & MLA Mechanism Deep-Dive", Step 5 (Chunked recurrence) solves each chunk
// of C = 64 tokens in closed form; with S the state entering a chunk,
//   gated: U = V;  delta ("HyMo-434M -- documentation portal", card 01):
//          (I + diag(beta) K) U = diag(beta) (V - Btil S),  U = Util - W S
//   O = Ctil S + P U,   S' = diag(E) S + Bhat^T U,
// with P, K the decay-weighted c.b and b.b scores, Ctil = c (.) exp(A G_t),
// Btil = b (.) exp(A G_t), Bhat = b (.) exp(A (G_63 - G_t)), E = exp(A G_63) and
// G_t the inclusive sum of g within the chunk.  The chunk's map of states is
// affine, S' = Phi S + Delta with Phi = diag(E) - Bhat^T W (gated: diag(E)) and
// Delta = Bhat^T Util (gated: Bhat^T V), and its outputs are O = Qc S + P Util
// with Qc = Ctil - P W (gated: Ctil).  So the adjoint of the entering state is
//   dS = Phi^T dS' + Y,   Y = Qc^T dO.
// The backward is therefore:
//   1. chunk_prep_kernel, one chunk at a time over every chunk of every head
//      (no chunk waits for another): Phi (delta), Delta and Y of each chunk;
//   2. the chain, one CTA per head: the states entering the chunks
//      (S_{k+1} = Phi_k S_k + Delta_k from h0) and the adjoints leaving them
//      (dS_k = Phi_k^T dS_{k+1} + Y_k from dh_T), fp32 records; in delta mode each
//      step is one tcgen05 product on Phi's tiles (chunk_chain_tc_kernel), in
//      gated mode an elementwise update (chunk_chain_gated_kernel);
//   3. chunk_grad_kernel, again one chunk at a time: with S and dS' of the
//      chunk known, every token gradient of the chunk by the reverse mode of its
//      closed form (the transposed contractions of the forward, on tcgen05).
//
// Decay split.  exp(A (G_t - G_s)) (s <= t) must be split into a row and a
// column factor without overflow (|A| up to 16 over 64 tokens reaches
// exp(+-1024)):
//   * tokens in different 16-blocks (t in block I > block of s): reference at
//     the last token before block I; both factors are <= 1, the operands fp16,
//     and one N = 96 product covers the three row blocks (their column operands
//     stacked: 16, 32 and 48 rows);
//   * tokens in the same 16-block ("near" pairs, the largest entries): fp32 on
//     the CUDA cores, exp(A (G_t - G_s)) = alpha_t / alpha_s with the anchor
//     alpha_t = exp(A (G_t - G_r)) at the 4th token r of t's 8-block (a factor
//     at most exp(|A| * sum of 4 g)), times exp(A (G_r' - G_r)) <= 1 when t and s
//     lie in different 8-halves.  A chunk whose anchors could overflow
//     (|A| log2(e) * 4-token span > 100) evaluates every near pair directly.
//
// Delta solve (WY form, as in the forward): D = the 32-blocks of I + M
// (M = diag(beta) K) is inverted in fp32 (16-blocks by forward substitution and
// their coupling block), L = the block below them, N = D^-1 L with N^2 = 0, so
//   (I + M)^-1 R = (I - N) D^-1 R   and   (I + M)^-T Z = D^-T (I - N^T) Z.
//
// Precision: the 16-block level's operands (factors <= 1) are fp16; every other
// product takes its derived operands as bf16 hi + lo pairs against exact bf16
// inputs (hi*x + lo*x), or hi*hi + hi*lo + lo*hi between two derived operands.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include "chunk_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace fwdtc;
using namespace chunk;

constexpr int kThreads = 256;
constexpr int kBS = 20;   // padded row stride of the fp32 16 x 16 blocks (conflict-free float4 rows)

struct CbParams {
    CUtensorMap tm_v, tm_b, tm_c, tm_do;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    const float* A_log;
    // delta: Phi of chunk q (S' = Phi S + Delta) as two bf16 tiles, hi then lo, each [64][64] (rows i, columns m)
    // in the 128-byte-swizzled layout of the MMA operands: 16 KB per chunk
    unsigned char* phi;
    // delta: the front's results that the gradient pass reuses (layout in namespace sv), 64 KB per chunk
    unsigned char* sv;
    // per chunk q = unit * nchunks + k, each 64 x 64 fp32 (rows = key channel i, columns = value column j), stored
    // column-group major (rec4)
    float* dlt;     // Delta
    float* ych;     // Y = Qc^T dO
    float* ec;      // gated: [q][64] exp(A G_63)
    float* st;      // the state entering the chunk
    float* dst;     // the adjoint of the state leaving the chunk
    const float* h0;
    const float* dhT;
    float* dh0;
    __nv_bfloat16 *dv, *db, *dc, *dg, *dbeta;
    float* dA_part;   // [q][64]: sum_t G_t dGam_t[i] of the chunk (times A in the reduction)
    uint32_t* status;
    int B, H, T, dk, dv_, nchunks, nq;
    uint64_t wait_ns;
    int starve;       // failure-path test hook: the chunk q whose loads are never issued (-1: none)
    int rev_only;     // the entering states came from the forward: the chain runs its reverse sweep only
    uint32_t sv_stride;   // bytes per chunk of the saved front (delta: sv::BYTES; gated residuals: P only, 16 KB)
    // delta, the chain as walks (few heads): nseg segments of seg_len chunks per unit (nseg = 1: no split)
    int nseg, seg_len;
    float* segrec;        // nseg > 1: per (direction, unit, segment) final X, final Pi, true start
    float* tvec;          // gated, nseg > 1: per (direction, chunk) the rows' decay product from the segment's start
    // the forward split in time by walks (delta): prep writes [Phi_hi | Qc_hi | Phi_lo | Qc_lo] per chunk to phi
    // and no Y; a saving forward's second walk writes D = T_k S_s to st for the residual fix-up
    int fwd_walks;
    int gated;            // prep from residuals, gated mode: Phi = diag(E) and Qc = Ctil come from g and c alone
    const float* fw_o32;  // the zero-start run's outputs, fp32 [B, T, H, d_v]
    __nv_bfloat16* fw_o;  // the outputs
    float* fw_st;         // saving: the residual states, made true by adding D (null: not saving)
};

// ---------------------------------------------------------------- shared memory
constexpr uint32_t OFF_STAGE = 0;                        // b, c, v, dO tiles (TMA)
constexpr uint32_t ST_B = 0, ST_C = 8192, ST_V = 16384, ST_DO = 24576;
constexpr int kAS = 68;                                  // padded row stride of ALPHA, YB (float4 rows, 2-way banks)
constexpr uint32_t OFF_ALPHA = 32768;                    // fp32 [64][kAS] anchors alpha_t[i]
constexpr uint32_t OFF_YB = OFF_ALPHA + 64 * kAS * 4;    // fp32 [64][kAS] b_t[i] / alpha_t[i]
constexpr uint32_t OFF_TAB = OFF_YB + 64 * kAS * 4;      // KU, KL [4][64], EC [64] (fp32)
constexpr uint32_t OFF_SMALL = OFF_TAB + 2560;
constexpr uint32_t OFF_X = 81920;                        // phase region

struct Small {
    float G[64];
    float A2[64];
    float g[64];
    float beta[64];
    float sd[4][64];     // grad: partial sums over value columns of dS'[i][j] S[i][j]
    float rs[2][2][64];  // grad: per (kind, column half) row partial sums
    float colsum[4][64];
    float dgp[4][64];    // grad: per channel quarter partial sums of dG_t
    uint64_t full, mma, full2;   // full2: the saved front (gradient pass, delta)
    uint32_t tmem_base, abort, unsafe;
    float a2max;
};
static_assert(sizeof(Small) <= OFF_X - OFF_SMALL, "small block");

// per 16-block J and channel: KU = 2^(A2 (G_{16J+11} - G_{16J+7})) and KL = 2^(A2 (G_{16J+7} - G_{16J+3})), both
// <= 1 and spanning 4 tokens; a pair (t in the upper 8-half, s in the lower one) has exp(A (G_t - G_s)) =
// (alpha_t KU) (KL / alpha_s) with both brackets <= 1 (an underflow in either means a negligible pair)
struct Tab {
    float KU[4][64];
    float KL[4][64];
    float EC[64];
};
static_assert(sizeof(Tab) <= OFF_SMALL - OFF_TAB, "tables");

// prep layout (offsets within the phase region)
namespace pl {
constexpr uint32_t A1 = 0, B1 = 16384, LR = 28672, LRL = 53248, NEAR = 69632, P = 78848, BH = 95232,
                   MS = 111616, DINV = 126976, BYTES = 143360;
constexpr uint32_t NA = 0, X0 = 28672, WU = 28672, QC = 0;
// gated: [Bhat | Ctil] hi, then lo
constexpr uint32_t GA = 0;
}  // namespace pl

// grad layout
namespace gl {
constexpr uint32_t A1 = 0, B1 = 16384, LR = 28672, LRL = 53248, NEAR = 69632, P = 78848,
                   MS = 103424, DINV = 118784, BYTES = 140288;
constexpr uint32_t NA = 0, X0 = 28672;
constexpr uint32_t NW = 16384, U = 28672, DSN = 61440;              // U_hi | S_hi | U_lo | S_lo
constexpr uint32_t BHH = 16384, BHL = 103424;
constexpr uint32_t DU = 78848, Z = 0, DOR = 78848, ZR = 0;
// the level operands of the reverse pass (A1H, A1L hi/lo; B1, B1L hi/lo) are written while [dO ; dR] [U | S]^T and
// U dS'^T run: clear of DOR, ZR, U and DSN, which those products read
constexpr uint32_t AD = 28672, NEARD = 61440, SEG = 28672, A1H = 95232, A1L = 111616, B1L = 128000;
static_assert(B1 >= ZR + 16384 && B1 + 96 * 128 <= U && A1H >= DOR + 16384 && B1L + 96 * 128 <= BYTES,
              "reverse-pass level operands clear of the products in flight");
// row stride of the epilogue's fp32 arrays: float4 rows, and a warp's 32 rows at one column map 8 rows of a
// quarter-warp onto disjoint bank groups (float4 access) or 32 consecutive banks (one row, 32 columns)
constexpr int kES = 68;
constexpr uint32_t SEG_END = SEG + 96 * kES * 4;
constexpr uint32_t DC = 78848, DB = DC + 64 * kES * 4, DG = DB + 64 * kES * 4, PB = SEG_END;
// (delta) the b-side rows' share of db, kept apart so that those rows run beside the dense terms; it also gives
// their share of dGam (times b)
constexpr uint32_t DB2 = 0;
static_assert(PB + 64 * kES * 4 <= DC && DG + 64 * kES * 4 <= BYTES && DB2 + 64 * kES * 4 <= SEG, "epilogue arrays");
}  // namespace gl

// The delta front's results that the gradient pass reuses, per chunk (byte offsets), written by the prep pass or
// by a saving forward (gdn_fwd_tc.cu, the same layout): P as hi, lo tiles; -N and Dinv, one half each of the
// stacked [-N ; -N] and [Dinv ; Dinv] operands; K (zero on and above the diagonal), fp32 64 x 64; -W, a bf16 tile
// [t][i] (its lo part after it: written by the saving forward only); at UT, fp32 [t][j], Util from the prep pass
// or U = Util - W S from the saving forward.  The fp32 matrices are column-group major like the records (rec4).
namespace sv {
constexpr uint32_t P = 0, NA = 16384, DINV = 24576, K = 32768, NW = 49152, NWL = 57344, UT = 65536, BYTES = 81920;
constexpr uint32_t GATED_BYTES = 16384;   // a gated saving forward keeps P only
}  // namespace sv

// fp32 sub-blocks inside MS: the diagonal 16-blocks of M, the 16-blocks below them inside each 32-block,
// the diagonal blocks' inverses and the 32-blocks' coupling blocks
constexpr uint32_t MS_M32 = 0, MS_C32 = 4 * 16 * kBS * 4, MS_DI32 = MS_C32 + 2 * 16 * kBS * 4,
                   MS_E32 = MS_DI32 + 4 * 16 * kBS * 4, MS_BYTES = MS_E32 + 2 * 16 * kBS * 4;
static_assert(MS_BYTES <= pl::DINV - pl::MS && MS_BYTES <= gl::DINV - gl::MS, "MS blocks");

// TMEM columns
constexpr uint32_t TM_D1 = 0;       // 16-block level [P ; K] (96 columns)
constexpr uint32_t TM_NX = 96;      // [N | X0V | X0W] -> [N | Util | W]
constexpr uint32_t TM_UT = TM_NX + 64, TM_W = TM_NX + 128;
constexpr uint32_t TM_COLS = 512;

#ifdef GDN_CHUNK_DEBUG
// debug builds only: cycles spent between the phase stamps of CTA 0, per kernel (0 prep, 1 grad, 2 delta chain),
// and its chunks (steps for the chain)
__device__ unsigned long long g_cb_stamps[3][32];
__device__ unsigned long long g_cb_last;
#define CB_STAMP(kid, k)                                                                  \
    do {                                                                                  \
        if (threadIdx.x == 0 && blockIdx.x == 0) {                                        \
            const unsigned long long now_ = clock64();                                    \
            g_cb_stamps[kid][k] += now_ - g_cb_last;                                      \
            g_cb_last = now_;                                                             \
        }                                                                                 \
    } while (0)
#define CB_STAMP_INIT                                                                     \
    do {                                                                                  \
        if (threadIdx.x == 0 && blockIdx.x == 0) g_cb_last = clock64();                   \
    } while (0)
#else
#define CB_STAMP(kid, k) do {} while (0)
#define CB_STAMP_INIT do {} while (0)
#endif

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ float* fptr(unsigned char* base, uint32_t off) { return reinterpret_cast<float*>(base + off); }

// The sum of 64 values x[s * stride] in a fixed order: four chains over s = 4 m + c, then (c0 + c1) + (c2 + c3)
__device__ __forceinline__ float sum64_fixed(const float* x, int stride)
{
    float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll 4
    for (int m = 0; m < 16; m++) {
        c0 += x[(4 * m) * stride];
        c1 += x[(4 * m + 1) * stride];
        c2 += x[(4 * m + 2) * stride];
        c3 += x[(4 * m + 3) * stride];
    }
    return (c0 + c1) + (c2 + c3);
}

// 4 bf16 of row `row`, columns col .. col + 3 (col a multiple of 4) of a swizzled tile, as fp32: one 8-byte load
__device__ __forceinline__ void ld4_bf16(const unsigned char* tile, int row, int col, float (&v)[4])
{
    const uint2 w = *reinterpret_cast<const uint2*>(tile + sw128(row, col));
    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xFFFF0000u);
    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xFFFF0000u);
}

// The fp32 records (Delta, Y, S, dS') are stored column-group major: the float4 of row `row`, columns col .. col + 3
// (col a multiple of 4) sits at index (col / 4) * 64 + row of the chunk's record, so the 32 rows of a warp read or
// write 512 contiguous bytes.
__device__ __forceinline__ float4* rec4(float* base, size_t q, int row, int col)
{
    return reinterpret_cast<float4*>(base + q * 4096) + ((col >> 2) * 64 + row);
}
__device__ __forceinline__ const float4* rec4(const float* base, size_t q, int row, int col)
{
    return reinterpret_cast<const float4*>(base + q * 4096) + ((col >> 2) * 64 + row);
}

__device__ __forceinline__ void tma_prefetch_l2(const void* tmap, int c0, int c1, int c2, int c3)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap), "r"(c0),
                 "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// ---------------------------------------------------------------- the common front of prep and grad
// Everything below runs with 256 threads: r = thread, trow = r & 127 = TMEM lane, q4 = lane quarter,
// wh = column half.
struct Ctx {
    unsigned char* sm;
    unsigned char* X;
    Small* S;
    Tab* KT;
    float* ALPHA;
    float* YB;
    uint32_t tbase, tl;
    int r, warp, lane, q4, wh, trow;
    uint32_t mma_phase;
};

__device__ __forceinline__ void bar_all() { named_bar_sync(1, kThreads); }

__device__ __forceinline__ void smem_to_tc()
{
    fence_proxy_async_smem();
    tc_fence_before();
    bar_all();
    tc_fence_after();
}

// one warp polls the MMA barrier, the others wait at the named barrier; an expired wait leaves `where` in
// status word 2
__device__ __forceinline__ bool mma_wait(Ctx& c, const CbParams& p, uint32_t where = 0)
{
    if (c.warp == 0 && !wait_or_abort(&c.S->mma, c.mma_phase, &c.S->abort, p.status, p.wait_ns) && c.lane == 0)
        atomicExch(p.status + 2, 100u + where);
    bar_all();
    c.mma_phase ^= 1;
    tc_fence_after();
    return *(volatile uint32_t*)&c.S->abort == 0;
}

// (1) scan of g (warp 0), overflow check of the anchors, decay tables
__device__ __forceinline__ void front_scan(Ctx& c)
{
    Small& S = *c.S;
    if (c.warp == 0) {
        const float ga = S.g[2 * c.lane], gb = S.g[2 * c.lane + 1];   // lane l scans tokens 2l, 2l + 1
        float x = ga + gb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (c.lane >= o) x += y;
        }
        const float ex = __shfl_up_sync(0xffffffffu, x, 1);
        S.G[2 * c.lane] = (c.lane > 0 ? ex : 0.f) + ga;
        S.G[2 * c.lane + 1] = x;
        float m = fmaxf(fabsf(S.A2[c.lane]), fabsf(S.A2[c.lane + 32]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        __syncwarp();
        // the 4-token spans of the anchors (first to 4th, 4th to 8th token of an 8-block) and of KU
        float span = 0.f;
        if (c.lane < 8) {
            const float g0 = S.G[8 * c.lane], g3 = S.G[8 * c.lane + 3], g7 = S.G[8 * c.lane + 7];
            span = fmaxf(g3 - g0, g7 - g3);
            if (c.lane & 1) span = fmaxf(span, g3 - S.G[8 * c.lane - 1]);
        }
        const bool bad = __any_sync(0xffffffffu, span * m > kSafeLog2);
        if (c.lane == 0) S.unsafe = bad ? 1u : 0u;
    }
    bar_all();
    {
        const int J = c.r >> 6, i = c.r & 63;
        const float a2 = S.A2[i];
        c.KT->KU[J][i] = fast_exp2(a2 * (S.G[16 * J + 11] - S.G[16 * J + 7]));
        c.KT->KL[J][i] = fast_exp2(a2 * (S.G[16 * J + 7] - S.G[16 * J + 3]));
        if (J == 0) c.KT->EC[i] = fast_exp2(a2 * S.G[63]);
    }
}

// (2) anchors of token t = r & 63 over channels 16 cq .. 16 cq + 15 (cq = r >> 6): ALPHA, YB; the 16-block level
// operands A1 = [c f1 ; b f1] (rows t >= 16) and B1 (the column operands of row blocks 1..3), fp16, and with
// A1lo, B1lo given their fp16 remainders (the backward's level products need the pairs: a pair (t, s) enters
// dGam_t through A1 and dGam_s through B1, and both must carry the same value)
__device__ __forceinline__ void front_operands(Ctx& c, unsigned char* A1, unsigned char* B1, bool with_b_rows,
                                               unsigned char* A1lo = nullptr, unsigned char* B1lo = nullptr,
                                               bool anchors = true)
{
    Small& S = *c.S;
    const int t = c.r & 63, cq = c.r >> 6, k8 = t >> 3, I = t >> 4;
    const float Gt = S.G[t], dG = Gt - S.G[8 * k8 + 3];
    const unsigned char* sB = c.sm + OFF_STAGE + ST_B;
    const unsigned char* sC = c.sm + OFF_STAGE + ST_C;
    float bv[16], cv[16];
    ld16_bf16(sB, t, cq, bv);
    ld16_bf16(sC, t, cq, cv);
    if (anchors) {
        float al[16], yb[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const float a2 = S.A2[16 * cq + e];
            al[e] = fast_exp2(a2 * dG);
            yb[e] = bv[e] * fast_exp2(-a2 * dG);
        }
        float* arow = c.ALPHA + t * kAS + 16 * cq;
        float* yrow = c.YB + t * kAS + 16 * cq;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            *reinterpret_cast<float4*>(arow + e) = make_float4(al[e], al[e + 1], al[e + 2], al[e + 3]);
            *reinterpret_cast<float4*>(yrow + e) = make_float4(yb[e], yb[e + 1], yb[e + 2], yb[e + 3]);
        }
    }
    // row factor of the 16-block level: exp(A (G_t - G_{16 I - 1})) <= 1
    float y[16], z[16];
    if (I >= 1) {
        const float Gref = S.G[16 * I - 1];
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const float f = fast_exp2(S.A2[16 * cq + e] * (Gt - Gref));
            y[e] = cv[e] * f;
            z[e] = bv[e] * f;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 16; e++) y[e] = z[e] = 0.f;
    }
    if (A1lo) {
        st16_f16_split(A1, A1lo, t, cq, y);
        if (with_b_rows) st16_f16_split(A1, A1lo, 64 + t, cq, z);
    } else {
        st16_f16(A1, t, cq, y);
        if (with_b_rows) st16_f16(A1, 64 + t, cq, z);
    }
    // column factors towards row blocks J > I: exp(A (G_{16 J - 1} - G_t)) <= 1
#pragma unroll 1
    for (int J = 1; J <= 3; J++) {
        if (t < 16 * J) {
            const float Gref = S.G[16 * J - 1];
#pragma unroll
            for (int e = 0; e < 16; e++) y[e] = bv[e] * fast_exp2(S.A2[16 * cq + e] * (Gref - Gt));
            if (B1lo) st16_f16_split(B1, B1lo, seg_base(J) + t, cq, y);
            else st16_f16(B1, seg_base(J) + t, cq, y);
        }
    }
}

// (3) the 16-block level product D1 = A1 B1^T (M = 128: rows 0..63 the c side, 64..127 the b side; N = 96)
__device__ __forceinline__ void issue_level(uint32_t tbase, const unsigned char* A1, const unsigned char* B1)
{
    mma_tiles(tbase + TM_D1, smem_u32(A1), false, 0, 0, smem_u32(B1), false, 0, 0, 4,
              idesc_f16(128, 96, false, false), false);
}

// (4) near pairs (same 16-block), fp32, register-blocked.  Per matrix (P: left = c, K: left = b) and 16-block J
// the pairs s <= t form three 8 x 8 quadrants: lower rows x lower columns, upper x upper (both same 8-half:
// x_t y_s with x = left alpha, y = b / alpha) and upper x lower (across: (x_t KU)(y_s KL)).  Task = (matrix,
// block, quadrant, 4-row block, 4-column block, channel half): 96 tasks per matrix, one per thread; the two
// channel halves of a 4 x 4 block sit in adjacent lanes and are added by one shuffle.  NEAR[mat][J][t][s]
// ([2][4][16][17]) receives every entry with s <= t (P) or s < t (K); entries above the diagonal are left
// unwritten and must not be read.
__device__ __forceinline__ void front_near(Ctx& c, float* NEAR, bool want_k)
{
    Small& S = *c.S;
    const int ntask = want_k ? 192 : 96;
    if (c.r >= ntask) return;   // whole warps (96, 192 are multiples of 32)
    const int mat = c.r / 96, rem = c.r % 96, J = rem / 24, rem2 = rem % 24, quad = rem2 >> 3, sub = rem2 & 7;
    const int tb = sub >> 2, sb = (sub >> 1) & 1, hh = sub & 1;
    const int t0 = (quad >= 1 ? 8 : 0) + 4 * tb, s0 = (quad == 1 ? 8 : 0) + 4 * sb;   // within the block
    const bool cross = quad == 2;
    const unsigned char* sL = c.sm + OFF_STAGE + (mat ? ST_B : ST_C);
    float acc[4][4];
#pragma unroll
    for (int ti = 0; ti < 4; ti++)
#pragma unroll
        for (int si = 0; si < 4; si++) acc[ti][si] = 0.f;
    if (!S.unsafe) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int ch0 = 32 * hh + 8 * q;
            float ku[8], kl[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                ku[e] = cross ? c.KT->KU[J][ch0 + e] : 1.f;
                kl[e] = cross ? c.KT->KL[J][ch0 + e] : 1.f;
            }
            float x[4][8], y[4][8];
#pragma unroll
            for (int ti = 0; ti < 4; ti++) {
                const int t = 16 * J + t0 + ti;
                float v8[8], a8[8];
                ld_row8(sL, t, ch0 >> 3, v8);
                ld_f8(c.ALPHA + t * kAS + ch0, a8);
#pragma unroll
                for (int e = 0; e < 8; e++) x[ti][e] = v8[e] * a8[e] * ku[e];
            }
#pragma unroll
            for (int si = 0; si < 4; si++) {
                const int s = 16 * J + s0 + si;
                float y8[8];
                ld_f8(c.YB + s * kAS + ch0, y8);
#pragma unroll
                for (int e = 0; e < 8; e++) y[si][e] = y8[e] * kl[e];
            }
#pragma unroll
            for (int ti = 0; ti < 4; ti++)
#pragma unroll
                for (int si = 0; si < 4; si++)
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[ti][si] = fmaf(x[ti][e], y[si][e], acc[ti][si]);
        }
    } else {
        // every factor evaluated directly (the anchors could overflow); the exponent is clamped at 0 for the
        // entries above the diagonal, which are discarded
        const unsigned char* sB = c.sm + OFF_STAGE + ST_B;
#pragma unroll 1
        for (int q = 0; q < 4; q++) {
            const int ch0 = 32 * hh + 8 * q;
#pragma unroll
            for (int ti = 0; ti < 4; ti++) {
                const int t = 16 * J + t0 + ti;
                float v8[8];
                ld_row8(sL, t, ch0 >> 3, v8);
#pragma unroll
                for (int si = 0; si < 4; si++) {
                    const int s = 16 * J + s0 + si;
                    float b8[8];
                    ld_row8(sB, s, ch0 >> 3, b8);
                    const float dG = fmaxf(S.G[t] - S.G[s], 0.f);
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[ti][si] = fmaf(v8[e] * b8[e], exp2f(S.A2[ch0 + e] * dG), acc[ti][si]);
                }
            }
        }
    }
#pragma unroll
    for (int ti = 0; ti < 4; ti++)
#pragma unroll
        for (int si = 0; si < 4; si++) acc[ti][si] += __shfl_xor_sync(0xffffffffu, acc[ti][si], 1);
    if (hh == 0) {
#pragma unroll
        for (int ti = 0; ti < 4; ti++) {
            float* out = NEAR + ((mat * 4 + J) * 16 + t0 + ti) * 17 + s0;
#pragma unroll
            for (int si = 0; si < 4; si++) out[si] = acc[ti][si];
        }
    }
}

// (5) P and K of row t = trow & 63 (lanes 0..63: P, 64..127: K), columns 32 wh .. 32 wh + 31, from the
// 16-block level (TMEM) and the near pairs.  v[0..31] receives the row part.
__device__ __forceinline__ void assemble_row(Ctx& c, const float* NEAR, float (&v)[32])
{
    const int t = c.trow & 63, isK = c.trow >> 6, I = t >> 4;
    // a warp's 32 rows span the 16-blocks Ia and Ia + 1; every TMEM load is warp-uniform, each lane then takes
    // the one of its block
    const int Ia = 2 * (c.q4 & 1), Ib = Ia + 1;
#pragma unroll
    for (int h2 = 0; h2 < 2; h2++) {
        const int cg = 2 * c.wh + h2;
        float da[16], db[16];
        if (cg < Ia) tmem_ld16(c.tl + TM_D1 + seg_base(Ia) + 16 * cg, da);
        if (cg < Ib) tmem_ld16(c.tl + TM_D1 + seg_base(Ib) + 16 * cg, db);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const int s = 16 * cg + e;
            float val = 0.f;
            if ((s >> 4) < I) val = (I == Ia) ? da[e] : db[e];
            else if ((s >> 4) == I && (isK ? s < t : s <= t)) val = NEAR[((isK * 4 + I) * 16 + (t & 15)) * 17 + (s & 15)];
            v[16 * h2 + e] = val;
        }
    }
}

// (6) the exact inverses of the diagonal 16-blocks of I + M (threads 0..63) and, per 32-block, its coupling
// block E = -B^-1 C A^-1 (warp w < 2 for 32-block w).  Reads M32, C32; writes DI32, E32.
__device__ __forceinline__ void solve_blocks(Ctx& c, unsigned char* MS)
{
    if (c.r >= 64) return;
    const int J = c.r >> 4, col = c.r & 15;
    const float* M32 = fptr(MS, MS_M32) + J * 16 * kBS;
    float xs[16];
#pragma unroll
    for (int q = 0; q < 16; q++) xs[q] = (q == col) ? 1.f : 0.f;
#pragma unroll
    for (int pp = 0; pp < 15; pp++) {
        if (pp >= col) {
            const float xp = xs[pp];
#pragma unroll
            for (int q = pp + 1; q < 16; q++) xs[q] = fmaf(-M32[q * kBS + pp], xp, xs[q]);
        }
    }
    float* DI32 = fptr(MS, MS_DI32) + J * 16 * kBS;
#pragma unroll
    for (int q = 0; q < 16; q++) DI32[q * kBS + col] = xs[q];
    __syncwarp();
    const int hf = c.lane >> 4, q0 = 8 * hf;
    const float* Ai = fptr(MS, MS_DI32) + (2 * c.warp) * 16 * kBS;
    const float* Bi = Ai + 16 * kBS;
    const float* Cb = fptr(MS, MS_C32) + c.warp * 16 * kBS;
    float acol[16];
#pragma unroll
    for (int m = 0; m < 16; m++) acol[m] = Ai[m * kBS + col];
    float f[8];
#pragma unroll
    for (int kq = 0; kq < 8; kq++) {
        float x = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 cr = *reinterpret_cast<const float4*>(Cb + (q0 + kq) * kBS + m);
            x = fmaf(cr.x, acol[m], x);
            x = fmaf(cr.y, acol[m + 1], x);
            x = fmaf(cr.z, acol[m + 2], x);
            x = fmaf(cr.w, acol[m + 3], x);
        }
        f[kq] = x;
    }
    float fc[16];
#pragma unroll
    for (int kq = 0; kq < 8; kq++) {
        const float o = __shfl_xor_sync(0xffffffffu, f[kq], 16);
        fc[kq] = hf ? o : f[kq];
        fc[8 + kq] = hf ? f[kq] : o;
    }
    float* Eb = fptr(MS, MS_E32) + c.warp * 16 * kBS;
#pragma unroll
    for (int kq = 0; kq < 8; kq++) {
        float x = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 br = *reinterpret_cast<const float4*>(Bi + (q0 + kq) * kBS + m);
            x = fmaf(br.x, fc[m], x);
            x = fmaf(br.y, fc[m + 1], x);
            x = fmaf(br.z, fc[m + 2], x);
            x = fmaf(br.w, fc[m + 3], x);
        }
        Eb[(q0 + kq) * kBS + col] = -x;
    }
}

// (6b) the tile [Dinv ; Dinv] (K-major, 128 rows; read MN-major it is [Dinv^T | Dinv^T])
__device__ __forceinline__ void write_dinv(Ctx& c, unsigned char* MS, unsigned char* DINV)
{
    const int t = c.trow & 63, J = t >> 4;
    const float* DI32 = fptr(MS, MS_DI32) + (J * 16 + (t & 15)) * kBS;
    const float* E32 = fptr(MS, MS_E32) + ((J >> 1) * 16 + (t & 15)) * kBS;
#pragma unroll 1
    for (int h2 = 0; h2 < 2; h2++) {
        const int cg = 2 * c.wh + h2;
        const float* src = (cg == J) ? DI32 : ((J & 1) && cg == J - 1) ? E32 : nullptr;
        float v16[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 x = src ? *reinterpret_cast<const float4*>(src + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            v16[e] = x.x; v16[e + 1] = x.y; v16[e + 2] = x.z; v16[e + 3] = x.w;
        }
        st16_bf16(DINV, c.trow, cg, v16);
    }
}

// The delta front after the level product: assemble P (into the hi/lo tile Pt) and M = diag(beta) K
// (L part into LR block 0, diagonal and coupling 16-blocks into MS, optionally K, fp32 column-group major, into
// KP), invert the 32-blocks, write [Dinv ; Dinv], run [N | X0] = Dinv [L | R] and
// [Util | W] = X0 - N X0 (both copies in TMEM lanes 0..63 and 64..127).  R was written by the operand step.
// Returns false on an abort.
template <bool DELTA>
__device__ bool front_solve(Ctx& c, const CbParams& p, unsigned char* NEARb, unsigned char* Pt, unsigned char* LR,
                            unsigned char* LRL, unsigned char* MS, unsigned char* DINV, unsigned char* NA,
                            unsigned char* X0, float* KP, int kid = 1)
{
    Small& S = *c.S;
    const int t = c.trow & 63, isK = c.trow >> 6, I = t >> 4;
    {
        float v[32];
        assemble_row(c, reinterpret_cast<const float*>(NEARb), v);
        if (!isK) {
#pragma unroll
            for (int h2 = 0; h2 < 2; h2++) {
                float w16[16];
#pragma unroll
                for (int e = 0; e < 16; e++) w16[e] = v[16 * h2 + e];
                st16_split(Pt, Pt + 8192, t, 2 * c.wh + h2, w16);
            }
        } else if (DELTA) {
            const float bet = S.beta[t];
#pragma unroll
            for (int h2 = 0; h2 < 2; h2++) {
                const int cg = 2 * c.wh + h2;
                float m16[16], l16[16];
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    m16[e] = bet * v[16 * h2 + e];
                    l16[e] = (I >= 2 && cg < 2) ? m16[e] : 0.f;
                }
                st16_bf16(LR, t, cg, l16);
                float* f32 = nullptr;
                if (cg == I) f32 = fptr(MS, MS_M32) + (I * 16 + (t & 15)) * kBS;
                else if ((I & 1) && cg == I - 1) f32 = fptr(MS, MS_C32) + ((I >> 1) * 16 + (t & 15)) * kBS;
                if (f32) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4*>(f32 + e) = make_float4(m16[e], m16[e + 1], m16[e + 2], m16[e + 3]);
                }
                if (KP) {
                    // K's row (zero on and above the diagonal), column-group major
                    float4* kr = reinterpret_cast<float4*>(KP) + (4 * cg) * 64 + t;
#pragma unroll
                    for (int e = 0; e < 4; e++)
                        kr[64 * e] = make_float4(v[16 * h2 + 4 * e], v[16 * h2 + 4 * e + 1], v[16 * h2 + 4 * e + 2],
                                                 v[16 * h2 + 4 * e + 3]);
                }
            }
        }
    }
    if (!DELTA) return true;
    bar_all();
    CB_STAMP(kid, 20);
    solve_blocks(c, MS);
    bar_all();
    CB_STAMP(kid, 21);
    write_dinv(c, MS, DINV);
    smem_to_tc();
    CB_STAMP(kid, 22);
    if (c.r == 0) {
        const uint32_t dinv = smem_u32(DINV);
        mma_tiles(c.tbase + TM_NX, dinv, false, 0, 0, smem_u32(LR), true, 8192, 0, 4,
                  idesc_bf16(128, 192, false, true), false);
        mma_tiles(c.tbase + TM_NX + 64, dinv, false, 0, 0, smem_u32(LRL), true, 8192, 0, 4,
                  idesc_bf16(128, 128, false, true), true);
        mma_commit(&S.mma);
    }
    if (!mma_wait(c, p, 1)) return false;
    CB_STAMP(kid, 23);
    // -N -> [-N ; -N] (K-major A); X0 -> hi/lo MN-major B blocks.  Twelve 16-column groups of token t:
    // groups 0..5 from lanes 0..63, 6..11 from their copy in lanes 64..127.
    {
        const int gb = (isK ? 6 : 0) + 3 * c.wh;
#pragma unroll 1
        for (int gg = 0; gg < 3; gg++) {
            const int g = gb + gg;
            float v[16];
            tmem_ld16(c.tl + TM_NX + 16 * g, v);
            tmem_wait_ld();
            if (g < 4) {
#pragma unroll
                for (int e = 0; e < 16; e++) v[e] = -v[e];
                st16_bf16(NA, t, g, v);
                st16_bf16(NA, 64 + t, g, v);
            } else {
                const int xg = g - 4;
                const uint32_t blk = (uint32_t)(xg >> 2) * 8192u;
                st16_split(X0 + blk, X0 + 16384 + blk, t, xg & 3, v);
            }
        }
    }
    smem_to_tc();
    CB_STAMP(kid, 24);
    if (c.r == 0) {
        const uint32_t id = idesc_bf16(128, 128, false, true);
        mma_tiles(c.tbase + TM_UT, smem_u32(NA), false, 0, 0, smem_u32(X0), true, 8192, 0, 4, id, true);
        mma_tiles(c.tbase + TM_UT, smem_u32(NA), false, 0, 0, smem_u32(X0 + 16384), true, 8192, 0, 4, id, true);
        mma_commit(&S.mma);
    }
    return mma_wait(c, p, 2);
}

// the operand step's R = [beta V | beta Btil] rows (thread t = r & 63, channels / columns 16 cq ..): hi in LR
// blocks 1, 2, lo in LRL blocks 0, 1
__device__ __forceinline__ void write_R(Ctx& c, unsigned char* LR, unsigned char* LRL)
{
    Small& S = *c.S;
    const int t = c.r & 63, cq = c.r >> 6;
    const float bet = S.beta[t], Gt = S.G[t];
    float vv[16], bv[16], y[16];
    ld16_bf16(c.sm + OFF_STAGE + ST_V, t, cq, vv);
    ld16_bf16(c.sm + OFF_STAGE + ST_B, t, cq, bv);
#pragma unroll
    for (int e = 0; e < 16; e++) y[e] = bet * vv[e];
    st16_split(LR + 8192, LRL, t, cq, y);
#pragma unroll
    for (int e = 0; e < 16; e++) y[e] = bet * bv[e] * fast_exp2(S.A2[16 * cq + e] * Gt);
    st16_split(LR + 16384, LRL + 8192, t, cq, y);
}

// per-chunk inputs: g, beta (threads 0..127) and A2 of the chunk's head (threads 128..191)
__device__ __forceinline__ void load_small(Ctx& c, const CbParams& p, int bb, int h, int t0)
{
    Small& S = *c.S;
    const int r = c.r;
    if (r < 64) {
        const int t = t0 + r;
        S.g[r] = t < p.T ? __bfloat162float(p.g[((size_t)bb * p.T + t) * p.H + h]) : 0.f;
    } else if (r < 128) {
        const int tt = r - 64, t = t0 + tt;
        S.beta[tt] = (p.beta && t < p.T) ? __bfloat162float(p.beta[((size_t)bb * p.T + t) * p.H + h]) : 0.f;
    } else if (r < 192) {
        const int i = r - 128;
        S.A2[i] = i < p.dk ? -expf(p.A_log[h * p.dk + i]) * kLog2e : 0.f;
    }
}

__device__ __forceinline__ void issue_tma(const CbParams& p, Small& S, unsigned char* sm, int q)
{
    if (q == p.starve) return;   // failure-path test hook: this chunk's loads never arrive
    const int u = q / p.nchunks, k = q - u * p.nchunks, bb = u / p.H, h = u - bb * p.H;
    unsigned char* st = sm + OFF_STAGE;
    mbar_arrive_expect_tx(&S.full, 4 * 8192);
    tma_load_4d(st + ST_B, &p.tm_b, &S.full, 0, h, 64 * k, bb);
    tma_load_4d(st + ST_C, &p.tm_c, &S.full, 0, h, 64 * k, bb);
    tma_load_4d(st + ST_V, &p.tm_v, &S.full, 0, h, 64 * k, bb);
    tma_load_4d(st + ST_DO, &p.tm_do, &S.full, 0, h, 64 * k, bb);
}

// the saved front of chunk q into the gradient pass's phase region (the stacked operands' halves twice; gated: P)
template <bool DELTA>
__device__ __forceinline__ void issue_saved(const CbParams& p, Small& S, unsigned char* sm, int q)
{
    if (q == p.starve) return;
    unsigned char* X = sm + OFF_X;
    const unsigned char* src = p.sv + (size_t)q * p.sv_stride;
    if (!DELTA) {
        mbar_arrive_expect_tx(&S.full2, 16384);
        bulk_g2s(X + gl::P, src + sv::P, 16384, &S.full2);
        return;
    }
    // -W only where U is still to be formed (a saving forward's record holds U itself)
    mbar_arrive_expect_tx(&S.full2, 16384 + 4 * 8192 + (p.rev_only ? 0 : 8192));
    bulk_g2s(X + gl::P, src + sv::P, 16384, &S.full2);
    bulk_g2s(X + gl::NA, src + sv::NA, 8192, &S.full2);
    bulk_g2s(X + gl::NA + 8192, src + sv::NA, 8192, &S.full2);
    bulk_g2s(X + gl::DINV, src + sv::DINV, 8192, &S.full2);
    bulk_g2s(X + gl::DINV + 8192, src + sv::DINV, 8192, &S.full2);
    if (!p.rev_only) bulk_g2s(X + gl::NW, src + sv::NW, 8192, &S.full2);
}

__device__ __forceinline__ void prefetch_tma(const CbParams& p, int q)
{
    const int u = q / p.nchunks, k = q - u * p.nchunks, bb = u / p.H, h = u - bb * p.H;
    tma_prefetch_l2(&p.tm_b, 0, h, 64 * k, bb);
    tma_prefetch_l2(&p.tm_c, 0, h, 64 * k, bb);
    tma_prefetch_l2(&p.tm_v, 0, h, 64 * k, bb);
    tma_prefetch_l2(&p.tm_do, 0, h, 64 * k, bb);
}

// kernel set-up shared by prep and grad; returns the context
__device__ __forceinline__ Ctx setup(unsigned char* smem_raw, const CbParams& p)
{
    Ctx c;
    c.sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    c.X = c.sm + OFF_X;
    c.S = reinterpret_cast<Small*>(c.sm + OFF_SMALL);
    c.KT = reinterpret_cast<Tab*>(c.sm + OFF_TAB);
    c.ALPHA = reinterpret_cast<float*>(c.sm + OFF_ALPHA);
    c.YB = reinterpret_cast<float*>(c.sm + OFF_YB);
    c.r = threadIdx.x;
    c.warp = c.r >> 5;
    c.lane = c.r & 31;
    c.q4 = c.warp & 3;
    c.wh = c.warp >> 2;
    c.trow = c.r & 127;
    c.mma_phase = 0;
    Small& S = *c.S;
    if (c.r == 0) {
        mbar_init(&S.full, 1);
        mbar_init(&S.mma, 1);
        mbar_init(&S.full2, 1);
        S.abort = 0;
        fence_mbar_init();
    }
    if (c.warp == 0) tmem_alloc(&S.tmem_base, TM_COLS);
    if (c.r == 0) {
        tma_prefetch_desc(&p.tm_b); tma_prefetch_desc(&p.tm_c); tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tbase = S.tmem_base;
    c.tl = c.tbase + ((uint32_t)(c.q4 * 32) << 16);
    return c;
}

__device__ __forceinline__ void teardown(Ctx& c, const CbParams& p, int issued_q, uint32_t full_phase,
                                         int issued_q2 = -1, uint32_t full2_phase = 0)
{
    // after an abort, let the copies still in flight land before exiting
    if (c.r == 0 && *(volatile uint32_t*)&c.S->abort && issued_q >= 0 && issued_q != p.starve)
        mbar_wait(&c.S->full, full_phase, nullptr, p.wait_ns);
    if (c.r == 0 && *(volatile uint32_t*)&c.S->abort && issued_q2 >= 0 && issued_q2 != p.starve)
        mbar_wait(&c.S->full2, full2_phase, nullptr, p.wait_ns);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (c.warp == 0) tmem_dealloc(c.tbase, TM_COLS);
}

// ================================================================= pass 1: prep
template <bool DELTA>
__global__ void __launch_bounds__(kThreads, 1) chunk_prep_kernel(const __grid_constant__ CbParams p)
{
    extern __shared__ unsigned char smem_raw[];
    Ctx c = setup(smem_raw, p);
    Small& S = *c.S;
    unsigned char* X = c.X;
    uint32_t full_phase = 0;
    int q = blockIdx.x;
    int pending = -1;   // chunk whose loads are in flight
    if (c.r == 0 && q < p.nq) { issue_tma(p, S, c.sm, q); pending = q; }
    CB_STAMP_INIT;
    for (; q < p.nq; q += gridDim.x) {
        CB_STAMP(0, 0);
        const int u = q / p.nchunks, k = q - u * p.nchunks, bb = u / p.H, h = u - bb * p.H;
        load_small(c, p, bb, h, 64 * k);
        if (c.r == 0 && q + (int)gridDim.x < p.nq) prefetch_tma(p, q + gridDim.x);
        if (c.warp == 0 && !wait_or_abort(&S.full, full_phase, &S.abort, p.status, p.wait_ns) && c.lane == 0)
            atomicExch(p.status + 2, 1u);
        bar_all();
        if (*(volatile uint32_t*)&S.abort) break;
        full_phase ^= 1;
        pending = -1;
        CB_STAMP(0, 1);
        front_scan(c);
        bar_all();
        const int t = c.r & 63, cq = c.r >> 6;
        if constexpr (!DELTA) {
            // [Bhat | Ctil] hi, lo: natural [t][i] tiles, read MN-major as [Bhat^T ; Ctil^T]
            float bv[16], cv[16], y[16], z[16];
            ld16_bf16(c.sm + OFF_STAGE + ST_B, t, cq, bv);
            ld16_bf16(c.sm + OFF_STAGE + ST_C, t, cq, cv);
            const float Gt = S.G[t], G63 = S.G[63];
#pragma unroll
            for (int e = 0; e < 16; e++) {
                const float a2 = S.A2[16 * cq + e];
                y[e] = bv[e] * fast_exp2(a2 * (G63 - Gt));
                z[e] = cv[e] * fast_exp2(a2 * Gt);
            }
            st16_split(X + pl::GA, X + pl::GA + 16384, t, cq, y);
            st16_split(X + pl::GA + 8192, X + pl::GA + 24576, t, cq, z);
            smem_to_tc();
            if (c.r == 0) {
                // [Bhat^T V | Bhat^T dO ; Ctil^T V | Ctil^T dO]
                const uint32_t id = idesc_bf16(128, 128, true, true);
                const uint32_t vd = smem_u32(c.sm + OFF_STAGE + ST_V);
                mma_tiles(c.tbase, smem_u32(X + pl::GA), true, 8192, 0, vd, true, 8192, 0, 4, id, false);
                mma_tiles(c.tbase, smem_u32(X + pl::GA + 16384), true, 8192, 0, vd, true, 8192, 0, 4, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_wait(c, p, 3)) break;
            // Delta = rows 0..63, columns 0..63; Y = rows 64..127, columns 64..127
            {
                const int i = c.trow & 63;
                float* dst = c.trow < 64 ? p.dlt : p.ych;
                const uint32_t col0 = c.trow < 64 ? 0u : 64u;
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    float v[16];
                    tmem_ld16(c.tl + col0 + 32 * c.wh + 16 * h2, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *rec4(dst, q, i, 32 * c.wh + 16 * h2 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                }
                if (c.r < 64) p.ec[(size_t)q * 64 + c.r] = c.KT->EC[c.r];
            }
        } else {
            front_operands(c, X + pl::A1, X + pl::B1, true);
            write_R(c, X + pl::LR, X + pl::LRL);
            {
                // Bhat natural [s][i] (read MN-major as Bhat^T)
                float bv[16], y[16];
                ld16_bf16(c.sm + OFF_STAGE + ST_B, t, cq, bv);
                const float Gt = S.G[t], G63 = S.G[63];
#pragma unroll
                for (int e = 0; e < 16; e++) y[e] = bv[e] * fast_exp2(S.A2[16 * cq + e] * (G63 - Gt));
                st16_split(X + pl::BH, X + pl::BH + 8192, t, cq, y);
            }
            smem_to_tc();
            if (c.r == 0) {
                issue_level(c.tbase, X + pl::A1, X + pl::B1);
                mma_commit(&S.mma);
            }
            front_near(c, fptr(X, pl::NEAR), true);
            bar_all();
            if (!mma_wait(c, p, 4)) break;
            unsigned char* svq = p.sv + (size_t)q * p.sv_stride;
            if (!front_solve<true>(c, p, X + pl::NEAR, X + pl::P, X + pl::LR, X + pl::LRL, X + pl::MS, X + pl::DINV,
                                   X + pl::NA, X + pl::X0, reinterpret_cast<float*>(svq + sv::K), 0))
                break;
            CB_STAMP(0, 4);
            // saved for the gradient pass: the P tiles and one half each of [-N ; -N] and [Dinv ; Dinv]
            {
                const uint4* sp = reinterpret_cast<const uint4*>(X + pl::P);
                const uint4* sn = reinterpret_cast<const uint4*>(X + pl::NA);
                const uint4* sd = reinterpret_cast<const uint4*>(X + pl::DINV);
                uint4* dp = reinterpret_cast<uint4*>(svq + sv::P);
                uint4* dn = reinterpret_cast<uint4*>(svq + sv::NA);
                uint4* dd = reinterpret_cast<uint4*>(svq + sv::DINV);
#pragma unroll
                for (int m = 0; m < 4; m++) dp[c.r + 256 * m] = sp[c.r + 256 * m];
#pragma unroll
                for (int m = 0; m < 2; m++) {
                    dn[c.r + 256 * m] = sn[c.r + 256 * m];
                    dd[c.r + 256 * m] = sd[c.r + 256 * m];
                }
            }
            // [Util | W] -> [W | Util] hi/lo MN-major B blocks (W block 0, Util block 1); saved: -W (bf16 tile)
            // and Util (fp32)
            {
                const bool isW = c.trow < 64;
                const int tt = c.trow & 63;
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int cg = 2 * c.wh + h2;
                    float v[16];
                    tmem_ld16(c.tl + (isW ? TM_W : TM_UT) + 16 * cg, v);
                    tmem_wait_ld();
                    const uint32_t blk = isW ? 0u : 8192u;
                    st16_split(X + pl::WU + blk, X + pl::WU + 16384 + blk, tt, cg, v);
                    if (isW) {
                        float nw[16];
#pragma unroll
                        for (int e = 0; e < 16; e++) nw[e] = -v[e];
                        st16_bf16(svq + sv::NW, tt, cg, nw);
                    } else {
                        float4* du = reinterpret_cast<float4*>(svq + sv::UT) + (4 * cg) * 64 + tt;
#pragma unroll
                        for (int e = 0; e < 4; e++)
                            du[64 * e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    }
                }
            }
            smem_to_tc();
            if (c.r == 0) {
                // [Phi' | Delta] = Bhat^T [W | Util] (TMEM 288..415), P W (416..479)
                const uint32_t idA = idesc_bf16(128, 128, true, true);
                const uint32_t bh = smem_u32(X + pl::BH), wu = smem_u32(X + pl::WU);
                mma_tiles(c.tbase + 288, bh, true, 8192, 0, wu, true, 8192, 0, 4, idA, false);
                mma_tiles(c.tbase + 288, bh, true, 8192, 0, wu + 16384, true, 8192, 0, 4, idA, true);
                mma_tiles(c.tbase + 288, bh + 8192, true, 8192, 0, wu, true, 8192, 0, 4, idA, true);
                const uint32_t idB = idesc_bf16(128, 64, false, true);
                const uint32_t pp = smem_u32(X + pl::P);
                mma_tiles(c.tbase + 416, pp, false, 0, 0, wu, true, 8192, 0, 4, idB, false);
                mma_tiles(c.tbase + 416, pp, false, 0, 0, wu + 16384, true, 8192, 0, 4, idB, true);
                mma_tiles(c.tbase + 416, pp + 8192, false, 0, 0, wu, true, 8192, 0, 4, idB, true);
                mma_commit(&S.mma);
            }
            if (!mma_wait(c, p, 5)) break;
            CB_STAMP(0, 5);
            // lanes 0..63: Phi = diag(E) - Bhat^T W and Delta out; lanes 64..127: Qc = Ctil - P W (hi/lo, natural)
            if (c.trow < 64) {
                const int i = c.trow;
                unsigned char* phq = p.phi + (size_t)q * 16384;

                const float eci = c.KT->EC[i];
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int c0 = 32 * c.wh + 16 * h2;
                    float a[16], b[16];
                    tmem_ld16(c.tl + 288 + c0, a);
                    tmem_ld16(c.tl + 352 + c0, b);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; e++) a[e] = (c0 + e == i ? eci : 0.f) - a[e];
                    st16_split(phq, phq + 8192, i, c0 >> 4, a);
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *rec4(p.dlt, q, i, c0 + e) = make_float4(b[e], b[e + 1], b[e + 2], b[e + 3]);
                }
            } else {
                // the P W rows sit in lanes 0..63; the lanes 64..127 threads read them through the copy below
            }
            bar_all();
            // Qc rows: token t in lanes 0..63 of the P W accumulator; threads of lanes 0..63 write them
            if (c.trow < 64) {
                const int tt = c.trow;
                float cv[16];
                const float Gt = S.G[tt];
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int cg = 2 * c.wh + h2;
                    float pw[16];
                    tmem_ld16(c.tl + 416 + 16 * cg, pw);
                    tmem_wait_ld();
                    ld16_bf16(c.sm + OFF_STAGE + ST_C, tt, cg, cv);
                    float y[16];
#pragma unroll
                    for (int e = 0; e < 16; e++) y[e] = cv[e] * fast_exp2(S.A2[16 * cg + e] * Gt) - pw[e];
                    st16_split(X + pl::QC, X + pl::QC + 8192, tt, cg, y);
                }
            }
            smem_to_tc();
            if (c.r == 0) {
                // Y = Qc^T dO (TMEM 96..159)
                const uint32_t id = idesc_bf16(128, 64, true, true);
                const uint32_t qc = smem_u32(X + pl::QC), dO = smem_u32(c.sm + OFF_STAGE + ST_DO);
                mma_tiles(c.tbase + 96, qc, true, 8192, 0, dO, true, 8192, 0, 4, id, false);
                mma_tiles(c.tbase + 96, qc + 8192, true, 8192, 0, dO, true, 8192, 0, 4, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_wait(c, p, 6)) break;
            CB_STAMP(0, 6);
            if (c.trow < 64) {
                const int i = c.trow;
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int c0 = 32 * c.wh + 16 * h2;
                    float v[16];
                    tmem_ld16(c.tl + 96 + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *rec4(p.ych, q, i, c0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                }
            }
        }
        CB_STAMP(0, 7);
#ifdef GDN_CHUNK_DEBUG
        if (c.r == 0 && blockIdx.x == 0) g_cb_stamps[0][31] += 1;
#endif
        // the stage is free: the next chunk's loads
        tc_fence_before();
        bar_all();
        tc_fence_after();
        if (q + (int)gridDim.x < p.nq) {
            if (c.r == 0) issue_tma(p, S, c.sm, q + gridDim.x);
            pending = q + gridDim.x;
        }
    }
    teardown(c, p, pending, full_phase);
}

// ================================================================= pass 1 from a saving forward's residuals (delta)
// With P and W of every chunk kept by the forward, the chain's inputs take three products per chunk:
//   Phi - diag(E) = Bhat^T (-W),   Qc - Ctil = P (-W),   Y = Qc^T dO,
// on hi/lo operands (hi*hi + hi*lo + lo*hi; dO exact).  Bhat and Ctil come from b, c and the chunk's decay (every
// factor <= 1).  74 KB of shared memory and 128 TMEM columns, so three CTAs share an SM.  The products have M = 128;
// the rows past 64 of an A operand read the next 8 KB (the lo tile, or the region after it), which hold other data
// and give TMEM rows that nobody reads.  Qc takes P's place once the first products are done, and Y takes their
// TMEM columns once Phi and Qc have been read out.
namespace ps {
constexpr uint32_t STB = 0, STC = 8192, STDO = 16384;   // b, c, dO tiles (TMA)
constexpr uint32_t BH = 24576;                           // Bhat hi, lo, natural [t][i]
constexpr uint32_t P = 40960;                            // P hi, lo (residuals)
constexpr uint32_t NW = 57344;                           // -W hi, lo (residuals)
constexpr uint32_t QC = P;                               // Qc hi, lo, natural [t][i] (after the first products)
constexpr uint32_t SMALL = 73728;
constexpr uint32_t SMEM = SMALL + 1024 + 1024;
constexpr uint32_t TM_COLS = 128;
static_assert(BH + 24576 <= SMALL && QC + 24576 <= SMALL && P + 24576 <= SMALL, "M = 128 reads stay inside");
}  // namespace ps

struct PsSmall {
    float G[64];
    float A2[64];
    float g[64];
    uint64_t full, mma;
    uint32_t tmem_base, abort;
};
static_assert(sizeof(PsSmall) <= 1024, "small block");

__global__ void __launch_bounds__(256, 3) chunk_prep_saved_kernel(const __grid_constant__ CbParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    PsSmall& S = *reinterpret_cast<PsSmall*>(sm + ps::SMALL);
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31, q4 = warp & 3, wh = warp >> 2, trow = r & 127;
    if (r == 0) {
        mbar_init(&S.full, 1);
        mbar_init(&S.mma, 1);
        S.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&p.tm_b); tma_prefetch_desc(&p.tm_c); tma_prefetch_desc(&p.tm_do);
    }
    if (warp == 0) tmem_alloc(&S.tmem_base, ps::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem_base, tl = tb + ((uint32_t)(q4 * 32) << 16);
    uint32_t full_phase = 0, mma_phase = 0;
    auto issue = [&](int q) {
        if (q == p.starve) return;   // failure-path test hook
        const int u = q / p.nchunks, k = q - u * p.nchunks, bb = u / p.H, h = u - bb * p.H;
        if (p.gated) {   // a gated chunk needs its c tile alone (and dO for Y)
            mbar_arrive_expect_tx(&S.full, p.fwd_walks ? 8192 : 16384);
            tma_load_4d(sm + ps::STC, &p.tm_c, &S.full, 0, h, 64 * k, bb);
            if (!p.fwd_walks) tma_load_4d(sm + ps::STDO, &p.tm_do, &S.full, 0, h, 64 * k, bb);
            return;
        }
        mbar_arrive_expect_tx(&S.full, (p.fwd_walks ? 2 : 3) * 8192 + 32768);
        tma_load_4d(sm + ps::STB, &p.tm_b, &S.full, 0, h, 64 * k, bb);
        tma_load_4d(sm + ps::STC, &p.tm_c, &S.full, 0, h, 64 * k, bb);
        if (!p.fwd_walks) tma_load_4d(sm + ps::STDO, &p.tm_do, &S.full, 0, h, 64 * k, bb);
        const unsigned char* rq = p.sv + (size_t)q * p.sv_stride;
        bulk_g2s(sm + ps::P, rq + sv::P, 16384, &S.full);
        bulk_g2s(sm + ps::NW, rq + sv::NW, 16384, &S.full);   // -W hi, then lo
    };
    auto sync_all = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 256);
        tc_fence_after();
    };
    auto wait_mma = [&](uint32_t where) -> bool {
        if (warp == 0 && !wait_or_abort(&S.mma, mma_phase, &S.abort, p.status, p.wait_ns) && lane == 0)
            atomicExch(p.status + 2, 400u + where);
        named_bar_sync(1, 256);
        mma_phase ^= 1;
        tc_fence_after();
        return *(volatile uint32_t*)&S.abort == 0;
    };
    int q = blockIdx.x, pending = -1;
    if (r == 0 && q < p.nq) issue(q);
    if (q < p.nq) pending = q;
    for (; q < p.nq; q += gridDim.x) {
        const int u = q / p.nchunks, k = q - u * p.nchunks, bb = u / p.H, h = u - bb * p.H, t0 = 64 * k;
        if (r < 64) {
            const int t = t0 + r;
            S.g[r] = t < p.T ? __bfloat162float(p.g[((size_t)bb * p.T + t) * p.H + h]) : 0.f;
        } else if (r < 128) {
            const int i = r - 64;
            S.A2[i] = i < p.dk ? -expf(p.A_log[h * p.dk + i]) * kLog2e : 0.f;
        } else if (r == 128 && q + (int)gridDim.x < p.nq) {
            // the next chunk's tiles and residuals towards L2 (its loads go out when this chunk is done)
            const int qn = q + gridDim.x, un = qn / p.nchunks, kn = qn - un * p.nchunks, bn = un / p.H,
                      hn = un - bn * p.H;
            tma_prefetch_l2(&p.tm_c, 0, hn, 64 * kn, bn);
            if (!p.fwd_walks) tma_prefetch_l2(&p.tm_do, 0, hn, 64 * kn, bn);
            if (!p.gated) {
                tma_prefetch_l2(&p.tm_b, 0, hn, 64 * kn, bn);
                const unsigned char* rq = p.sv + (size_t)qn * p.sv_stride;
                prefetch_l2_bulk(rq + sv::P, 16384);
                prefetch_l2_bulk(rq + sv::NW, 16384);
            }
        }
        if (warp == 0 && !wait_or_abort(&S.full, full_phase, &S.abort, p.status, p.wait_ns) && lane == 0)
            atomicExch(p.status + 2, 5u);
        named_bar_sync(1, 256);
        if (*(volatile uint32_t*)&S.abort) break;
        full_phase ^= 1;
        pending = -1;
        if (warp == 0) {
            // inclusive scan of g, two tokens per lane
            const float ga = S.g[2 * lane], gb = S.g[2 * lane + 1];
            float x = ga + gb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            S.G[2 * lane] = x - gb;
            S.G[2 * lane + 1] = x;
        }
        named_bar_sync(1, 256);
        if (!p.gated) {
            // Bhat = b (.) exp(A (G_63 - G_t)), thread = (token t, 16 channels)
            const int t = r & 63, cq = r >> 6;
            float bv[16], y[16];
            ld16_bf16(sm + ps::STB, t, cq, bv);
            const float Gt = S.G[t], G63 = S.G[63];
#pragma unroll
            for (int e = 0; e < 16; e++) y[e] = bv[e] * fast_exp2(S.A2[16 * cq + e] * (G63 - Gt));
            st16_split(sm + ps::BH, sm + ps::BH + 8192, t, cq, y);
        }
        sync_all();
        if (r == 0 && !p.gated) {
            const uint32_t bh = smem_u32(sm + ps::BH), pp = smem_u32(sm + ps::P), nw = smem_u32(sm + ps::NW);
            const uint32_t idA = idesc_bf16(128, 64, true, true), idB = idesc_bf16(128, 64, false, true);
            // Bhat^T (-W): TMEM columns 0..63, rows i
            mma_tiles(tb, bh, true, 8192, 0, nw, true, 8192, 0, 4, idA, false);
            mma_tiles(tb, bh, true, 8192, 0, nw + 8192, true, 8192, 0, 4, idA, true);
            mma_tiles(tb, bh + 8192, true, 8192, 0, nw, true, 8192, 0, 4, idA, true);
            // P (-W): columns 64..127, rows t
            mma_tiles(tb + 64, pp, false, 0, 0, nw, true, 8192, 0, 4, idB, false);
            mma_tiles(tb + 64, pp, false, 0, 0, nw + 8192, true, 8192, 0, 4, idB, true);
            mma_tiles(tb + 64, pp + 8192, false, 0, 0, nw, true, 8192, 0, 4, idB, true);
            mma_commit(&S.mma);
        }
        if (!p.gated && !wait_mma(0)) break;
        if (q4 < 2) {
            // lanes 0..63: Phi row i out (hi/lo tiles), Qc row t = i = Ctil + P (-W) into its tiles (gated: W = 0)
            const int i = trow;
            // the forward's walks take [Phi_hi | Qc_hi | Phi_lo | Qc_lo] (32 KB a chunk): the stacked A operand
            // [Phi ; Qc] gives the next state and the outputs' share in one product
            const uint32_t rb = p.fwd_walks ? 32768u : 16384u, lo = p.fwd_walks ? 16384u : 8192u;
            unsigned char* phq = p.phi + (size_t)q * rb;
            const float ec = fast_exp2(S.A2[i] * S.G[63]), Gt = S.G[i];
#pragma unroll 1
            for (int h2 = 0; h2 < 2; h2++) {
                const int cg = 2 * wh + h2;
                float a[16], b[16], cv[16];
                if (p.gated) {
#pragma unroll
                    for (int e = 0; e < 16; e++) a[e] = b[e] = 0.f;
                } else {
                    tmem_ld16(tl + 16 * cg, a);
                    tmem_ld16(tl + 64 + 16 * cg, b);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int e = 0; e < 16; e++) a[e] += (16 * cg + e == i) ? ec : 0.f;
                if (p.fwd_walks || !p.gated) st16_split(phq, phq + lo, i, cg, a);   // (the gated chain takes E)
                else if (h2 == 0 && wh == 0) p.ec[(size_t)q * 64 + i] = ec;
                ld16_bf16(sm + ps::STC, i, cg, cv);
#pragma unroll
                for (int e = 0; e < 16; e++) b[e] += cv[e] * fast_exp2(S.A2[16 * cg + e] * Gt);
                if (p.fwd_walks) st16_split(phq + 8192, phq + 8192 + lo, i, cg, b);
                else st16_split(sm + ps::QC, sm + ps::QC + 8192, i, cg, b);
            }
        }
        if (!p.fwd_walks) {   // Y = Qc^T dO
            sync_all();
            if (r == 0) {
                // Y = Qc^T dO: columns 0..63 (Phi's, read out), rows i
                const uint32_t qc = smem_u32(sm + ps::QC), dO = smem_u32(sm + ps::STDO);
                const uint32_t id = idesc_bf16(128, 64, true, true);
                mma_tiles(tb, qc, true, 8192, 0, dO, true, 8192, 0, 4, id, false);
                mma_tiles(tb, qc + 8192, true, 8192, 0, dO, true, 8192, 0, 4, id, true);
                mma_commit(&S.mma);
            }
            if (!wait_mma(1)) break;
            if (q4 < 2) {
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int c0 = 32 * wh + 16 * h2;
                    float v[16];
                    tmem_ld16(tl + c0, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *rec4(p.ych, q, trow, c0 + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                }
            }
        }
        // the tiles are free: the next chunk's loads
        tc_fence_before();
        named_bar_sync(1, 256);
        tc_fence_after();
        if (q + (int)gridDim.x < p.nq) {
            if (r == 0) issue(q + gridDim.x);
            pending = q + gridDim.x;
        }
    }
    // after an abort, let the loads in flight land before the CTA leaves
    if (r == 0 && *(volatile uint32_t*)&S.abort && pending >= 0 && pending != p.starve)
        mbar_wait(&S.full, full_phase, nullptr, p.wait_ns);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, ps::TM_COLS);
}

// ================================================================= pass 2: chain
// Gated mode: Phi = diag(E) and the chain is elementwise.  One CTA per (batch, head) unit, 256 threads, thread =
// rows 2 ip, 2 ip + 1 (ip = r >> 3) x value columns 8 (r & 7) .. + 7.  Forward: S_0 = h0, st[k] = S_k,
// S_{k+1} = E_k (.) S_k + Delta_k.  Reverse: dS = dhT, dst[k] = dS, dS <- E_k (.) dS + Y_k; dh0 = dS.
__global__ void __launch_bounds__(256) chunk_chain_gated_kernel(const __grid_constant__ CbParams p)
{
    const int u = blockIdx.x, r = threadIdx.x, i0 = 2 * (r >> 3), j0 = 8 * (r & 7);
    const int dk = p.dk, dv = p.dv_, nk = p.nchunks;
    const size_t qb = (size_t)u * nk;
    auto rec = [&](const float* base, int k, float4 (&v)[4]) {
        v[0] = *rec4(base, qb + k, i0, j0);
        v[1] = *rec4(base, qb + k, i0, j0 + 4);
        v[2] = *rec4(base, qb + k, i0 + 1, j0);
        v[3] = *rec4(base, qb + k, i0 + 1, j0 + 4);
    };
    auto put = [&](float* base, int k, const float2 (&x)[8]) {
        *rec4(base, qb + k, i0, j0) = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
        *rec4(base, qb + k, i0, j0 + 4) = make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
        *rec4(base, qb + k, i0 + 1, j0) = make_float4(x[4].x, x[4].y, x[5].x, x[5].y);
        *rec4(base, qb + k, i0 + 1, j0 + 4) = make_float4(x[6].x, x[6].y, x[7].x, x[7].y);
    };
    auto load_in = [&](const float* src, float2 (&s)[8]) {
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = i0 + (e >> 2), j = j0 + 2 * (e & 3);
            const bool in = src && i < dk;
            s[e] = make_float2(in && j < dv ? src[((size_t)u * dk + i) * dv + j] : 0.f,
                               in && j + 1 < dv ? src[((size_t)u * dk + i) * dv + j + 1] : 0.f);
        }
    };
    // s <- E (.) s + d, E = (e0, e1) of the chunk's rows i0, i0 + 1
    auto advance = [&](float e0, float e1, const float4 (&d)[4], float2 (&s)[8]) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float ec = e < 2 ? e0 : e1;
            const float4 dd = d[e];
            s[2 * e] = __ffma2_rn(make_float2(ec, ec), s[2 * e], make_float2(dd.x, dd.y));
            s[2 * e + 1] = __ffma2_rn(make_float2(ec, ec), s[2 * e + 1], make_float2(dd.z, dd.w));
        }
    };
    auto ec_of = [&](int k, float& e0, float& e1) {
        e0 = p.ec[(qb + k) * 64 + i0];
        e1 = p.ec[(qb + k) * 64 + i0 + 1];
    };
    float2 s[8];
    float4 d[4], dn[4];
    float e0, e1, en0 = 0.f, en1 = 0.f;   // the chunk's decays, and the next chunk's, loaded a step ahead
    if (!p.rev_only) {   // (with a saving forward's states only the reverse sweep runs)
        load_in(p.h0, s);
        rec(p.dlt, 0, d);
        ec_of(0, e0, e1);
        for (int k = 0; k < nk; k++) {
            put(p.st, k, s);
            if (k + 1 < nk) {
                rec(p.dlt, k + 1, dn);
                ec_of(k + 1, en0, en1);
            }
            advance(e0, e1, d, s);
#pragma unroll
            for (int e = 0; e < 4; e++) d[e] = dn[e];
            e0 = en0;
            e1 = en1;
        }
    }
    load_in(p.dhT, s);
    rec(p.ych, nk - 1, d);
    ec_of(nk - 1, e0, e1);
    for (int k = nk - 1; k >= 0; k--) {
        put(p.dst, k, s);
        if (k > 0) {
            rec(p.ych, k - 1, dn);
            ec_of(k - 1, en0, en1);
        }
        advance(e0, e1, d, s);
#pragma unroll
        for (int e = 0; e < 4; e++) d[e] = dn[e];
        e0 = en0;
        e1 = en1;
    }
    if (p.dh0) {
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = i0 + (e >> 2), j = j0 + 2 * (e & 3);
            if (i < dk && j < dv) p.dh0[((size_t)u * dk + i) * dv + j] = s[e].x;
            if (i < dk && j + 1 < dv) p.dh0[((size_t)u * dk + i) * dv + j + 1] = s[e].y;
        }
    }
}

// Delta mode: the chain on the tensor cores.  One CTA per (batch, head) unit.  The prep writes each chunk's Phi as
// two bf16 tiles, hi and lo (Phi ~ hi + lo to about 16 significant bits), in the 128-byte-swizzled [64][64] layout
// the MMA reads, 16 KB per chunk; one bulk copy moves them into a ring of CT_NS stages, in the order the two sweeps
// use them (chunks 0 .. nk - 1, then nk - 1 .. 0), CT_NS steps ahead.  The state (forward) or the adjoint
// (reverse), X, sits in two bf16 tiles (hi, lo; rows = state row m, read MN-major as the B operand).  A step is
//   D[:, 0:64 | 64:128] = Phi_hi [X_hi | X_lo]   (N = 128)    D[:, 0:64] += Phi_lo X_hi   (N = 64)
//   X' = D[:, 0:64] + D[:, 64:128] + R           (R = Delta_k forward, Y_k reverse, fp32 records)
// with Phi read K-major (Phi X) or MN-major (Phi^T X) from the same tiles; M = 128, rows 64 .. 127 are not used.
// Warps 0, 1, 4, 5 hold TMEM lanes 0 .. 63 (the state rows): thread = row i = 32 (warp & 1) + lane, columns
// 32 (warp >> 2) .. + 31.  Each reads its part of D, adds R (loaded a step ahead), writes the fp32 record
// (st forward, dst reverse) and rebuilds its part of the tiles; thread 0 issues the MMAs and the copies.  Warps 2
// and 3 exist only so that warps 4 and 5 map to TMEM lanes 0 .. 63; they leave after the set-up.
constexpr int CT_NS = 4;
constexpr uint32_t CT_STAGE = 16384;
constexpr uint32_t CT_X = CT_NS * CT_STAGE;       // X hi tile, then X lo tile
constexpr uint32_t CT_BAR = CT_X + 16384;          // full[CT_NS], mma, tmem base, abort
constexpr uint32_t CHAIN_TC_SMEM = CT_BAR + 128 + 1024;
constexpr int CT_THREADS = 192;

__global__ void __launch_bounds__(CT_THREADS, 1) chunk_chain_tc_kernel(const __grid_constant__ CbParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + CT_BAR);
    uint64_t* mmab = full + CT_NS;
    uint32_t* misc = reinterpret_cast<uint32_t*>(mmab + 1);   // [0] TMEM base, [1] abort
    unsigned char* Xhi = sm + CT_X;
    unsigned char* Xlo = Xhi + 8192;
    const int u = blockIdx.x, r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const int dk = p.dk, dv = p.dv_, nk = p.nchunks, nseq = 2 * nk;
    const int n0 = p.rev_only ? nk : 0;   // first sweep position (the forward sweep is skipped when states are given)
    const size_t qb = (size_t)u * nk;
    const unsigned char* phi = p.phi;
    // sweep position n -> chunk: 0 .. nk - 1 forward, then nk - 1 .. 0; the ring counts positions from n0
    auto chunk_of = [&](int n) { return n < nk ? n : nseq - 1 - n; };
    auto issue_copy = [&](int n) {
        const int s = (n - n0) % CT_NS;
        mbar_arrive_expect_tx(&full[s], CT_STAGE);
        bulk_g2s(sm + s * CT_STAGE, phi + (qb + chunk_of(n)) * CT_STAGE, CT_STAGE, &full[s]);
    };
    if (r == 0) {
        for (int s = 0; s < CT_NS; s++) mbar_init(&full[s], 1);
        mbar_init(mmab, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&misc[0], 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2 || warp == 3) return;
    const uint32_t tb = misc[0];
    int issued = n0 + (nseq - n0 < CT_NS ? nseq - n0 : CT_NS);
    if (r == 0) {
        for (int n = n0; n < issued; n++) issue_copy(n);
        for (int n = n0 + 1; n < n0 + 3 && n < nseq; n++)
            prefetch_l2_bulk((n < nk ? p.dlt : p.ych) + (qb + chunk_of(n)) * 4096, 16384);
    }
    const int i = 32 * (warp & 1) + lane, j0 = 32 * (warp >> 2);
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 1)) << 16);
    uint32_t* abortf = &misc[1];

    auto rec = [&](const float* base, int k, float (&v)[32]) {
        const float4* src = rec4(base, qb + k, i, j0);
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const float4 t = src[64 * e];
            v[4 * e] = t.x; v[4 * e + 1] = t.y; v[4 * e + 2] = t.z; v[4 * e + 3] = t.w;
        }
    };
    auto put = [&](float* base, int k, const float (&v)[32]) {
        float4* dst = rec4(base, qb + k, i, j0);
#pragma unroll
        for (int e = 0; e < 8; e++) dst[64 * e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
    };
    auto load_in = [&](const float* src, float (&v)[32]) {
#pragma unroll
        for (int e = 0; e < 32; e++) {
            const int j = j0 + e;
            v[e] = src && i < dk && j < dv ? src[((size_t)u * dk + i) * dv + j] : 0.f;
        }
    };
    auto tiles = [&](const float (&v)[32]) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float a[8];
#pragma unroll
            for (int e = 0; e < 8; e++) a[e] = v[8 * q + e];
            st_row8_split(Xhi, Xlo, i, (j0 >> 3) + q, a);
        }
    };
    // one step of either sweep: x <- P x + R with P = Phi (forward) or Phi^T (reverse); false after an abort
    auto step = [&](int n, float (&x)[32], const float (&R)[32]) -> bool {
        CB_STAMP(2, 0);
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 128);
        tc_fence_after();
        CB_STAMP(2, 1);
        const bool transpose = n >= nk;
        const int s = (n - n0) % CT_NS;
        if (r == 0) {
            if (wait_or_abort(&full[s], (uint32_t)((n - n0) / CT_NS) & 1u, abortf, p.status, p.wait_ns)) {
                tc_fence_after();
                const uint32_t a = smem_u32(sm + s * CT_STAGE), xb = smem_u32(Xhi);
                mma_tiles(tb, a, transpose, 8192, 0, xb, true, 8192, 0, 4, idesc_bf16(128, 128, transpose, true),
                          false);
                mma_tiles(tb, a + 8192, transpose, 8192, 0, xb, true, 8192, 0, 4,
                          idesc_bf16(128, 64, transpose, true), true);
                mma_commit(mmab);
            } else {
                atomicExch(p.status + 2, 300u + (uint32_t)n);
            }
        }
        CB_STAMP(2, 2);
        if (r == 0 && n + 3 < nseq) {
            // the fp32 record of step n + 3 into L2, so that its register loads (issued a step ahead) hit there
            const int m = n + 3;
            prefetch_l2_bulk((m < nk ? p.dlt : p.ych) + (qb + chunk_of(m)) * 4096, 16384);
        }
        CB_STAMP(2, 3);
        if (!wait_or_abort(mmab, (uint32_t)(n - n0) & 1u, abortf, p.status, p.wait_ns)) return false;
        tc_fence_after();
        CB_STAMP(2, 4);
        if (r == 0 && issued < nseq) issue_copy(issued++);   // the stage just read is free
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float a[16], b[16];
            tmem_ld16(tl + j0 + 16 * h, a);         // Phi_hi X_hi + Phi_lo X_hi
            tmem_ld16(tl + 64 + j0 + 16 * h, b);    // Phi_hi X_lo
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e++) x[16 * h + e] = (a[e] + b[e]) + R[16 * h + e];
        }
        CB_STAMP(2, 5);
        return true;
    };

    float x[32], R[32], Rn[32];
    bool ok = true;
    CB_STAMP_INIT;
    // ---- forward: st[k] = S_k, S_{k+1} = Phi_k S_k + Delta_k
    if (!p.rev_only) {
        load_in(p.h0, x);
        rec(p.dlt, 0, R);
        put(p.st, 0, x);
        tiles(x);
    }
    for (int k = 0; k < nk && ok && !p.rev_only; k++) {
        if (k + 1 < nk) rec(p.dlt, k + 1, Rn);
        ok = step(k, x, R);
        if (!ok) break;
        if (k + 1 < nk) {
            put(p.st, k + 1, x);
            CB_STAMP(2, 6);
            tiles(x);   // the step's MMAs have completed: the tiles are free
            CB_STAMP(2, 7);
#pragma unroll
            for (int e = 0; e < 32; e++) R[e] = Rn[e];
            CB_STAMP(2, 8);
        }
#ifdef GDN_CHUNK_DEBUG
        if (r == 0 && blockIdx.x == 0) g_cb_stamps[2][31] += 1;
#endif
    }
    // ---- reverse: dst[k] = dS_{k+1}, dS_k = Phi_k^T dS_{k+1} + Y_k, dh0 = dS_0
    if (ok) {
        load_in(p.dhT, x);
        rec(p.ych, nk - 1, R);
        put(p.dst, nk - 1, x);
        tiles(x);
        for (int k = nk - 1; k >= 0; k--) {
            if (k > 0) rec(p.ych, k - 1, Rn);
            ok = step(nseq - 1 - k, x, R);
            if (!ok) break;
            if (k > 0) {
                put(p.dst, k - 1, x);
                tiles(x);
#pragma unroll
                for (int e = 0; e < 32; e++) R[e] = Rn[e];
            }
        }
        if (ok && p.dh0) {
#pragma unroll
            for (int e = 0; e < 32; e++) {
                const int j = j0 + e;
                if (i < dk && j < dv) p.dh0[((size_t)u * dk + i) * dv + j] = x[e];
            }
        }
    }
    // wind down: after an abort, let the copies still in flight land before the CTA leaves
    if (r == 0 && *(volatile uint32_t*)abortf) {
        for (int n = issued - CT_NS < n0 ? n0 : issued - CT_NS; n < issued; n++)
            mbar_wait(&full[(n - n0) % CT_NS], (uint32_t)((n - n0) / CT_NS) & 1u, nullptr, p.wait_ns);
    }
    tc_fence_before();
    named_bar_sync(1, 128);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// ---------------------------------------------------------------- the chain as walks over segments (delta)
// With few heads over many chunks the chain above keeps few SMs busy.  Two changes spread it out.  (1) The two
// sweeps are independent (the reverse one reads Y and Phi only), so they run side by side: blockIdx.z = direction
// (0 forward, 1 reverse; with the forward's states given, the reverse one alone).  (2) The chunk map is affine
// ("GDN & MLA Mechanism Deep-Dive", Step 5: chunked recurrence), so a head's chunks are cut into nseg segments
// [k0, k1) of seg_len chunks: a first walk (TRANS) takes each segment once from zero, carrying beside the local
// state X the segment's transition Pi (from the identity),
//   forward: X <- Phi_k X + Delta_k,   Pi <- Phi_k Pi      (k = k0 .. k1 - 1)
//   reverse: X <- Phi_k^T X + Y_k,     Pi <- Phi_k^T Pi    (k = k1 - 1 .. k0)
// and leaves X and Pi in the segment records; chunk_walk_scan_kernel joins the segments (the true state entering
// segment s + 1 is Pi_s S_s + X_s, and the same for the adjoints backwards); a second walk (!TRANS) then takes each
// segment from its true start and writes the per-chunk records (st forward, dst reverse) as the chain above does,
// and in the reverse direction dh0 at the sequence's start.  The first walk skips the segment whose result nothing
// uses (the last one forward, the first one reverse).  A TRANS step is one product for both matrices:
//   D = Phi_hi [X_hi | Pi_hi | X_lo | Pi_lo] (N = 256),   D[:, 0:128] += Phi_lo [X_hi | Pi_hi]
//   X' = D[:, 0:64] + D[:, 128:192] + R,   Pi' = D[:, 64:128] + D[:, 192:256]
// and a !TRANS step is the chain's own (N = 128 then 64).  Thread roles and the copy ring are the chain's.  Two
// !TRANS walks fit an SM (83 KB of shared memory, 128 TMEM columns, at most 168 registers a thread).
__host__ __device__ constexpr uint32_t walk_tiles_bytes(bool trans) { return trans ? 32768u : 16384u; }
constexpr uint32_t walk_smem(bool trans) { return CT_NS * CT_STAGE + walk_tiles_bytes(trans) + 128 + 1024; }

// segment records of direction slot d, unit u, segment sg: [0] the final X, [1] the final Pi, [2] the true state
// entering the segment (forward) or the true adjoint leaving it (reverse); each 64 x 64 fp32, column-group major
__device__ __forceinline__ float* seg_rec(const CbParams& p, int d, int u, int sg, int which)
{
    const size_t units = (size_t)(p.nq / p.nchunks);
    return p.segrec + ((((size_t)d * units + u) * p.nseg + sg) * 3 + which) * 4096;
}

template <bool TRANS>
__global__ void __launch_bounds__(CT_THREADS, TRANS ? 1 : 2) chunk_chain_walk_kernel(const __grid_constant__ CbParams p)
{
    constexpr uint32_t XB = walk_tiles_bytes(TRANS);
    constexpr uint32_t LO = XB / 2;                    // offset of the lo tiles
    constexpr uint32_t XLO_COL = TRANS ? 128 : 64;     // TMEM column of Phi_hi X_lo
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* Xt = sm + CT_NS * CT_STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(Xt + XB);
    uint64_t* mmab = full + CT_NS;
    uint32_t* misc = reinterpret_cast<uint32_t*>(mmab + 1);   // [0] TMEM base, [1] abort
    const bool rev = p.rev_only || blockIdx.z == 1;
    const int dslot = p.rev_only ? 0 : (int)blockIdx.z;
    const int u = blockIdx.x, sg = TRANS && rev ? (int)blockIdx.y + 1 : (int)blockIdx.y;
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const int dk = p.dk, dv = p.dv_, nk = p.nchunks;
    const int k0 = sg * p.seg_len, k1 = min(k0 + p.seg_len, nk), ns = k1 - k0;
    const size_t qb = (size_t)u * nk;
    const unsigned char* phi = p.phi;
    auto chunk_of = [&](int n) { return rev ? k1 - 1 - n : k0 + n; };
    auto issue_copy = [&](int n) {
        const int s = n % CT_NS;
        mbar_arrive_expect_tx(&full[s], CT_STAGE);
        bulk_g2s(sm + s * CT_STAGE, phi + (qb + chunk_of(n)) * CT_STAGE, CT_STAGE, &full[s]);
    };
    if (r == 0) {
        for (int s = 0; s < CT_NS; s++) mbar_init(&full[s], 1);
        mbar_init(mmab, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&misc[0], TRANS ? 256 : 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2 || warp == 3) return;
    const uint32_t tb = misc[0];
    int issued = ns < CT_NS ? ns : CT_NS;
    const float* rec_in = rev ? p.ych : p.dlt;
    float* rec_out = rev ? p.dst : p.st;
    if (r == 0) {
        for (int n = 0; n < issued; n++) issue_copy(n);
        for (int n = 1; n < 3 && n < ns; n++) prefetch_l2_bulk(rec_in + (qb + chunk_of(n)) * 4096, 16384);
    }
    const int i = 32 * (warp & 1) + lane, j0 = 32 * (warp >> 2);
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 1)) << 16);
    uint32_t* abortf = &misc[1];

    auto rec = [&](const float* base, size_t q, float (&v)[32]) {
        const float4* src = rec4(base, q, i, j0);
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const float4 t = src[64 * e];
            v[4 * e] = t.x; v[4 * e + 1] = t.y; v[4 * e + 2] = t.z; v[4 * e + 3] = t.w;
        }
    };
    auto put = [&](float* base, size_t q, const float (&v)[32]) {
        float4* dst = rec4(base, q, i, j0);
#pragma unroll
        for (int e = 0; e < 8; e++) dst[64 * e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
    };
    auto tiles = [&](const float (&v)[32], uint32_t off) {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float a[8];
#pragma unroll
            for (int e = 0; e < 8; e++) a[e] = v[8 * q + e];
            st_row8_split(Xt + off, Xt + off + LO, i, (j0 >> 3) + q, a);
        }
    };
    float x[32], pi[TRANS ? 32 : 1], R[32], Rn[32];
    // one step: x <- P x + R (and pi <- P pi) with P = Phi (forward) or Phi^T (reverse); false after an abort
    auto step = [&](int n) -> bool {
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 128);
        tc_fence_after();
        const int s = n % CT_NS;
        if (r == 0) {
            if (wait_or_abort(&full[s], (uint32_t)(n / CT_NS) & 1u, abortf, p.status, p.wait_ns)) {
                tc_fence_after();
                const uint32_t a = smem_u32(sm + s * CT_STAGE), xb = smem_u32(Xt);
                mma_tiles(tb, a, rev, 8192, 0, xb, true, 8192, 0, 4, idesc_bf16(128, TRANS ? 256 : 128, rev, true),
                          false);
                mma_tiles(tb, a + 8192, rev, 8192, 0, xb, true, 8192, 0, 4,
                          idesc_bf16(128, TRANS ? 128 : 64, rev, true), true);
                mma_commit(mmab);
            } else {
                atomicExch(p.status + 2, (TRANS ? 500u : 600u) + (uint32_t)n);
            }
        }
        if (r == 0 && n + 3 < ns) prefetch_l2_bulk(rec_in + (qb + chunk_of(n + 3)) * 4096, 16384);
        if (!wait_or_abort(mmab, (uint32_t)n & 1u, abortf, p.status, p.wait_ns)) return false;
        tc_fence_after();
        if (r == 0 && issued < ns) issue_copy(issued++);   // the stage just read is free
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float a[16], b[16];
            tmem_ld16(tl + j0 + 16 * h, a);                 // Phi_hi X_hi + Phi_lo X_hi
            tmem_ld16(tl + XLO_COL + j0 + 16 * h, b);       // Phi_hi X_lo
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e++) x[16 * h + e] = (a[e] + b[e]) + R[16 * h + e];
            if constexpr (TRANS) {
                tmem_ld16(tl + 64 + j0 + 16 * h, a);        // Phi_hi Pi_hi + Phi_lo Pi_hi
                tmem_ld16(tl + 192 + j0 + 16 * h, b);       // Phi_hi Pi_lo
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e++) pi[16 * h + e] = a[e] + b[e];
            }
        }
        return true;
    };

    // the start: the sequence's own (h0 forward, dh_T reverse) at its end segment; zero elsewhere in the first
    // walk; the scan's true start elsewhere in the second
    const bool seq_start = rev ? sg == p.nseg - 1 : sg == 0;
    if (seq_start || TRANS) {
        const float* src0 = seq_start ? (rev ? p.dhT : p.h0) : nullptr;
#pragma unroll
        for (int e = 0; e < 32; e++) {
            const int j = j0 + e;
            x[e] = src0 && i < dk && j < dv ? src0[((size_t)u * dk + i) * dv + j] : 0.f;
        }
    } else {
        rec(seg_rec(p, dslot, u, sg, 2), 0, x);
    }
    if constexpr (TRANS) {
#pragma unroll
        for (int e = 0; e < 32; e++) pi[e] = i == j0 + e ? 1.f : 0.f;
    }
    rec(rec_in, qb + chunk_of(0), R);
    bool ok = true;
    for (int n = 0; n < ns; n++) {
        if constexpr (!TRANS) put(rec_out, qb + chunk_of(n), x);
        tiles(x, 0);
        if constexpr (TRANS) tiles(pi, 8192);
        if (n + 1 < ns) rec(rec_in, qb + chunk_of(n + 1), Rn);
        ok = step(n);
        if (!ok) break;
#pragma unroll
        for (int e = 0; e < 32; e++) R[e] = Rn[e];
    }
    if (ok) {
        if constexpr (TRANS) {
            put(seg_rec(p, dslot, u, sg, 0), 0, x);
            put(seg_rec(p, dslot, u, sg, 1), 0, pi);
        } else if (rev && sg == 0 && p.dh0) {
#pragma unroll
            for (int e = 0; e < 32; e++) {
                const int j = j0 + e;
                if (i < dk && j < dv) p.dh0[((size_t)u * dk + i) * dv + j] = x[e];
            }
        }
    }
    // wind down: after an abort, let the copies still in flight land before the CTA leaves
    if (r == 0 && *(volatile uint32_t*)abortf)
        for (int n = issued - CT_NS < 0 ? 0 : issued - CT_NS; n < issued; n++)
            mbar_wait(&full[n % CT_NS], (uint32_t)(n / CT_NS) & 1u, nullptr, p.wait_ns);
    tc_fence_before();
    named_bar_sync(1, 128);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, TRANS ? 256 : 128);
}

// One element (row i, column j) of a 64 x 64 column-group-major record (rec4)
__device__ __forceinline__ float& rec_at(float* base, int i, int j) { return base[(64 * (j >> 2) + i) * 4 + (j & 3)]; }
__device__ __forceinline__ float rec_at(const float* base, int i, int j)
{
    return base[(64 * (j >> 2) + i) * 4 + (j & 3)];
}

// The folds of a scan over segments, S <- Pi S + X, for one unit and the eight columns 8 blockIdx.y .. + 7 (the
// columns of a state never mix): 256 threads, thread = row i = r >> 2, columns j, j + 1 (j = 8 blockIdx.y +
// 2 (r & 3)), fp32 on the CUDA cores.  The next fold's Pi (this thread's four float4 of the shared tile) and X are
// loaded while the current one is computed.  fold(s) gives fold s's Pi and X; emit(s, c0, c1) takes the value
// entering step s (before its fold).
template <typename PiOf, typename XOf, typename Emit>
__device__ __forceinline__ void scan_columns(int nfold, int nemit, float& c0, float& c1, PiOf pi_of, XOf x_of,
                                             Emit emit)
{
    __shared__ __align__(16) float Pm[64][kAS];
    __shared__ float Cm[64][8];
    const int r = threadIdx.x, i = r >> 2, jj = 2 * (r & 3);
    float4 pn[4];
    float xn0 = 0.f, xn1 = 0.f;
    auto fetch = [&](int s) {
        const float* pim = pi_of(s);
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int f = r + 256 * e;
            pn[e] = *rec4(pim, 0, f & 63, 4 * (f >> 6));
        }
        x_of(s, xn0, xn1);
    };
    if (nfold > 0) fetch(0);
    for (int s = 0; s < nemit; s++) {
        emit(s, c0, c1);
        if (s >= nfold) break;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int f = r + 256 * e;
            *reinterpret_cast<float4*>(&Pm[f & 63][4 * (f >> 6)]) = pn[e];
        }
        Cm[i][jj] = c0;
        Cm[i][jj + 1] = c1;
        __syncthreads();
        float n0 = xn0, n1 = xn1;
        if (s + 1 < nfold) fetch(s + 1);
#pragma unroll 8
        for (int m = 0; m < 64; m++) {
            const float pv = Pm[i][m];
            n0 = fmaf(pv, Cm[m][jj], n0);
            n1 = fmaf(pv, Cm[m][jj + 1], n1);
        }
        c0 = n0;
        c1 = n1;
    }
}

// The scan over a unit's segments, one CTA of 256 threads per (unit, 8 columns, direction).  Forward: the first
// segment started from h0, so its X is the true state entering the second; then S_{s+1} = Pi_s S_s + X_s.
// Reverse: the last segment started from dh_T, so its X is the true adjoint leaving the one before; then
// E_{s-1} = Pi_s E_s + X_s.  Each value goes to record [2] of the segment it starts; the fold past the sequence's
// far end is not needed.
__global__ void __launch_bounds__(256) chunk_walk_scan_kernel(const __grid_constant__ CbParams p)
{
    const bool rev = p.rev_only || blockIdx.z == 1;
    const int dslot = p.rev_only ? 0 : (int)blockIdx.z;
    const int u = blockIdx.x, r = threadIdx.x, i = r >> 2, j = 8 * blockIdx.y + 2 * (r & 3);
    const int P = p.nseg;
    auto seg_of = [&](int t) { return rev ? P - 1 - t : t; };   // the t-th segment along the walk
    const float* x0 = seg_rec(p, dslot, u, seg_of(0), 0);
    float c0 = rec_at(x0, i, j), c1 = rec_at(x0, i, j + 1);
    // step t (1 .. P - 1) emits the start of segment seg_of(t); fold t - 1 + 1 = t uses segment seg_of(t)
    scan_columns(
        P - 2, P - 1, c0, c1, [&](int s) -> const float* { return seg_rec(p, dslot, u, seg_of(s + 1), 1); },
        [&](int s, float& a, float& b) {
            const float* xs = seg_rec(p, dslot, u, seg_of(s + 1), 0);
            a = rec_at(xs, i, j);
            b = rec_at(xs, i, j + 1);
        },
        [&](int s, float a, float b) {
            float* dst = seg_rec(p, dslot, u, seg_of(s + 1), 2);
            rec_at(dst, i, j) = a;
            rec_at(dst, i, j + 1) = b;
        });
}

// Gated mode, the chain split in time (few heads over many chunks): Phi = diag(E) acts on the rows, so a segment's
// transition is the vector of its decays' products and everything stays elementwise.  A walk per (unit, segment,
// sweep) from zero (the sequence's own start at its end segment) writes the local records and, per chunk, the
// product T_k of the decays walked so far (the rows' factor from the segment's start to the chunk); the scan
// joins the segments (S_{s+1} = Pi_s (.) S_s + X_s, likewise for the adjoints, and dh0 after the last fold); the
// fix-up adds T_k (.) S_s to every record of a segment that did not start from the sequence's own start.  Thread
// mapping as in chunk_chain_gated_kernel: rows 2 (r >> 3), + 1 x columns 8 (r & 7) .. + 7.
__device__ __forceinline__ float* gated_tvec(const CbParams& p, int d, size_t q)
{
    return p.tvec + ((size_t)d * p.nq + q) * 64;
}

__global__ void __launch_bounds__(256) chunk_chain_gated_seg_kernel(const __grid_constant__ CbParams p)
{
    const bool rev = p.rev_only || blockIdx.z == 1;
    const int dslot = p.rev_only ? 0 : (int)blockIdx.z;
    const int u = blockIdx.x, sg = blockIdx.y, r = threadIdx.x, i0 = 2 * (r >> 3), j0 = 8 * (r & 7);
    const int dk = p.dk, dv = p.dv_, nk = p.nchunks;
    const int k0 = sg * p.seg_len, k1 = min(k0 + p.seg_len, nk), ns = k1 - k0;
    const size_t qb = (size_t)u * nk;
    const float* rec_in = rev ? p.ych : p.dlt;
    float* rec_out = rev ? p.dst : p.st;
    auto chunk_of = [&](int n) { return rev ? k1 - 1 - n : k0 + n; };
    auto rec = [&](int k, float4 (&v)[4]) {
        v[0] = *rec4(rec_in, qb + k, i0, j0);
        v[1] = *rec4(rec_in, qb + k, i0, j0 + 4);
        v[2] = *rec4(rec_in, qb + k, i0 + 1, j0);
        v[3] = *rec4(rec_in, qb + k, i0 + 1, j0 + 4);
    };
    auto put = [&](float* base, size_t q, const float2 (&x)[8]) {
        *rec4(base, q, i0, j0) = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
        *rec4(base, q, i0, j0 + 4) = make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
        *rec4(base, q, i0 + 1, j0) = make_float4(x[4].x, x[4].y, x[5].x, x[5].y);
        *rec4(base, q, i0 + 1, j0 + 4) = make_float4(x[6].x, x[6].y, x[7].x, x[7].y);
    };
    // the local start: the sequence's own (h0 forward, dh_T reverse) at its end segment, zero elsewhere
    const float* src0 = rev ? (sg == p.nseg - 1 ? p.dhT : nullptr) : (sg == 0 ? p.h0 : nullptr);
    float2 s[8];
#pragma unroll
    for (int e = 0; e < 8; e++) {
        const int i = i0 + (e >> 2), j = j0 + 2 * (e & 3);
        const bool in = src0 && i < dk;
        s[e] = make_float2(in && j < dv ? src0[((size_t)u * dk + i) * dv + j] : 0.f,
                           in && j + 1 < dv ? src0[((size_t)u * dk + i) * dv + j + 1] : 0.f);
    }
    float t0 = 1.f, t1 = 1.f;   // T of rows i0, i0 + 1
    float4 d[4], dn[4];
    float e0 = 0.f, e1 = 0.f, en0 = 0.f, en1 = 0.f;
    rec(chunk_of(0), d);
    e0 = p.ec[(qb + chunk_of(0)) * 64 + i0];
    e1 = p.ec[(qb + chunk_of(0)) * 64 + i0 + 1];
    for (int n = 0; n < ns; n++) {
        const int k = chunk_of(n);
        put(rec_out, qb + k, s);
        if ((r & 7) == 0) {
            float* tv = gated_tvec(p, dslot, qb + k);
            tv[i0] = t0;
            tv[i0 + 1] = t1;
        }
        if (n + 1 < ns) {   // the next chunk's record and decays, a step ahead
            rec(chunk_of(n + 1), dn);
            en0 = p.ec[(qb + chunk_of(n + 1)) * 64 + i0];
            en1 = p.ec[(qb + chunk_of(n + 1)) * 64 + i0 + 1];
        }
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float ec = e < 2 ? e0 : e1;
            s[2 * e] = __ffma2_rn(make_float2(ec, ec), s[2 * e], make_float2(d[e].x, d[e].y));
            s[2 * e + 1] = __ffma2_rn(make_float2(ec, ec), s[2 * e + 1], make_float2(d[e].z, d[e].w));
        }
        t0 *= e0;
        t1 *= e1;
#pragma unroll
        for (int e = 0; e < 4; e++) d[e] = dn[e];
        e0 = en0;
        e1 = en1;
    }
    // the segment's final X and its transition Pi (record [1], its first 64 floats)
    put(seg_rec(p, dslot, u, sg, 0), 0, s);
    if ((r & 7) == 0) {
        float* pi = seg_rec(p, dslot, u, sg, 1);
        pi[i0] = t0;
        pi[i0 + 1] = t1;
    }
}

// The scan over a unit's segments, one CTA of 256 threads per (unit, sweep), elementwise: forward S_1 = X_0,
// S_{s+1} = Pi_s (.) S_s + X_s; reverse E_{P-2} = X_{P-1}, E_{s-1} = Pi_s (.) E_s + X_s, and dh0 = Pi_0 (.) E_0 + X_0.
// Each segment's start goes to its record [2].
__global__ void __launch_bounds__(256) chunk_gated_scan_kernel(const __grid_constant__ CbParams p)
{
    const bool rev = p.rev_only || blockIdx.y == 1;
    const int dslot = p.rev_only ? 0 : (int)blockIdx.y;
    const int u = blockIdx.x, r = threadIdx.x, i0 = 2 * (r >> 3), j0 = 8 * (r & 7);
    const int P = p.nseg;
    auto seg_of = [&](int t) { return rev ? P - 1 - t : t; };
    auto load = [&](const float* base, float4 (&v)[4]) {
        v[0] = *rec4(base, 0, i0, j0);
        v[1] = *rec4(base, 0, i0, j0 + 4);
        v[2] = *rec4(base, 0, i0 + 1, j0);
        v[3] = *rec4(base, 0, i0 + 1, j0 + 4);
    };
    float4 cur[4];
    load(seg_rec(p, dslot, u, seg_of(0), 0), cur);
    auto fold = [&](int sg) {   // cur <- Pi_sg (.) cur + X_sg
        const float* pi = seg_rec(p, dslot, u, sg, 1);
        const float p0 = pi[i0], p1 = pi[i0 + 1];
        float4 x[4];
        load(seg_rec(p, dslot, u, sg, 0), x);
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float pv = e < 2 ? p0 : p1;
            cur[e] = make_float4(fmaf(pv, cur[e].x, x[e].x), fmaf(pv, cur[e].y, x[e].y), fmaf(pv, cur[e].z, x[e].z),
                                 fmaf(pv, cur[e].w, x[e].w));
        }
    };
    for (int t = 1; t < P; t++) {
        float* dst = seg_rec(p, dslot, u, seg_of(t), 2);   // cur is this segment's true start
        *rec4(dst, 0, i0, j0) = cur[0];
        *rec4(dst, 0, i0, j0 + 4) = cur[1];
        *rec4(dst, 0, i0 + 1, j0) = cur[2];
        *rec4(dst, 0, i0 + 1, j0 + 4) = cur[3];
        if (t + 1 < P || rev) fold(seg_of(t));
    }
    if (rev && p.dh0) {
        // cur is the adjoint at the sequence's start
        const float v[2][8] = {{cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y, cur[1].z, cur[1].w},
                               {cur[2].x, cur[2].y, cur[2].z, cur[2].w, cur[3].x, cur[3].y, cur[3].z, cur[3].w}};
#pragma unroll
        for (int a = 0; a < 2; a++)
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int i = i0 + a, j = j0 + e;
                if (i < p.dk && j < p.dv_) p.dh0[((size_t)u * p.dk + i) * p.dv_ + j] = v[a][e];
            }
    }
}

// The fix-up, one CTA of 256 threads per (chunk, sweep): record += T_k (.) S_s for the chunks of every segment
// that did not start from the sequence's own start.
__global__ void __launch_bounds__(256) chunk_gated_fix_kernel(const __grid_constant__ CbParams p)
{
    const bool rev = p.rev_only || blockIdx.y == 1;
    const int dslot = p.rev_only ? 0 : (int)blockIdx.y;
    const int q = blockIdx.x, u = q / p.nchunks, k = q - u * p.nchunks, sg = k / p.seg_len;
    if (rev ? sg == p.nseg - 1 : sg == 0) return;   // those records are true already
    const int r = threadIdx.x, i0 = 2 * (r >> 3), j0 = 8 * (r & 7);
    const float* S = seg_rec(p, dslot, u, sg, 2);
    const float* tv = gated_tvec(p, dslot, (size_t)q);
    float* out = rev ? p.dst : p.st;
    const float ta = tv[i0], tb = tv[i0 + 1];
#pragma unroll
    for (int a = 0; a < 2; a++)
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const float t = a ? tb : ta;
            float4* o = rec4(out, (size_t)q, i0 + a, j0 + 4 * c);
            const float4 sv = *rec4(S, 0, i0 + a, j0 + 4 * c);
            const float4 x = *o;
            *o = make_float4(fmaf(t, sv.x, x.x), fmaf(t, sv.y, x.y), fmaf(t, sv.z, x.z), fmaf(t, sv.w, x.w));
        }
}

// ---------------------------------------------------------------- the forward split in time by walks (delta)
// A long sequence over few heads is cut into P segments of seg_len chunks.  The tcgen05 forward runs every segment
// from a zero state (the segments as batch rows) and keeps its residuals, so that the per-chunk maps are at hand:
// Phi_k = diag(E_k) + Bhat_k^T (-W_k) and Qc_k = Ctil_k + P_k (-W_k) (prep in its forward mode).  The chunk map is
// affine ("GDN & MLA Mechanism Deep-Dive", Step 5: chunked recurrence): with T_k = Phi_{k-1} ... Phi_{k0} the
// transition from the segment's start to chunk k, the true state entering chunk k is S_local,k + T_k S_s, and the
// chunk's outputs gain Qc_k T_k S_s.  So: a walk per segment carries T from the identity to the segment's
// transition Pi_s; fwd_walk_scan_kernel joins the segments (S_0 = h0, S_{s+1} = Pi_s S_s + X_s with X_s the
// zero-start run's final state) and writes h_T; a second walk per segment carries D_k = T_k S_s from S_s and writes
// o = o_zero-start + Qc_k D_k; for a saving forward, fwd_walk_res_kernel then makes the residuals true:
// S_k += D_k, U_k += (-W_k) D_k.

// The forward's scan over a unit's segments, one CTA of 256 threads per (unit, 8 columns): S_0 = h0,
// S_{s+1} = Pi_s S_s + X_s (X_s from Xb, the zero-start run's final states [B * P, H, d_k, d_v], segment view); each
// S_s goes to record [2] of segment s, and S_P is h_T.
__global__ void __launch_bounds__(256) fwd_walk_scan_kernel(const __grid_constant__ CbParams p, const float* Xb,
                                                            const float* h0, float* hT)
{
    const int u = blockIdx.x, r = threadIdx.x, i = r >> 2, j = 8 * blockIdx.y + 2 * (r & 3);
    const int P = p.nseg, dk = p.dk, dv = p.dv_, b = u / p.H, h = u - b * p.H;
    auto at = [&](const float* m, int jj) { return i < dk && jj < dv ? m[((size_t)u * dk + i) * dv + jj] : 0.f; };
    float c0 = h0 ? at(h0, j) : 0.f, c1 = h0 ? at(h0, j + 1) : 0.f;
    scan_columns(
        hT ? P : P - 1, P, c0, c1, [&](int s) -> const float* { return seg_rec(p, 0, u, s, 1); },
        [&](int s, float& a, float& bv) {
            const float* xs = Xb + ((size_t)(b * P + s) * p.H + h) * dk * dv;
            a = i < dk && j < dv ? xs[i * dv + j] : 0.f;
            bv = i < dk && j + 1 < dv ? xs[i * dv + j + 1] : 0.f;
        },
        [&](int s, float a, float bv) {
            float* dst = seg_rec(p, 0, u, s, 2);
            rec_at(dst, i, j) = a;
            rec_at(dst, i, j + 1) = bv;
        });
    if (hT) {
        if (i < dk && j < dv) hT[((size_t)u * dk + i) * dv + j] = c0;
        if (i < dk && j + 1 < dv) hT[((size_t)u * dk + i) * dv + j + 1] = c1;
    }
}

// The forward's walks over one segment each (blockIdx.x = unit, blockIdx.y = segment), on the records that prep
// writes in its forward mode, [Phi_hi | Qc_hi | Phi_lo | Qc_lo] (32 KB a chunk, one bulk copy into a ring of CT_NS
// stages).  A step is the chain's product with the stacked A operand [Phi ; Qc] (M = 128, rows 64..127 are Qc):
//   D[:, 0:64 | 64:128] = [Phi ; Qc]_hi [X_hi | X_lo] (N = 128),   D[:, 0:64] += [Phi ; Qc]_lo X_hi (N = 64)
// so TMEM lanes 0..63 hold Phi X (the next X) and lanes 64..127 Qc X.  OUT = false: X starts at the identity and
// the segment's transition Pi is left in its record [1].  OUT = true: X starts at the segment's true state S_s
// (record [2]) and is D_k = T_k S_s before chunk k's step; warps 2, 3, 6, 7 (lanes 64..127: token t of the chunk,
// 32 columns each) write o = o_zero-start + Qc D, and a saving forward's D goes to its records for the residual
// fix-up.  Warps 0, 1, 4, 5 hold X as in the chain (row i, 32 columns); thread 0 issues the copies and products.
// OUT = false launches 192 threads (warps 2 and 3 leave after the set-up), OUT = true 256.
constexpr uint32_t FW_STAGE = 32768;
constexpr uint32_t FW_X = CT_NS * FW_STAGE;                  // X hi, X lo tiles
constexpr uint32_t FW_BAR = FW_X + 16384;
constexpr uint32_t FW_SMEM = FW_BAR + 128 + 1024;

constexpr int fw_threads(bool out) { return out ? 256 : CT_THREADS; }

template <bool OUT>
__global__ void __launch_bounds__(fw_threads(OUT), 1) fwd_walk_kernel(const __grid_constant__ CbParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* Xt = sm + FW_X;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + FW_BAR);
    uint64_t* mmab = full + CT_NS;
    uint32_t* misc = reinterpret_cast<uint32_t*>(mmab + 1);   // [0] TMEM base, [1] abort
    const int u = blockIdx.x, sg = blockIdx.y, r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const int nk = p.nchunks, k0 = sg * p.seg_len, k1 = min(k0 + p.seg_len, nk), ns = k1 - k0;
    const int bb = u / p.H, h = u - bb * p.H;
    const size_t qb = (size_t)u * nk;
    // active threads: the X rows (warps 0, 1, 4, 5) and, with OUT, the output rows (warps 2, 3, 6, 7)
    const int nact = OUT ? 256 : 128;
    const bool orow = OUT && (warp & 2);
    auto issue_copy = [&](int n) {
        const int s = n % CT_NS;
        const unsigned char* src = p.phi + (qb + k0 + n) * FW_STAGE;
        if (OUT) {
            mbar_arrive_expect_tx(&full[s], FW_STAGE);
            bulk_g2s(sm + s * FW_STAGE, src, FW_STAGE, &full[s]);
        } else {
            // the transitions need Phi alone: its hi and lo tiles (the Qc rows of the stage feed TMEM rows
            // 64..127, which this walk never reads)
            mbar_arrive_expect_tx(&full[s], 16384);
            bulk_g2s(sm + s * FW_STAGE, src, 8192, &full[s]);
            bulk_g2s(sm + s * FW_STAGE + 16384, src + 16384, 8192, &full[s]);
        }
    };
    if (r == 0) {
        for (int s = 0; s < CT_NS; s++) mbar_init(&full[s], 1);
        mbar_init(mmab, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&misc[0], 128);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!OUT && (warp == 2 || warp == 3)) return;
    const uint32_t tb = misc[0];
    int issued = ns < CT_NS ? ns : CT_NS;
    if (r == 0)
        for (int n = 0; n < issued; n++) issue_copy(n);
    const int i = 32 * (warp & 1) + lane, j0 = 32 * (warp >> 2);
    const uint32_t tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    uint32_t* abortf = &misc[1];
    const int t = 32 * (warp & 1) + lane;   // output rows: the chunk's token, columns oc0 .. oc0 + 31
    const int oc0 = 32 * (warp >> 2);
    auto o_row = [&](int k) { return ((size_t)bb * p.T + 64 * k + t) * p.H + h; };
    if (orow && oc0 == 0)   // one prefetch per token row
        for (int n = 0; n < 2 && n < ns; n++)
            if (64 * (k0 + n) + t < p.T) prefetch_l2_bulk(p.fw_o32 + o_row(k0 + n) * p.dv_, (uint32_t)p.dv_ * 4u);
    float x[32];
    if (!orow) {
        if (OUT) {
            const float4* src = rec4(seg_rec(p, 0, u, sg, 2), 0, i, j0);
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const float4 v = src[64 * e];
                x[4 * e] = v.x; x[4 * e + 1] = v.y; x[4 * e + 2] = v.z; x[4 * e + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; e++) x[e] = i == j0 + e ? 1.f : 0.f;
        }
    }
    bool ok = true;
    float4 o0v[8];   // output rows: the zero-start outputs of token t, loaded before the step's product
    for (int n = 0; n < ns; n++) {
        const int k = k0 + n;
        if (orow) {
            const bool in = 64 * k + t < p.T;
            const float* o0 = p.fw_o32 + o_row(in ? k : k0) * p.dv_ + oc0;
#pragma unroll
            for (int e = 0; e < 8; e++)
                o0v[e] = oc0 + 4 * e < p.dv_ ? *reinterpret_cast<const float4*>(o0 + 4 * e)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!orow) {
            if (OUT && p.fw_st) {   // D_k for the residual fix-up
                float4* dst = rec4(p.st, qb + k, i, j0);
#pragma unroll
                for (int e = 0; e < 8; e++) dst[64 * e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
            }
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float a8[8];
#pragma unroll
                for (int e = 0; e < 8; e++) a8[e] = x[8 * q + e];
                st_row8_split(Xt, Xt + 8192, i, (j0 >> 3) + q, a8);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, nact);
        tc_fence_after();
        const int s = n % CT_NS;
        if (r == 0) {
            if (wait_or_abort(&full[s], (uint32_t)(n / CT_NS) & 1u, abortf, p.status, p.wait_ns)) {
                tc_fence_after();
                const uint32_t a = smem_u32(sm + s * FW_STAGE), xb = smem_u32(Xt);
                mma_tiles(tb, a, false, 0, 0, xb, true, 8192, 0, 4, idesc_bf16(128, 128, false, true), false);
                mma_tiles(tb, a + 16384, false, 0, 0, xb, true, 8192, 0, 4, idesc_bf16(128, 64, false, true), true);
                mma_commit(mmab);
            } else {
                atomicExch(p.status + 2, (OUT ? 820u : 810u) + (uint32_t)n);
            }
        }
        if (orow && oc0 == 0 && n + 2 < ns && 64 * (k + 2) + t < p.T)
            prefetch_l2_bulk(p.fw_o32 + o_row(k + 2) * p.dv_, (uint32_t)p.dv_ * 4u);
        if (!wait_or_abort(mmab, (uint32_t)n & 1u, abortf, p.status, p.wait_ns)) {
            ok = false;
            break;
        }
        tc_fence_after();
        if (r == 0 && issued < ns) issue_copy(issued++);   // the stage just read is free
        if (!orow) {
#pragma unroll
            for (int hh = 0; hh < 2; hh++) {
                float a[16], b[16];
                tmem_ld16(tl + j0 + 16 * hh, a);        // [Phi ; Qc]_hi X_hi + [Phi ; Qc]_lo X_hi
                tmem_ld16(tl + 64 + j0 + 16 * hh, b);   // [Phi ; Qc]_hi X_lo
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e++) x[16 * hh + e] = a[e] + b[e];
            }
        } else {
            // o = o_zero-start + Qc D, token t of chunk k (the TMEM loads are warp-uniform; the row may be past T)
            const bool in = 64 * k + t < p.T;
            __nv_bfloat16* o = p.fw_o + o_row(k) * p.dv_ + oc0;
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 16) {
                float a[16], b[16];
                tmem_ld16(tl + oc0 + c0, a);
                tmem_ld16(tl + 64 + oc0 + c0, b);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e += 8) {
                    if (in && oc0 + c0 + e < p.dv_) {
                        const float4 x0 = o0v[(c0 + e) >> 2];
                        const float4 x1 = o0v[((c0 + e) >> 2) + 1];
                        uint4 w;
                        w.x = pack_bf16(x0.x + a[e] + b[e], x0.y + a[e + 1] + b[e + 1]);
                        w.y = pack_bf16(x0.z + a[e + 2] + b[e + 2], x0.w + a[e + 3] + b[e + 3]);
                        w.z = pack_bf16(x1.x + a[e + 4] + b[e + 4], x1.y + a[e + 5] + b[e + 5]);
                        w.w = pack_bf16(x1.z + a[e + 6] + b[e + 6], x1.w + a[e + 7] + b[e + 7]);
                        *reinterpret_cast<uint4*>(o + c0 + e) = w;
                    }
                }
            }
        }
    }
    if (ok && !OUT && !orow) {   // the segment's transition
        float4* dst = rec4(seg_rec(p, 0, u, sg, 1), 0, i, j0);
#pragma unroll
        for (int e = 0; e < 8; e++) dst[64 * e] = make_float4(x[4 * e], x[4 * e + 1], x[4 * e + 2], x[4 * e + 3]);
    }
    // wind down: after an abort, let the copies still in flight land before the CTA leaves
    if (r == 0 && *(volatile uint32_t*)abortf)
        for (int n = issued - CT_NS < 0 ? 0 : issued - CT_NS; n < issued; n++)
            mbar_wait(&full[n % CT_NS], (uint32_t)(n / CT_NS) & 1u, nullptr, p.wait_ns);
    tc_fence_before();
    named_bar_sync(1, nact);
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// A saving forward's residual fix-up, chunk-parallel (persistent, three CTAs of 256 threads per SM): with D_k from
// the output walk, the residual state S_k += D_k and U_k += (-W_k) D_k, the latter one product on hi/lo operands:
// TMEM[:, 0:64 | 64:128] = (-W)_hi [D_hi | D_lo] (N = 128), TMEM[:, 0:64] += (-W)_lo D_hi; lanes 0..63 (tokens t)
// add it to U.  The products have M = 128; the rows past 64 of the A operands read the next 8 KB (the lo tile, and
// for the lo tile the D tiles), which give TMEM rows nobody reads.
namespace fx {
constexpr uint32_t NWH = 0, NWL = 8192;           // -W hi, lo (residuals, one bulk copy)
constexpr uint32_t DH = 16384, DL = 24576;        // D hi, lo [i][j] (MN-major B)
constexpr uint32_t SMALL = 32768;
constexpr uint32_t SMEM = SMALL + 1024 + 1024;
constexpr uint32_t TM_COLS = 128;
static_assert(NWL == NWH + 8192 && DH == NWL + 8192 && DL == DH + 8192, "stacked operands");
}  // namespace fx

struct FxSmall {
    uint64_t full, mma;
    uint32_t tmem_base, abort;
};

__global__ void __launch_bounds__(256, 3) fwd_walk_res_kernel(const __grid_constant__ CbParams p)
{
    if (p.gated) {
        // gated residuals keep no U: the state alone, S += D (thread = row i, 16 columns)
        const int i = threadIdx.x & 63, cq = threadIdx.x >> 6;
        for (int q = blockIdx.x; q < p.nq; q += gridDim.x)
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 d4 = *rec4(p.st, q, i, 16 * cq + e);
                float4* s4 = rec4(p.fw_st, q, i, 16 * cq + e);
                const float4 o = *s4;
                *s4 = make_float4(o.x + d4.x, o.y + d4.y, o.z + d4.z, o.w + d4.w);
            }
        return;
    }
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    FxSmall& S = *reinterpret_cast<FxSmall*>(sm + fx::SMALL);
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31, q4 = warp & 3, wh = warp >> 2, trow = r & 127;
    if (r == 0) {
        mbar_init(&S.full, 1);
        mbar_init(&S.mma, 1);
        S.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&S.tmem_base, fx::TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem_base, tl = tb + ((uint32_t)(q4 * 32) << 16);
    uint32_t full_phase = 0, mma_phase = 0;
    auto issue = [&](int q) {
        mbar_arrive_expect_tx(&S.full, 16384);
        bulk_g2s(sm + fx::NWH, p.sv + (size_t)q * p.sv_stride + sv::NW, 16384, &S.full);   // -W hi, then lo
    };
    int q = blockIdx.x, pending = -1;
    if (r == 0 && q < p.nq) issue(q);
    if (q < p.nq) pending = q;
    for (; q < p.nq; q += gridDim.x) {
        if (r == 0 && q + (int)gridDim.x < p.nq) {
            const int qn = q + gridDim.x;
            prefetch_l2_bulk(p.sv + (size_t)qn * p.sv_stride + sv::NW, 16384);
            prefetch_l2_bulk(p.sv + (size_t)qn * p.sv_stride + sv::UT, 16384);
            prefetch_l2_bulk(p.st + (size_t)qn * 4096, 16384);
            prefetch_l2_bulk(p.fw_st + (size_t)qn * 4096, 16384);
        }
        // D -> hi/lo tiles (thread = row i, 16 columns); the residual state S += D
        {
            const int i = r & 63, cq = r >> 6;
            float dv16[16];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 d4 = *rec4(p.st, q, i, 16 * cq + e);
                dv16[e] = d4.x; dv16[e + 1] = d4.y; dv16[e + 2] = d4.z; dv16[e + 3] = d4.w;
            }
            st16_split(sm + fx::DH, sm + fx::DL, i, cq, dv16);
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                float4* s4 = rec4(p.fw_st, q, i, 16 * cq + e);
                const float4 o = *s4;
                *s4 = make_float4(o.x + dv16[e], o.y + dv16[e + 1], o.z + dv16[e + 2], o.w + dv16[e + 3]);
            }
        }
        if (warp == 0 && !wait_or_abort(&S.full, full_phase, &S.abort, p.status, p.wait_ns) && lane == 0)
            atomicExch(p.status + 2, 6u);
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 256);
        tc_fence_after();
        if (*(volatile uint32_t*)&S.abort) break;
        full_phase ^= 1;
        pending = -1;
        if (r == 0) {
            const uint32_t nwh = smem_u32(sm + fx::NWH), nwl = smem_u32(sm + fx::NWL), dh = smem_u32(sm + fx::DH);
            mma_tiles(tb, nwh, false, 0, 0, dh, true, 8192, 0, 4, idesc_bf16(128, 128, false, true), false);
            mma_tiles(tb, nwl, false, 0, 0, dh, true, 8192, 0, 4, idesc_bf16(128, 64, false, true), true);
            mma_commit(&S.mma);
        }
        if (warp == 0 && !wait_or_abort(&S.mma, mma_phase, &S.abort, p.status, p.wait_ns) && lane == 0)
            atomicExch(p.status + 2, 710u);
        named_bar_sync(1, 256);
        mma_phase ^= 1;
        tc_fence_after();
        if (*(volatile uint32_t*)&S.abort) break;
        if (q4 < 2) {
            // the residual U += (-W) D, token trow
            float4* ur = reinterpret_cast<float4*>(p.sv + (size_t)q * p.sv_stride + sv::UT);
#pragma unroll 1
            for (int h2 = 0; h2 < 2; h2++) {
                const int c0 = 32 * wh + 16 * h2;
                float a[16], b[16];
                tmem_ld16(tl + c0, a);
                tmem_ld16(tl + 64 + c0, b);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    float4* u4 = ur + ((c0 + e) >> 2) * 64 + trow;
                    const float4 x = *u4;
                    *u4 = make_float4(x.x + a[e] + b[e], x.y + a[e + 1] + b[e + 1], x.z + a[e + 2] + b[e + 2],
                                      x.w + a[e + 3] + b[e + 3]);
                }
            }
        }
        // the tiles are free: the next chunk's -W
        tc_fence_before();
        named_bar_sync(1, 256);
        tc_fence_after();
        if (q + (int)gridDim.x < p.nq) {
            if (r == 0) issue(q + gridDim.x);
            pending = q + gridDim.x;
        }
    }
    if (r == 0 && *(volatile uint32_t*)&S.abort && pending >= 0) mbar_wait(&S.full, full_phase, nullptr, p.wait_ns);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tb, fx::TM_COLS);
}

// ================================================================= pass 3: gradients
// The near pairs' adjoint, one 4-column group sg of a 16-block at a time (rows tl0 .. tl0 + 3 of the block, channels
// nch .. nch + 3).  NQ / NK: the block's near dQ / dK entries ([16][20] fp32, zero above the diagonal).  Row side
// (t as row): aP[4 ti + e] += dQ[t][s] y_s[e] and aK likewise with dK, y = b / alpha (times KL across the halves).
// Column side (t as column): aP += dQ[s][t] c_s[e] x_s[e], aK += dK[s][t] b_s[e] x_s[e], x = left alpha (times KU
// across the halves, where both sums go into aP).  Every load of the group is issued before its products, and
// the accumulator each product feeds is fixed at compile time.
template <bool DELTA, bool CROSS>
__device__ __forceinline__ void near_rows_rev(const float* NQ, const float* NK, const float* yb, int tl0, int sg,
                                              const float* kl, float* aP, float* aK)
{
    float dq[4][4], dk[4][4], y[4][4];
#pragma unroll
    for (int ti = 0; ti < 4; ti++) {
        const float4 q4 = *reinterpret_cast<const float4*>(NQ + (tl0 + ti) * 20 + 4 * sg);
        dq[ti][0] = q4.x; dq[ti][1] = q4.y; dq[ti][2] = q4.z; dq[ti][3] = q4.w;
        if (DELTA) {
            const float4 k4 = *reinterpret_cast<const float4*>(NK + (tl0 + ti) * 20 + 4 * sg);
            dk[ti][0] = k4.x; dk[ti][1] = k4.y; dk[ti][2] = k4.z; dk[ti][3] = k4.w;
        }
    }
#pragma unroll
    for (int si = 0; si < 4; si++) {
        const float4 y4 = *reinterpret_cast<const float4*>(yb + (4 * sg + si) * kAS);
        y[si][0] = y4.x; y[si][1] = y4.y; y[si][2] = y4.z; y[si][3] = y4.w;
        if (CROSS) {
#pragma unroll
            for (int e = 0; e < 4; e++) y[si][e] *= kl[e];
        }
    }
#pragma unroll
    for (int si = 0; si < 4; si++)
#pragma unroll
        for (int ti = 0; ti < 4; ti++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                aP[4 * ti + e] = fmaf(dq[ti][si], y[si][e], aP[4 * ti + e]);
                if (DELTA) aK[4 * ti + e] = fmaf(dk[ti][si], y[si][e], aK[4 * ti + e]);
            }
}

template <bool DELTA, bool CROSS>
__device__ __forceinline__ void near_cols_rev(const float* NQ, const float* NK, const float* alpha,
                                              const unsigned char* sC, const unsigned char* sB, int tl0, int sb, int sg,
                                              int nch, const float* ku, float* aP, float* aK)
{
    float dq[4][4], dk[4][4], x[4][4], c4[4][4], b4[4][4];   // dq, dk: [si][ti] = dM[s][t]
#pragma unroll
    for (int si = 0; si < 4; si++) {
        const float4 q4 = *reinterpret_cast<const float4*>(NQ + (4 * sg + si) * 20 + tl0);
        dq[si][0] = q4.x; dq[si][1] = q4.y; dq[si][2] = q4.z; dq[si][3] = q4.w;
        if (DELTA) {
            const float4 k4 = *reinterpret_cast<const float4*>(NK + (4 * sg + si) * 20 + tl0);
            dk[si][0] = k4.x; dk[si][1] = k4.y; dk[si][2] = k4.z; dk[si][3] = k4.w;
        }
    }
#pragma unroll
    for (int si = 0; si < 4; si++) {
        const int s = sb + 4 * sg + si;
        const float4 a4 = *reinterpret_cast<const float4*>(alpha + s * kAS + nch);
        x[si][0] = a4.x; x[si][1] = a4.y; x[si][2] = a4.z; x[si][3] = a4.w;
        if (CROSS) {
#pragma unroll
            for (int e = 0; e < 4; e++) x[si][e] *= ku[e];
        }
        ld4_bf16(sC, s, nch, c4[si]);
        ld4_bf16(sB, s, nch, b4[si]);
    }
#pragma unroll
    for (int si = 0; si < 4; si++)
#pragma unroll
        for (int ti = 0; ti < 4; ti++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float xc = c4[si][e] * x[si][e], xb = b4[si][e] * x[si][e];
                if (CROSS) {
                    const float in = DELTA ? fmaf(dk[si][ti], xb, aP[4 * ti + e]) : aP[4 * ti + e];
                    aP[4 * ti + e] = fmaf(dq[si][ti], xc, in);
                } else {
                    aP[4 * ti + e] = fmaf(dq[si][ti], xc, aP[4 * ti + e]);
                    if (DELTA) aK[4 * ti + e] = fmaf(dk[si][ti], xb, aK[4 * ti + e]);
                }
            }
}

template <bool DELTA>
__global__ void __launch_bounds__(kThreads, 1) chunk_grad_kernel(const __grid_constant__ CbParams p)
{
    extern __shared__ unsigned char smem_raw[];
    Ctx c = setup(smem_raw, p);
    Small& S = *c.S;
    unsigned char* X = c.X;
    const unsigned char* sB = c.sm + OFF_STAGE + ST_B;
    const unsigned char* sC = c.sm + OFF_STAGE + ST_C;
    const unsigned char* sV = c.sm + OFF_STAGE + ST_V;
    const unsigned char* sDO = c.sm + OFF_STAGE + ST_DO;
    uint32_t full_phase = 0, full2_phase = 0;
    int q = blockIdx.x;
    int pending = -1, pending2 = -1;   // chunks whose loads (stage, saved front) are in flight
    // the saved front: delta always (from prep or a saving forward); gated only from a saving forward (P)
    const bool use_sv = DELTA || p.rev_only;
    if (c.r == 0 && q < p.nq) {
        issue_tma(p, S, c.sm, q);
        if (use_sv) issue_saved<DELTA>(p, S, c.sm, q);
    }
    if (q < p.nq) {
        pending = q;
        if (use_sv) pending2 = q;
    }
    const int trow = c.trow, tt = trow & 63, isK = trow >> 6, wh = c.wh;
    CB_STAMP_INIT;
    for (; q < p.nq; q += gridDim.x) {
        const int u = q / p.nchunks, k = q - u * p.nchunks, bb = u / p.H, h = u - bb * p.H;
        const int t0 = 64 * k, L = min(64, p.T - t0);
        CB_STAMP(1, 0);
        load_small(c, p, bb, h, t0);
        if (c.r == 0) {
            // this chunk's S, dS' (and Util) records and the next chunk's tiles towards L2
            prefetch_l2_bulk(p.st + (size_t)q * 4096, 16384);
            prefetch_l2_bulk(p.dst + (size_t)q * 4096, 16384);
            if (DELTA) {
                prefetch_l2_bulk(p.sv + (size_t)q * p.sv_stride + sv::UT, 16384);
                prefetch_l2_bulk(p.sv + (size_t)q * p.sv_stride + sv::K, 16384);
            }
            if (q + (int)gridDim.x < p.nq) {
                prefetch_tma(p, q + gridDim.x);
                // the next chunk's saved front (P, -N, Dinv, -W: the bulk copies at this chunk's end)
                if (use_sv) prefetch_l2_bulk(p.sv + (size_t)(q + gridDim.x) * p.sv_stride, DELTA ? sv::K : 16384);
                if (DELTA && !p.rev_only) prefetch_l2_bulk(p.sv + (size_t)(q + gridDim.x) * p.sv_stride + sv::NW, 8192);
            }
        }
        if (c.warp == 0 && !wait_or_abort(&S.full, full_phase, &S.abort, p.status, p.wait_ns) && c.lane == 0)
            atomicExch(p.status + 2, 2u);
        if (use_sv && c.warp == 1 && !wait_or_abort(&S.full2, full2_phase, &S.abort, p.status, p.wait_ns) &&
            c.lane == 0)
            atomicExch(p.status + 2, 3u);
        bar_all();
        if (*(volatile uint32_t*)&S.abort) break;
        full_phase ^= 1;
        pending = -1;
        if (use_sv) {
            full2_phase ^= 1;
            pending2 = -1;
        }
        CB_STAMP(1, 1);
        front_scan(c);
        bar_all();
        const int t = c.r & 63, cq = c.r >> 6;
        CB_STAMP(1, 2);

        // ---- front.  Delta: P, -N, Dinv, K and -W arrived with the saved front (the prep pass or the forward
        // computed them); gated: P from a saving forward, else the level operands, the level product, the near
        // pairs and P here
        if (!DELTA && !p.rev_only) {
            front_operands(c, X + gl::A1, X + gl::B1, true);
            smem_to_tc();
            if (c.r == 0) {
                issue_level(c.tbase, X + gl::A1, X + gl::B1);
                mma_commit(&S.mma);
            }
            front_near(c, fptr(X, gl::NEAR), false);
            bar_all();
            if (!mma_wait(c, p, 7)) break;
            front_solve<false>(c, p, X + gl::NEAR, X + gl::P, X + gl::LR, X + gl::LRL, X + gl::MS, X + gl::DINV,
                               X + gl::NA, X + gl::X0, nullptr);
            bar_all();
        }
        CB_STAMP(1, 4);

        // ---- S, dS' of the chunk (fp32 from the chain) -> hi/lo tiles [i][j]; sum_j dS'[i][j] S[i][j].  (Delta from
        // residuals: U, kept by the saving forward, is loaded here too, so that the loads share one wait.)
        float4 ures[8];
        if (DELTA && p.rev_only && !isK) {
            const float4* urow = reinterpret_cast<const float4*>(p.sv + (size_t)q * p.sv_stride + sv::UT) + tt;
#pragma unroll
            for (int e = 0; e < 8; e++) ures[e] = urow[(4 * (2 * wh + (e >> 2)) + (e & 3)) * 64];
        }
        {
            float sv[16], dv16[16];
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 a = *rec4(p.st, q, t, 16 * cq + e);
                const float4 b = *rec4(p.dst, q, t, 16 * cq + e);
                sv[e] = a.x; sv[e + 1] = a.y; sv[e + 2] = a.z; sv[e + 3] = a.w;
                dv16[e] = b.x; dv16[e + 1] = b.y; dv16[e + 2] = b.z; dv16[e + 3] = b.w;
            }
            float sdp = 0.f;
#pragma unroll
            for (int e = 0; e < 16; e++) sdp = fmaf(dv16[e], sv[e], sdp);
            S.sd[cq][t] = sdp;
            st16_split(X + gl::U + 8192, X + gl::U + 24576, t, cq, sv);
            st16_split(X + gl::DSN, X + gl::DSN + 8192, t, cq, dv16);
            if (!DELTA) {
                // U = V: the value tile copied into U_hi, U_lo = 0
                float vv[16];
                ld16_bf16(sV, t, cq, vv);
                st16_bf16(X + gl::U, t, cq, vv);
                zero16(X + gl::U + 16384, t, cq);
            }
        }
        if (DELTA && p.rev_only) {
            // a saving forward kept U itself: straight into its hi/lo tiles
            if (!isK) {
#pragma unroll
                for (int h2 = 0; h2 < 2; h2++) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float4 x = ures[4 * h2 + e];
                        v[4 * e] = x.x; v[4 * e + 1] = x.y; v[4 * e + 2] = x.z; v[4 * e + 3] = x.w;
                    }
                    st16_split(X + gl::U, X + gl::U + 16384, tt, 2 * wh + h2, v);
                }
            }
        } else if (DELTA) {
            // Util (saved fp32) into TMEM as the start of U = Util - W S; -W came with the saved front
            if (!isK) {
                const float4* urow = reinterpret_cast<const float4*>(p.sv + (size_t)q * p.sv_stride + sv::UT) + tt;
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int cg = 2 * wh + h2;
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const float4 x = urow[(4 * cg + e) * 64];
                        v[4 * e] = x.x; v[4 * e + 1] = x.y; v[4 * e + 2] = x.z; v[4 * e + 3] = x.w;
                    }
                    tmem_st16(c.tl + TM_UT + 16 * cg, v);
                }
                tmem_wait_st();
            }
            smem_to_tc();
            if (c.r == 0) {
                const uint32_t id = idesc_bf16(128, 64, false, true);
                const uint32_t nw = smem_u32(X + gl::NW), sh = smem_u32(X + gl::U + 8192);
                mma_tiles(c.tbase + TM_UT, nw, false, 0, 0, sh, true, 8192, 0, 4, id, true);
                mma_tiles(c.tbase + TM_UT, nw, false, 0, 0, sh + 16384, true, 8192, 0, 4, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_wait(c, p, 8)) break;
            // U -> hi/lo [s][j]
            if (!isK) {
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int cg = 2 * wh + h2;
                    float v[16];
                    tmem_ld16(c.tl + TM_UT + 16 * cg, v);
                    tmem_wait_ld();
                    st16_split(X + gl::U, X + gl::U + 16384, tt, cg, v);
                }
            }
        }
        // Bhat natural [t][i] hi/lo (K-major A of B^ dS')
        CB_STAMP(1, 5);
        {
            float bv[16], y[16];
            ld16_bf16(sB, t, cq, bv);
            const float Gt = S.G[t], G63 = S.G[63];
#pragma unroll
            for (int e = 0; e < 16; e++) y[e] = bv[e] * fast_exp2(S.A2[16 * cq + e] * (G63 - Gt));
            st16_split(X + gl::BHH, X + gl::BHL, t, cq, y);
        }
        smem_to_tc();
        // ---- dU = P^T dO + Bhat dS'  (TMEM 288)
        if (c.r == 0) {
            const uint32_t idA = idesc_bf16(128, 64, true, true), idB = idesc_bf16(128, 64, false, true);
            const uint32_t pt = smem_u32(X + gl::P), dO = smem_u32(sDO);
            const uint32_t bh = smem_u32(X + gl::BHH), bl = smem_u32(X + gl::BHL), dsn = smem_u32(X + gl::DSN);
            mma_tiles(c.tbase + 288, pt, true, 8192, 0, dO, true, 8192, 0, 4, idA, false);
            mma_tiles(c.tbase + 288, pt + 8192, true, 8192, 0, dO, true, 8192, 0, 4, idA, true);
            mma_tiles(c.tbase + 288, bh, false, 0, 0, dsn, true, 8192, 0, 4, idB, true);
            mma_tiles(c.tbase + 288, bh, false, 0, 0, dsn + 8192, true, 8192, 0, 4, idB, true);
            mma_tiles(c.tbase + 288, bl, false, 0, 0, dsn, true, 8192, 0, 4, idB, true);
            mma_commit(&S.mma);
        }
        if (!mma_wait(c, p, 9)) break;
        CB_STAMP(1, 6);
        const size_t tokrow = ((size_t)bb * p.T + t0 + tt) * p.H + h;   // (b, t0 + tt, h) row of the token tensors
        if (!DELTA) {
            // dv = dU (the TMEM loads are warp-uniform; only the stores depend on the row)
            if (!isK) {
#pragma unroll 1
                for (int h2 = 0; h2 < 2; h2++) {
                    const int c0 = 32 * wh + 16 * h2;
                    float v[16];
                    tmem_ld16(c.tl + 288 + c0, v);
                    tmem_wait_ld();
                    __nv_bfloat16* dst = p.dv + tokrow * p.dv_ + c0;
#pragma unroll
                    for (int e = 0; e < 16; e += 8) {
                        if (tt < L && c0 + e < p.dv_) {
                            uint4 w;
                            w.x = pack_bf16(v[e], v[e + 1]); w.y = pack_bf16(v[e + 2], v[e + 3]);
                            w.z = pack_bf16(v[e + 4], v[e + 5]); w.w = pack_bf16(v[e + 6], v[e + 7]);
                            *reinterpret_cast<uint4*>(dst + e) = w;
                        }
                    }
                }
            }
        } else {
            // dU -> hi/lo [s][j] (MN-major B)
            if (!isK) {
                float v0[16], v1[16];   // both column groups in one TMEM round trip
                tmem_ld16(c.tl + 288 + 32 * wh, v0);
                tmem_ld16(c.tl + 288 + 32 * wh + 16, v1);
                tmem_wait_ld();
                st16_split(X + gl::DU, X + gl::DU + 8192, tt, 2 * wh, v0);
                st16_split(X + gl::DU, X + gl::DU + 8192, tt, 2 * wh + 1, v1);
            }
            smem_to_tc();
            // Z = dU - N^T dU (accumulated onto dU)
            if (c.r == 0) {
                const uint32_t id = idesc_bf16(128, 64, true, true);
                const uint32_t na = smem_u32(X + gl::NA), du = smem_u32(X + gl::DU);
                mma_tiles(c.tbase + 288, na, true, 8192, 0, du, true, 8192, 0, 4, id, true);
                mma_tiles(c.tbase + 288, na, true, 8192, 0, du + 8192, true, 8192, 0, 4, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_wait(c, p, 10)) break;
            if (!isK) {
                float v0[16], v1[16];   // both column groups in one TMEM round trip
                tmem_ld16(c.tl + 288 + 32 * wh, v0);
                tmem_ld16(c.tl + 288 + 32 * wh + 16, v1);
                tmem_wait_ld();
                st16_split(X + gl::Z, X + gl::Z + 8192, tt, 2 * wh, v0);
                st16_split(X + gl::Z, X + gl::Z + 8192, tt, 2 * wh + 1, v1);
            }
            smem_to_tc();
            // dR = Dinv^T Z (TMEM 352; lanes 64..127 hold a copy)
            if (c.r == 0) {
                const uint32_t id = idesc_bf16(128, 64, true, true);
                const uint32_t di = smem_u32(X + gl::DINV), z = smem_u32(X + gl::Z);
                mma_tiles(c.tbase + 352, di, true, 8192, 0, z, true, 8192, 0, 4, id, false);
                mma_tiles(c.tbase + 352, di, true, 8192, 0, z + 8192, true, 8192, 0, 4, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_wait(c, p, 11)) break;
            // dR: lanes 0..63 -> dv = beta dR (global) and dR hi/lo rows of the A operands [dO ; dR_hi] and
            // [0 ; dR_lo]; lanes 64..127 -> the dO copy and zero rows, and sum_j dR[t][j] V[t][j]
            {
                const float bet = S.beta[tt];
                float part = 0.f;
                float vb[2][16];   // both column groups in one TMEM round trip
                tmem_ld16(c.tl + 352 + 32 * wh, vb[0]);
                tmem_ld16(c.tl + 352 + 32 * wh + 16, vb[1]);
                tmem_wait_ld();
#pragma unroll
                for (int h2 = 0; h2 < 2; h2++) {
                    const int cg = 2 * wh + h2, c0 = 16 * cg;
                    const float (&v)[16] = vb[h2];
                    if (!isK) {
                        st16_split(X + gl::DOR + 8192, X + gl::ZR + 8192, tt, cg, v);
                        if (tt < L) {
                            __nv_bfloat16* dst = p.dv + tokrow * p.dv_ + c0;
#pragma unroll
                            for (int e = 0; e < 16; e += 8) {
                                if (c0 + e < p.dv_) {
                                    uint4 w;
                                    w.x = pack_bf16(bet * v[e], bet * v[e + 1]);
                                    w.y = pack_bf16(bet * v[e + 2], bet * v[e + 3]);
                                    w.z = pack_bf16(bet * v[e + 4], bet * v[e + 5]);
                                    w.w = pack_bf16(bet * v[e + 6], bet * v[e + 7]);
                                    *reinterpret_cast<uint4*>(dst + e) = w;
                                }
                            }
                        }
                    } else {
                        float vv[16];
                        ld16_bf16(sV, tt, cg, vv);
#pragma unroll
                        for (int e = 0; e < 16; e++) part = fmaf(v[e], vv[e], part);
                        // dO row copy (same row, same swizzle) and the zero rows
                        const uint32_t o0 = sw128(tt, c0), o1 = sw128(tt, c0 + 8);
                        *reinterpret_cast<uint4*>(X + gl::DOR + o0) = *reinterpret_cast<const uint4*>(sDO + o0);
                        *reinterpret_cast<uint4*>(X + gl::DOR + o1) = *reinterpret_cast<const uint4*>(sDO + o1);
                        zero16(X + gl::ZR, tt, cg);
                    }
                }
                if (isK) S.rs[0][wh][tt] = part;
            }
        }
        smem_to_tc();
        // ---- [dO ; dR] [U | S]^T (TMEM 0..127) and dBhat = U dS'^T (TMEM 128..191)
        CB_STAMP(1, 7);
        if (c.r == 0) {
            const uint32_t id8 = idesc_bf16(128, 128, false, false), id9 = idesc_bf16(128, 64, false, false);
            const uint32_t uh = smem_u32(X + gl::U), ul = uh + 16384, dsn = smem_u32(X + gl::DSN);
            const uint32_t ah = DELTA ? smem_u32(X + gl::DOR) : smem_u32(sDO);
            mma_tiles(c.tbase + 0, ah, false, 0, 0, uh, false, 0, 0, 4, id8, false);
            mma_tiles(c.tbase + 0, ah, false, 0, 0, ul, false, 0, 0, 4, id8, true);
            if (DELTA) mma_tiles(c.tbase + 0, smem_u32(X + gl::ZR), false, 0, 0, uh, false, 0, 0, 4, id8, true);
            mma_tiles(c.tbase + 128, uh, false, 0, 0, dsn, false, 0, 0, 4, id9, false);
            mma_tiles(c.tbase + 128, uh, false, 0, 0, dsn + 8192, false, 0, 0, 4, id9, true);
            if (DELTA) mma_tiles(c.tbase + 128, ul, false, 0, 0, dsn, false, 0, 0, 4, id9, true);
            mma_commit(&S.mma);
        }
        // while they run: the 16-block level's operands again, as fp16 hi/lo pairs (and, delta, the anchors); they
        // depend on b, c and the decay only
        front_operands(c, X + gl::A1H, X + gl::B1, true, X + gl::A1L, X + gl::B1L, use_sv);
        if (!mma_wait(c, p, 12)) break;
        CB_STAMP(1, 8);
        // ---- dQ (lanes 0..63) and dK = -beta (dR U^T) below the diagonal (lanes 64..127): the 16-block level's
        // operand A_d = [dQ | dK] by segments (fp16, K-major [t][seg], two 64-wide K blocks), the near entries in
        // fp32
        {
            const int I = tt >> 4;
            const float bet = DELTA ? S.beta[tt] : 0.f;
            float row[64];
            {
                // the row's 64 columns in one TMEM round trip
                float v[4][16];
#pragma unroll
                for (int g4 = 0; g4 < 4; g4++) tmem_ld16(c.tl + 16 * g4, v[g4]);
                tmem_wait_ld();
#pragma unroll
                for (int g4 = 0; g4 < 4; g4++)
#pragma unroll
                    for (int e = 0; e < 16; e++) {
                        const int s = 16 * g4 + e;
                        row[s] = isK ? ((DELTA && s < tt) ? -bet * v[g4][e] : 0.f) : (s <= tt ? v[g4][e] : 0.f);
                    }
            }
            // A_d row trow: segment I's columns (lo .. lo + 16 I) hold the row's values for s < 16 I
            const int lo16 = seg_base(I) >> 4;
#pragma unroll 1
            for (int g4 = 0; g4 < 4; g4++) {
                const int sgrp = 4 * wh + g4 - lo16;   // 16-column group of s this segment group holds
                const bool valid = sgrp >= 0 && sgrp < I;
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    const float x = sgrp == 0 ? row[e] : (sgrp == 1 ? row[16 + e] : row[32 + e]);
                    v[e] = valid ? x : 0.f;
                }
                st16_f16(X + gl::AD + (uint32_t)wh * 16384u, trow, g4, v);
            }
            // near entries (same 16-block), by one of the row's two threads ([2][4][16][20]: float4 rows)
            if (wh == (I >> 1)) {
                float* nd = fptr(X, gl::NEARD) + ((isK * 4 + I) * 16 + (tt & 15)) * 20;
#pragma unroll
                for (int e = 0; e < 16; e++)
                    nd[e] = I == 0 ? row[e] : (I == 1 ? row[16 + e] : (I == 2 ? row[32 + e] : row[48 + e]));
            }
        }
        CB_STAMP(1, 9);
        smem_to_tc();
        if (c.r == 0) {
            // dA1 = A_d B1 (TMEM 192..255): rows 0..63 -> dc, 64..127 -> db (row side)
            const uint32_t ad = smem_u32(X + gl::AD), id10 = idesc_f16(128, 64, false, true);
            mma_tiles(c.tbase + 192, ad, false, 0, 16384, smem_u32(X + gl::B1), true, 8192, 0, 6, id10, false);
            mma_tiles(c.tbase + 192, ad, false, 0, 16384, smem_u32(X + gl::B1L), true, 8192, 0, 6, id10, true);
            // dB1 = A_d^T A1 (TMEM 256..319): rows = segments (column side)
            const uint32_t id11 = idesc_f16(128, 64, true, true);
            mma_tiles(c.tbase + 256, ad, true, 16384, 0, smem_u32(X + gl::A1H), true, 8192, 0, 8, id11, false);
            mma_tiles(c.tbase + 256, ad, true, 16384, 0, smem_u32(X + gl::A1L), true, 8192, 0, 8, id11, true);
            mma_commit(&S.mma);
        }
        CB_STAMP(1, 10);
        // ---- near pairs, reverse (fp32), register-blocked.  Thread = (16-block J, tokens 4 tq .. 4 tq + 3 of the
        // block, channels 4 cg .. 4 cg + 3); a warp's tokens share an 8-half (tq < 2: lower), so every branch is
        // warp-uniform.  Row side (t as row): sums over s of dM[t][s] y_s, column side (t as column): sums over s of
        // dM[s][t] x_s, with y = b / alpha, x = left alpha within an 8-half and the KL / KU factors across the
        // halves, kept in their own sums so that no factor leaves fp32's range.  The near dQ, dK are zero above
        // the diagonal, so no mask is needed: each side takes the two 4-column groups of its own 8-half, and the
        // upper rows (row side) or the lower columns (column side) the two of the other half.
        const int nJ = c.r >> 6, ntq = (c.r >> 4) & 3, ncg = c.r & 15;
        const int nt0 = 16 * nJ + 4 * ntq, nch = 4 * ncg;
        float nc[16], nb[16], ng[16];   // [token ti][channel e] at 4 ti + e
        {
            const float* ND = fptr(X, gl::NEARD);
            const float* NQ = ND + (0 * 4 + nJ) * 16 * 20;
            const float* NK = ND + (1 * 4 + nJ) * 16 * 20;
            const bool up = ntq >= 2;
            const int tl0 = 4 * ntq, sg0 = up ? 2 : 0;
            float ku[4], kl[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                ku[e] = c.KT->KU[nJ][nch + e];
                kl[e] = c.KT->KL[nJ][nch + e];
            }
            if (!S.unsafe) {
                // column side first: its three sums fold into dr at once, so that only dr (not nc, nb) is live
                // through the row side
                float dr[16];
                {
                    float cP[16], cK[16], cX[16];
#pragma unroll
                    for (int e = 0; e < 16; e++) cP[e] = cK[e] = cX[e] = 0.f;
#pragma unroll 1
                    for (int j = 0; j < 2; j++)
                        near_cols_rev<DELTA, false>(NQ, NK, c.ALPHA, sC, sB, tl0, 16 * nJ, sg0 + j, nch, ku, cP, cK);
                    if (!up) {
#pragma unroll 1
                        for (int j = 0; j < 2; j++)
                            near_cols_rev<DELTA, true>(NQ, NK, c.ALPHA, sC, sB, tl0, 16 * nJ, 2 + j, nch, ku, cX, nullptr);
                    }
#pragma unroll
                    for (int ti = 0; ti < 4; ti++) {
                        const int t = nt0 + ti;
                        const float dGa = S.G[t] - S.G[8 * (t >> 3) + 3];
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int k = 4 * ti + e;
                            const float ai = fast_exp2(-S.A2[nch + e] * dGa);
                            const float cx = up ? 0.f : ai * kl[e];   // KL / alpha_t
                            dr[k] = ai * (cP[k] + cK[k]) + cx * cX[k];
                        }
                    }
                }
                {
                    float rP[16], rK[16], rPx[16], rKx[16];
#pragma unroll
                    for (int e = 0; e < 16; e++) rP[e] = rK[e] = rPx[e] = rKx[e] = 0.f;
                    const float* yb = c.YB + 16 * nJ * kAS + nch;
#pragma unroll 1
                    for (int j = 0; j < 2; j++) near_rows_rev<DELTA, false>(NQ, NK, yb, tl0, sg0 + j, kl, rP, rK);
                    if (up) {
#pragma unroll 1
                        for (int j = 0; j < 2; j++) near_rows_rev<DELTA, true>(NQ, NK, yb, tl0, j, kl, rPx, rKx);
                    }
#pragma unroll
                    for (int ti = 0; ti < 4; ti++) {
                        const float4 a4 = *reinterpret_cast<const float4*>(c.ALPHA + (nt0 + ti) * kAS + nch);
                        const float al[4] = {a4.x, a4.y, a4.z, a4.w};
                        float cv[4], bv[4];
                        ld4_bf16(sC, nt0 + ti, nch, cv);
                        ld4_bf16(sB, nt0 + ti, nch, bv);
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int k = 4 * ti + e;
                            const float ax = up ? al[e] * ku[e] : 0.f;   // alpha_t KU
                            nc[k] = al[e] * rP[k] + ax * rPx[k];
                            nb[k] = al[e] * rK[k] + ax * rKx[k];
                            ng[k] = cv[e] * nc[k] + bv[e] * nb[k] - bv[e] * dr[k];
                            nb[k] += dr[k];
                        }
                    }
                }
            } else {
                // every factor evaluated directly (the anchors could overflow); exponents clamped at 0 where the
                // weight is zero anyway
                float rP[16], rK[16], cP[16], cK[16];
#pragma unroll
                for (int e = 0; e < 16; e++) rP[e] = rK[e] = cP[e] = cK[e] = 0.f;
#pragma unroll 1
                for (int sl = 0; sl < 16; sl++) {
                    const int s = 16 * nJ + sl;
                    float c4[4], b4[4];
                    ld4_bf16(sC, s, nch, c4);
                    ld4_bf16(sB, s, nch, b4);
#pragma unroll
                    for (int ti = 0; ti < 4; ti++) {
                        const int t = nt0 + ti;
                        const float wq = NQ[(tl0 + ti) * 20 + sl], wk = DELTA ? NK[(tl0 + ti) * 20 + sl] : 0.f;
                        const float vq = NQ[sl * 20 + tl0 + ti], vk = DELTA ? NK[sl * 20 + tl0 + ti] : 0.f;
                        const float dGr = fmaxf(S.G[t] - S.G[s], 0.f), dGc = fmaxf(S.G[s] - S.G[t], 0.f);
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const float a2 = S.A2[nch + e];
                            const float y = b4[e] * exp2f(a2 * dGr), x = exp2f(a2 * dGc);
                            rP[4 * ti + e] = fmaf(wq, y, rP[4 * ti + e]);
                            rK[4 * ti + e] = fmaf(wk, y, rK[4 * ti + e]);
                            cP[4 * ti + e] = fmaf(vq, c4[e] * x, cP[4 * ti + e]);
                            cK[4 * ti + e] = fmaf(vk, b4[e] * x, cK[4 * ti + e]);
                        }
                    }
                }
#pragma unroll
                for (int ti = 0; ti < 4; ti++) {
                    float cv[4], bv[4];
                    ld4_bf16(sC, nt0 + ti, nch, cv);
                    ld4_bf16(sB, nt0 + ti, nch, bv);
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int k = 4 * ti + e;
                        const float dr = cP[k] + cK[k];
                        nc[k] = rP[k];
                        nb[k] = rK[k] + dr;
                        ng[k] = cv[e] * rP[k] + bv[e] * rK[k] - bv[e] * dr;
                    }
                }
            }
        }
        bar_all();
        CB_STAMP(1, 15);
        if (!mma_wait(c, p, 13)) break;
        CB_STAMP(1, 11);
        // ---- epilogue: dense terms (lanes 0..63), the b-side rows (lanes 64..127), the segments' column side
        float* DC = fptr(X, gl::DC);
        float* DB = fptr(X, gl::DB);
        float* DG = fptr(X, gl::DG);
        float* PB = fptr(X, gl::PB);             // [64][gl::kES] dBhat Bhat, then G_t dGam
        float* SEGv = fptr(X, gl::SEG);          // [96][gl::kES] dB1 h1
        // (delta, b-side rows) K's row tt from the saved front (L2), column-group major, for dbeta below: the loads
        // run under the dense terms
        float4 krow[8];
        if (DELTA && isK) {
            const float4* kr = reinterpret_cast<const float4*>(p.sv + (size_t)q * p.sv_stride + sv::K) + tt;
#pragma unroll
            for (int e = 0; e < 8; e++) krow[e] = kr[(4 * (2 * wh + (e >> 2)) + (e & 3)) * 64];
        }
        if (!isK) {
            const int I = tt >> 4;
            const float Gt = S.G[tt], G63 = S.G[63], Gref = I >= 1 ? S.G[16 * I - 1] : 0.f;
#pragma unroll 1
            for (int h2 = 0; h2 < 2; h2++) {
                const int cg = 2 * wh + h2, c0 = 16 * cg;
                float dct[16], dbh[16], da1[16], cv[16], bv[16];
                tmem_ld16(c.tl + 64 + c0, dct);
                tmem_ld16(c.tl + 128 + c0, dbh);
                tmem_ld16(c.tl + 192 + c0, da1);
                tmem_wait_ld();
                ld16_bf16(sC, tt, cg, cv);
                ld16_bf16(sB, tt, cg, bv);
#pragma unroll
                for (int e4 = 0; e4 < 16; e4 += 4) {
                    float o1[4], o2[4], o3[4], o4[4];
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const int e = e4 + k;
                        const float a2 = S.A2[c0 + e];
                        const float Et = fast_exp2(a2 * Gt), Eh = fast_exp2(a2 * (G63 - Gt));
                        const float f1 = I >= 1 ? fast_exp2(a2 * (Gt - Gref)) : 0.f;
                        o1[k] = dct[e] * Et + da1[e] * f1;
                        o2[k] = dbh[e] * Eh;
                        o3[k] = dct[e] * cv[e] * Et - dbh[e] * bv[e] * Eh + da1[e] * f1 * cv[e];
                        o4[k] = dbh[e] * bv[e] * Eh;
                    }
                    const int at = tt * gl::kES + c0 + e4;
                    *reinterpret_cast<float4*>(DC + at) = make_float4(o1[0], o1[1], o1[2], o1[3]);
                    *reinterpret_cast<float4*>(DB + at) = make_float4(o2[0], o2[1], o2[2], o2[3]);
                    *reinterpret_cast<float4*>(DG + at) = make_float4(o3[0], o3[1], o3[2], o3[3]);
                    *reinterpret_cast<float4*>(PB + at) = make_float4(o4[0], o4[1], o4[2], o4[3]);
                }
            }
        }
        if (DELTA && isK) {
            // the b-side rows' share of db (into DB2; of dGam, b times it), beside the dense terms; and the rest of
            // dbeta, dbeta_t = sum_j dR V - sum_i Btil (dR S^T) - sum_{s<t} (dR U^T) K   (dMm = -dR U^T), whose
            // factors exp(Gam_t) are the same
            float* DB2 = fptr(X, gl::DB2);
            const int I = tt >> 4;
            const float Gt = S.G[tt], Gref = I >= 1 ? S.G[16 * I - 1] : 0.f, bet = S.beta[tt];
            float part = 0.f;
#pragma unroll 1
            for (int h2 = 0; h2 < 2; h2++) {
                const int cg = 2 * wh + h2, c0 = 16 * cg;
                float drs[16], da1[16], dru[16], bv[16], kv[16];
                tmem_ld16(c.tl + 64 + c0, drs);
                tmem_ld16(c.tl + 192 + c0, da1);
                tmem_ld16(c.tl + c0, dru);
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float4 x = h2 ? krow[4 + e] : krow[e];
                    kv[4 * e] = x.x; kv[4 * e + 1] = x.y; kv[4 * e + 2] = x.z; kv[4 * e + 3] = x.w;
                }
                tmem_wait_ld();
                ld16_bf16(sB, tt, cg, bv);
#pragma unroll
                for (int e4 = 0; e4 < 16; e4 += 4) {
                    float ob[4];
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const int e = e4 + k;
                        const float a2 = S.A2[c0 + e];
                        const float Et = fast_exp2(a2 * Gt);
                        const float f1 = I >= 1 ? fast_exp2(a2 * (Gt - Gref)) : 0.f;
                        const float dbt = -bet * drs[e];   // dBtil
                        ob[k] = dbt * Et + da1[e] * f1;
                        part -= bv[e] * Et * drs[e];
                        if (c0 + e < tt) part -= dru[e] * kv[e];
                    }
                    *reinterpret_cast<float4*>(DB2 + tt * gl::kES + c0 + e4) = make_float4(ob[0], ob[1], ob[2], ob[3]);
                }
            }
            S.rs[1][wh][tt] = part;
        }
        bar_all();
        if (c.r < 64) {
            // column sums over tokens of dBhat Bhat (fixed order: four interleaved chains, then their sum)
            S.colsum[0][c.r] = sum64_fixed(PB + c.r, gl::kES);
        }
        // segment rows (TMEM lanes 0..95): dB1[seg][i] times the column factor
        if (trow < 96) {
            const int I = trow < 16 ? 1 : (trow < 48 ? 2 : 3), s = trow - seg_base(I);
            const float Gref = S.G[16 * I - 1], Gs = S.G[s];
            float vb[2][16];   // both column groups in one TMEM round trip
            tmem_ld16(c.tl + 256 + 32 * wh, vb[0]);
            tmem_ld16(c.tl + 256 + 32 * wh + 16, vb[1]);
            tmem_wait_ld();
#pragma unroll
            for (int h2 = 0; h2 < 2; h2++) {
                const int c0 = 32 * wh + 16 * h2;
                const float (&v)[16] = vb[h2];
#pragma unroll
                for (int e4 = 0; e4 < 16; e4 += 4) {
                    float o[4];
#pragma unroll
                    for (int k = 0; k < 4; k++) o[k] = v[e4 + k] * fast_exp2(S.A2[c0 + e4 + k] * (Gref - Gs));
                    *reinterpret_cast<float4*>(SEGv + trow * gl::kES + c0 + e4) = make_float4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        bar_all();
        CB_STAMP(1, 12);
        // ---- gather, thread = (tokens nt0 .. nt0 + 3, channels nch .. nch + 3) as in the near pass: dc, db out;
        // dGam -> dG (summed over the sixteen channel groups of a token by shuffles in the half-warp), dA
        {
#pragma unroll
            for (int ti = 0; ti < 4; ti++) {
                const int t = nt0 + ti;
                float bv4[4];
                ld4_bf16(sB, t, nch, bv4);
                float dcv[4], dbv[4], pbv[4], gsum = 0.f;
                // this thread's four channels of the row's arrays (float4), the segments' shares summed in I order
                float sg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int I = 1; I <= 3; I++)
                    if (t < 16 * I) {
                        const float4 x = *reinterpret_cast<const float4*>(SEGv + (seg_base(I) + t) * gl::kES + nch);
                        sg[0] += x.x; sg[1] += x.y; sg[2] += x.z; sg[3] += x.w;
                    }
                const float4 c4 = *reinterpret_cast<const float4*>(DC + t * gl::kES + nch);
                const float4 b4 = *reinterpret_cast<const float4*>(DB + t * gl::kES + nch);
                const float4 g4 = *reinterpret_cast<const float4*>(DG + t * gl::kES + nch);
                const float4 k4 = DELTA ? *reinterpret_cast<const float4*>(fptr(X, gl::DB2) + t * gl::kES + nch)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                const float dcr[4] = {c4.x, c4.y, c4.z, c4.w}, dbr[4] = {b4.x, b4.y, b4.z, b4.w};
                const float dgr[4] = {g4.x, g4.y, g4.z, g4.w}, dbk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int i = nch + e, k = 4 * ti + e;
                    const float seg = sg[e];
                    dcv[e] = dcr[e] + nc[k];
                    dbv[e] = dbr[e] + dbk[e] + seg + nb[k];
                    float gam = dgr[e] + bv4[e] * dbk[e] - bv4[e] * seg + ng[k];
                    if (t == 63) {
                        const float sdi = S.sd[0][i] + S.sd[1][i] + S.sd[2][i] + S.sd[3][i];
                        gam += S.colsum[0][i] + sdi * c.KT->EC[i];
                    }
                    pbv[e] = S.G[t] * gam;
                    gsum = fmaf(S.A2[i], gam, gsum);
                }
                *reinterpret_cast<float4*>(PB + t * gl::kES + nch) = make_float4(pbv[0], pbv[1], pbv[2], pbv[3]);
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
                if (ncg == 0) S.dgp[0][t] = gsum / kLog2e;   // dG_t (A = A2 / log2 e)
                if (t < L && nch < p.dk) {
                    const size_t base = ((size_t)bb * p.T + t0 + t) * p.H + h;
                    uint2 w;
                    w.x = pack_bf16(dcv[0], dcv[1]);
                    w.y = pack_bf16(dcv[2], dcv[3]);
                    *reinterpret_cast<uint2*>(p.dc + base * p.dk + nch) = w;
                    w.x = pack_bf16(dbv[0], dbv[1]);
                    w.y = pack_bf16(dbv[2], dbv[3]);
                    *reinterpret_cast<uint2*>(p.db + base * p.dk + nch) = w;
                }
            }
        }
        bar_all();
        if (c.warp == 0) {
            // dg = reverse cumulative sum of dG over the chunk's tokens
            float a = 0.f, b = 0.f;
            const int t2 = 2 * c.lane;
            a = S.dgp[0][t2];
            b = S.dgp[0][t2 + 1];
            // suffix sums: x = a + b per lane, scan from the top
            float x = a + b;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, x, o);
                if (c.lane + o < 32) x += y;
            }
            const float after = __shfl_down_sync(0xffffffffu, x, 1);   // sum over pairs above this lane
            const float tail = c.lane < 31 ? after : 0.f;
            const float dg1 = b + tail, dg0 = a + dg1;
            if (t2 < L) p.dg[((size_t)bb * p.T + t0 + t2) * p.H + h] = __float2bfloat16_rn(dg0);
            if (t2 + 1 < L) p.dg[((size_t)bb * p.T + t0 + t2 + 1) * p.H + h] = __float2bfloat16_rn(dg1);
        } else if (c.r >= 64 && c.r < 128) {
            // dA partial: sum_t G_t dGam_t[i] (fixed order: four interleaved chains, then their sum)
            const int i = c.r - 64;
            p.dA_part[(size_t)q * 64 + i] = sum64_fixed(PB + i, gl::kES);
        } else if (DELTA && c.r >= 128 && c.r < 192) {
            // dbeta of the chunk's tokens (both column halves of every part)
            const int tq = c.r - 128;
            if (tq < L) {
                const float db_ = S.rs[0][0][tq] + S.rs[0][1][tq] + S.rs[1][0][tq] + S.rs[1][1][tq];
                p.dbeta[((size_t)bb * p.T + t0 + tq) * p.H + h] = __float2bfloat16_rn(db_);
            }
        }
        CB_STAMP(1, 13);
        // the stage is free: the next chunk's loads
        tc_fence_before();
        bar_all();
        tc_fence_after();
        if (q + (int)gridDim.x < p.nq) {
            if (c.r == 0) {
                issue_tma(p, S, c.sm, q + gridDim.x);
                if (use_sv) issue_saved<DELTA>(p, S, c.sm, q + gridDim.x);
            }
            pending = q + gridDim.x;
            if (use_sv) pending2 = q + gridDim.x;
        }
        CB_STAMP(1, 14);
#ifdef GDN_CHUNK_DEBUG
        if (c.r == 0 && blockIdx.x == 0) g_cb_stamps[1][31] += 1;
#endif
    }
    teardown(c, p, pending, full_phase, pending2, full2_phase);
}

// dA_log[h][i] = A[h][i] sum over batch rows and chunks of the chunk partials, in a fixed order: 1024 threads per
// head, thread (lane group g = threadIdx.x >> 6, channel i) sums the (batch, chunk) pairs n with n mod 16 = g in
// order, then the sixteen group sums are added in group order
constexpr int kDalogGroups = 16;
__global__ void __launch_bounds__(64 * kDalogGroups) chunk_dalog_kernel(const float* __restrict__ part,
                                                                        const float* __restrict__ A_log,
                                                                        float* __restrict__ dA_log, int B, int H,
                                                                        int dk, int nchunks)
{
    __shared__ float grp[kDalogGroups][64];
    const int h = blockIdx.x, i = threadIdx.x & 63, g = threadIdx.x >> 6;
    const int n_all = B * nchunks;
    float acc = 0.f;
#pragma unroll 4
    for (int n = g; n < n_all; n += kDalogGroups) {
        const int bb = n / nchunks, k = n - bb * nchunks;
        acc += part[(((size_t)bb * H + h) * nchunks + k) * 64 + i];
    }
    grp[g][i] = acc;
    __syncthreads();
    if (g == 0 && i < dk) {
        float sum = grp[0][i];
#pragma unroll
        for (int e = 1; e < kDalogGroups; e++) sum += grp[e][i];
        dA_log[h * dk + i] = -expf(A_log[h * dk + i]) * sum;
    }
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// ---------------------------------------------------------------- host side
cudaError_t launch_chunk_bwd(const Args& a, const WsLayout& Lw, cudaStream_t st)
{
    CbParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_v, a.v, a.B, a.T, a.H, a.dv) || !make_map(&p.tm_b, a.b, a.B, a.T, a.H, a.dk) ||
        !make_map(&p.tm_c, a.c, a.B, a.T, a.H, a.dk) || !make_map(&p.tm_do, a.dO, a.B, a.T, a.H, a.dv))
        return cudaErrorInvalidValue;
    unsigned char* ws = (unsigned char*)a.ws;
    p.g = (const __nv_bfloat16*)a.g;
    p.beta = (const __nv_bfloat16*)a.beta;
    p.A_log = a.A_log;
    p.phi = ws + Lw.cb_phi_off;
    p.sv = ws + Lw.cb_sv_off;
    p.dlt = (float*)(ws + Lw.cb_dlt_off);
    p.ych = (float*)(ws + Lw.cb_y_off);
    p.ec = (float*)(ws + Lw.cb_ec_off);
    p.st = (float*)(ws + Lw.cb_st_off);
    p.dst = (float*)(ws + Lw.cb_dst_off);
    p.dA_part = (float*)(ws + Lw.cb_da_off);
    p.h0 = a.h0;
    p.dhT = a.dhT;
    p.dh0 = a.dh0;
    p.dv = (__nv_bfloat16*)a.dv_;
    p.db = (__nv_bfloat16*)a.db;
    p.dc = (__nv_bfloat16*)a.dc;
    p.dg = (__nv_bfloat16*)a.dg;
    p.dbeta = (__nv_bfloat16*)a.dbeta;
    p.status = (uint32_t*)a.ws;
    p.B = a.B; p.H = a.H; p.T = a.T; p.dk = a.dk; p.dv_ = a.dv;
    p.nchunks = (a.T + 63) / 64;
    p.nq = a.B * a.H * p.nchunks;
    p.sv_stride = a.mode == GDN_DELTA ? sv::BYTES : sv::GATED_BYTES;
    p.nseg = chain_segments(a.mode, a.B * a.H, p.nchunks, a.saved ? 1 : 2, &p.seg_len);
    p.segrec = (float*)(ws + Lw.cb_seg_off);
    p.tvec = (float*)(ws + Lw.cb_tvec_off);
    if (a.saved) {
        // residuals of a saving forward: the entering states, then the solve's results (gated: P)
        p.st = (float*)a.saved;
        p.sv = (unsigned char*)a.saved + (size_t)p.nq * 16384;
        p.rev_only = 1;
    }
    p.starve = test_starve_chunk();
    p.wait_ns = p.starve >= 0 ? kTestWaitNs : kWaitNs;
    const bool delta = a.mode == GDN_DELTA;
    constexpr uint32_t prep_bytes = OFF_X + pl::BYTES + 1024, grad_bytes = OFF_X + gl::BYTES + 1024;
    static bool attr = false;
    if (!attr) {
        cudaError_t e;
        if ((e = set_smem(chunk_prep_kernel<true>, prep_bytes)) != cudaSuccess) return e;
        if ((e = set_smem(chunk_prep_kernel<false>, prep_bytes)) != cudaSuccess) return e;
        if ((e = set_smem(chunk_grad_kernel<true>, grad_bytes)) != cudaSuccess) return e;
        if ((e = set_smem(chunk_grad_kernel<false>, grad_bytes)) != cudaSuccess) return e;
        if ((e = set_smem(chunk_chain_tc_kernel, CHAIN_TC_SMEM)) != cudaSuccess) return e;
        if ((e = set_smem(chunk_prep_saved_kernel, ps::SMEM)) != cudaSuccess) return e;
        if ((e = set_smem(chunk_chain_walk_kernel<false>, walk_smem(false))) != cudaSuccess) return e;
        if ((e = set_smem(chunk_chain_walk_kernel<true>, walk_smem(true))) != cudaSuccess) return e;
        attr = true;
    }
    int sms = 152;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int grid = p.nq < sms ? p.nq : sms;
#ifdef GDN_CHUNK_DEBUG
#define CB_MARK(what) fprintf(stderr, "[chunk bwd] %s: %s\n", what, cudaGetErrorString(cudaStreamSynchronize(st)))
#else
#define CB_MARK(what)
#endif
    CB_MARK("start");
    if (a.saved) {
        // from the residuals: delta Phi and Y; gated Y and the chunks' decays E alone
        CbParams pg = p;
        pg.gated = !delta;
        chunk_prep_saved_kernel<<<p.nq < 3 * sms ? p.nq : 3 * sms, 256, ps::SMEM, st>>>(pg);
    } else if (delta) chunk_prep_kernel<true><<<grid, kThreads, prep_bytes, st>>>(p);
    else chunk_prep_kernel<false><<<grid, kThreads, prep_bytes, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CB_MARK("prep");
    const int units = a.B * a.H;
    const int dirs = p.rev_only ? 1 : 2;
    if (delta && (p.nseg > 1 || dirs * units <= 2 * sms)) {
        // the chain as walks: the two sweeps side by side; split in time, a first walk per segment and a scan
        if (p.nseg > 1) {
            chunk_chain_walk_kernel<true><<<dim3(units, p.nseg - 1, dirs), CT_THREADS, walk_smem(true), st>>>(p);
            chunk_walk_scan_kernel<<<dim3(units, 8, dirs), 256, 0, st>>>(p);
        }
        chunk_chain_walk_kernel<false><<<dim3(units, p.nseg, dirs), CT_THREADS, walk_smem(false), st>>>(p);
    } else if (delta) {
        chunk_chain_tc_kernel<<<units, CT_THREADS, CHAIN_TC_SMEM, st>>>(p);
    } else if (p.nseg > 1) {
        // gated, split in time: local walks per segment, an elementwise scan, the records' fix-up
        chunk_chain_gated_seg_kernel<<<dim3(units, p.nseg, dirs), 256, 0, st>>>(p);
        chunk_gated_scan_kernel<<<dim3(units, dirs), 256, 0, st>>>(p);
        chunk_gated_fix_kernel<<<dim3(p.nq, dirs), 256, 0, st>>>(p);
    } else {
        chunk_chain_gated_kernel<<<units, 256, 0, st>>>(p);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CB_MARK("chain");
    if (delta) chunk_grad_kernel<true><<<grid, kThreads, grad_bytes, st>>>(p);
    else chunk_grad_kernel<false><<<grid, kThreads, grad_bytes, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CB_MARK("grad");
    chunk_dalog_kernel<<<a.H, 64 * kDalogGroups, 0, st>>>(p.dA_part, a.A_log, a.dA_log, a.B, a.H, a.dk, p.nchunks);
    return cudaGetLastError();
}

// The forward split in time by walks (fwd_walks_apply): the zero-start saving run over the segment view, Phi per
// chunk, the transition walks, the scan over segments (with h_T), the walks of D = T_k S_s, the fix-up.  The
// residuals go to a.saved (a saving forward, made true by the fix-up) or to the workspace.
cudaError_t launch_fwd_walks(const Args& a, const WsLayout& Lw, cudaStream_t st)
{
    unsigned char* ws = (unsigned char*)a.ws;
    unsigned char* res = a.saved ? (unsigned char*)a.saved : ws + Lw.fw_res_off;
    float* Xb = (float*)(ws + Lw.ts_h_off);
    float* o32 = (float*)(ws + Lw.ts_o_off);
    gdn_shape_t sh = {a.B, a.H, a.T, a.dk, a.dv, a.mode, a.io};
    int L = 0;
    const int P = fwd_walk_split(sh, a.logits, a.norm, &L);
    const int nk = (a.T + 63) / 64, units = a.B * a.H;
    if (P < 2) return cudaErrorInvalidValue;
    // 1. every segment from a zero state, keeping the residuals (states entering the chunks, from zero)
    Args r = a;
    r.h0 = nullptr;
    r.hT = Xb;
    r.o32 = o32;
    r.saved = res;
    r.seg = P;
    r.seg_len = L;
    r.save_lite = a.saved ? 0 : 1;   // without a caller's residuals the walks need P and -W alone
    bool handled = false;
    cudaError_t e = launch_fwd_tc(r, st, &handled);
    if (e != cudaSuccess) return e;
    if (!handled) return cudaErrorInvalidValue;

    CbParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_b, a.b, a.B, a.T, a.H, a.dk) || !make_map(&p.tm_c, a.c, a.B, a.T, a.H, a.dk))
        return cudaErrorInvalidValue;
    p.g = (const __nv_bfloat16*)a.g;
    p.beta = (const __nv_bfloat16*)a.beta;
    p.A_log = a.A_log;
    p.phi = ws + Lw.cb_phi_off;
    p.sv = res + (size_t)units * nk * kSavedStateBytes;
    p.st = (float*)(ws + Lw.fw_d_off);   // the second walk's records D
    p.gated = a.mode == GDN_GATED;
    p.status = (uint32_t*)a.ws;
    p.B = a.B; p.H = a.H; p.T = a.T; p.dk = a.dk; p.dv_ = a.dv;
    p.nchunks = nk;
    p.nq = units * nk;
    p.sv_stride = (uint32_t)saved_solve_bytes(a.mode);
    p.nseg = P;
    p.seg_len = L;
    p.segrec = (float*)(ws + Lw.cb_seg_off);
    p.fwd_walks = 1;
    p.fw_o32 = o32;
    p.fw_o = (__nv_bfloat16*)a.o;
    p.fw_st = a.saved ? (float*)a.saved : nullptr;
    p.starve = -1;
    p.wait_ns = kWaitNs;
    static bool attr = false;
    if (!attr) {
        if ((e = set_smem(chunk_prep_saved_kernel, ps::SMEM)) != cudaSuccess) return e;
        if ((e = set_smem(fwd_walk_kernel<false>, FW_SMEM)) != cudaSuccess) return e;
        if ((e = set_smem(fwd_walk_kernel<true>, FW_SMEM)) != cudaSuccess) return e;
        if ((e = set_smem(fwd_walk_res_kernel, fx::SMEM)) != cudaSuccess) return e;
        attr = true;
    }
    int sms = 152;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int grid3 = p.nq < 3 * sms ? p.nq : 3 * sms;
    // 2. Phi and Qc of every chunk
    chunk_prep_saved_kernel<<<grid3, 256, ps::SMEM, st>>>(p);
    // 3. each segment's transition
    fwd_walk_kernel<false><<<dim3(units, P), fw_threads(false), FW_SMEM, st>>>(p);
    // 4. the segments' true starting states, and h_T
    fwd_walk_scan_kernel<<<dim3(units, 8), 256, 0, st>>>(p, Xb, a.h0, a.hT);
    // 5. D = T_k S_s through every segment, and the outputs o = o_zero-start + Qc D
    fwd_walk_kernel<true><<<dim3(units, P), fw_threads(true), FW_SMEM, st>>>(p);
    // 6. a saving forward's residuals made true
    if (a.saved) fwd_walk_res_kernel<<<grid3, 256, fx::SMEM, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn

#ifdef GDN_CHUNK_DEBUG
extern "C" int gdn_chunk_debug_stamps(unsigned long long* out, int clear)
{
    if (cudaMemcpyFromSymbol(out, gdn::g_cb_stamps, sizeof(gdn::g_cb_stamps)) != cudaSuccess) return 1;
    if (clear) {
        static const unsigned long long zero[3][32] = {};
        if (cudaMemcpyToSymbol(gdn::g_cb_stamps, zero, sizeof(zero)) != cudaSuccess) return 1;
    }
    return 0;
}
#endif
