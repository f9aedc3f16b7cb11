// gdn_fwd_tc.cu -- chunked forward of the gated delta rule on tcgen05 tensor
// cores, both modes (bf16 I/O, fp32 accumulation, fp32 state).
//
// "GDN & MLA Mechanism Deep-Dive", Step 5 (Chunked recurrence): chunks of
// C = 64 tokens are solved in closed form with 64 x 64 matrices and the state
// is carried serially from chunk to chunk.  Per (b, h) and chunk, with
// G_t = sum_{r<=t} g_r (inclusive, restarted per chunk), Gam_t[i] = A[i] G_t
// and S the state entering the chunk:
//   P[t,s] = sum_i c_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])            (s <= t)
//   Ctil_t = c_t (.) exp(Gam_t),  Bhat_s = b_s (.) exp(Gam_63 - Gam_s)
// gated ("GDN & MLA Mechanism Deep-Dive", Step 4):   U = V
// delta ("HyMo-434M -- documentation portal", card 01): with
//   M[t,s] = beta_t sum_i b_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])     (s < t),
//   Btil_t = b_t (.) exp(Gam_t), the written values solve
//   (I + M) U = diag(beta) (V - Btil S) = Util - W S
// and then   O = Ctil S + P U,   S' = exp(Gam_63) (.)rows S + Bhat^T U.
//
// Decay split.  exp(Gam_t - Gam_s) is factored into a row and a column factor
// around a reference point r between s and t, so no factor overflows (|A| up
// to 16 over a chunk reaches exp(+-1024)); secondary chunking after Yang et al.
// 2023 (Gated Linear Attention):
//   L1  different 16-blocks: r = last token before the row block; the three
//       row blocks' column operands (16, 32, 48 rows) form one N = 96 MMA;
//       factors <= 1;
//   L2  same 16-block, row in the upper and column in the lower 8-half:
//       r = last token of the lower half; factors <= 1;
//   L3  same 8-block: r = the block's 4th token; factors up to
//       exp(|A| * (sum of 4 g)).
// Every factor is an "anchor" exp(A (G_t - G_r8(t))) (its inverse for
// columns) times a per-(8-block, reference) constant <= 1, so a chunk costs
// two exponentials per (token, channel) plus the shared constants.  A
// per-chunk check (|A| log2(e) * span <= 100) guarantees finite anchors; when
// it fails every factor is evaluated directly and the L3 entries elementwise
// in fp32.
//
// Delta solve (WY form): D, the two 32x32 diagonal blocks of I + M, is
// inverted in fp32: its 16x16 diagonal blocks by forward substitution, and
// each 32-block [[A, 0], [C, B]] as [[A^-1, 0], [-B^-1 C A^-1, B^-1]].  With
// L = I + M - D (rows 32..63, columns 0..31 only), N = D^{-1} L has N^2 = 0, so
//   (I + M)^{-1} R = (I - N) D^{-1} R,   R = [beta V | beta Btil]
// as [N | X0] = D^{-1}[L | R], then [Util | W] = X0 - N X0 (X0 kept exactly in
// TMEM as the accumulator start).
//
// Precision: the L1/L2 operands (factors <= 1) are fp16; L3, P, Bhat^T, the
// state and, in delta mode, R, X0 and U enter their MMAs as bf16 hi + lo
// pairs (hi*hi + hi*lo + lo*hi); D^{-1}, L, N, W, Ctil are plain bf16.
//
// CTA = one (b, h), 8 warps (thread r <-> TMEM lane r & 127; warps w and
// w + 4 share a lane quarter and split the columns).  Thread 0 issues the MMAs
// and the TMA loads of v, b, c (128 B swizzle, zero fill past T and d) into a
// 2-stage ring: the load of chunk k + 2 goes out as soon as chunk k's last MMA
// has finished with its stage.  Threads 0..63 fetch g (and beta) one chunk
// ahead into registers.  The kernel is latency-bound, so independent work runs
// where warps would wait: chunk k's state update and output stores under
// chunk k+1's level products, chunk k+1's scan of g and decay constants on
// warps 2, 3, 6, 7 (the schedulers the critical path leaves free) under chunk
// k's diagonal-block inverse (delta) or output product (gated), and (delta)
// the Ctil rows of [-W ; Ctil] under the W products.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdlib.h>

#include "fwd_tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace fwdtc;

constexpr int kStages = 2;
constexpr int kMath = 256;
constexpr int kThreads = kMath;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_RING = 0;
constexpr uint32_t STAGE_BYTES = 3 * 8192;
constexpr uint32_t OFF_X = kStages * STAGE_BYTES;      // reused phase by phase (100 KB)
//   phase 1: the three decay levels (rows 0..63 c-side, rows 64..127 beta b-side)
constexpr uint32_t X_A1 = 0, X_B1a = 16384, X_B1b = 18432, X_B1c = 22528;
constexpr uint32_t X_A2 = 28672, X_B2 = 45056, X_A3 = 53248, X_A3L = 69632, X_B3 = 86016, X_B3L = 94208;
//   gated, after the levels: [0 ; Ctil]
constexpr uint32_t X_CH1 = 0;
//   delta phase 2: [N | X0] = Dinv [L | R], Dinv the inverse of the diagonal 32-blocks; fp32 staging of the
//   diagonal 16-blocks (M32), their inverses (DI32), the 16-blocks below them (C32) and the inverses' coupling
//   blocks (E32)
constexpr uint32_t X_DINV = 0, X_LRH = 16384, X_LRL = 40960;
constexpr uint32_t X_M32 = 57344, X_DI32 = 62464, X_C32 = 67584, X_E32 = 70144;
// fp32 16x16 blocks with a padded row stride (conflict-free float4 rows)
constexpr int kBS = 20;
//   delta phase 3: [Util | W] = X0 - N X0 (A = -N; X0 as hi/lo B blocks)
constexpr uint32_t X_NA = 0, X_X0H = 24576, X_X0L = 40960;
//   delta phase 4: the state products
//   (CW sits past the phase-3 operands so that its Ctil rows can be built while the phase-3 products run)
constexpr uint32_t X_CW = 57344, X_UH = 16384, X_UL = 24576;
constexpr uint32_t X_BYTES = 102400;
constexpr uint32_t OFF_CH0 = OFF_X + X_BYTES;          // [Bhat^T ; P] hi
constexpr uint32_t OFF_CH0L = OFF_CH0 + 16384;         // [Bhat^T ; P] lo
constexpr uint32_t OFF_S = OFF_CH0L + 16384;           // state bf16 [i][j], hi
constexpr uint32_t OFF_SL = OFF_S + 8192;              // state, lo
constexpr uint32_t OFF_K = OFF_SL + 8192;              // decay constants, 8 tables x [8][64] fp32
constexpr uint32_t OFF_SMALL = OFF_K + 16384;
constexpr uint32_t SMEM_BYTES = OFF_SMALL + 4096 + 1024;

// decay-constant tables (all entries <= 1), indexed [table][8-block][channel]
enum { K_A1 = 0, K_A2, K_0, K_B1_1, K_B1_2, K_B1_3, K_B2, K_BH };

// TMEM columns
constexpr uint32_t TM_D1a = 0, TM_D1b = 16, TM_D1c = 48, TM_D2 = 96, TM_D3 = 160;
constexpr uint32_t TM_CHG = 256;                       // gated: [dS ; O]
constexpr uint32_t TM_NX = 256;                        // delta: [N | X0V | X0W]
constexpr uint32_t TM_U = TM_NX + 64;                  // delta: X0V -> Util, then [U ; Ctil S]
constexpr uint32_t TM_W = TM_NX + 128;                 // delta: X0W -> W
constexpr uint32_t TM_CHD = TM_NX + 128;               // delta: [dS ; P U] (W is consumed by then)
constexpr uint32_t TM_COLS = 512;

struct Small {
    float G[2][64];         // inclusive scan of g within the chunk, by chunk parity
    float A2[64];
    float decay[2][64];     // exp(Gam_63) of the chunk, by chunk parity (read by the chunk's deferred epilogue)
    float g[kStages][64];
    float beta[kStages][64];
    float nb[64], nc[64];   // GDN_NORM_BC: 1 / max(||b_t||, floor), the same for c_t, of the current chunk
    uint64_t full[kStages], mma;
    uint32_t tmem_base;
    uint32_t unsafe[2];     // the chunk's anchors could overflow, by chunk parity
    uint32_t abort;
    float a2max;
};
static_assert(sizeof(Small) <= 4096, "the small-state block has a 4 KB slot");

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

__device__ __forceinline__ void st_split16(unsigned char* thi, unsigned char* tlo, int row, int col16,
                                           const float (&v)[16])
{
    float a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; k++) { a[k] = v[k]; b[k] = v[8 + k]; }
    st_row8_split(thi, tlo, row, 2 * col16, a);
    st_row8_split(thi, tlo, row, 2 * col16 + 1, b);
}

__device__ __forceinline__ void st_plain16(unsigned char* t, int row, int col16, const float (&v)[16])
{
    float a[8], b[8];
#pragma unroll
    for (int k = 0; k < 8; k++) { a[k] = v[k]; b[k] = v[8 + k]; }
    st_row8(t, row, 2 * col16, a);
    st_row8(t, row, 2 * col16 + 1, b);
}

__device__ __forceinline__ void zero_chunk(unsigned char* tile, int row, int q)
{
    *reinterpret_cast<uint4*>(tile + sw128(row, 8 * q)) = make_uint4(0, 0, 0, 0);
}

// The residuals a saving forward writes for the chunked backward (gdn_chunk_bwd.cu reads them with the same
// layout), per chunk q = unit * nchunks + k.  p.st: the state S entering the chunk, fp32 64 x 64 (rows = key
// channel, columns = value column).  p.sv, byte offsets in a chunk's record: P as hi, lo tiles; -N and Dinv (bf16
// tiles, the upper halves of the stacked solve operands); K (zero on and above the diagonal), fp32 64 x 64; -W as
// hi, lo tiles ([t][i]); U = Util - W S, fp32 [t][j].  Tiles are [64][64] 16-bit with the 128-byte swizzle of the
// MMA operands; the fp32 matrices are column-group major (row r, columns 4 g .. 4 g + 3 at float4 64 g + r), so a
// warp's 32 rows store 512 contiguous bytes.  Gated mode keeps the state and P only (a 16 KB record).
namespace svr {
constexpr uint32_t P = 0, NA = 16384, DINV = 24576, K = 32768, NW = 49152, NWL = 57344, U = 65536, BYTES = 81920;
constexpr uint32_t GATED_BYTES = 16384;   // gated: P only
// the record index of chunk k of unit u: u * nchunks + k, or, for the segments of a time split (SEG: unit
// u = (b * seg + s) * H + h runs chunks s * seg_len .. of (b, h)), the index of that chunk in the whole sequence
template <bool SEG>
__device__ __forceinline__ size_t rec_index(const TcParams& p, int u, int k)
{
    if (!SEG) return (size_t)u * p.nchunks + k;
    const int bs = u / p.H, h = u - bs * p.H, b = bs / p.seg, s = bs - b * p.seg;
    return ((size_t)b * p.H + h) * p.nchunks + (size_t)s * p.seg_len + k;
}
template <bool SEG>
__device__ __forceinline__ unsigned char* rec(const TcParams& p, int u, int k)
{
    return p.sv + rec_index<SEG>(p, u, k) * p.sv_stride;
}
// state row `row`, columns 32 wh .. 32 wh + 31; the record is column-group major (the float4 of row r, columns
// 4 g .. 4 g + 3 at index 64 g + r), so a warp's 32 rows write 512 contiguous bytes
template <bool SEG>
__device__ __forceinline__ void put_state(const TcParams& p, int u, int k, int row, int wh, const float (&v)[32])
{
    float4* d = reinterpret_cast<float4*>(p.st + rec_index<SEG>(p, u, k) * 4096) + (8 * wh) * 64 + row;
#pragma unroll
    for (int e = 0; e < 8; e++) d[64 * e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
}
}  // namespace svr

// D[d] (+)= A x B over K = 64 (four K = 16 steps); A K-major, B K- or MN-major
__device__ __forceinline__ void mma_k64(uint32_t d, uint32_t a, uint32_t b, bool b_mn, uint32_t idesc, bool acc)
{
#pragma unroll
    for (int ks = 0; ks < 4; ks++)
        mma_bf16(d, sdesc(a + ks * 32, 16, 1024), sdesc(b + (b_mn ? ks * 2048 : ks * 32), 8192, 1024), idesc,
                 (acc || ks > 0) ? 1u : 0u);
}

__device__ __forceinline__ const float* ktab(const unsigned char* sm, int tab, int k8)
{
    return reinterpret_cast<const float*>(sm + OFF_K) + (tab * 8 + k8) * 64;
}

// What a forward keeps for the chunked backward: nothing; the residuals of one pass; those of a time split's
// segment view (laid out by the chunks of the whole sequence); or only P and -W of them (what the split's walks read)
enum SaveMode { SAVE_NONE = 0, SAVE_FULL = 1, SAVE_SPLIT = 2, SAVE_SPLIT_LITE = 3 };

// NORM: b and c arrive before their L2 normalisation (a template flag, so the plain kernel carries no trace of it).
// SAVE (one 64-column slab; a SaveMode): the residuals of the chunked backward are written as well, per chunk q of
// the unit:
// the entering state (p.st, fp32 64 x 64, column-group major) and, in the layout of namespace svr, the delta
// solve's results (gated: P).  In delta mode the b-side level operands then leave beta out, so that the level
// products give K itself (M = beta K is formed when it is assembled).
template <bool DELTA, bool NORM, int SAVEM>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ TcParams p)
{
    constexpr bool SAVE = SAVEM != SAVE_NONE;
    constexpr bool LITE = SAVEM == SAVE_SPLIT_LITE;                        // P and -W only
    constexpr bool SEG = SAVEM == SAVE_SPLIT || SAVEM == SAVE_SPLIT_LITE;  // records of the whole sequence
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X = sm + OFF_X;
    Small& S = *reinterpret_cast<Small*>(sm + OFF_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u = blockIdx.x;
    // the unit's (batch, head) and its chunks: all of them, or (SEG) segment s of a time split, chunks
    // kbase .. kbase + nck - 1 of the sequence (the last segment may be shorter, its last chunk ragged)
    int bb, h, kbase = 0, nck = p.nchunks;
    if constexpr (SEG) {
        const int bs = u / p.H, sgi = bs % p.seg;
        h = u - bs * p.H;
        bb = bs / p.seg;
        kbase = sgi * p.seg_len;
        nck = min(p.seg_len, p.nchunks - kbase);
    } else {
        bb = u / p.H;
        h = u % p.H;
    }
    const int T = p.T, H = p.H, dk = p.dk, dv = p.dv;
    // value columns jc0 .. jc0 + nv - 1 of the unit (columns of the state never mix, so wider values are
    // split in 64-column slabs over blockIdx.y; the slabs repeat the decay and solve work of the keys)
    const int jc0 = 64 * (int)blockIdx.y, nv = min(64, dv - jc0);

    if (tid < 64) {
        const float A = tid < dk ? -expf(p.A_log[h * dk + tid]) : 0.f;
        S.A2[tid] = A * kLog2e;
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) mbar_init(&S.full[s], 1);
        mbar_init(&S.mma, 1);
        S.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&S.tmem_base, TM_COLS);
    if (tid == 0) {
        tma_prefetch_desc(&p.tm_v); tma_prefetch_desc(&p.tm_b); tma_prefetch_desc(&p.tm_c);
    }
    // g (and beta) of the first chunks
    for (int k = 0; k < kStages; k++)
        if (tid < kC) {
            const int t = (kbase + k) * kC + tid;
            const size_t row = ((size_t)bb * T + t) * H + h;
            S.g[k][tid] = t < T ? gate_in(__bfloat162float(p.g[row]), p.logits) : 0.f;
            if (DELTA) S.beta[k][tid] = t < T ? gate_in(__bfloat162float(p.beta[row]), p.logits) : 0.f;
        }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        float m = 0.f;
        for (int i = 0; i < 64; i++) m = fmaxf(m, fabsf(S.A2[i]));
        S.a2max = m;
    }
    const uint32_t tbase = S.tmem_base;
    auto issue_load = [&](int k) {   // thread 0: TMA of chunk k into its stage
        if (k == p.starve_chunk) return;   // failure-path test hook: this stage never fills
        const int s = k % kStages;
        unsigned char* st = sm + OFF_RING + s * STAGE_BYTES;
        mbar_arrive_expect_tx(&S.full[s], STAGE_BYTES);
        tma_load_4d(st, &p.tm_v, &S.full[s], jc0, h, (kbase + k) * kC, bb);
        tma_load_4d(st + 8192, &p.tm_b, &S.full[s], 0, h, (kbase + k) * kC, bb);
        tma_load_4d(st + 16384, &p.tm_c, &S.full[s], 0, h, (kbase + k) * kC, bb);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < kStages && issued < nck; issued++) issue_load(issued);

    {
        // ---------------------------------------------------------- math
        const int r = tid;                       // 0..255
        const int q4 = warp & 3, wh = warp >> 2;  // TMEM lane quarter, column half
        const int trow = r & 127;                // TMEM lane / accumulator row
        const uint32_t tl = tbase + ((uint32_t)(q4 * 32) << 16);
        const bool state_row = q4 < 2;           // rows 0..63 of the accumulators
        float Sreg[32];                          // state row trow, columns 32 wh .. 32 wh + 31
        if (state_row) {
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const int jj = 32 * wh + j;
                Sreg[j] = (p.h0 && trow < dk && jj < nv) ? p.h0[((size_t)u * dk + trow) * dv + jc0 + jj] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float v8[8];
#pragma unroll
                for (int e = 0; e < 8; e++) v8[e] = Sreg[8 * q + e];
                st_row8_split(sm + OFF_S, sm + OFF_SL, trow, 4 * wh + q, v8);
            }
            if (SAVE && !LITE) svr::put_state<SEG>(p, u, 0, trow, wh, Sreg);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kMath);
        // (15) chunk kk's state update (lanes 0..63) and output (lanes 64..127), 32 columns per thread.  It runs
        // while the next chunk's level products execute (they write TMEM columns 0..223 and read the operand
        // region; this reads the output columns and writes the state tiles, which only the tail products read).
        auto epilogue = [&](int kk) {
            const uint32_t tm_out = DELTA ? TM_CHD : TM_CHG;
            if (state_row) {
                const float dec = S.decay[kk & 1][trow];
#pragma unroll
                for (int cc = 0; cc < 2; cc++) {
                    float v[16];
                    tmem_ld16(tl + tm_out + 32 * wh + 16 * cc, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; c++) Sreg[16 * cc + c] = fmaf(dec, Sreg[16 * cc + c], v[c]);
                }
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float v8[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) v8[e] = Sreg[8 * q + e];
                    st_row8_split(sm + OFF_S, sm + OFF_SL, trow, 4 * wh + q, v8);
                }
                if (SAVE && !LITE && kk + 1 < nck) svr::put_state<SEG>(p, u, kk + 1, trow, wh, Sreg);
            } else {
                const int tg = (kbase + kk) * kC + (trow - 64);
                const size_t orow_at = (((size_t)bb * T + tg) * H + h) * dv + jc0;
                __nv_bfloat16* orow = p.o + orow_at;
#pragma unroll
                for (int cc = 0; cc < 2; cc++) {
                    const int col = 32 * wh + 16 * cc;
                    float v[16];
                    tmem_ld16(tl + tm_out + col, v);
                    if (DELTA) {
                        float w2[16];
                        tmem_ld16(tl + TM_U + col, w2);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; c++) v[c] += w2[c];
                    } else {
                        tmem_wait_ld();
                    }
                    if (tg < T) {
#pragma unroll
                        for (int hq = 0; hq < 2; hq++) {
                            const int j0 = col + 8 * hq;
                            if (j0 < nv && p.o32) {   // fp32 output (time-split intermediate runs)
                                float* q = p.o32 + orow_at + j0;
                                *reinterpret_cast<float4*>(q) =
                                    make_float4(v[8 * hq + 0], v[8 * hq + 1], v[8 * hq + 2], v[8 * hq + 3]);
                                *reinterpret_cast<float4*>(q + 4) =
                                    make_float4(v[8 * hq + 4], v[8 * hq + 5], v[8 * hq + 6], v[8 * hq + 7]);
                            } else if (j0 < nv) {
                                uint4 wv;
                                wv.x = pack_bf16(v[8 * hq + 0], v[8 * hq + 1]);
                                wv.y = pack_bf16(v[8 * hq + 2], v[8 * hq + 3]);
                                wv.z = pack_bf16(v[8 * hq + 4], v[8 * hq + 5]);
                                wv.w = pack_bf16(v[8 * hq + 6], v[8 * hq + 7]);
                                *reinterpret_cast<uint4*>(orow + j0) = wv;
                            }
                        }
                    }
                }
            }
        };
        // (1) chunk kk's inclusive scan of g and the overflow check of its anchors (one warp), into G[kk & 1] and
        // unsafe[kk & 1]; then its decay constants per (8-block, reference point), every exponent <= 0, into the
        // constant tables (read by the chunk's operand and Bhat steps only)
        auto scan = [&](int kk) {
            float* Gn = S.G[kk & 1];
            // lane l scans the pair (2l, 2l+1)
            const float ga = S.g[kk % kStages][2 * lane], gb = S.g[kk % kStages][2 * lane + 1];
            float x = ga + gb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const float ex = __shfl_up_sync(0xffffffffu, x, 1);
            Gn[2 * lane] = (lane > 0 ? ex : 0.f) + ga;
            Gn[2 * lane + 1] = x;
            __syncwarp();
            float span = 0.f;
            if (lane < 8) {
                const float g0 = Gn[8 * lane], g3 = Gn[8 * lane + 3], g7 = Gn[8 * lane + 7];
                span = fmaxf(g3 - g0, g7 - g3);
            }
            const bool bad = __any_sync(0xffffffffu, span * S.a2max > kSafeLog2);
            if (lane == 0) S.unsafe[kk & 1] = bad ? 1u : 0u;
        };
        auto table_entry = [&](const float* Gn, int pr) {   // pr = 64 k8 + i
            float* K = reinterpret_cast<float*>(sm + OFF_K);
            const int k8 = pr >> 6, i = pr & 63, J = k8 >> 1;
            const float a2 = S.A2[i], Gref = Gn[8 * k8 + 3];
            K[(K_A1 * 8 + k8) * 64 + i] = J >= 1 ? fast_exp2(a2 * (Gref - Gn[16 * J - 1])) : 0.f;
            K[(K_A2 * 8 + k8) * 64 + i] = (k8 & 1) ? fast_exp2(a2 * (Gref - Gn[16 * J + 7])) : 0.f;
            K[(K_0 * 8 + k8) * 64 + i] = fast_exp2(a2 * Gref);
            K[(K_B1_1 * 8 + k8) * 64 + i] = J < 1 ? fast_exp2(a2 * (Gn[15] - Gref)) : 0.f;
            K[(K_B1_2 * 8 + k8) * 64 + i] = J < 2 ? fast_exp2(a2 * (Gn[31] - Gref)) : 0.f;
            K[(K_B1_3 * 8 + k8) * 64 + i] = J < 3 ? fast_exp2(a2 * (Gn[47] - Gref)) : 0.f;
            K[(K_B2 * 8 + k8) * 64 + i] = (k8 & 1) ? 0.f : fast_exp2(a2 * (Gn[16 * J + 7] - Gref));
            K[(K_BH * 8 + k8) * 64 + i] = fast_exp2(a2 * (Gn[63] - Gref));
        };
        // all eight warps
        auto prep_all = [&](int kk) {
            if (warp == 0) scan(kk);
            named_bar_sync(1, kMath);   // G and the overflow flag
#pragma unroll
            for (int rep = 0; rep < 2; rep++) table_entry(S.G[kk & 1], r + rep * kMath);
        };
        // warps 2, 3, 6, 7 (the two schedulers the inverse step leaves idle), named barrier 2 among them
        auto prep_idle = [&](int kk) {
            const int gw = (warp & 1) + ((warp >> 2) << 1), gt = 32 * gw + lane;
            if (gw == 0) scan(kk);
            named_bar_sync(2, 128);
#pragma unroll
            for (int rep = 0; rep < 4; rep++) table_entry(S.G[kk & 1], gt + rep * 128);
        };
        int pending = -1;   // chunk whose epilogue has not run yet
        // token row of thread r in the decay-scaled operand step (and of its keep[] values)
        // (gated only: measured faster there, slower in delta mode, whose rows also store the b-side operands)
        auto op_row = [](int rr) { return DELTA ? (rr & 63) : (rr & 31) + 32 * (((rr >> 5) ^ (rr >> 7)) & 1); };
        uint32_t mma_phase = 0;
        // one warp polls the mbarrier; the others sleep in the named barrier
        auto mma_wait_all = [&]() -> bool {
            if (warp == 0) wait_or_abort(&S.mma, mma_phase, &S.abort, p.status, p.wait_ns);
            named_bar_sync(1, kMath);
            mma_phase ^= 1;
            tc_fence_after();
            return *(volatile uint32_t*)&S.abort == 0;
        };
        auto smem_to_tc = [&]() {   // generic-proxy smem writes -> visible to the tensor cores
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(1, kMath);
            tc_fence_after();
        };

        // chunk 0's scan and constants; later chunks' run on idle warps under the previous chunk's inverse step
        // (delta) or output product (gated)
        prep_all(0);
        named_bar_sync(1, kMath);
        for (int k = 0; k < nck; k++) {
            const int s = k % kStages;
            if (warp == 0) wait_or_abort(&S.full[s], (k / kStages) & 1, &S.abort, p.status, p.wait_ns);
            named_bar_sync(1, kMath);
            if (*(volatile uint32_t*)&S.abort) break;
            unsigned char* sV = sm + OFF_RING + s * STAGE_BYTES;
            unsigned char* sB = sV + 8192;
            unsigned char* sCt = sV + 16384;
            // g, beta of chunk k + kStages (threads 0..63), kept as raw bf16 until they are stored so that
            // nothing waits on the loads inside the chunk
            __nv_bfloat16 g_next = __float2bfloat16(0.f), beta_next = __float2bfloat16(0.f);
            if (r < kC && k + kStages < nck) {
                const int t = (kbase + k + kStages) * kC + r;
                const size_t row = ((size_t)bb * T + t) * H + h;
                if (t < T) {
                    g_next = p.g[row];
                    if (DELTA) beta_next = p.beta[row];
                }
            }

            // (1) the chunk's scan of g, overflow check and decay constants are ready (made by idle warps during the
            // previous chunk, or before the loop).  The inverse norms of b and c (GDN_NORM_BC) need the chunk's
            // tiles, so warps 1..4 compute them here.
            if (NORM && r >= 32 && r < 32 + 128) {
                const int vr = r - 32, t = vr & 63;
                float sq = 0.f;
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    float x8[8];
                    ld_row8(vr < 64 ? sB : sCt, t, q, x8);
#pragma unroll
                    for (int e = 0; e < 8; e++) sq = fmaf(x8[e], x8[e], sq);
                }
                const float inv = 1.f / fmaxf(sqrtf(sq), kNormFloor);
                if (vr < 64) S.nb[t] = inv;
                else S.nc[t] = inv;
            }
            if (NORM) named_bar_sync(1, kMath);   // the inverse norms
            const float* Gc = S.G[k & 1];

            // (2) decay-scaled operands; thread = (row t, 16 channels)
            const bool unsafe = S.unsafe[k & 1] != 0;
            float keep[16];   // gated: Ctil row part; delta: beta Btil row part
            {
                // gated: rows of blocks 0-1 store more operand tiles than rows of blocks 2-3; the row half
                // alternates with bit 2 of the warp so that each scheduler (warp mod 4) gets one of each
                const int t = op_row(r), cq = r >> 6, k8 = t >> 3, I = t >> 4;
                const bool upper = (t & 15) >= 8;
                const float Gt = Gc[t], Gr = Gc[8 * k8 + 3];
                const float dG = Gt - Gr;
                const float bet = DELTA ? S.beta[s][t] : 0.f;
                const float nbt = NORM ? S.nb[t] : 1.f, nct = NORM ? S.nc[t] : 1.f;
                if (!unsafe) {
                    // fast path: anchor exp(A (G_t - G_r8)) times per-block constants
#pragma unroll
                    for (int qq = 0; qq < 2; qq++) {
                        const int q = 2 * cq + qq;
                        float cv[8], bv[8], a2[8], ax[8], bxp[8], bbx[8], y[8], z[8];
                        ld_row8(sCt, t, q, cv);
                        ld_row8(sB, t, q, bv);
                        ld_f8(S.A2 + 8 * q, a2);
                        if (NORM) {
#pragma unroll
                            for (int e = 0; e < 8; e++) { cv[e] *= nct; bv[e] *= nbt; }
                        }
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const float an = fast_exp2(a2[e] * dG), ai = fast_exp2(-a2[e] * dG);
                            ax[e] = cv[e] * an;
                            bxp[e] = bv[e] * ai;
                            bbx[e] = (SAVE ? 1.f : bet) * bv[e] * an;
                        }
                        float kk[8];
                        if (I > 0) {
                            ld_f8(ktab(sm, K_A1, k8) + 8 * q, kk);
#pragma unroll
                            for (int e = 0; e < 8; e++) { y[e] = ax[e] * kk[e]; z[e] = bbx[e] * kk[e]; }
                            st_row8_f16(X + X_A1, t, q, y);
                            st_row8_f16(X + X_A1, 64 + t, q, *(DELTA ? &z : &y));
                        }
                        if (upper) {
                            ld_f8(ktab(sm, K_A2, k8) + 8 * q, kk);
#pragma unroll
                            for (int e = 0; e < 8; e++) { y[e] = ax[e] * kk[e]; z[e] = bbx[e] * kk[e]; }
                            st_row8_f16(X + X_A2, t, q, y);
                            st_row8_f16(X + X_A2, 64 + t, q, *(DELTA ? &z : &y));
                        }
                        st_row8_split(X + X_A3, X + X_A3L, t, q, ax);
                        st_row8_split(X + X_A3, X + X_A3L, 64 + t, q, *(DELTA ? &bbx : &ax));
                        if (I < 1) {
                            ld_f8(ktab(sm, K_B1_1, k8) + 8 * q, kk);
#pragma unroll
                            for (int e = 0; e < 8; e++) y[e] = bxp[e] * kk[e];
                            st_row8_f16(X + X_B1a, t, q, y);
                        }
                        if (I < 2) {
                            ld_f8(ktab(sm, K_B1_2, k8) + 8 * q, kk);
#pragma unroll
                            for (int e = 0; e < 8; e++) y[e] = bxp[e] * kk[e];
                            st_row8_f16(X + X_B1b, t, q, y);
                        }
                        if (I < 3) {
                            ld_f8(ktab(sm, K_B1_3, k8) + 8 * q, kk);
#pragma unroll
                            for (int e = 0; e < 8; e++) y[e] = bxp[e] * kk[e];
                            st_row8_f16(X + X_B1c, t, q, y);
                        }
                        if (!upper) {
                            ld_f8(ktab(sm, K_B2, k8) + 8 * q, kk);
#pragma unroll
                            for (int e = 0; e < 8; e++) y[e] = bxp[e] * kk[e];
                            st_row8_f16(X + X_B2, t, q, y);
                        }
                        st_row8_split(X + X_B3, X + X_B3L, t, q, bxp);
                        ld_f8(ktab(sm, K_0, k8) + 8 * q, kk);
#pragma unroll
                        for (int e = 0; e < 8; e++) keep[8 * qq + e] = (DELTA ? (SAVE ? bet : 1.f) * bbx[e] : ax[e]) * kk[e];
                    }
                } else {
                    // fallback: every factor evaluated directly (all exponents <= 0 except L3's,
                    // whose entries the assembly step replaces by exact sums)
                    const float GI = I > 0 ? Gc[16 * I - 1] : 0.f, GJ7 = Gc[16 * I + 7];
#pragma unroll
                    for (int qq = 0; qq < 2; qq++) {
                        const int q = 2 * cq + qq;
                        float cv[8], bv[8], bbv[8], y[8], z[8];
                        ld_row8(sCt, t, q, cv);
                        ld_row8(sB, t, q, bv);
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            cv[e] *= nct;
                            bv[e] *= nbt;
                            bbv[e] = (SAVE ? 1.f : bet) * bv[e];
                        }
                        if (I > 0) {
                            scale8(cv, S.A2, q, Gt - GI, y); st_row8_f16(X + X_A1, t, q, y);
                            if (DELTA) { scale8(bbv, S.A2, q, Gt - GI, z); st_row8_f16(X + X_A1, 64 + t, q, z); }
                            else st_row8_f16(X + X_A1, 64 + t, q, y);
                        }
                        if (upper) {
                            scale8(cv, S.A2, q, Gt - GJ7, y); st_row8_f16(X + X_A2, t, q, y);
                            if (DELTA) { scale8(bbv, S.A2, q, Gt - GJ7, z); st_row8_f16(X + X_A2, 64 + t, q, z); }
                            else st_row8_f16(X + X_A2, 64 + t, q, y);
                        }
                        if (I < 1) { scale8(bv, S.A2, q, Gc[15] - Gt, y); st_row8_f16(X + X_B1a, t, q, y); }
                        if (I < 2) { scale8(bv, S.A2, q, Gc[31] - Gt, y); st_row8_f16(X + X_B1b, t, q, y); }
                        if (I < 3) { scale8(bv, S.A2, q, Gc[47] - Gt, y); st_row8_f16(X + X_B1c, t, q, y); }
                        if (!upper) { scale8(bv, S.A2, q, GJ7 - Gt, y); st_row8_f16(X + X_B2, t, q, y); }
                        scale8(DELTA ? bbv : cv, S.A2, q, Gt, y);
#pragma unroll
                        for (int e = 0; e < 8; e++) keep[8 * qq + e] = (DELTA && SAVE ? bet : 1.f) * y[e];
                    }
                }
            }
            smem_to_tc();

            // (3) level MMAs
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                // L1 for all three row blocks in one N = 96 product: the column operands B1a | B1b | B1c
                // (16, 32, 48 rows) are contiguous, and so are their accumulators D1a | D1b | D1c
                static_assert(X_B1b == X_B1a + 16 * 128 && X_B1c == X_B1b + 32 * 128, "L1 column operands");
                static_assert(TM_D1b == TM_D1a + 16 && TM_D1c == TM_D1b + 32, "L1 accumulators");
                mma_k64(tbase + TM_D1a, x0 + X_A1, x0 + X_B1a, false, idesc_f16(128, 96, false, false), false);
                mma_k64(tbase + TM_D2, x0 + X_A2, x0 + X_B2, false, idesc_f16(128, 64, false, false), false);
                const uint32_t id3 = idesc_bf16(128, 64, false, false);
                mma_k64(tbase + TM_D3, x0 + X_A3, x0 + X_B3, false, id3, false);
                mma_k64(tbase + TM_D3, x0 + X_A3, x0 + X_B3L, false, id3, true);
                mma_k64(tbase + TM_D3, x0 + X_A3L, x0 + X_B3, false, id3, true);
                mma_commit(&S.mma);
            }
            // (2b) Bhat^T rows (i = channel), from the L3 column operand; decay vector.  Runs while the
            // level MMAs execute: it reads their operands and writes only [Bhat^T ; P] rows 0..63.
            {
                const int i = r & 63, sq = r >> 6;
                const float a2 = S.A2[i], G63 = Gc[63];
                if (!unsafe) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; h2++) {
                        float y8[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const int sc = 16 * sq + 8 * h2 + e;
                            const float b3 = bf2f(*reinterpret_cast<const uint16_t*>(X + X_B3 + sw128(sc, i))) +
                                             bf2f(*reinterpret_cast<const uint16_t*>(X + X_B3L + sw128(sc, i)));
                            y8[e] = b3 * ktab(sm, K_BH, sc >> 3)[i];
                        }
                        st_row8_split(sm + OFF_CH0, sm + OFF_CH0L, i, 2 * sq + h2, y8);
                    }
                } else {
#pragma unroll 1
                    for (int h2 = 0; h2 < 2; h2++) {
                        float y8[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const int sc = 16 * sq + 8 * h2 + e;
                            const float bval = bf2f(*reinterpret_cast<const uint16_t*>(sB + sw128(sc, i))) *
                                               (NORM ? S.nb[sc] : 1.f);
                            y8[e] = bval * exp2f(a2 * (G63 - Gc[sc]));
                        }
                        st_row8_split(sm + OFF_CH0, sm + OFF_CH0L, i, 2 * sq + h2, y8);
                    }
                }
                if (r < 64) S.decay[k & 1][r] = fast_exp2(S.A2[r] * Gc[63]);
            }
            if (pending >= 0) epilogue(pending), pending = -1;   // the previous chunk's, under the level products
            if (!mma_wait_all()) break;

            // (4) assemble P (lanes 0..63) and M (lanes 64..127); thread = (row, 32 columns).  Gated: lanes
            // 64..127 hold a copy of P (the level operands repeat the c-side rows there), and every thread takes
            // one 16-column group of its row
            {
                const bool isM = DELTA && q4 >= 2;
                // two instances: the common one without the elementwise L3 entries of a chunk whose anchors could
                // overflow (their registers and code stay out of it)
                auto assemble = [&](auto us) {
                    constexpr bool US = decltype(us)::value;
                    const int t = trow & 63, wl = q4 & 1, tb = t >> 4;
                    float ew[8];
                    if (US) {
                        const int s0 = 8 * (t >> 3);
                        const float bet = DELTA ? S.beta[s][t] : 0.f;
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            float acc = 0.f;
                            const int sc = s0 + e;
                            if (sc < t || (sc == t && !isM)) {
                                for (int q = 0; q < 8; q++) {
                                    float xv[8], bv[8];
                                    ld_row8(isM ? sB : sCt, t, q, xv);
                                    ld_row8(sB, sc, q, bv);
#pragma unroll
                                    for (int kk = 0; kk < 8; kk++)
                                        acc += xv[kk] * bv[kk] * exp2f(S.A2[8 * q + kk] * (Gc[t] - Gc[sc]));
                                }
                                if (NORM) acc *= (isM ? S.nb[t] : S.nc[t]) * S.nb[sc];
                            }
                            ew[e] = (isM && !SAVE) ? bet * acc : acc;
                        }
                    }
                    const int Ia = 2 * wl, Ib = 2 * wl + 1;
                    const uint32_t colA = wl == 0 ? 0u : TM_D1b, colB = wl == 0 ? TM_D1a : TM_D1c;
                    float* M32 = reinterpret_cast<float*>(X + X_M32);
                    // gated: the four threads of a row (two lane halves x two column halves) take one group each,
                    // so that the TMEM loads of the lower triangle (rows 0..31: 3, 2, 0, 0 per group; rows 32..63:
                    // 4, 4, 3, 2) come to at most 7 per scheduler instead of 13
                    const int lo = q4 >> 1;
#pragma unroll
                    for (int cc = 0; cc < (DELTA ? 2 : 1); cc++) {
                        const int cg = DELTA ? 2 * wh + cc : (wh ? (wl ? 3 - lo : 2 + lo) : lo);
                        float out[16];
                        if (16 * cg > 32 * wl + 31) {
#pragma unroll
                            for (int c = 0; c < 16; c++) out[c] = 0.f;
                        } else {
                            float v1a[16], v1b[16], v2[16], v3[16];
                            if (Ia >= 1 && cg < Ia) tmem_ld16(tl + colA + 16 * cg, v1a);
                            if (cg < Ib) tmem_ld16(tl + colB + 16 * cg, v1b);
                            tmem_ld16(tl + TM_D2 + 16 * cg, v2);
                            tmem_ld16(tl + TM_D3 + 16 * cg, v3);
                            tmem_wait_ld();
#pragma unroll
                            for (int c = 0; c < 16; c++) {
                                const int sc = 16 * cg + c;
                                float val;
                                if (sc > t || (isM && sc == t)) val = 0.f;
                                else if ((sc >> 4) < tb) val = (tb == Ia) ? v1a[c] : v1b[c];
                                else if ((sc >> 3) < (t >> 3)) val = v2[c];
                                else val = US ? ew[c & 7] : v3[c];
                                out[c] = val;
                            }
                        }
                        if (SAVE && isM) {
                            // the level products gave K (zero on and above the diagonal): a residual; M = beta K
                            float4* kr = reinterpret_cast<float4*>(svr::rec<SEG>(p, u, k) + svr::K) + (4 * cg) * 64 + t;
                            const float bet = S.beta[s][t];
                            if (!LITE) {
#pragma unroll
                                for (int e = 0; e < 4; e++)
                                    kr[64 * e] = make_float4(out[4 * e], out[4 * e + 1], out[4 * e + 2], out[4 * e + 3]);
                            }
#pragma unroll
                            for (int c = 0; c < 16; c++) out[c] *= bet;
                        }
                        if (!isM) {
                            st_split16(sm + OFF_CH0, sm + OFF_CH0L, 64 + t, cg, out);
                            if (SAVE) {
                                unsigned char* pr = svr::rec<SEG>(p, u, k) + svr::P;
                                st_split16(pr, pr + 8192, t, cg, out);
                            }
                        } else {
                            // L: the column blocks left of the row's 32-block; the diagonal 16-block (M32) and,
                            // in the upper 16-block of a 32-block, the one below the diagonal (C32) in fp32
                            float lpart[16];
#pragma unroll
                            for (int c = 0; c < 16; c++) lpart[c] = (cg < (tb & 2)) ? out[c] : 0.f;
                            st_plain16(X + X_LRH, t, cg, lpart);
                            float* f32 = nullptr;
                            if (cg == tb) f32 = M32 + (tb * 16 + (t & 15)) * kBS;
                            else if ((tb & 1) && cg == tb - 1)
                                f32 = reinterpret_cast<float*>(X + X_C32) + ((tb >> 1) * 16 + (t & 15)) * kBS;
                            if (f32) {
#pragma unroll
                                for (int c = 0; c < 16; c += 4)
                                    *reinterpret_cast<float4*>(f32 + c) =
                                        make_float4(out[c], out[c + 1], out[c + 2], out[c + 3]);
                            }
                        }
                    }
                };
                if (unsafe) assemble(BoolTag<true>{});
                else assemble(BoolTag<false>{});
            }
            {
                const int t = op_row(r), cq = r >> 6;   // the rows whose keep[] this thread holds
                if (!DELTA) {
                    // [0 ; Ctil] for the output MMA (the levels' space is free now)
#pragma unroll
                    for (int qq = 0; qq < 2; qq++) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) y[e] = keep[8 * qq + e];
                        st_row8(X + X_CH1, 64 + t, 2 * cq + qq, y);
                        zero_chunk(X + X_CH1, t, 2 * cq + qq);
                    }
                } else {
                    // R = [beta V | beta Btil]: hi in LRH blocks 1-2, lo in LRL blocks 0-1
                    const float bet = S.beta[s][t];
#pragma unroll
                    for (int qq = 0; qq < 2; qq++) {
                        const int q = 2 * cq + qq;
                        float vv[8], y[8];
                        ld_row8(sV, t, q, vv);
#pragma unroll
                        for (int e = 0; e < 8; e++) y[e] = bet * vv[e];
                        st_row8_split(X + X_LRH + 8192, X + X_LRL, t, q, y);
#pragma unroll
                        for (int e = 0; e < 8; e++) y[e] = keep[8 * qq + e];
                        st_row8_split(X + X_LRH + 16384, X + X_LRL + 8192, t, q, y);
                    }
                }
            }

            if constexpr (!DELTA) {
                smem_to_tc();
                // (5g) [dS ; O] = [[Bhat^T, 0], [P, Ctil]] x [V ; S]  (hi/lo parts)
                if (r == 0) {
                    const uint32_t ch0 = smem_u32(sm + OFF_CH0), ch0l = smem_u32(sm + OFF_CH0L);
                    const uint32_t ch1 = smem_u32(X + X_CH1);
                    const uint32_t vt = smem_u32(sV), st = smem_u32(sm + OFF_S), stl = smem_u32(sm + OFF_SL);
                    const uint32_t id = idesc_bf16(128, 64, false, true);
                    mma_k64(tbase + TM_CHG, ch0, vt, true, id, false);
                    mma_k64(tbase + TM_CHG, ch0l, vt, true, id, true);
                    mma_k64(tbase + TM_CHG, ch1, st, true, id, true);
                    mma_k64(tbase + TM_CHG, ch1, stl, true, id, true);
                    mma_commit(&S.mma);
                }
                // meanwhile warps 2, 3, 6, 7: the next chunk's scan and constants (G and the tables are the
                // current chunk's no longer: both were last read before this product)
                if ((warp & 2) && k + 1 < nck) prep_idle(k + 1);
                if (!mma_wait_all()) break;
            } else {
                named_bar_sync(1, kMath);
                // (5) exact inverse of the diagonal 16-blocks of I + M
                if (r < 64) {
                    const int J = r >> 4, c = r & 15;
                    const float* M32 = reinterpret_cast<const float*>(X + X_M32) + J * 16 * kBS;
                    // column c of (I + M_JJ)^{-1}, right-looking: once x_p is final,
                    // subtract M[q][p] x_p from every later row q (independent FMAs)
                    float xs[16];
#pragma unroll
                    for (int q = 0; q < 16; q++) xs[q] = (q == c) ? 1.f : 0.f;
#pragma unroll
                    for (int pp = 0; pp < 15; pp++) {
                        if (pp >= c) {
                            const float xp = xs[pp];
#pragma unroll
                            for (int q = pp + 1; q < 16; q++) xs[q] = fmaf(-M32[q * kBS + pp], xp, xs[q]);
                        }
                    }
                    float* DI32 = reinterpret_cast<float*>(X + X_DI32) + J * 16 * kBS;
#pragma unroll
                    for (int q = 0; q < 16; q++) DI32[q * kBS + c] = xs[q];
                    // (5b) the 32-block [[A, 0], [C, B]] of I + M formed by the 16-blocks 2 w, 2 w + 1 (this warp's)
                    // has the inverse [[A^-1, 0], [E, B^-1]], E = -B^-1 C A^-1: lane (half hf, column c) forms
                    // F = C A^-1 on rows 8 hf .. 8 hf + 7 of column c, trades them with lane ^ 16, then E on the
                    // same rows.  It runs while the idle warps prepare the next chunk.
                    __syncwarp();
                    {
                        const int hf = lane >> 4, q0 = 8 * hf;
                        const float* Ai = reinterpret_cast<const float*>(X + X_DI32) + (2 * warp) * 16 * kBS;
                        const float* Bi = Ai + 16 * kBS;
                        const float* Cb = reinterpret_cast<const float*>(X + X_C32) + warp * 16 * kBS;
                        float acol[16];
#pragma unroll
                        for (int m = 0; m < 16; m++) acol[m] = Ai[m * kBS + c];
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
                        float fc[16];   // column c of F
#pragma unroll
                        for (int kq = 0; kq < 8; kq++) {
                            const float o = __shfl_xor_sync(0xffffffffu, f[kq], 16);
                            fc[kq] = hf ? o : f[kq];
                            fc[8 + kq] = hf ? f[kq] : o;
                        }
                        float* Eb = reinterpret_cast<float*>(X + X_E32) + warp * 16 * kBS;
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
                            Eb[(q0 + kq) * kBS + c] = -x;
                        }
                    }
                } else if ((warp & 2) && k + 1 < nck) {
                    prep_idle(k + 1);   // meanwhile warps 2, 3, 6, 7: the next chunk's scan and constants
                }
                named_bar_sync(1, kMath);
                {
                    // [Dinv ; Dinv]: row trow, 32 columns of half wh.  The copy in rows 64..127 puts a copy of
                    // [N | X0] in TMEM lanes 64..127, so that the output-lane warps convert half of it.
                    const int J = (trow & 63) >> 4;
                    const float* DI32 = reinterpret_cast<const float*>(X + X_DI32) + (J * 16 + (trow & 15)) * kBS;
                    const float* E32 = reinterpret_cast<const float*>(X + X_E32) + ((J >> 1) * 16 + (trow & 15)) * kBS;
#pragma unroll
                    for (int cc = 0; cc < 2; cc++) {
                        const int cg = 2 * wh + cc;
                        const float* src = (cg == J) ? DI32 : ((J & 1) && cg == J - 1) ? E32 : nullptr;
                        float v16[16];
#pragma unroll
                        for (int c = 0; c < 16; c += 4) {
                            const float4 x = src ? *reinterpret_cast<const float4*>(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                            v16[c] = x.x; v16[c + 1] = x.y; v16[c + 2] = x.z; v16[c + 3] = x.w;
                        }
                        st_plain16(X + X_DINV, trow, cg, v16);
                        if (SAVE && !LITE && trow < 64) st_plain16(svr::rec<SEG>(p, u, k) + svr::DINV, trow, cg, v16);
                    }
                }
                smem_to_tc();

                // (6) [N | X0] = Dinv [L | R]
                if (r == 0) {
                    const uint32_t x0 = smem_u32(X);
                    mma_k64(tbase + TM_NX, x0 + X_DINV, x0 + X_LRH, true, idesc_bf16(128, 192, false, true), false);
                    mma_k64(tbase + TM_NX + 64, x0 + X_DINV, x0 + X_LRL, true, idesc_bf16(128, 128, false, true),
                            true);
                    mma_commit(&S.mma);
                }
                if (!mma_wait_all()) break;

                // (7) -N -> A operand; X0 -> hi/lo B blocks.  Twelve 16-column groups of token t: groups 0..5 from
                // the state lanes, 6..11 from their copy in the output lanes.  The output lanes then clear their
                // rows of the A operand and of TMEM columns TM_U .. TM_U + 127 (each thread only columns that it
                // has read itself, or that nobody reads), so that [U ; Ctil S] starts from [Util ; 0].
                {
                    const int t = trow & 63;
                    const int gb = (state_row ? 0 : 6) + 3 * wh;
#pragma unroll
                    for (int gg = 0; gg < 3; gg++) {
                        const int g = gb + gg;
                        float v[16];
                        tmem_ld16(tl + TM_NX + 16 * g, v);
                        tmem_wait_ld();
                        if (g < 4) {
#pragma unroll
                            for (int c = 0; c < 16; c++) v[c] = -v[c];
                            st_plain16(X + X_NA, t, g, v);
                            if (SAVE && !LITE) st_plain16(svr::rec<SEG>(p, u, k) + svr::NA, t, g, v);
                        } else {
                            const int xg = g - 4;
                            const uint32_t blk = (uint32_t)(xg >> 2) * 8192u;
                            st_split16(X + X_X0H + blk, X + X_X0L + blk, t, xg & 3, v);
                        }
                    }
                    if (!state_row) {
#pragma unroll
                        for (int q = 0; q < 4; q++) zero_chunk(X + X_NA, trow, 4 * wh + q);
                        float zz[16];
#pragma unroll
                        for (int c = 0; c < 16; c++) zz[c] = 0.f;
                        // half 0 read X0 groups 2..4 (columns TM_U + 32 .. + 79), half 1 groups 5..7
                        if (wh == 0) {
#pragma unroll
                            for (int xg = 0; xg < 5; xg++) tmem_st16(tl + TM_U + 16 * xg, zz);
                        } else {
#pragma unroll
                            for (int xg = 5; xg < 8; xg++) tmem_st16(tl + TM_U + 16 * xg, zz);
                        }
                        tmem_wait_st();
                    }
                }
                smem_to_tc();

                // (8) [Util | W] = X0 - N X0, accumulated onto X0 (exact in TMEM)
                if (r == 0) {
                    const uint32_t x0 = smem_u32(X);
                    const uint32_t id = idesc_bf16(128, 128, false, true);
                    mma_k64(tbase + TM_U, x0 + X_NA, x0 + X_X0H, true, id, true);
                    mma_k64(tbase + TM_U, x0 + X_NA, x0 + X_X0L, true, id, true);
                    mma_commit(&S.mma);
                }
                // (11) CW = [-W ; Ctil]: the Ctil rows (output lanes) while the products run
                static_assert(X_CW >= X_X0L + 16384 && X_CW + 16384 <= X_BYTES, "CW clear of the phase-3 operands");
                static_assert(X_E32 + 2 * 16 * kBS * 4 <= X_CW + 16384, "fp32 staging inside the operand region");
                if (!state_row) {
                    const int t = trow - 64;
                    const float Gt = Gc[t];
#pragma unroll
                    for (int qq = 0; qq < 4; qq++) {
                        const int q = 4 * wh + qq;
                        float cv[8], y[8];
                        ld_row8(sCt, t, q, cv);
                        if (NORM) {
#pragma unroll
                            for (int e = 0; e < 8; e++) cv[e] *= S.nc[t];
                        }
                        scale8(cv, S.A2, q, Gt, y);
                        st_row8(X + X_CW, trow, q, y);
                    }
                }
                if (!mma_wait_all()) break;
                if (state_row) {   // the -W rows
#pragma unroll
                    for (int cc = 0; cc < 2; cc++) {
                        const int cg = 2 * wh + cc;
                        float v[16];
                        tmem_ld16(tl + TM_W + 16 * cg, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; c++) v[c] = -v[c];
                        st_plain16(X + X_CW, trow, cg, v);
                        if (SAVE) {
                            unsigned char* rq = svr::rec<SEG>(p, u, k);
                            st_split16(rq + svr::NW, rq + svr::NWL, trow, cg, v);
                        }
                    }
                }
                smem_to_tc();

                // (12) [U ; Ctil S] = [Util ; 0] + [-W ; Ctil] S
                if (r == 0) {
                    const uint32_t x0 = smem_u32(X);
                    const uint32_t id = idesc_bf16(128, 64, false, true);
                    mma_k64(tbase + TM_U, x0 + X_CW, smem_u32(sm + OFF_S), true, id, true);
                    mma_k64(tbase + TM_U, x0 + X_CW, smem_u32(sm + OFF_SL), true, id, true);
                    mma_commit(&S.mma);
                }
                if (!mma_wait_all()) break;

                // (13) U -> hi/lo B tiles
                if (state_row) {
#pragma unroll
                    for (int cc = 0; cc < 2; cc++) {
                        const int cg = 2 * wh + cc;
                        float v[16];
                        tmem_ld16(tl + TM_U + 16 * cg, v);
                        tmem_wait_ld();
                        st_split16(X + X_UH, X + X_UL, trow, cg, v);
                        if (SAVE && !LITE) {
                            // U itself (the state already folded in) is a residual
                            float4* du = reinterpret_cast<float4*>(svr::rec<SEG>(p, u, k) + svr::U) + (4 * cg) * 64 + trow;
#pragma unroll
                            for (int e = 0; e < 4; e++)
                                du[64 * e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                        }
                    }
                }
                smem_to_tc();

                // (14) [dS ; P U] = [Bhat^T ; P] U
                if (r == 0) {
                    const uint32_t x0 = smem_u32(X);
                    const uint32_t ch0 = smem_u32(sm + OFF_CH0), ch0l = smem_u32(sm + OFF_CH0L);
                    const uint32_t id = idesc_bf16(128, 64, false, true);
                    mma_k64(tbase + TM_CHD, ch0, x0 + X_UH, true, id, false);
                    mma_k64(tbase + TM_CHD, ch0l, x0 + X_UH, true, id, true);
                    mma_k64(tbase + TM_CHD, ch0, x0 + X_UL, true, id, true);
                    mma_commit(&S.mma);
                }
                if (!mma_wait_all()) break;
            }

            pending = k;   // its state update and outputs run under the next chunk's level products
            smem_to_tc();
            // stage s is free again (every read of it, and the last MMA, are done)
            if (k + kStages < nck) {
                if (r < kC) {
                    // (the sigmoid of a logit is taken here, where the loaded value is first used,
                    // so the load's latency stays hidden behind the chunk)
                    // tokens past T keep g = beta = 0 (an identity step)
                    const bool tok = (kbase + k + kStages) * kC + r < T;
                    S.g[s][r] = tok ? gate_in(__bfloat162float(g_next), p.logits) : 0.f;
                    if (DELTA) S.beta[s][r] = tok ? gate_in(__bfloat162float(beta_next), p.logits) : 0.f;
                }
                if (r == 0) issue_load(k + kStages), issued = k + kStages + 1;
            }
        }
        if (pending >= 0 && *(volatile uint32_t*)&S.abort == 0) epilogue(pending);
        if (state_row && p.hT && trow < dk) {
            float* hrow = p.hT + ((size_t)u * dk + trow) * dv + jc0;
#pragma unroll
            for (int j = 0; j < 32; j++)
                if (32 * wh + j < nv) hrow[32 * wh + j] = Sreg[j];
        }
        // after an abort, let the copies already issued land before exiting
        if (tid == 0 && *(volatile uint32_t*)&S.abort)
            for (int k = issued > kStages ? issued - kStages : 0; k < issued; k++)
                mbar_wait(&S.full[k % kStages], (k / kStages) & 1, nullptr, p.wait_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

template <bool DELTA, bool NORM, int SAVEM = SAVE_NONE>
cudaError_t launch_t(const TcParams& p, dim3 grid, cudaStream_t st)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<DELTA, NORM, SAVEM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    fwd_tc_kernel<DELTA, NORM, SAVEM><<<grid, kThreads, SMEM_BYTES, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const Args& a, cudaStream_t st, bool* handled)
{
    *handled = false;
    if (a.io != GDN_BF16 || a.T <= 0 || a.dk > 64) return cudaSuccess;
    TcParams p;
    memset(&p, 0, sizeof(p));
    if (!make_map(&p.tm_v, a.v, a.B, a.T, a.H, a.dv) || !make_map(&p.tm_b, a.b, a.B, a.T, a.H, a.dk) ||
        !make_map(&p.tm_c, a.c, a.B, a.T, a.H, a.dk))
        return cudaErrorInvalidValue;
    p.g = (const __nv_bfloat16*)a.g;
    p.beta = (const __nv_bfloat16*)a.beta;
    p.A_log = a.A_log;
    p.h0 = a.h0;
    p.o = (__nv_bfloat16*)a.o;
    p.o32 = a.o32;
    p.hT = a.hT;
    p.status = (uint32_t*)a.ws;
    p.B = a.B; p.H = a.H; p.T = a.T; p.dk = a.dk; p.dv = a.dv;
    p.logits = a.logits;
    p.nchunks = (a.T + kC - 1) / kC;
    // failure-path test hook (read once per process, see test_starve_chunk): the loads of that chunk are never
    // issued, so its bounded wait expires after kTestWaitNs and the status word reads GDN_ERR_TIMEOUT
    p.starve_chunk = test_starve_chunk();
    p.wait_ns = p.starve_chunk >= 0 ? kTestWaitNs : kWaitNs;
    *handled = true;
    const int nseg = a.saved && a.seg > 1 ? a.seg : 1;
    const dim3 grid(a.B * a.H * nseg, (a.dv + 63) / 64);
    if (a.saved) {
        // the residuals of the chunked backward: one slab, no option bits (the host checks); on a time split's
        // segment view (a.seg segments per sequence) they are laid out by the chunks of the whole sequence
        if (a.dv > 64 || a.norm || a.logits) return cudaErrorInvalidValue;
        const size_t nq = (size_t)a.B * a.H * p.nchunks;
        p.seg = nseg;
        p.seg_len = a.seg_len;
        p.st = (float*)a.saved;
        p.sv = (unsigned char*)a.saved + nq * 16384;
        p.sv_stride = a.mode == GDN_DELTA ? svr::BYTES : svr::GATED_BYTES;
        if (a.mode != GDN_DELTA) {
            if (p.seg <= 1) return launch_t<false, false, SAVE_FULL>(p, grid, st);
            return a.save_lite ? launch_t<false, false, SAVE_SPLIT_LITE>(p, grid, st)
                               : launch_t<false, false, SAVE_SPLIT>(p, grid, st);
        }
        if (p.seg <= 1) return launch_t<true, false, SAVE_FULL>(p, grid, st);
        return a.save_lite ? launch_t<true, false, SAVE_SPLIT_LITE>(p, grid, st)
                           : launch_t<true, false, SAVE_SPLIT>(p, grid, st);
    }
    if (a.norm)
        return a.mode == GDN_DELTA ? launch_t<true, true>(p, grid, st) : launch_t<false, true>(p, grid, st);
    return a.mode == GDN_DELTA ? launch_t<true, false>(p, grid, st) : launch_t<false, false>(p, grid, st);
}

}  // namespace gdn
