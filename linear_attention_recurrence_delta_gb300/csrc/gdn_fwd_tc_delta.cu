// gdn_fwd_tc_delta.cu -- chunked forward of the delta mode on tcgen05 tensor
// cores (bf16 I/O, fp32 accumulation and fp32 state).
//
// Delta rule ("HyMo-434M -- documentation portal", card 01): per token
//   h' = alpha_t (.)rows h_{t-1},  u_t = beta_t (v_t - h'^T b_t),
//   h_t = h' + b_t u_t^T,          o_t = h_t^T c_t.
// Chunked ("GDN & MLA Mechanism Deep-Dive", Step 5, chunk C = 64): with G, Gam,
// P, Ctil, Bhat as in the gated kernel, Btil_t = b_t (.) exp(Gam_t) and the
//   M[t,s] = beta_t sum_i b_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])   (s < t)
// the values written into the state solve the unit lower-triangular system
//   (I + M) U = diag(beta) V - diag(beta) Btil S  =:  Util - W S
// with Util = (I+M)^{-1} diag(beta) V and W = (I+M)^{-1} diag(beta) Btil
// (the WY / UT-transform form), after which
//   O = Ctil S + P U,    S' = exp(Gam_63) (.)rows S + Bhat^T U.
//
// The inverse is applied with three tensor-core products.  Split I + M into
// its 16x16 diagonal blocks D (unit lower triangular, inverted exactly in fp32
// by forward substitution on the CUDA cores) and the strictly block-lower rest
// L.  With N = D^{-1} L, which is nilpotent (N^4 = 0, four block rows):
//   (I + M)^{-1} R = (I + N^2)(I - N) D^{-1} R,
// evaluated as  [N | X0] = D^{-1} [L | R],  [N^2 | N X0] = N [N | X0],
// Z = X0 - N X0,  X = Z + N^2 Z  for R = [beta V | beta Btil], X = [Util | W].
//
// P and M come from the same three decay-safe levels as in the gated kernel
// (rows 0..63 of the M = 128 MMAs hold the c-side, rows 64..127 the
// beta b-side).  Precision: level-1/2 operands fp16; the level-3, P, R, X0, Z,
// U and state operands as bf16 hi + lo pairs; D^{-1}, L, N, N^2, W and Ctil
// plain bf16; Z is also kept exactly (fp32) in TMEM as the accumulator X
// starts from.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fwd_tc_common.cuh"

namespace gdn {
namespace {

using namespace tc;
using namespace fwdtc;

constexpr int kStages = 2;
constexpr int kThreads = 160;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_RING = 0;
constexpr uint32_t STAGE_BYTES = 3 * 8192;
constexpr uint32_t OFF_X = kStages * STAGE_BYTES;      // region reused phase by phase (100 KB)
//   phase 1: decay levels of P and M
constexpr uint32_t X_A1 = 0, X_B1a = 16384, X_B1b = 18432, X_B1c = 22528;
constexpr uint32_t X_A2 = 28672, X_B2 = 45056, X_A3 = 53248, X_A3L = 69632, X_B3 = 86016, X_B3L = 94208;
//   phase 2: [N | X0] = Dinv [L | R]
constexpr uint32_t X_DINV = 0, X_LRH = 16384, X_LRL = 40960, X_M32 = 57344, X_DI32 = 61440;
//   phase 3: [N^2 | N X0] = N [N | X0]
constexpr uint32_t X_NA = 0, X_NXH = 16384, X_NXL = 40960;
//   phase 4: X = Z + N^2 Z
constexpr uint32_t X_N2A = 0, X_ZH = 16384, X_ZL = 32768;
//   phase 5: the two state products
constexpr uint32_t X_CW = 0, X_UH = 16384, X_UL = 24576;
constexpr uint32_t X_BYTES = 102400;
constexpr uint32_t OFF_CH0 = OFF_X + X_BYTES;          // [Bhat^T ; P] hi
constexpr uint32_t OFF_CH0L = OFF_CH0 + 16384;         // [Bhat^T ; P] lo
constexpr uint32_t OFF_S = OFF_CH0L + 16384;           // state bf16 [i][j] hi
constexpr uint32_t OFF_SL = OFF_S + 8192;              // state lo
constexpr uint32_t OFF_SMALL = OFF_SL + 8192;
constexpr uint32_t SMEM_BYTES = OFF_SMALL + 4096 + 1024;

// TMEM columns
constexpr uint32_t TM_D1a = 0, TM_D1b = 16, TM_D1c = 48, TM_D2 = 96, TM_D3 = 160;
constexpr uint32_t TM_NX = 256;    // [N | X0V | X0W]    192 columns
constexpr uint32_t TM_N2X = 0;     // [N^2 | N X0]       192 columns (after the levels)
constexpr uint32_t TM_X = 256;     // [Util | W], then [U ; Ctil S] in columns 0..63
constexpr uint32_t TM_CH = 384;    // [dS ; P U]
constexpr uint32_t TM_COLS = 512;

struct Small {
    float G[64];
    float A2[64];
    float decay[64];
    float scan[64];
    float g[kStages][64];
    float beta[kStages][64];
    uint64_t full[kStages], empty[kStages], mma;
    uint32_t tmem_base;
    uint32_t unsafe;
    uint32_t abort;
    float a2max;
};

__device__ __forceinline__ void ld_tm16(uint32_t taddr, float (&v)[16])
{
    tmem_ld16(taddr, v);
    tmem_wait_ld();
}

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

__device__ __forceinline__ void zero_rows(unsigned char* tile, int row)
{
#pragma unroll
    for (int q = 0; q < 8; q++) *reinterpret_cast<uint4*>(tile + sw128(row, 8 * q)) = make_uint4(0, 0, 0, 0);
}

// one MMA group: D[d] (+)= A x B over K = 64 (four K = 16 steps)
__device__ __forceinline__ void mma_k64(uint32_t d, uint32_t a, bool a_mn, uint32_t b, bool b_mn, uint32_t lbo_b,
                                        uint32_t idesc, bool acc)
{
#pragma unroll
    for (int ks = 0; ks < 4; ks++)
        mma_bf16(d, sdesc(a + (a_mn ? ks * 2048 : ks * 32), 16, 1024),
                 sdesc(b + (b_mn ? ks * 2048 : ks * 32), lbo_b, 1024), idesc, (acc || ks > 0) ? 1u : 0u);
}

__global__ void __launch_bounds__(kThreads, 1) fwd_tc_delta_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* X = sm + OFF_X;
    Small& S = *reinterpret_cast<Small*>(sm + OFF_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u = blockIdx.x, bb = u / p.H, h = u % p.H;
    const int T = p.T, H = p.H, dk = p.dk, dv = p.dv;

    if (tid < 64) {
        const float A = tid < dk ? -expf(p.A_log[h * dk + tid]) : 0.f;
        S.A2[tid] = A * kLog2e;
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) { mbar_init(&S.full[s], 1); mbar_init(&S.empty[s], 1); }
        mbar_init(&S.mma, 1);
        S.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&S.tmem_base, TM_COLS);
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&p.tm_v); tma_prefetch_desc(&p.tm_b); tma_prefetch_desc(&p.tm_c);
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

    if (warp == 4) {
        // ---------------------------------------------------------- producer
        int issued = 0;
        for (int k = 0; k < p.nchunks; k++) {
            const int s = k % kStages;
            if (k >= kStages && !wait_or_abort(&S.empty[s], ((k / kStages) - 1) & 1, &S.abort, p.status)) break;
            issued = k + 1;
            for (int tt = lane; tt < kC; tt += 32) {
                const int t = k * kC + tt;
                const size_t row = ((size_t)bb * T + t) * H + h;
                S.g[s][tt] = t < T ? __bfloat162float(p.g[row]) : 0.f;
                S.beta[s][tt] = t < T ? __bfloat162float(p.beta[row]) : 0.f;
            }
            __syncwarp();
            if (lane == 0) {
                unsigned char* st = sm + OFF_RING + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&S.full[s], STAGE_BYTES);
                tma_load_4d(st, &p.tm_v, &S.full[s], 0, h, k * kC, bb);
                tma_load_4d(st + 8192, &p.tm_b, &S.full[s], 0, h, k * kC, bb);
                tma_load_4d(st + 16384, &p.tm_c, &S.full[s], 0, h, k * kC, bb);
            }
            __syncwarp();
        }
        if (*(volatile uint32_t*)&S.abort && lane == 0)
            for (int k = issued > kStages ? issued - kStages : 0; k < issued; k++)
                mbar_wait(&S.full[k % kStages], (k / kStages) & 1, nullptr, 1u << 20);
    } else {
        // ---------------------------------------------------------- math
        const int r = tid;
        const int t = r & 63, hc = r >> 6;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const uint32_t tl = tbase + lane_base;     // this warp's TMEM lanes
        float Sreg[64];
        if (r < 64) {
#pragma unroll
            for (int j = 0; j < 64; j++)
                Sreg[j] = (p.h0 && r < dk && j < dv) ? p.h0[((size_t)u * dk + r) * dv + j] : 0.f;
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float v8[8];
#pragma unroll
                for (int e = 0; e < 8; e++) v8[e] = Sreg[8 * q + e];
                st_row8_split(sm + OFF_S, sm + OFF_SL, r, q, v8);
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        uint32_t mma_phase = 0;
        auto mma_sync_all = [&]() -> bool {
            if (!wait_or_abort(&S.mma, mma_phase, &S.abort, p.status)) return false;
            mma_phase ^= 1;
            tc_fence_after();
            return true;
        };
        auto smem_to_tc = [&]() {   // make generic-proxy smem writes visible to the MMAs
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(1, 128);
            tc_fence_after();
        };

        for (int k = 0; k < p.nchunks; k++) {
            const int s = k % kStages;
            if (!wait_or_abort(&S.full[s], (k / kStages) & 1, &S.abort, p.status)) break;
            unsigned char* sV = sm + OFF_RING + s * STAGE_BYTES;
            unsigned char* sB = sV + 8192;
            unsigned char* sCt = sV + 16384;

            // (1) inclusive scan of g
            if (r < 64) {
                float x = S.g[s][r];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                S.scan[r] = x;
            }
            named_bar_sync(1, 128);
            if (r < 64) S.G[r] = S.scan[r] + (r >= 32 ? S.scan[31] : 0.f);
            named_bar_sync(1, 128);
            if (warp == 0) {
                float span = 0.f;
                if (lane < 8) {
                    const float g0 = S.G[8 * lane], g3 = S.G[8 * lane + 3], g7 = S.G[8 * lane + 7];
                    span = fmaxf(g3 - g0, g7 - g3);
                }
                const bool bad = __any_sync(0xffffffffu, span * S.a2max > kSafeLog2);
                if (lane == 0) S.unsafe = bad ? 1u : 0u;
            }

            // (2) decay-scaled operands of the three levels (rows 0..63 c-side,
            //     rows 64..127 beta b-side) and Bhat^T
            {
                const float Gt = S.G[t];
                const int I = t >> 4;
                const float Gr1 = I > 0 ? S.G[16 * I - 1] : 0.f;
                const float Gr2 = S.G[16 * I + 7];
                const float Gr3 = S.G[8 * (t >> 3) + 3];
                const bool upper = (t & 15) >= 8;
                const float bet = S.beta[s][t];
#pragma unroll 1
                for (int qq = 0; qq < 4; qq++) {
                    const int q = hc * 4 + qq;
                    float cv[8], bv[8], bbv[8], y[8], z[8];
                    ld_row8(sCt, t, q, cv);
                    ld_row8(sB, t, q, bv);
#pragma unroll
                    for (int e = 0; e < 8; e++) bbv[e] = bet * bv[e];
                    if (I > 0) {
                        scale8(cv, S.A2, q, Gt - Gr1, y); st_row8_f16(X + X_A1, t, q, y);
                        scale8(bbv, S.A2, q, Gt - Gr1, z); st_row8_f16(X + X_A1, 64 + t, q, z);
                    }
                    if (upper) {
                        scale8(cv, S.A2, q, Gt - Gr2, y); st_row8_f16(X + X_A2, t, q, y);
                        scale8(bbv, S.A2, q, Gt - Gr2, z); st_row8_f16(X + X_A2, 64 + t, q, z);
                    }
                    scale8(cv, S.A2, q, Gt - Gr3, y); st_row8_split(X + X_A3, X + X_A3L, t, q, y);
                    scale8(bbv, S.A2, q, Gt - Gr3, z); st_row8_split(X + X_A3, X + X_A3L, 64 + t, q, z);
                    if (I < 1) { scale8(bv, S.A2, q, S.G[15] - Gt, y); st_row8_f16(X + X_B1a, t, q, y); }
                    if (I < 2) { scale8(bv, S.A2, q, S.G[31] - Gt, y); st_row8_f16(X + X_B1b, t, q, y); }
                    if (I < 3) { scale8(bv, S.A2, q, S.G[47] - Gt, y); st_row8_f16(X + X_B1c, t, q, y); }
                    if (!upper) { scale8(bv, S.A2, q, Gr2 - Gt, y); st_row8_f16(X + X_B2, t, q, y); }
                    scale8(bv, S.A2, q, Gr3 - Gt, y); st_row8_split(X + X_B3, X + X_B3L, t, q, y);
                }
                {
                    const int i = t;
                    const float a2 = S.A2[i], G63 = S.G[63];
#pragma unroll 1
                    for (int qq = 0; qq < 4; qq++) {
                        float y8[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            const int sc = 32 * hc + 8 * qq + e;
                            const float bval = bf2f(*reinterpret_cast<const uint16_t*>(sB + sw128(sc, i)));
                            y8[e] = bval * exp2f(a2 * (G63 - S.G[sc]));
                        }
                        st_row8_split(sm + OFF_CH0, sm + OFF_CH0L, i, 4 * hc + qq, y8);
                    }
                }
                if (r < 64) S.decay[r] = exp2f(S.A2[r] * S.G[63]);
            }
            smem_to_tc();

            // (3) level MMAs
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                const uint32_t b1[3] = {x0 + X_B1a, x0 + X_B1b, x0 + X_B1c};
                const uint32_t d1[3] = {TM_D1a, TM_D1b, TM_D1c};
#pragma unroll
                for (int I = 1; I <= 3; I++)
                    mma_k64(tbase + d1[I - 1], x0 + X_A1, false, b1[I - 1], false, 16, idesc_f16(128, 16 * I, false, false),
                            false);
                mma_k64(tbase + TM_D2, x0 + X_A2, false, x0 + X_B2, false, 16, idesc_f16(128, 64, false, false), false);
                const uint32_t id3 = idesc_bf16(128, 64, false, false);
                mma_k64(tbase + TM_D3, x0 + X_A3, false, x0 + X_B3, false, 16, id3, false);
                mma_k64(tbase + TM_D3, x0 + X_A3, false, x0 + X_B3L, false, 16, id3, true);
                mma_k64(tbase + TM_D3, x0 + X_A3L, false, x0 + X_B3, false, 16, id3, true);
                mma_commit(&S.mma);
            }
            if (!mma_sync_all()) break;

            // (4) assemble P (warps 0,1) and M (warps 2,3)
            {
                const bool unsafe = S.unsafe != 0;
                const bool isM = warp >= 2;
                const int wl = warp & 1;                 // 0: rows 0..31, 1: rows 32..63
                const int tb = t >> 4;
                float ew[8];
                if (unsafe) {
                    const int s0 = 8 * (t >> 3);
                    const float bet = S.beta[s][t];
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
                                    acc += xv[kk] * bv[kk] * exp2f(S.A2[8 * q + kk] * (S.G[t] - S.G[sc]));
                            }
                        }
                        ew[e] = isM ? bet * acc : acc;
                    }
                }
                const int Ia = 2 * wl, Ib = 2 * wl + 1;
                const uint32_t colA = wl == 0 ? 0u : TM_D1b, colB = wl == 0 ? TM_D1a : TM_D1c;
                float* M32 = reinterpret_cast<float*>(X + X_M32);
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
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
                            else val = unsafe ? ew[c & 7] : v3[c];
                            out[c] = val;
                        }
                    }
                    if (!isM) {
                        st_split16(sm + OFF_CH0, sm + OFF_CH0L, 64 + t, cg, out);
                    } else {
                        // L: strictly block-lower part; diagonal 16-blocks go to fp32
                        float lpart[16];
#pragma unroll
                        for (int c = 0; c < 16; c++) lpart[c] = (cg < tb) ? out[c] : 0.f;
                        st_plain16(X + X_LRH, t, cg, lpart);
                        if (cg == tb) {
#pragma unroll
                            for (int c = 0; c < 16; c++) M32[(tb * 16 + (t & 15)) * 16 + c] = out[c];
                        }
                    }
                }
            }
            // R = [beta V | beta Btil], hi into LRH blocks 1-2, lo into LRL blocks 0-1
            {
                const float bet = S.beta[s][t];
                const float Gt = S.G[t];
#pragma unroll 1
                for (int qq = 0; qq < 4; qq++) {
                    const int q = hc * 4 + qq;
                    float vv[8], bv[8], y[8];
                    ld_row8(sV, t, q, vv);
#pragma unroll
                    for (int e = 0; e < 8; e++) y[e] = bet * vv[e];
                    st_row8_split(X + X_LRH + 8192, X + X_LRL, t, q, y);
                    ld_row8(sB, t, q, bv);
#pragma unroll
                    for (int e = 0; e < 8; e++) y[e] = bet * bv[e];
                    scale8(y, S.A2, q, Gt, bv);
                    st_row8_split(X + X_LRH + 16384, X + X_LRL + 8192, t, q, bv);
                }
            }
            named_bar_sync(1, 128);

            // (5) inverse of the diagonal 16-blocks of I + M (fp32 forward substitution)
            if (r < 64) {
                const int J = r >> 4, c = r & 15;
                const float* M32 = reinterpret_cast<const float*>(X + X_M32) + J * 256;
                float xs[16];
#pragma unroll
                for (int q = 0; q < 16; q++) {
                    float acc = 0.f;
#pragma unroll
                    for (int pp = 0; pp < q; pp++)
                        if (pp >= c) acc = fmaf(M32[q * 16 + pp], xs[pp], acc);
                    xs[q] = (q < c) ? 0.f : (q == c ? 1.f : -acc);
                }
                float* DI32 = reinterpret_cast<float*>(X + X_DI32) + J * 256;
#pragma unroll
                for (int q = 0; q < 16; q++) DI32[q * 16 + c] = xs[q];
            }
            named_bar_sync(1, 128);
            if (r < 64) {
                const int J = t >> 4;
                const float* DI32 = reinterpret_cast<const float*>(X + X_DI32) + J * 256 + (t & 15) * 16;
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v16[16];
#pragma unroll
                    for (int c = 0; c < 16; c++) v16[c] = (cg == J) ? DI32[c] : 0.f;
                    st_plain16(X + X_DINV, t, cg, v16);
                }
            } else {
                zero_rows(X + X_DINV, r);
            }
            smem_to_tc();

            // (6) [N | X0] = Dinv [L | R]
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                mma_k64(tbase + TM_NX, x0 + X_DINV, false, x0 + X_LRH, true, 8192, idesc_bf16(128, 192, false, true),
                        false);
                mma_k64(tbase + TM_NX + 64, x0 + X_DINV, false, x0 + X_LRL, true, 8192,
                        idesc_bf16(128, 128, false, true), true);
                mma_commit(&S.mma);
            }
            if (!mma_sync_all()) break;

            // (7) N -> A operand and B block; X0 -> hi/lo B blocks
            if (r < 64) {
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v[16];
                    ld_tm16(tl + TM_NX + 16 * cg, v);
                    st_plain16(X + X_NA, t, cg, v);
                    st_plain16(X + X_NXH, t, cg, v);
                }
#pragma unroll
                for (int cg = 0; cg < 8; cg++) {
                    float v[16];
                    ld_tm16(tl + TM_NX + 64 + 16 * cg, v);
                    const uint32_t blk = (uint32_t)(cg >> 2) * 8192u;
                    st_split16(X + X_NXH + 8192 + blk, X + X_NXL + blk, t, cg & 3, v);
                }
            } else {
                zero_rows(X + X_NA, r);
            }
            smem_to_tc();

            // (8) [N^2 | N X0] = N [N | X0]
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                mma_k64(tbase + TM_N2X, x0 + X_NA, false, x0 + X_NXH, true, 8192, idesc_bf16(128, 192, false, true),
                        false);
                mma_k64(tbase + TM_N2X + 64, x0 + X_NA, false, x0 + X_NXL, true, 8192,
                        idesc_bf16(128, 128, false, true), true);
                mma_commit(&S.mma);
            }
            if (!mma_sync_all()) break;

            // (9) N^2 -> A operand; Z = X0 - N X0 -> hi/lo B blocks and, exactly, into TMEM
            if (r < 64) {
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v[16];
                    ld_tm16(tl + TM_N2X + 16 * cg, v);
                    st_plain16(X + X_N2A, t, cg, v);
                }
#pragma unroll
                for (int cg = 0; cg < 8; cg++) {
                    float x0v[16], nx[16];
                    tmem_ld16(tl + TM_NX + 64 + 16 * cg, x0v);
                    tmem_ld16(tl + TM_N2X + 64 + 16 * cg, nx);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; c++) x0v[c] -= nx[c];
                    const uint32_t blk = (uint32_t)(cg >> 2) * 8192u;
                    st_split16(X + X_ZH + blk, X + X_ZL + blk, t, cg & 3, x0v);
                    tmem_st16(tl + TM_X + 16 * cg, x0v);
                }
            } else {
                zero_rows(X + X_N2A, r);
                float zz[16];
#pragma unroll
                for (int c = 0; c < 16; c++) zz[c] = 0.f;
#pragma unroll
                for (int cg = 0; cg < 8; cg++) tmem_st16(tl + TM_X + 16 * cg, zz);
            }
            tmem_wait_st();
            smem_to_tc();

            // (10) X = Z + N^2 Z  ->  [Util | W]
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                const uint32_t id = idesc_bf16(128, 128, false, true);
                mma_k64(tbase + TM_X, x0 + X_N2A, false, x0 + X_ZH, true, 8192, id, true);
                mma_k64(tbase + TM_X, x0 + X_N2A, false, x0 + X_ZL, true, 8192, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_sync_all()) break;

            // (11) CW = [-W ; Ctil]
            if (r < 64) {
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v[16];
                    ld_tm16(tl + TM_X + 64 + 16 * cg, v);
#pragma unroll
                    for (int c = 0; c < 16; c++) v[c] = -v[c];
                    st_plain16(X + X_CW, t, cg, v);
                }
            } else {
                const float Gt = S.G[t];
#pragma unroll 1
                for (int q = 0; q < 8; q++) {
                    float cv[8], y[8];
                    ld_row8(sCt, t, q, cv);
                    scale8(cv, S.A2, q, Gt, y);
                    st_row8(X + X_CW, 64 + t, q, y);
                }
            }
            smem_to_tc();

            // (12) [U ; Ctil S] = [Util ; 0] + [-W ; Ctil] S
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                const uint32_t id = idesc_bf16(128, 64, false, true);
                mma_k64(tbase + TM_X, x0 + X_CW, false, smem_u32(sm + OFF_S), true, 8192, id, true);
                mma_k64(tbase + TM_X, x0 + X_CW, false, smem_u32(sm + OFF_SL), true, 8192, id, true);
                mma_commit(&S.mma);
            }
            if (!mma_sync_all()) break;

            // (13) U -> hi/lo B tiles
            if (r < 64) {
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v[16];
                    ld_tm16(tl + TM_X + 16 * cg, v);
                    st_split16(X + X_UH, X + X_UL, t, cg, v);
                }
            }
            smem_to_tc();

            // (14) [dS ; P U] = [Bhat^T ; P] U
            if (r == 0) {
                const uint32_t x0 = smem_u32(X);
                const uint32_t ch0 = smem_u32(sm + OFF_CH0), ch0l = smem_u32(sm + OFF_CH0L);
                const uint32_t id = idesc_bf16(128, 64, false, true);
                mma_k64(tbase + TM_CH, ch0, false, x0 + X_UH, true, 8192, id, false);
                mma_k64(tbase + TM_CH, ch0l, false, x0 + X_UH, true, 8192, id, true);
                mma_k64(tbase + TM_CH, ch0, false, x0 + X_UL, true, 8192, id, true);
                mma_commit(&S.empty[s]);
                mma_commit(&S.mma);
            }
            if (!mma_sync_all()) break;

            // (15) state update (rows 0..63) and output (rows 64..127)
            if (r < 64) {
                const float dec = S.decay[r];
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v[16];
                    ld_tm16(tl + TM_CH + 16 * cg, v);
#pragma unroll
                    for (int c = 0; c < 16; c++) Sreg[16 * cg + c] = fmaf(dec, Sreg[16 * cg + c], v[c]);
                }
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    float v8[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) v8[e] = Sreg[8 * q + e];
                    st_row8_split(sm + OFF_S, sm + OFF_SL, r, q, v8);
                }
            } else {
                const int tg = k * kC + t;
                __nv_bfloat16* orow = p.o + (((size_t)bb * T + tg) * H + h) * dv;
#pragma unroll
                for (int cg = 0; cg < 4; cg++) {
                    float v[16], w2[16];
                    tmem_ld16(tl + TM_CH + 16 * cg, v);
                    tmem_ld16(tl + TM_X + 16 * cg, w2);
                    tmem_wait_ld();
                    if (tg < T) {
#pragma unroll
                        for (int hq = 0; hq < 2; hq++) {
                            const int j0 = 16 * cg + 8 * hq;
                            if (j0 < dv) {
                                uint4 wv;
                                wv.x = pack_bf16(v[8 * hq + 0] + w2[8 * hq + 0], v[8 * hq + 1] + w2[8 * hq + 1]);
                                wv.y = pack_bf16(v[8 * hq + 2] + w2[8 * hq + 2], v[8 * hq + 3] + w2[8 * hq + 3]);
                                wv.z = pack_bf16(v[8 * hq + 4] + w2[8 * hq + 4], v[8 * hq + 5] + w2[8 * hq + 5]);
                                wv.w = pack_bf16(v[8 * hq + 6] + w2[8 * hq + 6], v[8 * hq + 7] + w2[8 * hq + 7]);
                                *reinterpret_cast<uint4*>(orow + j0) = wv;
                            }
                        }
                    }
                }
            }
            smem_to_tc();
        }
        if (r < 64 && p.hT && r < dk) {
            float* hrow = p.hT + ((size_t)u * dk + r) * dv;
#pragma unroll
            for (int j = 0; j < 64; j++)
                if (j < dv) hrow[j] = Sreg[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

}  // namespace

cudaError_t launch_fwd_tc_delta(const Args& a, cudaStream_t st)
{
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
    p.hT = a.hT;
    p.status = (uint32_t*)a.ws;
    p.B = a.B; p.H = a.H; p.T = a.T; p.dk = a.dk; p.dv = a.dv;
    p.nchunks = (a.T + kC - 1) / kC;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fwd_tc_delta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    fwd_tc_delta_kernel<<<a.B * a.H, kThreads, SMEM_BYTES, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
