// gdn_serial_bwd.cu -- token-serial backward of the gated delta rule on the
// CUDA cores (fp32 state and adjoint, packed fp32x2 arithmetic).
//
// The forward per token (gated: "GDN & MLA Mechanism Deep-Dive", Step 4;
// delta: the delta-rule card of "HyMo-434M -- documentation portal"):
//   h' = alpha_t (.) h_{t-1},  alpha_t = exp(g_t A),  A = -exp(A_log)
//   x  = v_t                        (gated)
//   x  = beta_t (v_t - h'^T b_t)    (delta)
//   h_t = h' + b_t x^T,   o_t = h_t^T c_t.
// Its adjoint, walked from the last token back with dH = dL/dh_t:
//   dH  += c_t do_t^T;         dc_t = h_t do_t
//   du   = dH^T b_t;           dv_t = beta du (delta) | du (gated)
//   dr   = -beta du;           dbeta_t = du . (v_t - h'^T b_t)
//   db_t = dH x + h' dr;       dH += b_t dr^T   (now dH = dL/dh')
//   q = dH (.) h';  dg_t = sum_ij A_i q_ij;  dA_log_i += A_i g_t sum_j q_ij
//   dH <- alpha_t (.) dH.
//
// One CTA per (batch, head) unit and slab of value columns, 256 threads.
// KIG lanes of a warp share a column pair, each holding eight rows: KIG = 8
// covers d_k <= 64 with 64 columns per CTA, KIG = 16 covers d_k <= 128 with 32
// columns per CTA.  Warp w owns columns 2 NJ w .. 2 NJ w + 2 NJ - 1 of its slab
// (NJ = 32 / KIG column pairs per warp); lane = KIG jl + ig holds columns
// j0 = 2 NJ w + 2 jl and j0 + 1 and the rows 8 ig .. 8 ig + 7, stored as four
// packed row pairs in an order permuted by jl so that the sums over columns
// (dc, db) need no selects.  Columns of the state never mix, so slabs are
// independent except for the sums over columns (db, dc, dg, dbeta, dA_log):
// with more than one slab each writes fp32 partials that a second kernel adds
// in a fixed order.
// Recompute: the forward sweep writes the state every 8 tokens (and, delta,
// x and v - h'^T b of every token) to the workspace; the reverse walk brings
// back one 32-token block of them at a time by cp.async, recomputes each
// 4-token window into registers from its snapshot and walks it backwards.
// Per-warp row partials are summed across warps once per window.
#include "gdn_internal.h"
#include "serial_common.cuh"

namespace gdn {
namespace {

using namespace rec;

constexpr int kBT = kSerialBlock;  // tokens per staged block = checkpoint interval
constexpr int kSub = kSerialSnap;  // tokens per state snapshot
constexpr int kWin = 4;            // tokens per register window
constexpr int kNQ = 2;             // row quantities summed over columns: dc, db

template <int KIG>
struct Cfg {
    static constexpr int ROWS = 8 * KIG;           // state rows covered (d_k <= ROWS)
    static constexpr int NJ = 32 / KIG;            // column pairs per warp
    static constexpr int COLS = 16 * NJ;           // value columns per CTA
    static constexpr int PBUF = KIG == 8 ? 2 : 1;  // row-partial buffers (one, and a barrier more, at 128 rows)
};

template <typename IO, int KIG>
struct BwdSmem {
    static constexpr int R = Cfg<KIG>::ROWS, NC = Cfg<KIG>::COLS;
    float A[kBT][R], Bv[kBT][R], Cv[kBT][R];                     // alpha_t, b_t, c_t
    float V[kBT][NC], DO[kBT][NC];                               // v_t, do_t on the slab's columns
    float XV[2][2][kBT][NC];      // two buffers of [x ; v_t - h'^T b_t] (the next block's arrives early)
    float beta[kBT], g[kBT];
    float Arow[R], Arow2[R];      // A and A log2(e)
    float2 snap[kBT / kSub][8][256];                             // per-thread state snapshots
    float part[Cfg<KIG>::PBUF][8][kWin][kNQ][R];                 // per-warp row partials
    float dvb[2][kWin][NC];
    float bpart[2][8][kWin], gpart[2][8][kWin];
    float red[8][R];
    float rg[kBT], rbeta[kBT];
    float nb[kBT], nc[kBT];       // GDN_NORM_BC: 1 / max(||b_t||, floor), the same for c_t
    IO rb[kBT][R], rc[kBT][R], rv[kBT][NC], rdo[kBT][NC];       // raw bytes of the next block
};

// eight consecutive staged values: raw I/O (16 bytes of bf16, 32 of fp32) -> fp32, and fp32 -> shared
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8])
{
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; k++) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8])
{
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

struct Ctx {
    int tid, lane, w, ig, jl, j0, m2, u, bb, h;
    int jc0, nv;  // first value column of the slab, columns in it
    int roff[4];  // float offset of register pair p inside a row vector
};

// where the sums over columns go: the outputs themselves (one slab) or fp32
// per-slab partials [slab][...] that reduce_slabs_kernel adds up
struct Outs {
    float *db, *dc, *dg, *dbeta;  // partial buffers, or NULL for direct output
};

__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }

template <typename IO, bool DELTA, int KIG>
__device__ __forceinline__ void issue_block(const Args& a, BwdSmem<IO, KIG>& s, const Ctx& C, int t0, bool grad,
                                            bool vec, IO& greg, IO& breg)
{
    constexpr int R = Cfg<KIG>::ROWS;
    const int tid = C.tid, dk = a.dk, dv = a.dv, T = a.T, H = a.H, nv = C.nv;
    const IO* vs = (const IO*)a.v + C.jc0;     // the slab's columns
    const IO* dOs = (const IO*)a.dO + C.jc0;
    const int nt = min(kBT, T - t0);
    const IO* bk = (const IO*)a.b;
    const IO* c = (const IO*)a.c;
    constexpr int E = 16 / sizeof(IO);
    if (vec) {
        const int cb = dk / E, cv = nv / E;
        const int per = grad ? 2 * (cb + cv) : cb + cv;
        for (int idx = tid; idx < nt * per; idx += 256) {
            const int tt = idx / per;
            int r = idx - tt * per;
            const size_t row = ((size_t)C.bb * T + t0 + tt) * H + C.h;
            if (r < cb) { cp_async16(&s.rb[tt][r * E], bk + row * dk + r * E); continue; }
            r -= cb;
            if (r < cv) { cp_async16(&s.rv[tt][r * E], vs + row * dv + r * E); continue; }
            r -= cv;
            if (r < cb) { cp_async16(&s.rc[tt][r * E], c + row * dk + r * E); continue; }
            r -= cb;
            cp_async16(&s.rdo[tt][r * E], dOs + row * dv + r * E);
        }
        cp_async_commit();
    } else {
        for (int idx = tid; idx < nt * R; idx += 256) {
            const int tt = idx / R, i = idx % R;
            const size_t row = ((size_t)C.bb * T + t0 + tt) * H + C.h;
            if (i < dk) {
                s.rb[tt][i] = bk[row * dk + i];
                if (grad) s.rc[tt][i] = c[row * dk + i];
            }
            if (i < nv) {
                s.rv[tt][i] = vs[row * dv + i];
                if (grad) s.rdo[tt][i] = dOs[row * dv + i];
            }
        }
    }
    // g, beta stay raw until finish_block stores them: nothing waits on these loads meanwhile
    if (tid < nt) greg = ((const IO*)a.g)[((size_t)C.bb * T + t0 + tid) * H + C.h];
    if (DELTA && tid >= 32 && tid - 32 < nt)
        breg = ((const IO*)a.beta)[((size_t)C.bb * T + t0 + tid - 32) * H + C.h];
}

// Make the block issued last the current one.  Tokens past T become identity
// steps (alpha = 1, every other input 0), so a block is always 32 tokens.
template <typename IO, bool DELTA, int KIG>
__device__ __forceinline__ void finish_block(const Args& a, BwdSmem<IO, KIG>& s, const Ctx& C, int t0, bool grad,
                                             IO greg, IO breg, bool leave_newest = false)
{
    constexpr int R = Cfg<KIG>::ROWS, NC = Cfg<KIG>::COLS;
    const int tid = C.tid, dk = a.dk, nv = C.nv;
    const int nt = min(kBT, a.T - t0);
    if (tid < 32) s.rg[tid] = gate(to_f(greg), a.logits);
    else if (tid < 64) s.rbeta[tid - 32] = gate(to_f(breg), a.logits);
    if (leave_newest) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    else cp_async_wait_all();
    __syncthreads();
    if (a.norm) {   // inverse norms of the block's b_t (and c_t), one thread per vector
        if (tid < 2 * nt) {
            const int tt = tid >> 1;
            const IO* x = (tid & 1) ? s.rc[tt] : s.rb[tt];
            float q = 0.f;
            if (!(tid & 1) || grad)
                for (int k = 0, i = tt % dk; k < dk; k++, i = i + 1 < dk ? i + 1 : 0)   // rotated: fewer bank conflicts
                    q = fmaf(to_f(x[i]), to_f(x[i]), q);
            (tid & 1 ? s.nc : s.nb)[tt] = 1.f / fmaxf(sqrtf(q), kNormFloor);
        }
        __syncthreads();
    }
    if (sizeof(IO) == 4) {   // fp32 I/O: element by element (measured faster than the 8-wide form here)
        for (int idx = tid; idx < kBT * R; idx += 256) {
            const int tt = idx / R, i = idx % R;
            const bool ok = tt < nt;
            const float sb = a.norm && ok ? s.nb[tt] : 1.f, sc = a.norm && ok ? s.nc[tt] : 1.f;
            s.A[tt][i] = ok ? decay<IO>(s.rg[tt], s.Arow[i], s.Arow2[i]) : 1.f;
            s.Bv[tt][i] = ok && i < dk ? to_f(s.rb[tt][i]) * sb : 0.f;
            s.Cv[tt][i] = grad && ok && i < dk ? to_f(s.rc[tt][i]) * sc : 0.f;
        }
        for (int idx = tid; idx < kBT * NC; idx += 256) {
            const int tt = idx / NC, i = idx % NC;
            const bool ok = tt < nt;
            s.V[tt][i] = ok && i < nv ? to_f(s.rv[tt][i]) : 0.f;
            s.DO[tt][i] = grad && ok && i < nv ? to_f(s.rdo[tt][i]) : 0.f;
        }
    } else {
    // bf16: eight consecutive values per thread, one 16-byte raw load and two 16-byte stores per array
    for (int ch = tid; ch < kBT * (R / 8); ch += 256) {
        const int tt = ch / (R / 8), i0 = (ch % (R / 8)) * 8;
        const bool ok = tt < nt;
        const float sb = a.norm && ok ? s.nb[tt] : 1.f, sc = a.norm && ok ? s.nc[tt] : 1.f;
        const float gt = s.rg[tt];
        float av[8], bv[8], cv[8];
        load8(&s.rb[tt][i0], bv);
        if (grad) load8(&s.rc[tt][i0], cv);
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = i0 + e;
            const bool live = ok && i < dk;
            av[e] = ok ? decay<IO>(gt, s.Arow[i], s.Arow2[i]) : 1.f;
            bv[e] = live ? bv[e] * sb : 0.f;
            cv[e] = grad && live ? cv[e] * sc : 0.f;
        }
        store8(&s.A[tt][i0], av);
        store8(&s.Bv[tt][i0], bv);
        store8(&s.Cv[tt][i0], cv);
    }
    for (int ch = tid; ch < kBT * (NC / 8); ch += 256) {
        const int tt = ch / (NC / 8), j0 = (ch % (NC / 8)) * 8;
        const bool ok = tt < nt;
        float vv[8], dd[8];
        load8(&s.rv[tt][j0], vv);
        if (grad) load8(&s.rdo[tt][j0], dd);
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const bool live = ok && j0 + e < nv;
            vv[e] = live ? vv[e] : 0.f;
            dd[e] = grad && live ? dd[e] : 0.f;
        }
        store8(&s.V[tt][j0], vv);
        store8(&s.DO[tt][j0], dd);
    }
    }
    if (tid < kBT) {
        const bool ok = tid < nt;
        s.g[tid] = ok ? s.rg[tid] : 0.f;
        s.beta[tid] = DELTA && ok ? s.rbeta[tid] : 0.f;
    }
    __syncthreads();
}

// one token's staged row vectors as this thread uses them (loaded a token ahead in the forward sweep)
struct TokRows {
    float2 a2[4], b2[4], v2;
    float be;
};

__device__ __forceinline__ void load_tok(TokRows& r, const float* A, const float* Bv, const float* V, float be,
                                         const Ctx& C)
{
#pragma unroll
    for (int p = 0; p < 4; p++) {
        r.a2[p] = ld2(A + C.roff[p]);
        r.b2[p] = ld2(Bv + C.roff[p]);
    }
    r.v2 = ld2(V + C.j0);
    r.be = be;
}

// one forward step with the row reduction h'^T b (delta); optionally caches
// x and v - h'^T b for the window recompute and the adjoint
template <bool DELTA, bool CACHE, int KIG>
__device__ __forceinline__ void fwd_full(float2 (&S)[2][4], const TokRows& r, float* X, float* VR, const Ctx& C)
{
    const float2 (&a2)[4] = r.a2;
    const float2 (&b2)[4] = r.b2;
    const float2 v2 = r.v2;
    const float be = r.be;
    float2 hp[2][4];
#pragma unroll
    for (int c = 0; c < 2; c++)
#pragma unroll
        for (int p = 0; p < 4; p++) hp[c][p] = mul2(S[c][p], a2[p]);
    float x0, x1;
    if (DELTA) {
        float2 r0 = mul2(hp[0][0], b2[0]), r1 = mul2(hp[1][0], b2[0]);
#pragma unroll
        for (int p = 1; p < 4; p++) {
            r0 = fma2(hp[0][p], b2[p], r0);
            r1 = fma2(hp[1][p], b2[p], r1);
        }
        float q0 = r0.x + r0.y, q1 = r1.x + r1.y;
#pragma unroll
        for (int o = 1; o < KIG; o <<= 1) {
            q0 += __shfl_xor_sync(kFull, q0, o);
            q1 += __shfl_xor_sync(kFull, q1, o);
        }
        const float vr0 = v2.x - q0, vr1 = v2.y - q1;
        x0 = be * vr0;
        x1 = be * vr1;
        if (CACHE && C.ig == 0) {
            *reinterpret_cast<float2*>(X + C.j0) = f2(x0, x1);
            *reinterpret_cast<float2*>(VR + C.j0) = f2(vr0, vr1);
        }
    } else {
        x0 = v2.x;
        x1 = v2.y;
    }
    const float2 xx0 = f2(x0, x0), xx1 = f2(x1, x1);
#pragma unroll
    for (int p = 0; p < 4; p++) {
        S[0][p] = fma2(b2[p], xx0, hp[0][p]);
        S[1][p] = fma2(b2[p], xx1, hp[1][p]);
    }
}

// one forward step with x already known (window recompute)
__device__ __forceinline__ void fwd_cached(const float2 (&Si)[2][4], float2 (&So)[2][4], const float* A,
                                           const float* Bv, const float* X, const Ctx& C)
{
    float2 a2[4], b2[4];
#pragma unroll
    for (int p = 0; p < 4; p++) {
        a2[p] = ld2(A + C.roff[p]);
        b2[p] = ld2(Bv + C.roff[p]);
    }
    const float2 x2 = ld2(X + C.j0);
    const float2 xx0 = f2(x2.x, x2.x), xx1 = f2(x2.y, x2.y);
#pragma unroll
    for (int p = 0; p < 4; p++) {
        So[0][p] = fma2(b2[p], xx0, mul2(Si[0][p], a2[p]));
        So[1][p] = fma2(b2[p], xx1, mul2(Si[1][p], a2[p]));
    }
}

// Sum four packed row pairs over the four column-pair lanes jl of a row
// group (KIG = 8: lanes ig, ig+8, ig+16, ig+24).  Pair p of lane (jl) holds
// rows 2 (p ^ m2) of the group with m2 = 2 (jl & 1) + (jl >> 1); the result
// holds rows 2 m2, 2 m2 + 1.
__device__ __forceinline__ float2 colsum_pairs(const float2 (&x)[4])
{
    float2 y0, y1;
    y0.x = x[0].x + __shfl_xor_sync(kFull, x[2].x, 8);
    y0.y = x[0].y + __shfl_xor_sync(kFull, x[2].y, 8);
    y1.x = x[1].x + __shfl_xor_sync(kFull, x[3].x, 8);
    y1.y = x[1].y + __shfl_xor_sync(kFull, x[3].y, 8);
    float2 z;
    z.x = y0.x + __shfl_xor_sync(kFull, y1.x, 16);
    z.y = y0.y + __shfl_xor_sync(kFull, y1.y, 16);
    return z;
}

// The same over the two column-pair lanes of a row group at KIG = 16 (lanes
// ig, ig+16), with m2 = 2 jl: lane jl ends with rows 4 jl .. 4 jl + 3.
__device__ __forceinline__ float4 colsum_pairs2(const float2 (&x)[4])
{
    float4 z;
    z.x = x[0].x + __shfl_xor_sync(kFull, x[2].x, 16);
    z.y = x[0].y + __shfl_xor_sync(kFull, x[2].y, 16);
    z.z = x[1].x + __shfl_xor_sync(kFull, x[3].x, 16);
    z.w = x[1].y + __shfl_xor_sync(kFull, x[3].y, 16);
    return z;
}

// the warp's sum over its columns of four packed row pairs, into a row vector
template <int KIG>
__device__ __forceinline__ void colsum_store(const float2 (&x)[4], float* rowvec, const Ctx& C)
{
    if (KIG == 8) *reinterpret_cast<float2*>(rowvec + 8 * C.ig + 2 * C.m2) = colsum_pairs(x);
    else *reinterpret_cast<float4*>(rowvec + 8 * C.ig + 4 * C.jl) = colsum_pairs2(x);
}

template <typename IO, bool DELTA, int KIG>
__global__ void __launch_bounds__(256, 1) serial_bwd_kernel(Args a, WsLayout L, Outs out, bool vec)
{
    constexpr int R = Cfg<KIG>::ROWS, NJ = Cfg<KIG>::NJ, NC = Cfg<KIG>::COLS, PBUF = Cfg<KIG>::PBUF;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem<IO, KIG>& s = *reinterpret_cast<BwdSmem<IO, KIG>*>(smem_raw);
    Ctx C;
    C.tid = threadIdx.x;
    C.lane = C.tid & 31;
    C.w = C.tid >> 5;
    C.ig = C.lane % KIG;
    C.jl = C.lane / KIG;
    C.j0 = 2 * NJ * C.w + 2 * C.jl;
    C.m2 = KIG == 8 ? 2 * (C.jl & 1) + (C.jl >> 1) : 2 * C.jl;
#pragma unroll
    for (int p = 0; p < 4; p++) C.roff[p] = 8 * C.ig + 2 * (p ^ C.m2);
    C.u = blockIdx.x;
    C.bb = C.u / a.H;
    C.h = C.u % a.H;
    C.jc0 = NC * (int)blockIdx.y;
    C.nv = min(NC, a.dv - C.jc0);
    const int tid = C.tid, lane = C.lane, w = C.w;
    const int dk = a.dk, dv = a.dv, T = a.T, H = a.H, nv = C.nv;
    const int nblk = (T + kBT - 1) / kBT;
    const size_t cta = (size_t)C.u * gridDim.y + blockIdx.y;   // this CTA's workspace slot
    constexpr int kSnapPerBlk = kBT / kSub;
    float2* gsnap = reinterpret_cast<float2*>((unsigned char*)a.ws + L.snap_off) + cta * nblk * kSnapPerBlk * 2048;
    float* gxvr = reinterpret_cast<float*>((unsigned char*)a.ws + L.xvr_off) + cta * nblk * kBT * 2 * NC;
    float* dA_part = reinterpret_cast<float*>((unsigned char*)a.ws + L.dalog_off) + cta * dk;
    const size_t slab_tok = (size_t)blockIdx.y * a.B * T * H;   // offset of this slab's partials, in tokens

    if (tid < R) {
        const float Ai = tid < dk ? -expf(a.A_log[C.h * dk + tid]) : 0.f;
        s.Arow[tid] = Ai;
        s.Arow2[tid] = Ai * 1.4426950408889634f;
    }

    // load a [B,H,dk,dv] fp32 matrix in this thread's register layout
    auto load_state = [&](const float* src, float2 (&S)[2][4]) {
#pragma unroll
        for (int c = 0; c < 2; c++)
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const int i0 = C.roff[p], j = C.j0 + c;
                float x0 = 0.f, x1 = 0.f;
                if (src && j < nv) {
                    if (i0 < dk) x0 = src[((size_t)C.u * dk + i0) * dv + C.jc0 + j];
                    if (i0 + 1 < dk) x1 = src[((size_t)C.u * dk + i0 + 1) * dv + C.jc0 + j];
                }
                S[c][p] = f2(x0, x1);
            }
    };

    float2 S[2][4];
    load_state(a.h0, S);

    // ---------------- forward sweep: state entering every block ----------------
    IO greg = from_f<IO>(0.f), breg = from_f<IO>(0.f);
    __syncthreads();  // Arow
    issue_block<IO, DELTA, KIG>(a, s, C, 0, false, vec, greg, breg);
    for (int n = 0; n < nblk; n++) {
        finish_block<IO, DELTA, KIG>(a, s, C, n * kBT, false, greg, breg);
        if (n + 1 < nblk) issue_block<IO, DELTA, KIG>(a, s, C, (n + 1) * kBT, false, vec, greg, breg);
        else issue_block<IO, DELTA, KIG>(a, s, C, n * kBT, true, vec, greg, breg);  // first block of the reverse walk
        float2* snap_n = gsnap + (size_t)n * kSnapPerBlk * 2048;
        float* xvr_n = gxvr + (size_t)n * kBT * 2 * NC;
        // the next token's row vectors are loaded while this one computes
        TokRows cur, nxt;
        load_tok(nxt, s.A[0], s.Bv[0], s.V[0], s.beta[0], C);
#pragma unroll 2
        for (int tt = 0; tt < kBT; tt++) {
            cur = nxt;
            if (tt + 1 < kBT) load_tok(nxt, s.A[tt + 1], s.Bv[tt + 1], s.V[tt + 1], s.beta[tt + 1], C);
            if ((tt & (kSub - 1)) == 0) {
#pragma unroll
                for (int q = 0; q < 8; q++) snap_n[((tt / kSub) * 8 + q) * 256 + tid] = S[q >> 2][q & 3];
            }
            fwd_full<DELTA, DELTA, KIG>(S, cur, xvr_n + tt * NC, xvr_n + kBT * NC + tt * NC, C);
        }
    }

    // the reverse walk reads back what other threads stored in the sweep
    __syncthreads();

    // ---------------- adjoint: dH = dh_T ----------------
    float2 dS[2][4];
    load_state(a.dhT, dS);
    float2 Ap[4], dA_acc[4];  // A of this thread's row pairs; sum_t g_t sum_j q over its columns
#pragma unroll
    for (int p = 0; p < 4; p++) {
        Ap[p] = ld2(&s.Arow[C.roff[p]]);
        dA_acc[p] = f2(0.f, 0.f);
    }
    int wbuf = 0;

    // Snapshots and x cache of block n come back from the workspace: the x cache one block ahead into the other
    // buffer, snapshot sb of block n-1 as soon as block n's windows are done with slot sb.
    auto fetch_snap = [&](int n, int sb) {
        const float4* src = reinterpret_cast<const float4*>(gsnap + ((size_t)n * kSnapPerBlk + sb) * 2048);
        float4* dst = reinterpret_cast<float4*>(&s.snap[sb][0][0]);
        for (int idx = tid; idx < 2048 / 2; idx += 256) cp_async16(dst + idx, src + idx);
    };
    auto fetch_xv = [&](int n) {
        if (!DELTA) return;
        const float4* sx = reinterpret_cast<const float4*>(gxvr + (size_t)n * kBT * 2 * NC);
        float4* dx = reinterpret_cast<float4*>(&s.XV[n & 1][0][0][0]);
        for (int idx = tid; idx < kBT * 2 * NC / 4; idx += 256) cp_async16(dx + idx, sx + idx);
    };
    for (int sb = 0; sb < kSnapPerBlk; sb++) fetch_snap(nblk - 1, sb);
    fetch_xv(nblk - 1);
    cp_async_commit();

    // ---------------- reverse walk over blocks ----------------
    for (int n = nblk - 1; n >= 0; n--) {
        const int t0 = n * kBT;
        // waits for this block's inputs, x cache and snapshots but the last (slot 0, needed from window 1 on)
        finish_block<IO, DELTA, KIG>(a, s, C, t0, true, greg, breg, n < nblk - 1);
        if (n > 0) {
            issue_block<IO, DELTA, KIG>(a, s, C, t0 - kBT, true, vec, greg, breg);
            fetch_xv(n - 1);
            cp_async_commit();
        }
        const float* Xsrc = DELTA ? &s.XV[n & 1][0][0][0] : &s.V[0][0];
        const float* VRsrc = &s.XV[n & 1][1][0][0];

#pragma unroll 1
        for (int wi = kBT / kWin - 1; wi >= 0; wi--) {
            const int tw = kWin * wi;  // first token of the window inside the block
            const int pb = PBUF == 2 ? wbuf : 0;
            float gsv[kWin], pbv[kWin];   // this lane's dg and dbeta partials of the window's tokens
            float2 W[kWin + 1][2][4];
            {
                const int sb = tw / kSub;
#pragma unroll
                for (int q = 0; q < 8; q++) W[0][q >> 2][q & 3] = s.snap[sb][q][tid];
                if (tw & (kSub - 1)) {
                    // advance from the snapshot to the window start
#pragma unroll
                    for (int k = 0; k < kWin; k++) {
                        const int tt = sb * kSub + k;
                        float2 Tm[2][4];
                        fwd_cached(W[0], Tm, s.A[tt], s.Bv[tt], Xsrc + tt * NC, C);
#pragma unroll
                        for (int q = 0; q < 8; q++) W[0][q >> 2][q & 3] = Tm[q >> 2][q & 3];
                    }
                }
#pragma unroll
                for (int k = 0; k < kWin; k++) {
                    const int tt = tw + k;
                    fwd_cached(W[k], W[k + 1], s.A[tt], s.Bv[tt], Xsrc + tt * NC, C);
                }
            }
#pragma unroll
            for (int k = kWin - 1; k >= 0; k--) {
                const int tt = tw + k;
                float2 a2[4], b2[4], c2[4];
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    a2[p] = ld2(&s.A[tt][C.roff[p]]);
                    b2[p] = ld2(&s.Bv[tt][C.roff[p]]);
                    c2[p] = ld2(&s.Cv[tt][C.roff[p]]);
                }
                const float2 do2 = ld2(&s.DO[tt][C.j0]);
                const float2 d0 = f2(do2.x, do2.x), d1 = f2(do2.y, do2.y);
                float2 pdc[4];
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    dS[0][p] = fma2(c2[p], d0, dS[0][p]);
                    dS[1][p] = fma2(c2[p], d1, dS[1][p]);
                    pdc[p] = fma2(W[k + 1][0][p], d0, mul2(W[k + 1][1][p], d1));
                }
                float du0, du1;
                {
                    float2 r0 = mul2(dS[0][0], b2[0]), r1 = mul2(dS[1][0], b2[0]);
#pragma unroll
                    for (int p = 1; p < 4; p++) {
                        r0 = fma2(dS[0][p], b2[p], r0);
                        r1 = fma2(dS[1][p], b2[p], r1);
                    }
                    du0 = r0.x + r0.y;
                    du1 = r1.x + r1.y;
#pragma unroll
                    for (int o = 1; o < KIG; o <<= 1) {
                        du0 += __shfl_xor_sync(kFull, du0, o);
                        du1 += __shfl_xor_sync(kFull, du1, o);
                    }
                }
                const float2 x2 = ld2(Xsrc + tt * NC + C.j0);
                const float2 xx0 = f2(x2.x, x2.x), xx1 = f2(x2.y, x2.y);
                float2 pdb[4];
                float pbeta = 0.f, dv0, dv1;
                const float2 gg = f2(s.g[tt], s.g[tt]);
                float2 gq = f2(0.f, 0.f);
                if (DELTA) {
                    const float be = s.beta[tt];
                    const float2 vr2 = ld2(VRsrc + tt * NC + C.j0);
                    const float dr0 = -be * du0, dr1 = -be * du1;
                    dv0 = be * du0;
                    dv1 = be * du1;
                    pbeta = du0 * vr2.x + du1 * vr2.y;
                    const float2 e0 = f2(dr0, dr0), e1 = f2(dr1, dr1);
#pragma unroll
                    for (int p = 0; p < 4; p++) {
                        const float2 hp0 = mul2(W[k][0][p], a2[p]), hp1 = mul2(W[k][1][p], a2[p]);
                        pdb[p] = fma2(hp0, e0, fma2(hp1, e1, fma2(dS[0][p], xx0, mul2(dS[1][p], xx1))));
                        const float2 g0 = fma2(b2[p], e0, dS[0][p]), g1 = fma2(b2[p], e1, dS[1][p]);
                        const float2 qs = fma2(g0, hp0, mul2(g1, hp1));
                        dA_acc[p] = fma2(gg, qs, dA_acc[p]);
                        gq = fma2(Ap[p], qs, gq);
                        dS[0][p] = mul2(g0, a2[p]);
                        dS[1][p] = mul2(g1, a2[p]);
                    }
                } else {
                    dv0 = du0;
                    dv1 = du1;
#pragma unroll
                    for (int p = 0; p < 4; p++) {
                        const float2 hp0 = mul2(W[k][0][p], a2[p]), hp1 = mul2(W[k][1][p], a2[p]);
                        pdb[p] = fma2(dS[0][p], xx0, mul2(dS[1][p], xx1));
                        const float2 qs = fma2(dS[0][p], hp0, mul2(dS[1][p], hp1));
                        dA_acc[p] = fma2(gg, qs, dA_acc[p]);
                        gq = fma2(Ap[p], qs, gq);
                        dS[0][p] = mul2(dS[0][p], a2[p]);
                        dS[1][p] = mul2(dS[1][p], a2[p]);
                    }
                }
                colsum_store<KIG>(pdc, s.part[pb][w][k][0], C);
                colsum_store<KIG>(pdb, s.part[pb][w][k][1], C);
                gsv[k] = gq.x + gq.y;   // warp sums taken for the whole window below
                pbv[k] = pbeta;
                if (C.ig == 0) *reinterpret_cast<float2*>(&s.dvb[wbuf][k][C.j0]) = f2(dv0, dv1);
            }
            // the window's four dg (and dbeta) warp sums at once: a reduce-scatter over lane bits 4 and 3 leaves
            // token (lane >> 3) & 3 in lanes 8 (lane >> 3), then the remaining lanes are summed (dg only; dbeta's
            // partials are equal across the row lanes)
            {
                static_assert(kWin == 4, "the window reduce-scatter is written for four tokens");
                const bool h16 = lane & 16, h8 = lane & 8;
                float a0 = (h16 ? gsv[2] : gsv[0]) + __shfl_xor_sync(kFull, h16 ? gsv[0] : gsv[2], 16);
                float a1 = (h16 ? gsv[3] : gsv[1]) + __shfl_xor_sync(kFull, h16 ? gsv[1] : gsv[3], 16);
                float g1 = (h8 ? a1 : a0) + __shfl_xor_sync(kFull, h8 ? a0 : a1, 8);
#pragma unroll
                for (int o = 4; o > 0; o >>= 1) g1 += __shfl_xor_sync(kFull, g1, o);
                if ((lane & 7) == 0) s.gpart[wbuf][w][(lane >> 3) & 3] = g1;
                if (DELTA) {
                    float b0 = (h16 ? pbv[2] : pbv[0]) + __shfl_xor_sync(kFull, h16 ? pbv[0] : pbv[2], 16);
                    float b1 = (h16 ? pbv[3] : pbv[1]) + __shfl_xor_sync(kFull, h16 ? pbv[1] : pbv[3], 16);
                    if (KIG == 8) {   // jl = lane >> 3: sum over lane bits 4 and 3
                        const float bb = (h8 ? b1 : b0) + __shfl_xor_sync(kFull, h8 ? b0 : b1, 8);
                        if ((lane & 7) == 0) s.bpart[wbuf][w][(lane >> 3) & 3] = bb;
                    } else {          // jl = lane >> 4: sum over lane bit 4 only
                        if ((lane & 15) == 0) {
                            s.bpart[wbuf][w][2 * (lane >> 4)] = b0;
                            s.bpart[wbuf][w][2 * (lane >> 4) + 1] = b1;
                        }
                    }
                }
            }
            if (wi == 2 && n < nblk - 1) cp_async_wait_all();   // snapshot slot 0, read from window 1 on
            __syncthreads();
            if (n > 0 && (tw & (kSub - 1)) == 0) {   // slot tw / kSub is done for this block
                fetch_snap(n - 1, tw / kSub);
                cp_async_commit();
            }

            // ---- reduction phase: thread (row ri, token rk) of this window ----
            {
#pragma unroll
                for (int e0 = 0; e0 < kWin * R; e0 += 256) {   // one pass at 64 rows, two at 128
                    const int e = e0 + tid, ri = e % R, rk = e / R;
                    const int tt = tw + rk, t = t0 + tt;
                    const bool live = t < T;
                    float dc = 0.f, db = 0.f;
#pragma unroll
                    for (int ww = 0; ww < 8; ww++) {
                        dc += s.part[pb][ww][rk][0][ri];
                        db += s.part[pb][ww][rk][1][ri];
                    }
                    const size_t row = ((size_t)C.bb * T + t) * H + C.h;
                    if (live && ri < dk) {
                        if (out.db) {
                            out.dc[(slab_tok + row) * dk + ri] = dc;
                            out.db[(slab_tok + row) * dk + ri] = db;
                        } else {
                            ((IO*)a.dc)[row * dk + ri] = from_f<IO>(dc);
                            ((IO*)a.db)[row * dk + ri] = from_f<IO>(db);
                        }
                    }
                    if (live && ri < nv) ((IO*)a.dv_)[row * dv + C.jc0 + ri] = from_f<IO>(s.dvb[wbuf][rk][ri]);
                }
                if (tid < kWin && t0 + tw + tid < T) {
                    const size_t rowk = ((size_t)C.bb * T + t0 + tw + tid) * H + C.h;
                    float sg = 0.f, sb = 0.f;
#pragma unroll
                    for (int ww = 0; ww < 8; ww++) {
                        sg += s.gpart[wbuf][ww][tid];
                        sb += s.bpart[wbuf][ww][tid];
                    }
                    if (a.logits) {   // through the sigmoid: d sigma(z) / dz = sigma (1 - sigma)
                        const float gv = s.g[tw + tid], bv = s.beta[tw + tid];
                        sg *= gv * (1.f - gv);
                        sb *= bv * (1.f - bv);
                    }
                    if (out.dg) {
                        out.dg[slab_tok + rowk] = sg;
                        if (DELTA) out.dbeta[slab_tok + rowk] = sb;
                    } else {
                        ((IO*)a.dg)[rowk] = from_f<IO>(sg);
                        if (DELTA) ((IO*)a.dbeta)[rowk] = from_f<IO>(sb);
                    }
                }
            }
            if (PBUF == 1) __syncthreads();   // the single partial buffer is read out before the next window
            wbuf ^= 1;
        }
    }
    if (a.dh0) {
#pragma unroll
        for (int c = 0; c < 2; c++)
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const int i0 = C.roff[p], j = C.j0 + c;
                if (j < nv) {
                    if (i0 < dk) a.dh0[((size_t)C.u * dk + i0) * dv + C.jc0 + j] = dS[c][p].x;
                    if (i0 + 1 < dk) a.dh0[((size_t)C.u * dk + i0 + 1) * dv + C.jc0 + j] = dS[c][p].y;
                }
            }
    }
    // dA_log partial of this unit: A_i sum_t g_t sum_j q_ij
    {
        colsum_store<KIG>(dA_acc, s.red[w], C);
        __syncthreads();
        for (int i = tid; i < dk; i += 256) {
            float acc = 0.f;
#pragma unroll
            for (int ww = 0; ww < 8; ww++) acc += s.red[ww][i];
            dA_part[i] = acc * s.Arow[i];
        }
    }
}

// dA_log[h, i] = sum_b sum_slab partial[b, h, slab, i]  (fixed order, deterministic)
__global__ void reduce_dalog_kernel(const float* part, float* dA_log, int B, int H, int dk, int nslab)
{
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= H * dk) return;
    const int h = idx / dk, i = idx % dk;
    float acc = 0.f;
    for (int b = 0; b < B; b++)
        for (int sl = 0; sl < nslab; sl++) acc += part[(((size_t)b * H + h) * nslab + sl) * dk + i];
    dA_log[idx] = acc;
}

// out[i] = sum_slab part[slab][i], slabs in order (deterministic)
template <typename IO>
__global__ void reduce_slabs_kernel(const float* part, IO* outp, size_t n, int nslab)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        float acc = part[i];
        for (int sl = 1; sl < nslab; sl++) acc += part[(size_t)sl * n + i];
        outp[i] = from_f<IO>(acc);
    }
}

// db or dc of each (token, head) row: the column slabs' fp32 partials added in order, then, with
// GDN_NORM_BC, taken through the normalisation y = x / max(||x||, floor) of the vector x as given:
// dL/dx = (d - y <y, d>) / ||x|| (d / floor below the floor).  One warp per row, d_k <= 128.
template <typename IO>
__global__ void finish_keys_kernel(const float* part, const IO* x, IO* outp, size_t nrows, int dk, int nslab,
                                   size_t slab_stride, int norm)
{
    const int lane = threadIdx.x & 31;
    const size_t wpb = blockDim.x / 32;
    for (size_t row = blockIdx.x * wpb + (threadIdx.x >> 5); row < nrows; row += (size_t)gridDim.x * wpb) {
        float d[4], xv[4];
        float q = 0.f;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = lane + 32 * k;
            d[k] = xv[k] = 0.f;
            if (i < dk) {
                const size_t at = row * dk + i;
                float acc = part[at];
                for (int sl = 1; sl < nslab; sl++) acc += part[(size_t)sl * slab_stride + at];
                d[k] = acc;
                xv[k] = to_f(x[at]);
                q = fmaf(xv[k], xv[k], q);
            }
        }
        if (norm) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(kFull, q, o);
            const float n = sqrtf(q), inv = 1.f / fmaxf(n, kNormFloor);
            float yd = 0.f;
#pragma unroll
            for (int k = 0; k < 4; k++) yd = fmaf(xv[k] * inv, d[k], yd);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) yd += __shfl_xor_sync(kFull, yd, o);
            const bool big = n > kNormFloor;
#pragma unroll
            for (int k = 0; k < 4; k++) d[k] = big ? (d[k] - xv[k] * inv * yd) * inv : d[k] * inv;
        }
#pragma unroll
        for (int k = 0; k < 4; k++)
            if (lane + 32 * k < dk) outp[row * dk + lane + 32 * k] = from_f<IO>(d[k]);
    }
}

static bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

template <typename IO, bool DELTA, int KIG>
cudaError_t launch_t(const Args& a, const WsLayout& L, int nslab, cudaStream_t st)
{
    const size_t smem = sizeof(BwdSmem<IO, KIG>);
    cudaError_t e = cudaFuncSetAttribute(serial_bwd_kernel<IO, DELTA, KIG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const size_t sz = sizeof(IO);
    const bool vec = (a.dk * sz) % 16 == 0 && (a.dv * sz) % 16 == 0 && al16(a.b) && al16(a.c) && al16(a.v) &&
                     al16(a.dO);
    Outs out{nullptr, nullptr, nullptr, nullptr};
    const size_t ntok = (size_t)a.B * a.T * a.H;
    const bool partials = bwd_partials(a.dk, a.dv, a.norm);
    if (partials) {
        unsigned char* w = (unsigned char*)a.ws + L.slab_off;
        out.db = reinterpret_cast<float*>(w);
        out.dc = out.db + nslab * ntok * a.dk;
        out.dg = out.dc + nslab * ntok * a.dk;
        out.dbeta = out.dg + nslab * ntok;
    }
    serial_bwd_kernel<IO, DELTA, KIG><<<dim3(a.B * a.H, nslab), 256, smem, st>>>(a, L, out, vec);
    if ((e = cudaGetLastError()) != cudaSuccess || !partials) return e;
    const int blocks = 4 * 152;
    const size_t slab_keys = ntok * a.dk;
    finish_keys_kernel<IO><<<blocks, 256, 0, st>>>(out.db, (const IO*)a.b, (IO*)a.db, ntok, a.dk, nslab, slab_keys,
                                                   a.norm);
    finish_keys_kernel<IO><<<blocks, 256, 0, st>>>(out.dc, (const IO*)a.c, (IO*)a.dc, ntok, a.dk, nslab, slab_keys,
                                                   a.norm);
    reduce_slabs_kernel<IO><<<blocks, 256, 0, st>>>(out.dg, (IO*)a.dg, ntok, nslab);
    if (DELTA) reduce_slabs_kernel<IO><<<blocks, 256, 0, st>>>(out.dbeta, (IO*)a.dbeta, ntok, nslab);
    return cudaGetLastError();
}

template <typename IO, bool DELTA>
cudaError_t launch_rows(const Args& a, const WsLayout& L, cudaStream_t st)
{
    const int nslab = bwd_slabs(a.dk, a.dv);
    return a.dk <= 64 ? launch_t<IO, DELTA, 8>(a, L, nslab, st) : launch_t<IO, DELTA, 16>(a, L, nslab, st);
}

}  // namespace

cudaError_t launch_serial_bwd(const Args& a, cudaStream_t st)
{
    gdn_shape_t sh{a.B, a.H, a.T, a.dk, a.dv, a.mode, a.io};
    const WsLayout L = ws_layout_bwd_core(sh, a.norm);
    cudaError_t e;
    if (a.io == GDN_BF16)
        e = a.mode == GDN_DELTA ? launch_rows<__nv_bfloat16, true>(a, L, st) : launch_rows<__nv_bfloat16, false>(a, L, st);
    else
        e = a.mode == GDN_DELTA ? launch_rows<float, true>(a, L, st) : launch_rows<float, false>(a, L, st);
    if (e != cudaSuccess) return e;
    const int n = a.H * a.dk;
    reduce_dalog_kernel<<<(n + 127) / 128, 128, 0, st>>>(
        reinterpret_cast<const float*>((const unsigned char*)a.ws + L.dalog_off), a.dA_log, a.B, a.H, a.dk,
        bwd_slabs(a.dk, a.dv));
    return cudaGetLastError();
}

}  // namespace gdn
