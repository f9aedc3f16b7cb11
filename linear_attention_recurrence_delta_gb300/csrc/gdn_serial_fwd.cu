// gdn_serial_fwd.cu -- token-serial forward of the gated delta rule on the
// CUDA cores (fp32 state, packed fp32x2 arithmetic).
//
// Follows the per-token recurrence of "GDN & MLA Mechanism Deep-Dive", Step 4
// (gated: h_t = alpha_t (.) h_{t-1} + b_t v_t^T) and the delta-rule card of
// "HyMo-434M -- documentation portal" (h_t = h' + beta_t b_t (v_t - h'^T b_t)^T
// with h' = alpha_t (.) h_{t-1}); both read o_t = h_t^T c_t, and
// alpha_t = exp(g_t A), A = -exp(A_log).
//
// Columns j of the state never mix (the erase term acts on rows), so a CTA
// owns a slab of columns of one (batch, head) unit and needs no other CTA.
// Thread layout: LPC lanes share a column, each holding 16 consecutive rows
// as 8 packed pairs (LPC = 4 covers d_k <= 64 with 32 columns per CTA, LPC = 8
// covers d_k <= 128 with 16); warp w owns columns (32 / LPC) w + jl, and
// lane = LPC jl + ig holds rows 16 ig .. 16 ig + 15.  A sum over rows is 8
// packed products in-thread plus log2(LPC) shuffles.  Inputs stream through shared memory in blocks of 32 tokens: the
// next block's raw bytes arrive by cp.async while the current one computes.
#include "gdn_internal.h"
#include "serial_common.cuh"

namespace gdn {
namespace {

using namespace rec;

template <int LPC>
struct FCfg {
    static constexpr int ROWS = 16 * LPC;          // state rows covered
    static constexpr int PAD = ROWS + ROWS / 4;    // padded row-vector length (see prow)
    static constexpr int COLS = 128 / LPC;         // state columns per CTA (4 warps)
    // tokens per staged block: 16 at 128 rows keeps the CTA near 42 KB of shared memory, five per SM
    static constexpr int TB = LPC == 4 ? 32 : 16;
};

template <typename IO, int LPC>
struct FwdSmem {
    static constexpr int R = FCfg<LPC>::ROWS, NC = FCfg<LPC>::COLS, PAD = FCfg<LPC>::PAD, kTB = FCfg<LPC>::TB;
    float A[kTB][PAD];       // alpha_t per state row
    float Bv[kTB][PAD];      // b_t
    float Cv[kTB][PAD];      // c_t
    float V[kTB][NC];        // v_t on this CTA's columns
    float O[kTB][NC];        // o_t staging for coalesced stores
    float beta[kTB];
    float Arow[R];           // A = -exp(A_log) of this head
    float rg[kTB], rbeta[kTB];
    float nb[kTB], nc[kTB];  // GDN_NORM_BC: 1 / max(||b_t||, floor), the same for c_t
    IO rb[kTB][R], rc[kTB][R], rv[kTB][NC];  // raw bytes of the next block (rc directly after rb)
};

struct Unit {
    int bb, h, u, jc0, ncols;
};

// Start fetching block [t0, t0+nt): row vectors by cp.async (or plain loads
// when rows are not 16-byte aligned), g and beta into registers.
template <typename IO, bool DELTA, int LPC>
__device__ __forceinline__ void issue_block(const Args& a, FwdSmem<IO, LPC>& s, const Unit& U, int t0, int nt,
                                            bool vec, IO& greg, IO& breg)
{
    constexpr int R = FCfg<LPC>::ROWS;
    const int tid = threadIdx.x, dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    const IO* bk = (const IO*)a.b;
    const IO* c = (const IO*)a.c;
    const IO* v = (const IO*)a.v;
    constexpr int E = 16 / sizeof(IO);
    if (vec) {
        const int cb = dk / E, cv = U.ncols / E, per = 2 * cb + cv;
        for (int idx = tid; idx < nt * per; idx += blockDim.x) {
            const int tt = idx / per, r = idx - tt * per;
            const size_t row = ((size_t)U.bb * T + t0 + tt) * H + U.h;
            if (r < cb) cp_async16(&s.rb[tt][r * E], bk + row * dk + r * E);
            else if (r < 2 * cb) cp_async16(&s.rc[tt][(r - cb) * E], c + row * dk + (r - cb) * E);
            else cp_async16(&s.rv[tt][(r - 2 * cb) * E], v + row * dv + U.jc0 + (r - 2 * cb) * E);
        }
        cp_async_commit();
    } else {
        for (int idx = tid; idx < nt * R; idx += blockDim.x) {
            const int tt = idx / R, i = idx % R;
            const size_t row = ((size_t)U.bb * T + t0 + tt) * H + U.h;
            if (i < dk) {
                s.rb[tt][i] = bk[row * dk + i];
                s.rc[tt][i] = c[row * dk + i];
            }
            if (i < U.ncols) s.rv[tt][i] = v[row * dv + U.jc0 + i];
        }
    }
    // g, beta stay raw until they are stored at the end of the block: nothing waits on these loads meanwhile
    if (tid < nt) greg = ((const IO*)a.g)[((size_t)U.bb * T + t0 + tid) * H + U.h];
    if (DELTA && tid >= 32 && tid - 32 < nt)
        breg = ((const IO*)a.beta)[((size_t)U.bb * T + t0 + tid - 32) * H + U.h];
}

// raw block -> fp32 staged arrays (alpha computed here, once per row and token)
template <typename IO, bool DELTA, int LPC>
__device__ __forceinline__ void convert_block(const Args& a, FwdSmem<IO, LPC>& s, const Unit& U, int nt)
{
    constexpr int R = FCfg<LPC>::ROWS, NC = FCfg<LPC>::COLS;
    const int tid = threadIdx.x, dk = a.dk;
    if (a.norm) {   // inverse norms of the block's b_t and c_t, one thread per vector
        for (int v = tid; v < 2 * nt; v += blockDim.x) {
            const int tt = v >> 1;
            const IO* x = &s.rb[0][0] + (size_t)((v & 1) * FCfg<LPC>::TB + tt) * R;   // rc follows rb
            float q = 0.f;
            for (int k = 0, i = tt % dk; k < dk; k++, i = i + 1 < dk ? i + 1 : 0)   // rotated: fewer bank conflicts
                q = fmaf(to_f(x[i]), to_f(x[i]), q);
            const float inv = 1.f / fmaxf(sqrtf(q), kNormFloor);
            if (v & 1) s.nc[tt] = inv;
            else s.nb[tt] = inv;
        }
        __syncthreads();
    }
    for (int idx = tid; idx < nt * R; idx += blockDim.x) {
        const int tt = idx / R, i = idx % R;
        float xa = 0.f, xb = 0.f, xc = 0.f;
        if (i < dk) {
            xa = expf(s.rg[tt] * s.Arow[i]);
            xb = to_f(s.rb[tt][i]);
            xc = to_f(s.rc[tt][i]);
            if (a.norm) {
                xb *= s.nb[tt];
                xc *= s.nc[tt];
            }
        }
        const int p = prow(i);
        s.A[tt][p] = xa;
        s.Bv[tt][p] = xb;
        s.Cv[tt][p] = xc;
    }
    for (int idx = tid; idx < nt * NC; idx += blockDim.x) {
        const int tt = idx / NC, q = idx - tt * NC;
        s.V[tt][q] = q < U.ncols ? to_f(s.rv[tt][q]) : 0.f;
    }
    if (tid < nt) s.beta[tid] = DELTA ? s.rbeta[tid] : 0.f;
}

template <typename IO, bool DELTA, int LPC>
__global__ void __launch_bounds__(128) serial_fwd_kernel(Args a, bool vec)
{
    constexpr int R = FCfg<LPC>::ROWS, NC = FCfg<LPC>::COLS, kTB = FCfg<LPC>::TB;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    FwdSmem<IO, LPC>& s = *reinterpret_cast<FwdSmem<IO, LPC>*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int ig = lane % LPC, jl = lane / LPC, cl = (32 / LPC) * w + jl;
    // one flat index over (unit, column slab), a unit's slabs adjacent so that they share b and c in L2
    const int nslab = (a.dv + NC - 1) / NC;
    Unit U;
    U.u = blockIdx.x / nslab;
    U.bb = U.u / a.H;
    U.h = U.u % a.H;
    U.jc0 = (blockIdx.x % nslab) * NC;
    U.ncols = min(NC, a.dv - U.jc0);
    const int j = U.jc0 + cl, dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    const int nblk = (T + kTB - 1) / kTB;

    for (int i = tid; i < R; i += 128) s.Arow[i] = i < dk ? -expf(a.A_log[U.h * dk + i]) : 0.f;

    // state: rows 16 ig + 2p, 16 ig + 2p + 1 of column j in h[p]
    float2 h[8];
#pragma unroll
    for (int p = 0; p < 8; p++) {
        const int i0 = 16 * ig + 2 * p;
        float x0 = 0.f, x1 = 0.f;
        if (a.h0 && j < dv) {
            if (i0 < dk) x0 = a.h0[((size_t)U.u * dk + i0) * dv + j];
            if (i0 + 1 < dk) x1 = a.h0[((size_t)U.u * dk + i0 + 1) * dv + j];
        }
        h[p] = f2(x0, x1);
    }

    IO greg = from_f<IO>(0.f), breg = from_f<IO>(0.f);
    issue_block<IO, DELTA, LPC>(a, s, U, 0, min(kTB, T), vec, greg, breg);
    if (tid < kTB) s.rg[tid] = gate(to_f(greg), a.logits);
    else if (tid >= 32 && tid < 32 + kTB) s.rbeta[tid - 32] = gate(to_f(breg), a.logits);
    cp_async_wait_all();
    __syncthreads();
    convert_block<IO, DELTA, LPC>(a, s, U, min(kTB, T));
    __syncthreads();
    if (nblk > 1) issue_block<IO, DELTA, LPC>(a, s, U, kTB, min(kTB, T - kTB), vec, greg, breg);

    IO* o = (IO*)a.o;
    for (int n = 0; n < nblk; n++) {
        const int t0 = n * kTB, nt = min(kTB, T - t0);
        // the next token's row vectors load while this one computes (they do not depend on the state)
        float2 avn[8], bvn[8], cvn[8];
        ld_rows16(&s.A[0][20 * ig], avn);
        ld_rows16(&s.Bv[0][20 * ig], bvn);
        ld_rows16(&s.Cv[0][20 * ig], cvn);
        float vn = s.V[0][cl], betn = s.beta[0];
#pragma unroll 4
        for (int tt = 0; tt < nt; tt++) {
            float2 av[8], bv[8], cv[8];
#pragma unroll
            for (int p = 0; p < 8; p++) {
                av[p] = avn[p];
                bv[p] = bvn[p];
                cv[p] = cvn[p];
            }
            const float vt = vn, bet = betn;
            const int tn = tt + 1 < nt ? tt + 1 : tt;
            ld_rows16(&s.A[tn][20 * ig], avn);
            ld_rows16(&s.Bv[tn][20 * ig], bvn);
            ld_rows16(&s.Cv[tn][20 * ig], cvn);
            vn = s.V[tn][cl];
            betn = s.beta[tn];
            float2 hp[8];
#pragma unroll
            for (int p = 0; p < 8; p++) hp[p] = mul2(h[p], av[p]);
            float x;
            if (DELTA) {
                float r = dot8x2(hp, bv);
#pragma unroll
                for (int o = 1; o < LPC; o <<= 1) r += __shfl_xor_sync(kFull, r, o);
                x = bet * (vt - r);
            } else {
                x = vt;
            }
            const float2 xx = f2(x, x);
#pragma unroll
            for (int p = 0; p < 8; p++) h[p] = fma2(bv[p], xx, hp[p]);
            float ov = dot8x2(h, cv);
#pragma unroll
            for (int o = 1; o < LPC; o <<= 1) ov += __shfl_xor_sync(kFull, ov, o);
            if (ig == 0) s.O[tt][cl] = ov;
        }
        __syncthreads();
        for (int idx = tid; idx < nt * U.ncols; idx += blockDim.x) {
            const int tt = idx / U.ncols, q = idx - tt * U.ncols;
            o[(((size_t)U.bb * T + t0 + tt) * H + U.h) * dv + U.jc0 + q] = from_f<IO>(s.O[tt][q]);
        }
        if (n + 1 < nblk) {
            if (tid < kTB) s.rg[tid] = gate(to_f(greg), a.logits);
            else if (tid >= 32 && tid < 32 + kTB) s.rbeta[tid - 32] = gate(to_f(breg), a.logits);
            cp_async_wait_all();
            __syncthreads();
            convert_block<IO, DELTA, LPC>(a, s, U, min(kTB, T - t0 - kTB));
            __syncthreads();
            if (n + 2 < nblk)
                issue_block<IO, DELTA, LPC>(a, s, U, t0 + 2 * kTB, min(kTB, T - t0 - 2 * kTB), vec, greg, breg);
        }
    }

    if (a.hT && j < dv) {
#pragma unroll
        for (int p = 0; p < 8; p++) {
            const int i0 = 16 * ig + 2 * p;
            if (i0 < dk) a.hT[((size_t)U.u * dk + i0) * dv + j] = h[p].x;
            if (i0 + 1 < dk) a.hT[((size_t)U.u * dk + i0 + 1) * dv + j] = h[p].y;
        }
    }
}

static bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

template <typename IO, bool DELTA, int LPC>
cudaError_t launch_lpc(const Args& a, cudaStream_t st)
{
    const size_t smem = sizeof(FwdSmem<IO, LPC>);
    cudaError_t e = cudaFuncSetAttribute(serial_fwd_kernel<IO, DELTA, LPC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const size_t sz = sizeof(IO);
    const bool vec = (a.dk * sz) % 16 == 0 && (a.dv * sz) % 16 == 0 && al16(a.b) && al16(a.c) && al16(a.v);
    constexpr int NC = FCfg<LPC>::COLS;
    const unsigned grid = (unsigned)((a.dv + NC - 1) / NC) * (unsigned)(a.B * a.H);
    serial_fwd_kernel<IO, DELTA, LPC><<<grid, 128, smem, st>>>(a, vec);
    return cudaGetLastError();
}

template <typename IO, bool DELTA>
cudaError_t launch_t(const Args& a, cudaStream_t st)
{
    return a.dk <= 64 ? launch_lpc<IO, DELTA, 4>(a, st) : launch_lpc<IO, DELTA, 8>(a, st);
}

}  // namespace

cudaError_t launch_serial_fwd(const Args& a, cudaStream_t st)
{
    if (a.io == GDN_BF16)
        return a.mode == GDN_DELTA ? launch_t<__nv_bfloat16, true>(a, st) : launch_t<__nv_bfloat16, false>(a, st);
    return a.mode == GDN_DELTA ? launch_t<float, true>(a, st) : launch_t<float, false>(a, st);
}

}  // namespace gdn
