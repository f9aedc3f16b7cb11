// gdn_serial.cu -- token-serial gated delta rule on the CUDA cores (fp32 math).
//
// This is the float32-I/O path of the library and the reference-precision
// backward: it follows the recurrence of "GDN & MLA Mechanism Deep-Dive",
// Step 4 (gated) and the delta-rule card of "HyMo-434M -- documentation
// portal" one token at a time, with no chunking and no tensor cores.
//
// Thread layout (both kernels): a warp owns 8 state columns j and all rows i;
// lane = 4*jl + ig holds rows i = ig + 4k (k = 0..15) of column j = 8w + jl.
// Columns of the state never mix in the recurrence (the erase term of the
// delta rule, b_t b_t^T, acts on rows), so the forward needs no cross-warp
// traffic at all; sums over rows are 16 in-thread terms plus two shuffles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float x) { *p = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

constexpr int kFwdTok = 32;   // tokens staged per block in the forward
constexpr int kSeg = kSerialSeg;

// ---------------------------------------------------------------------------
// forward: grid (ceil(dv/32), B*H), 128 threads; a CTA owns 32 state columns
// ---------------------------------------------------------------------------
template <typename IO, bool DELTA>
__global__ void __launch_bounds__(128) serial_fwd_kernel(Args a)
{
    __shared__ float sA[64];
    __shared__ float sb[kFwdTok][64], sc[kFwdTok][64], sa[kFwdTok][64];
    __shared__ float sv[kFwdTok][32], so[kFwdTok][32];
    __shared__ float sbeta[kFwdTok];

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int ig = lane & 3, jl = lane >> 2;
    const int u = blockIdx.y, bb = u / a.H, h = u % a.H;
    const int jc0 = blockIdx.x * 32;
    const int jj = w * 8 + jl, j = jc0 + jj;
    const int dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    const IO* v = (const IO*)a.v;
    const IO* bk = (const IO*)a.b;
    const IO* c = (const IO*)a.c;
    const IO* g = (const IO*)a.g;
    const IO* beta = (const IO*)a.beta;
    IO* o = (IO*)a.o;

    if (tid < 64) sA[tid] = tid < dk ? -expf(a.A_log[h * dk + tid]) : 0.f;

    float hs[16];
#pragma unroll
    for (int k = 0; k < 16; k++) {
        const int i = ig + 4 * k;
        hs[k] = (a.h0 && i < dk && j < dv) ? a.h0[((size_t)u * dk + i) * dv + j] : 0.f;
    }
    __syncthreads();

    for (int t0 = 0; t0 < T; t0 += kFwdTok) {
        const int nt = min(kFwdTok, T - t0);
        for (int idx = tid; idx < kFwdTok * 64; idx += 128) {
            const int tt = idx >> 6, i = idx & 63;
            float xb = 0.f, xc = 0.f, xa = 0.f;
            if (tt < nt && i < dk) {
                const size_t row = ((size_t)bb * T + t0 + tt) * H + h;
                xb = ld(bk + row * dk + i);
                xc = ld(c + row * dk + i);
                xa = expf(ld(g + row) * sA[i]);
            }
            sb[tt][i] = xb; sc[tt][i] = xc; sa[tt][i] = xa;
        }
        for (int idx = tid; idx < kFwdTok * 32; idx += 128) {
            const int tt = idx >> 5, q = idx & 31;
            float xv = 0.f;
            if (tt < nt && jc0 + q < dv) xv = ld(v + (((size_t)bb * T + t0 + tt) * H + h) * dv + jc0 + q);
            sv[tt][q] = xv;
        }
        if (DELTA && tid < kFwdTok)
            sbeta[tid] = tid < nt ? ld(beta + ((size_t)bb * T + t0 + tid) * H + h) : 0.f;
        __syncthreads();

        for (int tt = 0; tt < nt; tt++) {
            float x;
            if (DELTA) {
                float r = 0.f;
#pragma unroll
                for (int k = 0; k < 16; k++) {
                    hs[k] *= sa[tt][ig + 4 * k];
                    r = fmaf(hs[k], sb[tt][ig + 4 * k], r);
                }
                r += __shfl_xor_sync(0xffffffffu, r, 1);
                r += __shfl_xor_sync(0xffffffffu, r, 2);
                x = sbeta[tt] * (sv[tt][jj] - r);
            } else {
#pragma unroll
                for (int k = 0; k < 16; k++) hs[k] *= sa[tt][ig + 4 * k];
                x = sv[tt][jj];
            }
            float ov = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k++) {
                hs[k] = fmaf(sb[tt][ig + 4 * k], x, hs[k]);
                ov = fmaf(hs[k], sc[tt][ig + 4 * k], ov);
            }
            ov += __shfl_xor_sync(0xffffffffu, ov, 1);
            ov += __shfl_xor_sync(0xffffffffu, ov, 2);
            if (ig == 0) so[tt][jj] = ov;
        }
        __syncthreads();
        for (int idx = tid; idx < kFwdTok * 32; idx += 128) {
            const int tt = idx >> 5, q = idx & 31;
            if (tt < nt && jc0 + q < dv)
                st(o + (((size_t)bb * T + t0 + tt) * H + h) * dv + jc0 + q, so[tt][q]);
        }
        __syncthreads();
    }
    if (a.hT && j < dv) {
#pragma unroll
        for (int k = 0; k < 16; k++) {
            const int i = ig + 4 * k;
            if (i < dk) a.hT[((size_t)u * dk + i) * dv + j] = hs[k];
        }
    }
}

// ---------------------------------------------------------------------------
// backward: grid (B*H), 256 threads; a CTA owns all 64 state columns
// ---------------------------------------------------------------------------
struct BwdSmem {
    float A[64];
    float b[kSeg][64], c[kSeg][64], a[kSeg][64];
    float v[kSeg][64], dO[kSeg][64], dvo[kSeg][64];
    float g[kSeg], beta[kSeg];
    float part[8][kSeg][3][64];     // per-warp row sums: db, dc, q
    float partB[8][kSeg];           // per-warp dbeta sums
    float q[kSeg][64];
};

// Sum a 16-vector over the 8 columns of a warp (lane bits 2..4).  On return
// lane keeps rows k0 = 8*b2 + 4*b3 + 2*b4 and k0 + 1 of the reduced vector.
__device__ __forceinline__ void colsum16(float (&x)[16], int lane, float& out0, float& out1)
{
    const bool b2 = lane & 4, b3 = lane & 8, b4 = lane & 16;
    float y[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const float send = b2 ? x[k] : x[k + 8];
        const float keep = b2 ? x[k + 8] : x[k];
        y[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float z[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const float send = b3 ? y[k] : y[k + 4];
        const float keep = b3 ? y[k + 4] : y[k];
        z[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int k = 0; k < 2; k++) {
        const float send = b4 ? z[k] : z[k + 2];
        const float keep = b4 ? z[k + 2] : z[k];
        (k == 0 ? out0 : out1) = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
}

template <typename IO, bool DELTA>
__device__ void stage_segment(const Args& a, BwdSmem& s, int bb, int h, int t0, int nt, bool with_grad)
{
    const int tid = threadIdx.x, dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    for (int idx = tid; idx < kSeg * 64; idx += blockDim.x) {
        const int tt = idx >> 6, i = idx & 63;
        const size_t row = ((size_t)bb * T + t0 + tt) * H + h;
        float xb = 0.f, xc = 0.f, xa = 0.f, xv = 0.f, xo = 0.f;
        if (tt < nt) {
            if (i < dk) {
                xb = ld((const IO*)a.b + row * dk + i);
                xc = ld((const IO*)a.c + row * dk + i);
                xa = expf(ld((const IO*)a.g + row) * s.A[i]);
            }
            if (i < dv) {
                xv = ld((const IO*)a.v + row * dv + i);
                if (with_grad) xo = ld((const IO*)a.dO + row * dv + i);
            }
        }
        s.b[tt][i] = xb; s.c[tt][i] = xc; s.a[tt][i] = xa; s.v[tt][i] = xv; s.dO[tt][i] = xo;
    }
    if (tid < kSeg) {
        const size_t row = ((size_t)bb * T + t0 + tid) * H + h;
        s.g[tid] = tid < nt ? ld((const IO*)a.g + row) : 0.f;
        s.beta[tid] = (DELTA && tid < nt) ? ld((const IO*)a.beta + row) : 0.f;
    }
}

// One forward step on the thread's 16 state entries; returns r (delta) via rr.
template <bool DELTA>
__device__ __forceinline__ float fwd_step(float (&hs)[16], const BwdSmem& s, int tt, int ig, int j, float& rr)
{
    float x;
    if (DELTA) {
        float r = 0.f;
#pragma unroll
        for (int k = 0; k < 16; k++) {
            hs[k] *= s.a[tt][ig + 4 * k];
            r = fmaf(hs[k], s.b[tt][ig + 4 * k], r);
        }
        r += __shfl_xor_sync(0xffffffffu, r, 1);
        r += __shfl_xor_sync(0xffffffffu, r, 2);
        rr = r;
        x = s.beta[tt] * (s.v[tt][j] - r);
    } else {
#pragma unroll
        for (int k = 0; k < 16; k++) hs[k] *= s.a[tt][ig + 4 * k];
        rr = 0.f;
        x = s.v[tt][j];
    }
#pragma unroll
    for (int k = 0; k < 16; k++) hs[k] = fmaf(s.b[tt][ig + 4 * k], x, hs[k]);
    return x;
}

template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) serial_bwd_kernel(Args a, WsLayout L)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BwdSmem& s = *reinterpret_cast<BwdSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int ig = lane & 3, jl = lane >> 2, j = w * 8 + jl;
    const int u = blockIdx.x, bb = u / a.H, h = u % a.H;
    const int dk = a.dk, dv = a.dv, T = a.T;
    const int nseg = (T + kSeg - 1) / kSeg;
    unsigned char* ws = (unsigned char*)a.ws;
    float* ck = (float*)(ws + L.ck_off) + (size_t)u * (size_t)nseg * (kStateSlot / 4);
    float* scr = (float*)(ws + L.scratch_off) + (size_t)u * kSeg * (kStateSlot / 4);
    float* dA_part = (float*)(ws + L.dalog_off) + (size_t)u * dk;

    if (tid < 64) s.A[tid] = tid < dk ? -expf(a.A_log[h * dk + tid]) : 0.f;
    float hs[16];
#pragma unroll
    for (int k = 0; k < 16; k++) {
        const int i = ig + 4 * k;
        hs[k] = (a.h0 && i < dk && j < dv) ? a.h0[((size_t)u * dk + i) * dv + j] : 0.f;
    }
    __syncthreads();

    // 1) forward sweep: keep the state entering every segment
    for (int n = 0; n < nseg; n++) {
        const int t0 = n * kSeg, nt = min(kSeg, T - t0);
#pragma unroll
        for (int k = 0; k < 16; k++) ck[(size_t)n * (kStateSlot / 4) + k * 256 + tid] = hs[k];
        stage_segment<IO, DELTA>(a, s, bb, h, t0, nt, false);
        __syncthreads();
        for (int tt = 0; tt < nt; tt++) { float r; fwd_step<DELTA>(hs, s, tt, ig, j, r); }
        __syncthreads();
    }

    // 2) reverse walk, one segment at a time
    float dS[16];
#pragma unroll
    for (int k = 0; k < 16; k++) {
        const int i = ig + 4 * k;
        dS[k] = (a.dhT && i < dk && j < dv) ? a.dhT[((size_t)u * dk + i) * dv + j] : 0.f;
    }
    float dA_acc = 0.f;   // thread tid < dk owns row tid
    for (int n = nseg - 1; n >= 0; n--) {
        const int t0 = n * kSeg, nt = min(kSeg, T - t0);
        stage_segment<IO, DELTA>(a, s, bb, h, t0, nt, true);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; k++) hs[k] = ck[(size_t)n * (kStateSlot / 4) + k * 256 + tid];
        for (int tt = 0; tt < nt; tt++) {
#pragma unroll
            for (int k = 0; k < 16; k++) scr[(size_t)tt * (kStateSlot / 4) + k * 256 + tid] = hs[k];
            float r; fwd_step<DELTA>(hs, s, tt, ig, j, r);
        }
        for (int tt = nt - 1; tt >= 0; tt--) {
            float hp[16], hc[16];
#pragma unroll
            for (int k = 0; k < 16; k++) hp[k] = scr[(size_t)tt * (kStateSlot / 4) + k * 256 + tid];
            // rebuild h', r, u, h_t
            float r = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k++) {
                hp[k] *= s.a[tt][ig + 4 * k];
                r = fmaf(hp[k], s.b[tt][ig + 4 * k], r);
            }
            r += __shfl_xor_sync(0xffffffffu, r, 1);
            r += __shfl_xor_sync(0xffffffffu, r, 2);
            const float be = s.beta[tt], vj = s.v[tt][j], doj = s.dO[tt][j];
            const float x = DELTA ? be * (vj - r) : vj;
            float pdc[16], pdb[16], pq[16];
            float du = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k++) {
                const float bi = s.b[tt][ig + 4 * k], ci = s.c[tt][ig + 4 * k];
                hc[k] = fmaf(bi, x, hp[k]);
                dS[k] = fmaf(ci, doj, dS[k]);        // read o_t = h_t^T c_t
                pdc[k] = hc[k] * doj;
                du = fmaf(dS[k], bi, du);
                pdb[k] = dS[k] * x;
            }
            du += __shfl_xor_sync(0xffffffffu, du, 1);
            du += __shfl_xor_sync(0xffffffffu, du, 2);
            float pbeta = 0.f;
            if (DELTA) {
                const float dr = -be * du;
                pbeta = du * (vj - r);
                if (ig == 0) s.dvo[tt][j] = be * du;
#pragma unroll
                for (int k = 0; k < 16; k++) {
                    pdb[k] = fmaf(hp[k], dr, pdb[k]);
                    dS[k] = fmaf(s.b[tt][ig + 4 * k], dr, dS[k]);
                }
            } else {
                if (ig == 0) s.dvo[tt][j] = du;
            }
#pragma unroll
            for (int k = 0; k < 16; k++) {
                pq[k] = dS[k] * hp[k];
                dS[k] *= s.a[tt][ig + 4 * k];
            }
            float o0, o1;
            const int k0 = ((lane & 4) ? 8 : 0) + ((lane & 8) ? 4 : 0) + ((lane & 16) ? 2 : 0);
            colsum16(pdb, lane, o0, o1);
            s.part[w][tt][0][ig + 4 * k0] = o0; s.part[w][tt][0][ig + 4 * (k0 + 1)] = o1;
            colsum16(pdc, lane, o0, o1);
            s.part[w][tt][1][ig + 4 * k0] = o0; s.part[w][tt][1][ig + 4 * (k0 + 1)] = o1;
            colsum16(pq, lane, o0, o1);
            s.part[w][tt][2][ig + 4 * k0] = o0; s.part[w][tt][2][ig + 4 * (k0 + 1)] = o1;
            if (DELTA) {
                pbeta += __shfl_xor_sync(0xffffffffu, pbeta, 4);
                pbeta += __shfl_xor_sync(0xffffffffu, pbeta, 8);
                pbeta += __shfl_xor_sync(0xffffffffu, pbeta, 16);
                if (lane == 0) s.partB[w][tt] = pbeta;
            }
        }
        __syncthreads();
        // reduce the per-warp partials of this segment (fixed order)
        for (int idx = tid; idx < kSeg * 64; idx += 256) {
            const int tt = idx >> 6, i = idx & 63;
            float sdb = 0.f, sdc = 0.f, sq = 0.f;
#pragma unroll
            for (int ww = 0; ww < 8; ww++) {
                sdb += s.part[ww][tt][0][i];
                sdc += s.part[ww][tt][1][i];
                sq += s.part[ww][tt][2][i];
            }
            s.q[tt][i] = sq;
            if (tt < nt) {
                const size_t row = ((size_t)bb * T + t0 + tt) * a.H + h;
                if (i < dk) {
                    st((IO*)a.db + row * dk + i, sdb);
                    st((IO*)a.dc + row * dk + i, sdc);
                }
                if (i < dv) st((IO*)a.dv_ + row * dv + i, s.dvo[tt][i]);
            }
        }
        __syncthreads();
        if (tid < nt) {
            float dg = 0.f;
            for (int i = 0; i < dk; i++) dg = fmaf(s.A[i], s.q[tid][i], dg);
            const size_t row = ((size_t)bb * T + t0 + tid) * a.H + h;
            st((IO*)a.dg + row, dg);
            if (DELTA) {
                float sb = 0.f;
#pragma unroll
                for (int ww = 0; ww < 8; ww++) sb += s.partB[ww][tid];
                st((IO*)a.dbeta + row, sb);
            }
        }
        if (tid < dk)
            for (int tt = 0; tt < nt; tt++) dA_acc = fmaf(s.g[tt], s.q[tt][tid], dA_acc);
        __syncthreads();
    }
    if (a.dh0 && j < dv) {
#pragma unroll
        for (int k = 0; k < 16; k++) {
            const int i = ig + 4 * k;
            if (i < dk) a.dh0[((size_t)u * dk + i) * dv + j] = dS[k];
        }
    }
    if (tid < dk) dA_part[tid] = dA_acc * s.A[tid];
}

// dA_log[h, i] = sum_b partial[b, h, i]  (fixed order, deterministic)
__global__ void reduce_dalog_kernel(const float* part, float* dA_log, int B, int H, int dk)
{
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= H * dk) return;
    const int h = idx / dk, i = idx % dk;
    float s = 0.f;
    for (int b = 0; b < B; b++) s += part[((size_t)b * H + h) * dk + i];
    dA_log[idx] = s;
}

}  // namespace

cudaError_t launch_serial_fwd(const Args& a, cudaStream_t st)
{
    dim3 grid((a.dv + 31) / 32, a.B * a.H);
    if (a.io == GDN_BF16) {
        if (a.mode == GDN_DELTA) serial_fwd_kernel<__nv_bfloat16, true><<<grid, 128, 0, st>>>(a);
        else serial_fwd_kernel<__nv_bfloat16, false><<<grid, 128, 0, st>>>(a);
    } else {
        if (a.mode == GDN_DELTA) serial_fwd_kernel<float, true><<<grid, 128, 0, st>>>(a);
        else serial_fwd_kernel<float, false><<<grid, 128, 0, st>>>(a);
    }
    return cudaGetLastError();
}

template <typename IO, bool DELTA>
static cudaError_t launch_bwd_t(const Args& a, const WsLayout& L, cudaStream_t st)
{
    const size_t smem = sizeof(BwdSmem);
    cudaError_t e = cudaFuncSetAttribute(serial_bwd_kernel<IO, DELTA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    serial_bwd_kernel<IO, DELTA><<<a.B * a.H, 256, smem, st>>>(a, L);
    return cudaGetLastError();
}

cudaError_t launch_serial_bwd(const Args& a, cudaStream_t st)
{
    gdn_shape_t s{a.B, a.H, a.T, a.dk, a.dv, a.mode, a.io};
    const WsLayout L = ws_layout(s, 1);
    cudaError_t e;
    if (a.io == GDN_BF16) e = a.mode == GDN_DELTA ? launch_bwd_t<__nv_bfloat16, true>(a, L, st)
                                                  : launch_bwd_t<__nv_bfloat16, false>(a, L, st);
    else e = a.mode == GDN_DELTA ? launch_bwd_t<float, true>(a, L, st) : launch_bwd_t<float, false>(a, L, st);
    if (e != cudaSuccess) return e;
    const int n = a.H * a.dk;
    reduce_dalog_kernel<<<(n + 127) / 128, 128, 0, st>>>(
        (const float*)((unsigned char*)a.ws + L.dalog_off), a.dA_log, a.B, a.H, a.dk);
    return cudaGetLastError();
}

}  // namespace gdn
