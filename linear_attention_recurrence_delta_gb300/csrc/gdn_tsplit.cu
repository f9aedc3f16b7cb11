// gdn_tsplit.cu -- forward of long sequences over few heads, split in time.
//
// With few (batch, head) units the forward kernels leave most SMs idle while
// each unit walks its chunks one after another ("GDN & MLA Mechanism
// Deep-Dive", Step 5: the state is carried serially between chunks).  The map
// from a segment's entering state to its leaving state is affine,
//   h_end = A_s h_start + H_s,
// with H_s the leaving state from a zero start and A_s the d_k x d_k
// transition: the product of the per-token factors (I - beta b b^T) diag(alpha)
// in delta mode, diag(exp(A sum_seg g)) in gated mode.  So the sequence is cut
// into P equal segments and:
//   1. every segment runs from a zero state          -> H_s      (parallel)
//   2. delta: every segment runs with v = 0 from I   -> A_s      (parallel)
//   3. a scan over segments  S_{p+1} = A_p S_p + H_p             (serial, small)
//   4. every segment runs again from its S_p         -> o        (parallel)
// A [B, T, H, d] tensor cut into P segments of T/P tokens is, byte for byte,
// a [B*P, T/P, H, d] tensor, so steps 1, 2 and 4 are the ordinary forward on
// that shape and no input moves.
//
// The backward splits the same way.  With the segments' entering states S_p
// from steps 1-3, the adjoint dL/dS_p of a segment is G_p + A_p^T E_p, where
// G_p is the segment's own backward started from a zero end gradient and E_p
// the gradient at its end (dh_T for the last one, dL/dS_{p+1} otherwise):
//   5. every segment's backward from S_p with a zero end gradient -> G_p
//   6. a reverse scan  E_{p-1} = G_p + A_p^T E_p,  dh0 = G_0 + A_0^T E_0
//   7. every segment's backward again from S_p with end gradient E_p
// Step 7's gradients are the true ones; dA_log sums over all (batch,
// segment) pairs, which the backward's own reduction over its batch does.
#include <cuda_bf16.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

// identity d_k x d_k states for the transition runs
__global__ void eye_kernel(float* I, size_t n_units, int dk)
{
    const size_t n = n_units * dk * dk;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)((idx / dk) % dk), c = (int)(idx % dk);
        I[idx] = r == c ? 1.f : 0.f;
    }
}

// Step 3 for one (batch, head): S_0 = h0; S_{p+1} = A_p S_p + H_p; stores every
// S_p (the entering states of step 4) and, if asked, S_P as h_T.
template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) scan_kernel(const float* Abuf, const float* Hbuf, const float* h0, float* Sst,
                                                   float* hT, const IO* g, const float* A_log, int B, int H, int T,
                                                   int P, int dk, int dv, int logits)
{
    __shared__ float S[64][65];
    __shared__ float At[64][65];
    __shared__ float dec[64];
    const int u = blockIdx.x, bb = u / H, h = u % H, tid = threadIdx.x;
    const int Ts = T / P;
    for (int idx = tid; idx < dk * dv; idx += 256) {
        const int i = idx / dv, j = idx % dv;
        S[i][j] = h0 ? h0[(size_t)u * dk * dv + idx] : 0.f;
    }
    __syncthreads();
    for (int p = 0; p < P; p++) {
        const size_t vu = ((size_t)(bb * P + p) * H + h);  // unit of the [B*P, T/P, H] view
        for (int idx = tid; idx < dk * dv; idx += 256) Sst[vu * dk * dv + idx] = S[idx / dv][idx % dv];
        if (DELTA) {
            for (int idx = tid; idx < dk * dk; idx += 256) At[idx / dk][idx % dk] = Abuf[vu * dk * dk + idx];
        } else if (tid < dk) {
            // decay of the whole segment: exp(A_i sum_t g_t)
            float gs = 0.f;
            for (int t = 0; t < Ts; t++) {
                const float gv = (float)g[((size_t)bb * T + (size_t)p * Ts + t) * H + h];
                gs += logits ? 1.f / (1.f + expf(-gv)) : gv;
            }
            dec[tid] = expf(gs * -expf(A_log[h * dk + tid]));
        }
        __syncthreads();
        float acc[16];
#pragma unroll
        for (int q = 0; q < 16; q++) {
            const int idx = tid + 256 * q;
            if (idx < dk * dv) {
                const int i = idx / dv, j = idx % dv;
                float v = Hbuf[vu * dk * dv + idx];
                if (DELTA) {
                    for (int k = 0; k < dk; k++) v = fmaf(At[i][k], S[k][j], v);
                } else {
                    v = fmaf(dec[i], S[i][j], v);
                }
                acc[q] = v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 16; q++) {
            const int idx = tid + 256 * q;
            if (idx < dk * dv) S[idx / dv][idx % dv] = acc[q];
        }
        __syncthreads();
    }
    if (hT)
        for (int idx = tid; idx < dk * dv; idx += 256) hT[(size_t)u * dk * dv + idx] = S[idx / dv][idx % dv];
}

// Step 6 for one (batch, head): E_{P-1} = dh_T; E_{p-1} = G_p + A_p^T E_p;
// stores every E_p (the end gradients of step 7) and dh0 = G_0 + A_0^T E_0.
template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) bscan_kernel(const float* Abuf, const float* Gbuf, const float* dhT,
                                                    float* Ebuf, float* dh0, const IO* g, const float* A_log, int B,
                                                    int H, int T, int P, int dk, int dv, int logits)
{
    __shared__ float E[64][65];
    __shared__ float At[64][65];
    __shared__ float dec[64];
    const int u = blockIdx.x, bb = u / H, h = u % H, tid = threadIdx.x;
    const int Ts = T / P;
    for (int idx = tid; idx < dk * dv; idx += 256) E[idx / dv][idx % dv] = dhT ? dhT[(size_t)u * dk * dv + idx] : 0.f;
    __syncthreads();
    for (int p = P - 1; p >= 0; p--) {
        const size_t vu = ((size_t)(bb * P + p) * H + h);
        for (int idx = tid; idx < dk * dv; idx += 256) Ebuf[vu * dk * dv + idx] = E[idx / dv][idx % dv];
        if (DELTA) {
            for (int idx = tid; idx < dk * dk; idx += 256) At[idx / dk][idx % dk] = Abuf[vu * dk * dk + idx];
        } else if (tid < dk) {
            float gs = 0.f;
            for (int t = 0; t < Ts; t++) {
                const float gv = (float)g[((size_t)bb * T + (size_t)p * Ts + t) * H + h];
                gs += logits ? 1.f / (1.f + expf(-gv)) : gv;
            }
            dec[tid] = expf(gs * -expf(A_log[h * dk + tid]));
        }
        __syncthreads();
        float acc[16];
#pragma unroll
        for (int q = 0; q < 16; q++) {
            const int idx = tid + 256 * q;
            if (idx < dk * dv) {
                const int i = idx / dv, j = idx % dv;
                float v = Gbuf[vu * dk * dv + idx];
                if (DELTA) {
                    for (int k = 0; k < dk; k++) v = fmaf(At[k][i], E[k][j], v);
                } else {
                    v = fmaf(dec[i], E[i][j], v);
                }
                acc[q] = v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 16; q++) {
            const int idx = tid + 256 * q;
            if (idx < dk * dv) E[idx / dv][idx % dv] = acc[q];
        }
        __syncthreads();
    }
    if (dh0)
        for (int idx = tid; idx < dk * dv; idx += 256) dh0[(size_t)u * dk * dv + idx] = E[idx / dv][idx % dv];
}

}  // namespace

int tsplit_factor(const gdn_shape_t& s, int backward)
{
    const long units = (long)s.B * s.H;
    // forward: three passes (delta) or two (gated) must still pay; backward: two backward passes, the
    // forward passes are cheap beside them
    const int min_p = backward ? 3 : (s.mode == GDN_DELTA ? 4 : 3);
    const long cap = kSplitSMs / units;
    for (long p = cap; p >= min_p; p--) {
        if (s.T % p) continue;
        if (s.T / p < kSplitMinTokens) continue;
        return (int)p;
    }
    return 1;
}

// Steps 1-3: the entering state of every segment into L.ts_s_off and, if
// hT is given, the leaving state of the whole sequence.  `a.o` receives the
// outputs of step 1, which are not the final ones.
static cudaError_t tsplit_states(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                                 cudaError_t (*fwd_core)(const Args&, cudaStream_t))
{
    unsigned char* ws = (unsigned char*)a.ws;
    float* Hbuf = (float*)(ws + L.ts_h_off);
    float* Abuf = (float*)(ws + L.ts_a_off);
    float* Sst = (float*)(ws + L.ts_s_off);
    float* Ibuf = (float*)(ws + L.ts_i_off);
    void* zv = ws + L.ts_zv_off;
    void* so = ws + L.ts_so_off;
    const int Ts = a.T / P;
    const size_t vunits = (size_t)a.B * P * a.H;
    cudaError_t e;

    // 1. leaving states from a zero start
    Args r = a;
    r.B = a.B * P;
    r.T = Ts;
    r.h0 = nullptr;
    r.hT = Hbuf;
    if ((e = fwd_core(r, st)) != cudaSuccess) return e;

    // 2. delta: transitions A_s = h_end with v = 0 from the identity
    if (a.mode == GDN_DELTA) {
        const size_t esz = a.io == GDN_BF16 ? 2 : 4;
        if ((e = cudaMemsetAsync(zv, 0, (size_t)a.B * a.T * a.H * a.dk * esz, st)) != cudaSuccess) return e;
        eye_kernel<<<256, 256, 0, st>>>(Ibuf, vunits, a.dk);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        Args t = r;
        t.dv = a.dk;
        t.v = zv;
        t.o = so;
        t.h0 = Ibuf;
        t.hT = Abuf;
        if ((e = fwd_core(t, st)) != cudaSuccess) return e;
    }

    // 3. scan over segments
    const int units = a.B * a.H;
    if (a.io == GDN_BF16) {
        if (a.mode == GDN_DELTA)
            scan_kernel<__nv_bfloat16, true><<<units, 256, 0, st>>>(Abuf, Hbuf, a.h0, Sst, a.hT,
                                                                     (const __nv_bfloat16*)a.g, a.A_log, a.B, a.H,
                                                                     a.T, P, a.dk, a.dv, a.logits);
        else
            scan_kernel<__nv_bfloat16, false><<<units, 256, 0, st>>>(Abuf, Hbuf, a.h0, Sst, a.hT,
                                                                      (const __nv_bfloat16*)a.g, a.A_log, a.B, a.H,
                                                                      a.T, P, a.dk, a.dv, a.logits);
    } else {
        if (a.mode == GDN_DELTA)
            scan_kernel<float, true><<<units, 256, 0, st>>>(Abuf, Hbuf, a.h0, Sst, a.hT, (const float*)a.g, a.A_log,
                                                            a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
        else
            scan_kernel<float, false><<<units, 256, 0, st>>>(Abuf, Hbuf, a.h0, Sst, a.hT, (const float*)a.g,
                                                             a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
    }
    return cudaGetLastError();
}

cudaError_t launch_fwd_tsplit(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                              cudaError_t (*fwd_core)(const Args&, cudaStream_t))
{
    cudaError_t e = tsplit_states(a, L, P, st, fwd_core);
    if (e != cudaSuccess) return e;
    // 4. every segment again from its true entering state: the outputs
    Args f = a;
    f.B = a.B * P;
    f.T = a.T / P;
    f.h0 = (const float*)((unsigned char*)a.ws + L.ts_s_off);
    f.hT = nullptr;
    return fwd_core(f, st);
}

cudaError_t launch_bwd_tsplit(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                              cudaError_t (*fwd_core)(const Args&, cudaStream_t))
{
    unsigned char* ws = (unsigned char*)a.ws;
    const float* Sst = (const float*)(ws + L.ts_s_off);
    float* Gbuf = (float*)(ws + L.ts_g_off);
    float* Ebuf = (float*)(ws + L.ts_e_off);
    cudaError_t e;

    // 1-3. entering states of the segments (outputs of step 1 go to scratch)
    Args fa = a;
    fa.o = ws + L.ts_o_off;
    fa.hT = nullptr;
    if ((e = tsplit_states(fa, L, P, st, fwd_core)) != cudaSuccess) return e;

    // 5. every segment's backward from a zero end gradient: G_p in Gbuf
    Args b = a;
    b.B = a.B * P;
    b.T = a.T / P;
    b.h0 = Sst;
    b.dhT = nullptr;
    b.dh0 = Gbuf;
    if ((e = launch_serial_bwd(b, st)) != cudaSuccess) return e;

    // 6. reverse scan of the end gradients; dh0 of the whole sequence
    const int units = a.B * a.H;
    const float* Abuf = (const float*)(ws + L.ts_a_off);
    if (a.io == GDN_BF16) {
        if (a.mode == GDN_DELTA)
            bscan_kernel<__nv_bfloat16, true><<<units, 256, 0, st>>>(Abuf, Gbuf, a.dhT, Ebuf, a.dh0,
                                                                      (const __nv_bfloat16*)a.g, a.A_log, a.B, a.H,
                                                                      a.T, P, a.dk, a.dv, a.logits);
        else
            bscan_kernel<__nv_bfloat16, false><<<units, 256, 0, st>>>(Abuf, Gbuf, a.dhT, Ebuf, a.dh0,
                                                                       (const __nv_bfloat16*)a.g, a.A_log, a.B, a.H,
                                                                       a.T, P, a.dk, a.dv, a.logits);
    } else {
        if (a.mode == GDN_DELTA)
            bscan_kernel<float, true><<<units, 256, 0, st>>>(Abuf, Gbuf, a.dhT, Ebuf, a.dh0, (const float*)a.g,
                                                             a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
        else
            bscan_kernel<float, false><<<units, 256, 0, st>>>(Abuf, Gbuf, a.dhT, Ebuf, a.dh0, (const float*)a.g,
                                                              a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // 7. every segment's backward again with its true end gradient
    b.dhT = Ebuf;
    b.dh0 = nullptr;
    return launch_serial_bwd(b, st);
}

}  // namespace gdn
