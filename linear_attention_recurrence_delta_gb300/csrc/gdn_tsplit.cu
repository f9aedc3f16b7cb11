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
//   4. the outputs: the forward is linear in the entering state, so with
//      Phi_t the transition from the segment start through token t,
//        o_t = o0_t + S_p^T (Phi_t^T c_t),
//      o0_t the zero-start output of step 1 and Phi_t^T c_t the output of the
//      transition run of step 2 (delta) or c_t (.) exp(A Gam_t), Gam_t the sum
//      of g over the segment through t (gated); both runs keep their outputs
//      in fp32 for this                                          (parallel)
// A [B, T, H, d] tensor cut into P segments of T/P tokens is, byte for byte,
// a [B*P, T/P, H, d] tensor, so steps 1 and 2 are the ordinary forward on that
// shape and no input moves.
//
// The backward splits the same way.  With the segments' entering states S_p
// from steps 1-3, the adjoint dL/dS_p of a segment is G_p + A_p^T E_p, where
// G_p is its adjoint with a zero end gradient and E_p the gradient at its end
// (dh_T for the last one, dL/dS_{p+1} otherwise).  The outputs depend on S_p
// only through o_t = S_p^T (Phi_t^T c_t) + (terms free of S_p), so
//   5. G_p = sum_t (Phi_t^T c_t) do_t^T over the segment: the transition
//      run's outputs (delta) or c_t (.) exp(A Gam_t) (gated) against dO
//   6. a reverse scan  E_{p-1} = G_p + A_p^T E_p,  dh0 = G_0 + A_0^T E_0
//   7. every segment's backward from S_p with end gradient E_p
// Step 7's gradients are the true ones; dA_log sums over all (batch,
// segment) pairs, which the backward's own reduction over its batch does.
#include <cuda_bf16.h>

#include "gdn_internal.h"
#include "serial_common.cuh"

namespace gdn {
namespace {

using rec::cp_async16;
using rec::cp_async_commit;

// identity d_k x d_k states for the transition runs
__global__ void eye_kernel(float* I, size_t n_units, int dk)
{
    const size_t n = n_units * dk * dk;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)((idx / dk) % dk), c = (int)(idx % dk);
        I[idx] = r == c ? 1.f : 0.f;
    }
}

// Step 4 for one (view batch, head) unit and a run of kOutRun of its segment's tokens: o_t = o0_t + S_p^T q_t
// with q_t = Phi_t^T c_t (delta: from the transition run; gated: c_t (.) exp(A Gam_t)).  Thread (j, r) holds
// column j of S_p in registers; the run goes in sub-tiles of 64 tokens whose q and o0 rows are staged in
// shared memory, thread (j, r) computing tokens r, r + 4, ... of each.  With rows of whole 16-byte quads the
// next sub-tile's o0 (and, delta, q) rows stream in by cp.async into a second buffer while one computes.
// Gated: the gates of the segment before the run are a fixed-order block sum, then a running inclusive scan
// over the sub-tiles.
constexpr int kOutTile = 64;
constexpr int kOutRun = 512;

struct OutSmem {
    float q[2][kOutTile][64];
    float oz[2][kOutTile][64];
};


template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) tsplit_out_kernel(const float* o0, const float* so, const IO* c, const IO* g,
                                                         const float* A_log, const float* Sst, IO* o, int H, int Ts,
                                                         int dk, int dv, int logits, int norm)
{
    extern __shared__ __align__(16) unsigned char out_smem[];
    OutSmem& sm = *reinterpret_cast<OutSmem*>(out_smem);
    __shared__ float Gam[kOutTile];
    __shared__ float red[8];
    __shared__ float Arow[64];
    const int u = blockIdx.x, bv = u / H, h = u % H, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int j = tid & 63, r = tid >> 6;
    const int run0 = kOutRun * blockIdx.y, run_end = min(Ts, run0 + kOutRun);
    auto row = [&](int t) { return ((size_t)bv * Ts + t) * H + h; };   // token row of the [B*P, T/P, H] view
    auto gate_at = [&](int t) {
        const float gv = (float)g[row(t)];
        return logits ? 1.f / (1.f + expf(-gv)) : gv;
    };

    float2 Scol[32];   // rows 2k, 2k + 1 of column j, for packed fp32x2 products
#pragma unroll
    for (int k = 0; k < 32; k++) {
        const int i = 2 * k;
        Scol[k].x = (i < dk && j < dv) ? Sst[((size_t)u * dk + i) * dv + j] : 0.f;
        Scol[k].y = (i + 1 < dk && j < dv) ? Sst[((size_t)u * dk + i + 1) * dv + j] : 0.f;
    }

    float base = 0.f;   // gated: sum of the segment's gates before the current sub-tile
    if (!DELTA) {
        if (tid < 64) Arow[tid] = tid < dk ? -expf(A_log[h * dk + tid]) : 0.f;
        float part = 0.f;
        for (int t = tid; t < run0; t += 256) part += gate_at(t);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) red[w] = part;
        __syncthreads();
#pragma unroll
        for (int ww = 0; ww < 8; ww++) base += red[ww];
    }

    // the sub-tile from t0 into buffer sb by cp.async (zeros past the run and the row width), one commit group
    const bool quads = (dv & 3) == 0 && (!DELTA || (dk & 3) == 0);
    auto stage_async = [&](int t0, int sb) {
        const int nt = min(kOutTile, run_end - t0);
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int idx = tid + 256 * m, tt = idx >> 4, c4 = 4 * (idx & 15);
            const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
            float* od = &sm.oz[sb][tt][c4];
            if (tt < nt && c4 < dv) cp_async16(od, o0 + row(t0 + tt) * dv + c4);
            else *reinterpret_cast<float4*>(od) = z4;
            if (DELTA) {
                float* qd = &sm.q[sb][tt][c4];
                if (tt < nt && c4 < dk) cp_async16(qd, so + row(t0 + tt) * dk + c4);
                else *reinterpret_cast<float4*>(qd) = z4;
            }
        }
        cp_async_commit();
    };
    if (quads) stage_async(run0, 0);

    for (int t0 = run0, sb = 0; t0 < run_end; t0 += kOutTile, sb ^= 1) {
        const int nt = min(kOutTile, run_end - t0);
        float (*q)[64] = sm.q[sb];
        float (*oz)[64] = sm.oz[sb];
        __syncthreads();   // the previous sub-tile's rows are consumed: its buffer takes the next sub-tile's
        if (quads) {
            if (t0 + kOutTile < run_end) stage_async(t0 + kOutTile, sb ^ 1);
            else cp_async_commit();
        }
        if (!DELTA && w == 0) {   // inclusive scan of the sub-tile's gates (two per lane) on top of `base`
            const float ga = 2 * lane < nt ? gate_at(t0 + 2 * lane) : 0.f;
            const float gb = 2 * lane + 1 < nt ? gate_at(t0 + 2 * lane + 1) : 0.f;
            float x = ga + gb;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            const float ex = __shfl_up_sync(0xffffffffu, x, 1);
            Gam[2 * lane] = base + (lane > 0 ? ex : 0.f) + ga;
            Gam[2 * lane + 1] = base + x;
        }
        // the sub-tile's o0 (and, delta, q) rows: in flight since the previous sub-tile, or (rows not of whole
        // quads) element by element now
        if (!quads) {
            for (int idx = tid; idx < kOutTile * 64; idx += 256) {
                const int tt = idx >> 6, jj = idx & 63;
                oz[tt][jj] = (tt < nt && jj < dv) ? o0[row(t0 + tt) * dv + jj] : 0.f;
                if (DELTA) q[tt][jj] = (tt < nt && jj < dk) ? so[row(t0 + tt) * dk + jj] : 0.f;
            }
        }
        if (!DELTA) {
            float cv[16];   // the sub-tile's c rows, all loads in flight before the exponentials
#pragma unroll
            for (int m = 0; m < 16; m++) {
                const int idx = tid + 256 * m, tt = idx >> 6, i = idx & 63;
                cv[m] = (tt < nt && i < dk) ? (float)c[row(t0 + tt) * dk + i] : 0.f;
            }
            __syncthreads();   // Gam
#pragma unroll
            for (int m = 0; m < 16; m++) {
                const int idx = tid + 256 * m, tt = idx >> 6, i = idx & 63;
                q[tt][i] = cv[m] * expf(Arow[i] * Gam[tt]);
            }
            if (norm) {   // c_t / max(||c_t||, floor): one warp per token row
                __syncthreads();
                for (int tt = w; tt < nt; tt += 8) {
                    float sq = 0.f;
                    for (int i = lane; i < dk; i += 32) {
                        const float x = (float)c[row(t0 + tt) * dk + i];
                        sq = fmaf(x, x, sq);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
                    const float inv = 1.f / fmaxf(sqrtf(sq), kNormFloor);
                    for (int i = lane; i < 64; i += 32) q[tt][i] *= inv;
                }
            }
            base = Gam[kOutTile - 1];   // (tokens past the run's end add zero)
        }
        if (quads) asm volatile("cp.async.wait_group 1;\n" ::: "memory");   // this sub-tile's group
        __syncthreads();
        if (j < dv) {
            for (int tt = r; tt < nt; tt += 4) {
                // two chains of packed fp32x2 FMAs, added in a fixed order
                float2 acc0 = make_float2(oz[tt][j], 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    const float4 qq = *reinterpret_cast<const float4*>(&q[tt][i]);
                    acc0 = __ffma2_rn(Scol[i / 2], make_float2(qq.x, qq.y), acc0);
                    acc1 = __ffma2_rn(Scol[i / 2 + 1], make_float2(qq.z, qq.w), acc1);
                }
                o[row(t0 + tt) * dv + j] = (IO)((acc0.x + acc0.y) + (acc1.x + acc1.y));
            }
        }
    }
}

template <typename IO>
cudaError_t out_smem_attr(int bytes)
{
    cudaError_t e = cudaFuncSetAttribute(tsplit_out_kernel<IO, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tsplit_out_kernel<IO, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

// Step 5 for one (view batch, head) unit and a run of kGpRun of its segment's tokens: the run's share
// sum_t q_t do_t^T of G_p, q_t as in tsplit_out_kernel.  Thread t accumulates rows 4 (t >> 4) .. + 3, columns
// 4 (t & 15) .. + 3 in fp32 (packed pairs) over 64-token sub-tiles of q and dO staged in shared memory, in
// token order; with rows of whole 16-byte pieces the next sub-tile streams in by cp.async while one computes.
// One run per segment writes G_p itself; otherwise each run writes a partial that gp_reduce_kernel adds up in
// run order (deterministic).
constexpr int kGpRun = 512;

struct GpSmem {
    float q[2][kOutTile][64];
    float d[2][kOutTile][64];   // dO rows as stored (bf16 use the first half of each row's bytes)
};

__device__ __forceinline__ void ld4(const float* p, float (&x)[4])
{
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16* p, float (&x)[4])
{
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
}

template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) tsplit_gp_kernel(const float* so, const IO* c, const IO* g, const IO* dO,
                                                        const float* A_log, float* G, int H, int Ts, int dk, int dv,
                                                        int logits, int norm)
{
    extern __shared__ __align__(16) unsigned char gp_smem[];
    GpSmem& sm = *reinterpret_cast<GpSmem*>(gp_smem);
    __shared__ float Gam[kOutTile];
    __shared__ float red[8];
    __shared__ float Arow[64];
    const int u = blockIdx.x, bv = u / H, h = u % H, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int i0 = 4 * (tid >> 4), j0 = 4 * (tid & 15);
    const int run0 = kGpRun * blockIdx.y, run_end = min(Ts, run0 + kGpRun);
    auto row = [&](int t) { return ((size_t)bv * Ts + t) * H + h; };   // token row of the [B*P, T/P, H] view
    auto gate_at = [&](int t) {
        const float gv = (float)g[row(t)];
        return logits ? 1.f / (1.f + expf(-gv)) : gv;
    };
    constexpr int E = 16 / sizeof(IO);   // dO elements per 16-byte piece

    float base = 0.f;   // gated: sum of the segment's gates before the current sub-tile
    if (!DELTA) {
        if (tid < 64) Arow[tid] = tid < dk ? -expf(A_log[h * dk + tid]) : 0.f;
        float part = 0.f;
        for (int t = tid; t < run0; t += 256) part += gate_at(t);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) red[w] = part;
        __syncthreads();
#pragma unroll
        for (int ww = 0; ww < 8; ww++) base += red[ww];
    }

    // rows past the sub-tile are never read and columns past d_k / d_v only reach accumulators that are not
    // stored, so the staging leaves them as they are
    const bool pieces = (dv % E) == 0 && ((uintptr_t)dO & 15) == 0 && (!DELTA || (dk & 3) == 0);
    auto stage_async = [&](int t0, int sb) {
        const int nt = min(kOutTile, run_end - t0);
        IO* dd = reinterpret_cast<IO*>(&sm.d[sb][0][0]);
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int idx = tid + 256 * m;
            if (DELTA) {
                const int tt = idx >> 4, c4 = 4 * (idx & 15);
                if (tt < nt && c4 < dk) cp_async16(&sm.q[sb][tt][c4], so + row(t0 + tt) * dk + c4);
            }
            const int tt = idx / (64 / E), ce = E * (idx % (64 / E));
            if (tt < nt && ce < dv) cp_async16(dd + tt * 64 + ce, dO + row(t0 + tt) * dv + ce);
        }
        cp_async_commit();
    };
    if (pieces) stage_async(run0, 0);

    float2 acc[4][2];
#pragma unroll
    for (int a = 0; a < 4; a++) acc[a][0] = acc[a][1] = make_float2(0.f, 0.f);
    for (int t0 = run0, sb = 0; t0 < run_end; t0 += kOutTile, sb ^= 1) {
        const int nt = min(kOutTile, run_end - t0);
        float (*q)[64] = sm.q[sb];
        const IO* dd = reinterpret_cast<const IO*>(&sm.d[sb][0][0]);
        __syncthreads();   // the previous sub-tile is consumed: its buffer takes the next one
        if (pieces) {
            if (t0 + kOutTile < run_end) stage_async(t0 + kOutTile, sb ^ 1);
            else cp_async_commit();
        } else {
            IO* dw = reinterpret_cast<IO*>(&sm.d[sb][0][0]);
            for (int idx = tid; idx < kOutTile * 64; idx += 256) {
                const int tt = idx >> 6, jj = idx & 63;
                if (tt < nt && jj < dv) dw[tt * 64 + jj] = dO[row(t0 + tt) * dv + jj];
                if (DELTA && tt < nt) q[tt][jj] = jj < dk ? so[row(t0 + tt) * dk + jj] : 0.f;
            }
        }
        if (!DELTA) {
            if (w == 0) {   // inclusive scan of the sub-tile's gates (two per lane) on top of `base`
                const float ga = 2 * lane < nt ? gate_at(t0 + 2 * lane) : 0.f;
                const float gb = 2 * lane + 1 < nt ? gate_at(t0 + 2 * lane + 1) : 0.f;
                float x = ga + gb;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                const float ex = __shfl_up_sync(0xffffffffu, x, 1);
                Gam[2 * lane] = base + (lane > 0 ? ex : 0.f) + ga;
                Gam[2 * lane + 1] = base + x;
            }
            float cv[16];   // the sub-tile's c rows, all loads in flight before the exponentials
#pragma unroll
            for (int m = 0; m < 16; m++) {
                const int idx = tid + 256 * m, tt = idx >> 6, i = idx & 63;
                cv[m] = (tt < nt && i < dk) ? (float)c[row(t0 + tt) * dk + i] : 0.f;
            }
            __syncthreads();   // Gam
#pragma unroll
            for (int m = 0; m < 16; m++) {
                const int idx = tid + 256 * m, tt = idx >> 6, i = idx & 63;
                q[tt][i] = cv[m] * expf(Arow[i] * Gam[tt]);
            }
            if (norm) {   // c_t / max(||c_t||, floor): one warp per token row
                __syncthreads();
                for (int tt = w; tt < nt; tt += 8) {
                    float sq = 0.f;
                    for (int i = lane; i < dk; i += 32) {
                        const float x = (float)c[row(t0 + tt) * dk + i];
                        sq = fmaf(x, x, sq);
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
                    const float inv = 1.f / fmaxf(sqrtf(sq), kNormFloor);
                    for (int i = lane; i < 64; i += 32) q[tt][i] *= inv;
                }
            }
            base = Gam[kOutTile - 1];   // (tokens past the run's end add zero)
        }
        if (pieces) asm volatile("cp.async.wait_group 1;\n" ::: "memory");   // this sub-tile's group
        __syncthreads();
        for (int tt = 0; tt < nt; tt++) {
            float qv[4], dv4[4];
            ld4(&q[tt][i0], qv);
            ld4(dd + tt * 64 + j0, dv4);
            const float2 d01 = make_float2(dv4[0], dv4[1]), d23 = make_float2(dv4[2], dv4[3]);
#pragma unroll
            for (int a = 0; a < 4; a++) {
                const float2 qa = make_float2(qv[a], qv[a]);
                acc[a][0] = __ffma2_rn(qa, d01, acc[a][0]);
                acc[a][1] = __ffma2_rn(qa, d23, acc[a][1]);
            }
        }
    }
    float* Gout = G + (size_t)(u * gridDim.y + blockIdx.y) * dk * dv;
#pragma unroll
    for (int a = 0; a < 4; a++) {
        const float r[4] = {acc[a][0].x, acc[a][0].y, acc[a][1].x, acc[a][1].y};
#pragma unroll
        for (int b = 0; b < 4; b++)
            if (i0 + a < dk && j0 + b < dv) Gout[(size_t)(i0 + a) * dv + j0 + b] = r[b];
    }
}

// G_p = the runs' partials [unit][run][d_k x d_v] added in run order
__global__ void gp_reduce_kernel(const float* part, float* G, int units, int runs, int n)
{
    const size_t total = (size_t)units * n;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const size_t u = e / n, k = e - u * n;
        const float* p = part + u * runs * n + k;
        float x = 0.f;
        for (int r = 0; r < runs; r++) x += p[(size_t)r * n];
        G[e] = x;
    }
}

template <typename IO>
cudaError_t gp_smem_attr(int bytes)
{
    cudaError_t e = cudaFuncSetAttribute(tsplit_gp_kernel<IO, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tsplit_gp_kernel<IO, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e;
}

// The scans over segments, one CTA per (batch, head), P sequential steps of a
// 64 x 64 x 64 fp32 product:
//   forward (steps 3):  X_0 = h0;   X_{p+1} = A_p X_p + H_p;     stores X_p, ends with h_T
//   reverse (step 6):   X = dh_T;   X <- A_p^T X + G_p (p = P-1 .. 0); stores X before
//                                   each update (the end gradients), ends with dh0
// Delta: A_p from the transition runs; gated: A_p = diag(exp(A sum_{t in p} g_t)).
// Thread t owns the 4 x 4 output tile rows 4 (t >> 4) .., columns 4 (t & 15) ..;
// the product reads one float4 of A (transposed in shared memory) and one of X
// per 16 FMAs.  The segment sums of g are fixed-order block reductions.
constexpr int kSP = 68;   // padded row stride of the 64 x 64 tiles
constexpr int kMaxSeg = 152;

template <typename IO, bool DELTA, bool REVERSE>
__global__ void __launch_bounds__(256) seg_scan_kernel(const float* Abuf, const float* Add, const float* X0,
                                                       float* Xst, float* Xend, const IO* g, const float* A_log,
                                                       int B, int H, int T, int P, int dk, int dv, int logits)
{
    __shared__ __align__(16) float Xs[64][kSP];
    __shared__ __align__(16) float MT[64][kSP];   // MT[k][i] = M[i][k], M = A_p (forward) or A_p^T (reverse)
    __shared__ float dec[64];
    __shared__ float gseg[kMaxSeg];
    __shared__ float red[8][kMaxSeg];
    const int u = blockIdx.x, bb = u / H, h = u % H, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int Ts = T / P, i0 = 4 * (tid >> 4), j0 = 4 * (tid & 15);
    const size_t S = (size_t)dk * dv;

    for (int idx = tid; idx < 64 * kSP; idx += 256) {
        const int i = idx / kSP, j = idx % kSP;
        Xs[i][j] = (X0 && i < dk && j < dv) ? X0[(size_t)u * S + (size_t)i * dv + j] : 0.f;
        if (!DELTA) MT[i][j] = 0.f;
    }
    if (!DELTA) {
        // sum of the gates of every segment: each thread its strided tokens, then the warps in order
        for (int p = 0; p < P; p++) {
            float part = 0.f;
            for (int t = tid; t < Ts; t += 256) {
                const float gv = (float)g[((size_t)bb * T + (size_t)p * Ts + t) * H + h];
                part += logits ? 1.f / (1.f + expf(-gv)) : gv;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (lane == 0) red[w][p] = part;
        }
        __syncthreads();
        for (int p = tid; p < P; p += 256) {
            float sum = 0.f;
#pragma unroll
            for (int ww = 0; ww < 8; ww++) sum += red[ww][p];
            gseg[p] = sum;
        }
    }
    __syncthreads();

    for (int step = 0; step < P; step++) {
        const int p = REVERSE ? P - 1 - step : step;
        const size_t vu = ((size_t)(bb * P + p) * H + h);   // unit of the [B*P, T/P, H] view
        for (int idx = tid; idx < dk * dv; idx += 256) Xst[vu * S + idx] = Xs[idx / dv][idx % dv];
        if (DELTA) {
            const float* A = Abuf + vu * dk * dk;
            for (int idx = tid; idx < 64 * 64; idx += 256) {
                const int r = idx >> 6, c = idx & 63;    // MT[r][c]
                float x = 0.f;
                if (r < dk && c < dk) x = REVERSE ? A[r * dk + c] : A[c * dk + r];
                MT[r][c] = x;
            }
        } else if (tid < 64) {
            dec[tid] = tid < dk ? expf(gseg[p] * -expf(A_log[h * dk + tid])) : 0.f;
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int i = i0 + a, j = j0 + c;
                acc[a][c] = (i < dk && j < dv) ? Add[vu * S + (size_t)i * dv + j] : 0.f;
            }
        if (DELTA) {
            for (int k = 0; k < dk; k++) {
                const float4 m = *reinterpret_cast<const float4*>(&MT[k][i0]);
                const float4 x = *reinterpret_cast<const float4*>(&Xs[k][j0]);
                const float mv[4] = {m.x, m.y, m.z, m.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int a = 0; a < 4; a++)
#pragma unroll
                    for (int c = 0; c < 4; c++) acc[a][c] = fmaf(mv[a], xv[c], acc[a][c]);
            }
        } else {
#pragma unroll
            for (int a = 0; a < 4; a++) {
                const float4 x = *reinterpret_cast<const float4*>(&Xs[i0 + a][j0]);
                acc[a][0] = fmaf(dec[i0 + a], x.x, acc[a][0]);
                acc[a][1] = fmaf(dec[i0 + a], x.y, acc[a][1]);
                acc[a][2] = fmaf(dec[i0 + a], x.z, acc[a][2]);
                acc[a][3] = fmaf(dec[i0 + a], x.w, acc[a][3]);
            }
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < 4; a++)
            *reinterpret_cast<float4*>(&Xs[i0 + a][j0]) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        __syncthreads();
    }
    if (Xend)
        for (int idx = tid; idx < dk * dv; idx += 256) Xend[(size_t)u * S + idx] = Xs[idx / dv][idx % dv];
}

template <bool REVERSE>
static void launch_seg_scan(const Args& a, int P, const float* Abuf, const float* Add, const float* X0, float* Xst,
                            float* Xend, cudaStream_t st)
{
    const int units = a.B * a.H;
    if (a.io == GDN_BF16) {
        if (a.mode == GDN_DELTA)
            seg_scan_kernel<__nv_bfloat16, true, REVERSE><<<units, 256, 0, st>>>(
                Abuf, Add, X0, Xst, Xend, (const __nv_bfloat16*)a.g, a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
        else
            seg_scan_kernel<__nv_bfloat16, false, REVERSE><<<units, 256, 0, st>>>(
                Abuf, Add, X0, Xst, Xend, (const __nv_bfloat16*)a.g, a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
    } else {
        if (a.mode == GDN_DELTA)
            seg_scan_kernel<float, true, REVERSE><<<units, 256, 0, st>>>(
                Abuf, Add, X0, Xst, Xend, (const float*)a.g, a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
        else
            seg_scan_kernel<float, false, REVERSE><<<units, 256, 0, st>>>(
                Abuf, Add, X0, Xst, Xend, (const float*)a.g, a.A_log, a.B, a.H, a.T, P, a.dk, a.dv, a.logits);
    }
}

}  // namespace

int tsplit_factor(const gdn_shape_t& s, int backward)
{
    const long units = (long)s.B * s.H;
    // the segment scan keeps 64 x 64 tiles: wider heads are not split
    if (s.dk > 64 || s.dv > 64) return 1;
    // forward: three passes (delta) or two (gated) must still pay; backward: one backward pass over T / P,
    // the forward passes and the G_p reduction are cheap beside it
    const int min_p = backward ? 2 : (s.mode == GDN_DELTA ? 4 : 3);
    const long cap = kSplitSMs / units;
    for (long p = cap; p >= min_p; p--) {
        if (s.T % p) continue;
        if (s.T / p < kSplitMinTokens) continue;
        return (int)p;
    }
    return 1;
}

// Steps 1-3: the entering state of every segment into L.ts_s_off and, if
// hT is given, the leaving state of the whole sequence; the zero-start outputs
// (step 1) into L.ts_o_off and, delta, the transition run's (step 2) into
// L.ts_so_off, both fp32.
static cudaError_t tsplit_states(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                                 cudaError_t (*fwd_core)(const Args&, cudaStream_t))
{
    unsigned char* ws = (unsigned char*)a.ws;
    float* Hbuf = (float*)(ws + L.ts_h_off);
    float* Abuf = (float*)(ws + L.ts_a_off);
    float* Sst = (float*)(ws + L.ts_s_off);
    float* Ibuf = (float*)(ws + L.ts_i_off);
    void* zv = ws + L.ts_zv_off;
    float* so = (float*)(ws + L.ts_so_off);
    float* o0 = (float*)(ws + L.ts_o_off);
    const bool bf = a.io == GDN_BF16;
    const int Ts = a.T / P;
    const size_t vunits = (size_t)a.B * P * a.H;
    cudaError_t e;

    // 1. leaving states from a zero start
    Args r = a;
    r.B = a.B * P;
    r.T = Ts;
    r.h0 = nullptr;
    r.hT = Hbuf;
    r.o = bf ? a.o : (void*)o0;   // the zero-start outputs, in fp32 (o0)
    r.o32 = bf ? o0 : nullptr;
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
        t.o = bf ? a.o : (void*)so;   // Phi_t^T c_t, in fp32 (so)
        t.o32 = bf ? so : nullptr;
        t.h0 = Ibuf;
        t.hT = Abuf;
        if ((e = fwd_core(t, st)) != cudaSuccess) return e;
    }

    // 3. scan over segments
    launch_seg_scan<false>(a, P, Abuf, Hbuf, a.h0, Sst, a.hT, st);
    return cudaGetLastError();
}

cudaError_t launch_fwd_tsplit(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                              cudaError_t (*fwd_core)(const Args&, cudaStream_t))
{
    cudaError_t e = tsplit_states(a, L, P, st, fwd_core);
    if (e != cudaSuccess) return e;
    // 4. o_t = o0_t + S_p^T Phi_t^T c_t
    const unsigned char* ws = (const unsigned char*)a.ws;
    const float* o0 = (const float*)(ws + L.ts_o_off);
    const float* so = (const float*)(ws + L.ts_so_off);
    const float* Sst = (const float*)(ws + L.ts_s_off);
    const int Ts = a.T / P;
    const dim3 grid(a.B * P * a.H, (Ts + kOutRun - 1) / kOutRun);
    const int osm = (int)sizeof(OutSmem);
    cudaError_t e2;
    if ((e2 = out_smem_attr<__nv_bfloat16>(osm)) != cudaSuccess || (e2 = out_smem_attr<float>(osm)) != cudaSuccess)
        return e2;
    if (a.io == GDN_BF16) {
        if (a.mode == GDN_DELTA)
            tsplit_out_kernel<__nv_bfloat16, true><<<grid, 256, osm, st>>>(
                o0, so, (const __nv_bfloat16*)a.c, (const __nv_bfloat16*)a.g, a.A_log, Sst, (__nv_bfloat16*)a.o, a.H,
                Ts, a.dk, a.dv, a.logits, a.norm);
        else
            tsplit_out_kernel<__nv_bfloat16, false><<<grid, 256, osm, st>>>(
                o0, so, (const __nv_bfloat16*)a.c, (const __nv_bfloat16*)a.g, a.A_log, Sst, (__nv_bfloat16*)a.o, a.H,
                Ts, a.dk, a.dv, a.logits, a.norm);
    } else {
        if (a.mode == GDN_DELTA)
            tsplit_out_kernel<float, true><<<grid, 256, osm, st>>>(o0, so, (const float*)a.c, (const float*)a.g, a.A_log,
                                                                 Sst, (float*)a.o, a.H, Ts, a.dk, a.dv, a.logits,
                                                                 a.norm);
        else
            tsplit_out_kernel<float, false><<<grid, 256, osm, st>>>(o0, so, (const float*)a.c, (const float*)a.g,
                                                                  a.A_log, Sst, (float*)a.o, a.H, Ts, a.dk, a.dv,
                                                                  a.logits, a.norm);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_tsplit(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                              cudaError_t (*fwd_core)(const Args&, cudaStream_t))
{
    unsigned char* ws = (unsigned char*)a.ws;
    const float* Sst = (const float*)(ws + L.ts_s_off);
    float* Gbuf = (float*)(ws + L.ts_g_off);
    float* Ebuf = (float*)(ws + L.ts_e_off);
    cudaError_t e;

    // 1-3. entering states of the segments (the runs' outputs are not needed here)
    Args fa = a;
    fa.hT = nullptr;
    if ((e = tsplit_states(fa, L, P, st, fwd_core)) != cudaSuccess) return e;

    // 5. G_p = sum_t (Phi_t^T c_t) do_t^T over each segment, by runs of kGpRun tokens; with several runs their
    //    partials go where the zero-start outputs were (dead in the backward: at most 2 T/P / kGpRun * d_k <=
    //    T/P * d_v / 4 floats per unit, within its T/P * d_v)
    const float* so = (const float*)(ws + L.ts_so_off);
    const int Ts = a.T / P;
    const int vunits = a.B * P * a.H;
    const int runs = (Ts + kGpRun - 1) / kGpRun;
    float* Gpart = runs > 1 ? (float*)(ws + L.ts_o_off) : Gbuf;
    const dim3 ggrid(vunits, runs);
    const int gsm = (int)sizeof(GpSmem);
    if ((e = gp_smem_attr<__nv_bfloat16>(gsm)) != cudaSuccess || (e = gp_smem_attr<float>(gsm)) != cudaSuccess)
        return e;
    if (a.io == GDN_BF16) {
        if (a.mode == GDN_DELTA)
            tsplit_gp_kernel<__nv_bfloat16, true><<<ggrid, 256, gsm, st>>>(
                so, (const __nv_bfloat16*)a.c, (const __nv_bfloat16*)a.g, (const __nv_bfloat16*)a.dO, a.A_log, Gpart,
                a.H, Ts, a.dk, a.dv, a.logits, a.norm);
        else
            tsplit_gp_kernel<__nv_bfloat16, false><<<ggrid, 256, gsm, st>>>(
                so, (const __nv_bfloat16*)a.c, (const __nv_bfloat16*)a.g, (const __nv_bfloat16*)a.dO, a.A_log, Gpart,
                a.H, Ts, a.dk, a.dv, a.logits, a.norm);
    } else {
        if (a.mode == GDN_DELTA)
            tsplit_gp_kernel<float, true><<<ggrid, 256, gsm, st>>>(so, (const float*)a.c, (const float*)a.g,
                                                                   (const float*)a.dO, a.A_log, Gpart, a.H, Ts, a.dk,
                                                                   a.dv, a.logits, a.norm);
        else
            tsplit_gp_kernel<float, false><<<ggrid, 256, gsm, st>>>(so, (const float*)a.c, (const float*)a.g,
                                                                    (const float*)a.dO, a.A_log, Gpart, a.H, Ts, a.dk,
                                                                    a.dv, a.logits, a.norm);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (runs > 1) {
        gp_reduce_kernel<<<256, 256, 0, st>>>(Gpart, Gbuf, vunits, runs, a.dk * a.dv);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    Args b = a;
    b.B = a.B * P;
    b.T = a.T / P;
    b.h0 = Sst;

    // 6. reverse scan of the end gradients; dh0 of the whole sequence
    const float* Abuf = (const float*)(ws + L.ts_a_off);
    launch_seg_scan<true>(a, P, Abuf, Gbuf, a.dhT, Ebuf, a.dh0, st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // 7. every segment's backward with its true end gradient
    b.dhT = Ebuf;
    b.dh0 = nullptr;
    return launch_serial_bwd(b, st);
}

}  // namespace gdn
