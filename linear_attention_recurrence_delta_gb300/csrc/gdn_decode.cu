// gdn_decode.cu -- forward for short sequences (1 <= T <= 8 tokens), the
// token-by-token decoding case: the state comes in through h0 and leaves
// through hT, possibly the same buffer.
//
// The recurrence is the per-token one of "GDN & MLA Mechanism Deep-Dive",
// Step 4 (gated) and the delta-rule card of "HyMo-434M -- documentation
// portal" (delta); the pages motivate the linear state by this use: a fixed
// d_k x d_v state per head instead of a growing cache.  With T this small the
// work is moving the fp32 state (16 KB per head each way at d = 64), so the
// kernel is laid out for coalesced state traffic: one CTA per (batch, head),
// 256 threads; thread t owns columns 4 (t & 15) .. +3 of rows (t >> 4) + 16 k,
// k = 0..3, so a warp reads two full 256-byte state rows per access.  Sums
// over rows go through registers, one shuffle and a fixed-order pass over
// eight per-warp partials in shared memory.
#include "gdn_internal.h"
#include "serial_common.cuh"

namespace gdn {
namespace {

using namespace rec;

constexpr int kDecMaxT = 8;

template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) decode_kernel(Args a, bool vec4)
{
    __shared__ float sAl[kDecMaxT][64], sB[kDecMaxT][64], sC[kDecMaxT][64], sV[kDecMaxT][64];
    __shared__ float sbeta[kDecMaxT];
    __shared__ float redR[8][64], redO[8][64];
    __shared__ float xcol[64];

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int cq = tid & 15, rg = tid >> 4;
    const int u = blockIdx.x, bb = u / a.H, h = u % a.H;
    const int dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    const int j0 = 4 * cq;

    for (int idx = tid; idx < T * 64; idx += 256) {
        const int tt = idx >> 6, i = idx & 63;
        const size_t row = ((size_t)bb * T + tt) * H + h;
        float xa = 0.f, xb = 0.f, xc = 0.f, xv = 0.f;
        if (i < dk) {
            const float g = to_f(((const IO*)a.g)[row]);
            xa = expf(g * -expf(a.A_log[h * dk + i]));
            xb = to_f(((const IO*)a.b)[row * dk + i]);
            xc = to_f(((const IO*)a.c)[row * dk + i]);
        }
        if (i < dv) xv = to_f(((const IO*)a.v)[row * dv + i]);
        sAl[tt][i] = xa;
        sB[tt][i] = xb;
        sC[tt][i] = xc;
        sV[tt][i] = xv;
    }
    if (DELTA && tid < T) sbeta[tid] = to_f(((const IO*)a.beta)[((size_t)bb * T + tid) * H + h]);

    // state entries (row rg + 16 k, columns j0 .. j0 + 3)
    float hs[4][4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int i = rg + 16 * k;
        const float* src = a.h0 ? a.h0 + ((size_t)u * dk + i) * dv + j0 : nullptr;
        if (src && i < dk && vec4 && j0 < dv) {
            const float4 q = *reinterpret_cast<const float4*>(src);
            hs[k][0] = q.x; hs[k][1] = q.y; hs[k][2] = q.z; hs[k][3] = q.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; c++) hs[k][c] = (src && i < dk && j0 + c < dv) ? src[c] : 0.f;
        }
    }
    __syncthreads();

    IO* o = (IO*)a.o;
    for (int tt = 0; tt < T; tt++) {
        float al[4], bk[4], ck[4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            al[k] = sAl[tt][rg + 16 * k];
            bk[k] = sB[tt][rg + 16 * k];
            ck[k] = sC[tt][rg + 16 * k];
        }
        float hp[4][4];
#pragma unroll
        for (int k = 0; k < 4; k++)
#pragma unroll
            for (int c = 0; c < 4; c++) hp[k][c] = hs[k][c] * al[k];
        if (DELTA) {
            // r_j = sum_i h'[i, j] b_i over this thread's 4 rows, then the 16 row groups
#pragma unroll
            for (int c = 0; c < 4; c++) {
                float r = hp[0][c] * bk[0];
#pragma unroll
                for (int k = 1; k < 4; k++) r = fmaf(hp[k][c], bk[k], r);
                r += __shfl_xor_sync(kFull, r, 16);
                if (lane < 16) redR[w][j0 + c] = r;
            }
        }
        __syncthreads();
        if (tid < 64) {
            if (DELTA) {
                float r = 0.f;
#pragma unroll
                for (int ww = 0; ww < 8; ww++) r += redR[ww][tid];
                xcol[tid] = sbeta[tt] * (sV[tt][tid] - r);
            }
            if (tt > 0 && tid < dv) {  // output of the previous token (its partials are complete now)
                float ov = 0.f;
#pragma unroll
                for (int ww = 0; ww < 8; ww++) ov += redO[ww][tid];
                o[(((size_t)bb * T + tt - 1) * H + h) * dv + tid] = from_f<IO>(ov);
            }
        }
        __syncthreads();
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const float x = DELTA ? xcol[j0 + c] : sV[tt][j0 + c];
#pragma unroll
            for (int k = 0; k < 4; k++) hs[k][c] = fmaf(bk[k], x, hp[k][c]);
            float ov = hs[0][c] * ck[0];
#pragma unroll
            for (int k = 1; k < 4; k++) ov = fmaf(hs[k][c], ck[k], ov);
            ov += __shfl_xor_sync(kFull, ov, 16);
            if (lane < 16) redO[w][j0 + c] = ov;
        }
    }
    __syncthreads();
    if (tid < dv) {
        float ov = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ww++) ov += redO[ww][tid];
        o[(((size_t)bb * T + T - 1) * H + h) * dv + tid] = from_f<IO>(ov);
    }
    if (a.hT) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = rg + 16 * k;
            if (i >= dk || j0 >= dv) continue;
            float* dst = a.hT + ((size_t)u * dk + i) * dv + j0;
            if (vec4) {
                *reinterpret_cast<float4*>(dst) = make_float4(hs[k][0], hs[k][1], hs[k][2], hs[k][3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; c++)
                    if (j0 + c < dv) dst[c] = hs[k][c];
            }
        }
    }
}

template <typename IO, bool DELTA>
cudaError_t launch_t(const Args& a, cudaStream_t st)
{
    // float4 state access needs whole 16-byte column quads in every row
    const bool vec4 = (a.dv % 4) == 0 && (!a.h0 || ((uintptr_t)a.h0 & 15) == 0) &&
                      (!a.hT || ((uintptr_t)a.hT & 15) == 0);
    decode_kernel<IO, DELTA><<<a.B * a.H, 256, 0, st>>>(a, vec4);
    return cudaGetLastError();
}

}  // namespace

int decode_max_tokens() { return kDecMaxT; }

cudaError_t launch_decode(const Args& a, cudaStream_t st)
{
    if (a.io == GDN_BF16)
        return a.mode == GDN_DELTA ? launch_t<__nv_bfloat16, true>(a, st) : launch_t<__nv_bfloat16, false>(a, st);
    return a.mode == GDN_DELTA ? launch_t<float, true>(a, st) : launch_t<float, false>(a, st);
}

}  // namespace gdn
