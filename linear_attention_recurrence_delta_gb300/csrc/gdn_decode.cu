// gdn_decode.cu -- forward for short sequences (1 <= T <= 8 tokens), the
// token-by-token decoding case: the state comes in through h0 and leaves
// through hT, possibly the same buffer.
//
// The recurrence is the per-token one of "GDN & MLA Mechanism Deep-Dive",
// Step 4 (gated) and the delta-rule card of "HyMo-434M -- documentation
// portal" (delta); the pages motivate the linear state by this use: a fixed
// d_k x d_v state per head instead of a growing cache.  With T this small the
// work is moving the fp32 state (16 KB per head each way at d = 64), so the
// kernel is laid out for state traffic: persistent CTAs (four per SM) walk
// the (batch, head) units; while one unit computes, the next unit's state
// streams into a second shared buffer by cp.async and its tokens into
// registers, so every CTA keeps bytes in flight.  256 threads; thread t owns
// columns 4 (t & 15) .. +3 of rows (t >> 4) + 16 k, k = 0..3.  Sums over rows
// go through registers, one shuffle and a fixed-order pass over eight
// per-warp partials in shared memory.
#include "gdn_internal.h"
#include "serial_common.cuh"

namespace gdn {
namespace {

using namespace rec;

constexpr int kDecMaxT = 8;
constexpr int kDecCtasPerSm = 4;   // 64 registers x 256 threads: four CTAs fill an SM's register file

// One unit's token inputs held in registers until they are staged: thread t
// owns elements idx = t + 256 q of the [T][64] rows (T <= 8, so q < 2).
template <typename IO>
struct TokRegs {   // raw I/O values: converted when staged, so nothing waits on the loads meanwhile
    IO g[2], b[2], c[2], v[2];
    IO beta;
};

template <typename IO, bool DELTA>
__device__ __forceinline__ void load_tokens(const Args& a, int u, TokRegs<IO>& r)
{
    const int tid = threadIdx.x, bb = u / a.H, h = u % a.H, dk = a.dk, dv = a.dv, T = a.T, H = a.H;
#pragma unroll
    for (int q = 0; q < 2; q++) {
        const int idx = tid + 256 * q, tt = idx >> 6, i = idx & 63;
        r.g[q] = r.b[q] = r.c[q] = r.v[q] = from_f<IO>(0.f);
        if (tt < T) {
            const size_t row = ((size_t)bb * T + tt) * H + h;
            r.g[q] = ((const IO*)a.g)[row];
            if (i < dk) {
                r.b[q] = ((const IO*)a.b)[row * dk + i];
                r.c[q] = ((const IO*)a.c)[row * dk + i];
            }
            if (i < dv) r.v[q] = ((const IO*)a.v)[row * dv + i];
        }
    }
    r.beta = (DELTA && tid < T) ? ((const IO*)a.beta)[((size_t)bb * T + tid) * H + h] : from_f<IO>(0.f);
}

// the unit's fp32 state (d_k x d_v, contiguous) into a shared buffer by cp.async
__device__ __forceinline__ void issue_state(const Args& a, int u, float* dst)
{
    const size_t n16 = (size_t)a.dk * a.dv / 4;
    const float4* src = reinterpret_cast<const float4*>(a.h0 + (size_t)u * a.dk * a.dv);
    for (size_t idx = threadIdx.x; idx < n16; idx += 256) cp_async16(reinterpret_cast<float4*>(dst) + idx, src + idx);
    cp_async_commit();
}

template <typename IO, bool DELTA>
__global__ void __launch_bounds__(256) decode_kernel(Args a, bool vec4)
{
    __shared__ __align__(16) float snext[2][64 * 64];   // double-buffered incoming states
    __shared__ float sAl[kDecMaxT][64], sB[kDecMaxT][64], sC[kDecMaxT][64], sV[kDecMaxT][64];
    __shared__ float sbeta[kDecMaxT];
    __shared__ float redR[8][64], redO[8][64];
    __shared__ float xcol[64];

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int cq = tid & 15, rg = tid >> 4;
    const int dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    const int units = a.B * a.H, G = gridDim.x;
    const int j0 = 4 * cq;
    const bool pre = vec4 && a.h0 != nullptr;   // state prefetch by cp.async (rows of whole 16-byte quads)
    IO* o = (IO*)a.o;

    TokRegs<IO> tr;
    int u = blockIdx.x;
    load_tokens<IO, DELTA>(a, u, tr);
    if (pre) issue_state(a, u, snext[0]);

    for (int it = 0; u < units; u += G, it++) {
        const int buf = it & 1, un = u + G, bb = u / H, h = u % H;
        // stage this unit's tokens (decay factors computed here), then fetch the next unit's
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int idx = tid + 256 * q, tt = idx >> 6, i = idx & 63;
            if (tt < kDecMaxT) {
                sAl[tt][i] = i < dk ? expf(gate(to_f(tr.g[q]), a.logits) * -expf(a.A_log[h * dk + i])) : 0.f;
                sB[tt][i] = to_f(tr.b[q]);
                sC[tt][i] = to_f(tr.c[q]);
                sV[tt][i] = to_f(tr.v[q]);
            }
        }
        if (DELTA && tid < kDecMaxT) sbeta[tid] = gate(to_f(tr.beta), a.logits);
        if (un < units) {
            load_tokens<IO, DELTA>(a, un, tr);
            if (pre) issue_state(a, un, snext[buf ^ 1]);
        }
        if (pre) {
            if (un < units) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
            else cp_async_wait_all();
        }
        __syncthreads();

        // state entries (row rg + 16 k, columns j0 .. j0 + 3)
        float hs[4][4];
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int i = rg + 16 * k;
            if (pre) {
                if (i < dk && j0 < dv) {
                    const float4 q = *reinterpret_cast<const float4*>(&snext[buf][i * dv + j0]);
                    hs[k][0] = q.x; hs[k][1] = q.y; hs[k][2] = q.z; hs[k][3] = q.w;
                } else {
                    hs[k][0] = hs[k][1] = hs[k][2] = hs[k][3] = 0.f;
                }
            } else {
                const float* src = a.h0 ? a.h0 + ((size_t)u * dk + i) * dv + j0 : nullptr;
                if (src && i < dk && vec4 && j0 < dv) {
                    const float4 q = *reinterpret_cast<const float4*>(src);
                    hs[k][0] = q.x; hs[k][1] = q.y; hs[k][2] = q.z; hs[k][3] = q.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; c++) hs[k][c] = (src && i < dk && j0 + c < dv) ? src[c] : 0.f;
                }
            }
        }

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
        __syncthreads();   // staged tokens, partials and this state buffer are free for the next unit
    }
}

template <typename IO, bool DELTA>
cudaError_t launch_t(const Args& a, cudaStream_t st)
{
    // float4 state access needs whole 16-byte column quads in every row
    const bool vec4 = (a.dv % 4) == 0 && (!a.h0 || ((uintptr_t)a.h0 & 15) == 0) &&
                      (!a.hT || ((uintptr_t)a.hT & 15) == 0);
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    const int units = a.B * a.H;
    const int grid = units < sms * kDecCtasPerSm ? units : sms * kDecCtasPerSm;
    decode_kernel<IO, DELTA><<<grid, 256, 0, st>>>(a, vec4);
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
