// gdn_decode.cu -- forward for short sequences (1 <= T <= 8 tokens), the
// token-by-token decoding case: the state comes in through h0 and leaves
// through hT, possibly the same buffer.
//
// The recurrence is the per-token one of "GDN & MLA Mechanism Deep-Dive",
// Step 4 (gated) and the delta-rule card of "HyMo-434M -- documentation
// portal" (delta); the pages motivate the linear state by this use: a fixed
// d_k x d_v state per head instead of a growing cache.  With T this small the
// work is moving the fp32 state (16 KB per head each way at d = 64), so the
// kernel is laid out for state traffic: persistent CTAs (as many per SM as
// fit) walk the items, one (batch, head) unit and 64-column slab of the value
// each (columns of the state never mix); while one item computes, the next
// item's state streams into a second shared buffer by cp.async and its tokens
// into registers, so every CTA keeps bytes in flight.  256 threads; thread t
// owns columns 4 (t & 15) .. +3 of rows (t >> 4) + 16 k, k < d_k rows / 16
// (64 or 128 rows).  Sums over rows go through registers, one shuffle and a
// fixed-order pass over eight per-warp partials in shared memory.
#include "gdn_internal.h"
#include "serial_common.cuh"

namespace gdn {
namespace {

using namespace rec;

constexpr int kDecMaxT = 8;

// One work item's token inputs held in registers until they are staged.  The
// key-side rows [T][ROWS] are spread as elements idx = t + 256 q (q < NQ), the
// value rows [T][64] of the item's column slab as idx = t + 256 q (q < 2).
template <typename IO, int ROWS>
struct TokRegs {   // raw I/O values: converted when staged, so nothing waits on the loads meanwhile
    static constexpr int NQ = kDecMaxT * ROWS / 256;
    IO g[NQ], b[NQ], c[NQ], v[2];
    IO beta;
};

struct Item {
    int u, bb, h, jc0, nv;   // unit, its batch and head, value columns jc0 .. jc0 + nv - 1
};

__device__ __forceinline__ Item item_of(const Args& a, int it, int nslab)
{
    Item r;
    r.u = it / nslab;
    r.bb = r.u / a.H;
    r.h = r.u % a.H;
    r.jc0 = 64 * (it % nslab);
    r.nv = min(64, a.dv - r.jc0);
    return r;
}

template <typename IO, bool DELTA, int ROWS>
__device__ __forceinline__ void load_tokens(const Args& a, const Item& I, TokRegs<IO, ROWS>& r)
{
    constexpr int NQ = TokRegs<IO, ROWS>::NQ;
    const int tid = threadIdx.x, dk = a.dk, dv = a.dv, T = a.T, H = a.H;
#pragma unroll
    for (int q = 0; q < NQ; q++) {
        const int idx = tid + 256 * q, tt = idx / ROWS, i = idx % ROWS;
        r.g[q] = r.b[q] = r.c[q] = from_f<IO>(0.f);
        if (tt < T) {
            const size_t row = ((size_t)I.bb * T + tt) * H + I.h;
            r.g[q] = ((const IO*)a.g)[row];
            if (i < dk) {
                r.b[q] = ((const IO*)a.b)[row * dk + i];
                r.c[q] = ((const IO*)a.c)[row * dk + i];
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 2; q++) {
        const int idx = tid + 256 * q, tt = idx >> 6, i = idx & 63;
        r.v[q] = from_f<IO>(0.f);
        if (tt < T && i < I.nv) r.v[q] = ((const IO*)a.v)[(((size_t)I.bb * T + tt) * H + I.h) * dv + I.jc0 + i];
    }
    r.beta = (DELTA && tid < T) ? ((const IO*)a.beta)[((size_t)I.bb * T + tid) * H + I.h] : from_f<IO>(0.f);
}

// the item's fp32 state (d_k rows x its nv columns) into a shared buffer [ROWS][64] by cp.async
__device__ __forceinline__ void issue_state(const Args& a, const Item& I, float* dst)
{
    if (a.dv == 64) {   // the slab is the whole row: one contiguous 16-byte stream
        const float4* src = reinterpret_cast<const float4*>(a.h0 + (size_t)I.u * a.dk * 64);
        for (int idx = threadIdx.x; idx < a.dk * 16; idx += 256) cp_async16(reinterpret_cast<float4*>(dst) + idx, src + idx);
    } else {
        const int nq = I.nv / 4, n16 = a.dk * nq;
        for (int idx = threadIdx.x; idx < n16; idx += 256) {
            const int i = idx / nq, q = idx - i * nq;
            cp_async16(dst + i * 64 + 4 * q, a.h0 + ((size_t)I.u * a.dk + i) * a.dv + I.jc0 + 4 * q);
        }
    }
    cp_async_commit();
}

template <int ROWS>
struct DecSmem {
    float snext[2][ROWS * 64];   // double-buffered incoming states
    float sAl[kDecMaxT][ROWS], sB[kDecMaxT][ROWS], sC[kDecMaxT][ROWS], sV[kDecMaxT][64];
    float sbeta[kDecMaxT];
    float nb[kDecMaxT], nc[kDecMaxT];   // GDN_NORM_BC: 1 / max(||b_t||, floor), the same for c_t
    float redR[8][64], redO[8][64];
    float xcol[64];
};

// NORM: b and c arrive before their L2 normalisation (a template flag, so the plain kernel carries no trace of it)
template <typename IO, bool DELTA, int ROWS, bool NORM>
__global__ void __launch_bounds__(256) decode_kernel(Args a, bool vec4, int nslab)
{
    constexpr int K = ROWS / 16;   // state rows per thread
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ __align__(16) DecSmem<ROWS == 64 ? 64 : 1> s64;
    DecSmem<ROWS>& S = *reinterpret_cast<DecSmem<ROWS>*>(ROWS == 64 ? reinterpret_cast<unsigned char*>(&s64)
                                                                       : smem_raw);

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int cq = tid & 15, rg = tid >> 4;
    const int dk = a.dk, dv = a.dv, T = a.T, H = a.H;
    const int items = a.B * a.H * nslab, G = gridDim.x;
    const int j0 = 4 * cq;
    const bool pre = vec4 && a.h0 != nullptr;   // state prefetch by cp.async (rows of whole 16-byte quads)
    IO* o = (IO*)a.o;

    TokRegs<IO, ROWS> tr;
    int it = blockIdx.x;
    Item I = item_of(a, it, nslab);
    load_tokens<IO, DELTA, ROWS>(a, I, tr);
    if (pre) issue_state(a, I, S.snext[0]);

    for (int n = 0; it < items; it += G, n++) {
        const int buf = n & 1, itn = it + G;
        const Item In = item_of(a, itn < items ? itn : it, nslab);
        // stage this item's tokens (decay factors computed here), then fetch the next item's
#pragma unroll
        for (int q = 0; q < TokRegs<IO, ROWS>::NQ; q++) {
            const int idx = tid + 256 * q, tt = idx / ROWS, i = idx % ROWS;
            if (tt < kDecMaxT) {
                S.sAl[tt][i] = i < dk ? expf(gate(to_f(tr.g[q]), a.logits) * -expf(a.A_log[I.h * dk + i])) : 0.f;
                S.sB[tt][i] = to_f(tr.b[q]);
                S.sC[tt][i] = to_f(tr.c[q]);
            }
        }
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int idx = tid + 256 * q, tt = idx >> 6, i = idx & 63;
            if (tt < kDecMaxT) S.sV[tt][i] = to_f(tr.v[q]);
        }
        if (DELTA && tid < kDecMaxT) S.sbeta[tid] = gate(to_f(tr.beta), a.logits);
        if (itn < items) {
            load_tokens<IO, DELTA, ROWS>(a, In, tr);
            if (pre) issue_state(a, In, S.snext[buf ^ 1]);
        }
        if (pre) {
            if (itn < items) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
            else cp_async_wait_all();
        }
        __syncthreads();
        if (NORM) {   // inverse norms of the staged b_t and c_t, one thread per vector
            if (tid < 2 * T) {
                const int tt = tid >> 1;
                const float* x = (tid & 1) ? S.sC[tt] : S.sB[tt];
                float q = 0.f;
                for (int i = 0; i < dk; i++) q = fmaf(x[i], x[i], q);
                (tid & 1 ? S.nc : S.nb)[tt] = 1.f / fmaxf(sqrtf(q), kNormFloor);
            }
            __syncthreads();
        }

        // state entries (row rg + 16 k, columns j0 .. j0 + 3 of the slab)
        float hs[K][4];
#pragma unroll
        for (int k = 0; k < K; k++) {
            const int i = rg + 16 * k;
            if (pre) {
                if (i < dk && j0 < I.nv) {
                    const float4 q = *reinterpret_cast<const float4*>(&S.snext[buf][i * 64 + j0]);
                    hs[k][0] = q.x; hs[k][1] = q.y; hs[k][2] = q.z; hs[k][3] = q.w;
                } else {
                    hs[k][0] = hs[k][1] = hs[k][2] = hs[k][3] = 0.f;
                }
            } else {
                const float* src = a.h0 ? a.h0 + ((size_t)I.u * dk + i) * dv + I.jc0 + j0 : nullptr;
                if (src && i < dk && vec4 && j0 < I.nv) {
                    const float4 q = *reinterpret_cast<const float4*>(src);
                    hs[k][0] = q.x; hs[k][1] = q.y; hs[k][2] = q.z; hs[k][3] = q.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; c++) hs[k][c] = (src && i < dk && j0 + c < I.nv) ? src[c] : 0.f;
                }
            }
        }

        for (int tt = 0; tt < T; tt++) {
            float al[K], bk[K], ck[K];
#pragma unroll
            for (int k = 0; k < K; k++) {
                al[k] = S.sAl[tt][rg + 16 * k];
                bk[k] = S.sB[tt][rg + 16 * k];
                ck[k] = S.sC[tt][rg + 16 * k];
            }
            if (NORM) {
#pragma unroll
                for (int k = 0; k < K; k++) {
                    bk[k] *= S.nb[tt];
                    ck[k] *= S.nc[tt];
                }
            }
            float hp[K][4];
#pragma unroll
            for (int k = 0; k < K; k++)
#pragma unroll
                for (int c = 0; c < 4; c++) hp[k][c] = hs[k][c] * al[k];
            if (DELTA) {
                // r_j = sum_i h'[i, j] b_i over this thread's rows, then the 16 row groups
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    float r = hp[0][c] * bk[0];
#pragma unroll
                    for (int k = 1; k < K; k++) r = fmaf(hp[k][c], bk[k], r);
                    r += __shfl_xor_sync(kFull, r, 16);
                    if (lane < 16) S.redR[w][j0 + c] = r;
                }
            }
            __syncthreads();
            if (tid < 64) {
                if (DELTA) {
                    float r = 0.f;
#pragma unroll
                    for (int ww = 0; ww < 8; ww++) r += S.redR[ww][tid];
                    S.xcol[tid] = S.sbeta[tt] * (S.sV[tt][tid] - r);
                }
                if (tt > 0 && tid < I.nv) {  // output of the previous token (its partials are complete now)
                    float ov = 0.f;
#pragma unroll
                    for (int ww = 0; ww < 8; ww++) ov += S.redO[ww][tid];
                    o[(((size_t)I.bb * T + tt - 1) * H + I.h) * dv + I.jc0 + tid] = from_f<IO>(ov);
                }
            }
            __syncthreads();
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const float x = DELTA ? S.xcol[j0 + c] : S.sV[tt][j0 + c];
#pragma unroll
                for (int k = 0; k < K; k++) hs[k][c] = fmaf(bk[k], x, hp[k][c]);
                float ov = hs[0][c] * ck[0];
#pragma unroll
                for (int k = 1; k < K; k++) ov = fmaf(hs[k][c], ck[k], ov);
                ov += __shfl_xor_sync(kFull, ov, 16);
                if (lane < 16) S.redO[w][j0 + c] = ov;
            }
        }
        __syncthreads();
        if (tid < I.nv) {
            float ov = 0.f;
#pragma unroll
            for (int ww = 0; ww < 8; ww++) ov += S.redO[ww][tid];
            o[(((size_t)I.bb * T + T - 1) * H + I.h) * dv + I.jc0 + tid] = from_f<IO>(ov);
        }
        if (a.hT) {
#pragma unroll
            for (int k = 0; k < K; k++) {
                const int i = rg + 16 * k;
                if (i >= dk || j0 >= I.nv) continue;
                float* dst = a.hT + ((size_t)I.u * dk + i) * dv + I.jc0 + j0;
                if (vec4) {
                    *reinterpret_cast<float4*>(dst) = make_float4(hs[k][0], hs[k][1], hs[k][2], hs[k][3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        if (j0 + c < I.nv) dst[c] = hs[k][c];
                }
            }
        }
        __syncthreads();   // staged tokens, partials and this state buffer are free for the next item
        I = In;
    }
}

template <typename IO, bool DELTA, int ROWS, bool NORM>
cudaError_t launch_rows(const Args& a, cudaStream_t st)
{
    // float4 state access needs whole 16-byte column quads in every row
    const bool vec4 = (a.dv % 4) == 0 && (!a.h0 || ((uintptr_t)a.h0 & 15) == 0) &&
                      (!a.hT || ((uintptr_t)a.hT & 15) == 0);
    const size_t smem = ROWS == 64 ? 0 : sizeof(DecSmem<ROWS>);   // 64 rows: static shared memory
    if (smem) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<IO, DELTA, ROWS, NORM>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int sms = 0, dev = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<IO, DELTA, ROWS, NORM>, 256, smem) !=
            cudaSuccess)
        return cudaErrorUnknown;
    if (per_sm < 1) per_sm = 1;
    // persistent CTAs, as many as fit at once, walk the (unit, 64-column slab) items
    const int nslab = (a.dv + 63) / 64;
    const int items = a.B * a.H * nslab;
    const int grid = items < sms * per_sm ? items : sms * per_sm;
    decode_kernel<IO, DELTA, ROWS, NORM><<<grid, 256, smem, st>>>(a, vec4, nslab);
    return cudaGetLastError();
}

template <typename IO, bool DELTA>
cudaError_t launch_t(const Args& a, cudaStream_t st)
{
    if (a.norm) return a.dk <= 64 ? launch_rows<IO, DELTA, 64, true>(a, st) : launch_rows<IO, DELTA, 128, true>(a, st);
    return a.dk <= 64 ? launch_rows<IO, DELTA, 64, false>(a, st) : launch_rows<IO, DELTA, 128, false>(a, st);
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
