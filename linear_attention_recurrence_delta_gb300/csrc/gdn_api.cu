// gdn_api.cu -- the C ABI of libgdn: argument checks, workspace carve-up and
// dispatch to the kernels.  Nothing here allocates or synchronises, except
// gdn_last_device_status, whose job is to synchronise and read back.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gdn_internal.h"

namespace gdn {

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool shape_ok(const gdn_shape_t& s)
{
    if (s.B < 1 || s.H < 1 || s.T < 0) return false;
    // (batch, head) units index grids and int unit counters: at most 2^26 of them
    if ((double)s.B * s.H > (double)(1 << 26)) return false;
    if (s.dk < 1 || s.dk > 128 || s.dv < 1 || s.dv > 128) return false;
    if (s.io == GDN_BF16 && ((s.dk % 8) || (s.dv % 8))) return false;
    // keep every element offset inside a signed 64-bit range with margin
    const double elems = (double)s.B * s.T * s.H * 64.0;
    if (elems > 9.0e15) return false;
    return true;
}

// the serial backward's buffers for shape s, placed from `off`
static size_t place_bwd_core(const gdn_shape_t& s, WsLayout& L, size_t off, int norm)
{
    const size_t nslab = (size_t)bwd_slabs(s.dk, s.dv);
    const size_t ctas = (size_t)s.B * s.H * nslab;   // one CTA per unit and column slab
    const size_t nblk = (size_t)((s.T + kSerialBlock - 1) / kSerialBlock);
    L.snap_off = off;
    off = round_up(off + ctas * nblk * (kSerialBlock / kSerialSnap) * kStateSlot, 256);
    L.xvr_off = off;
    if (s.mode == GDN_DELTA)
        off = round_up(off + ctas * nblk * kSerialBlock * 2 * bwd_cols(s.dk) * sizeof(float), 256);
    L.dalog_off = off;
    off = round_up(off + ctas * (size_t)s.dk * 4, 256);
    L.slab_off = off;
    if (bwd_partials(s.dk, s.dv, norm)) {
        const size_t ntok = (size_t)s.B * s.T * s.H;
        off = round_up(off + nslab * ntok * (2 * (size_t)s.dk + 2) * sizeof(float), 256);
    }
    return off;
}

// buffers of a time split into P segments (see gdn_tsplit.cu), placed from `off`
static size_t place_tsplit(const gdn_shape_t& s, int P, bool backward, WsLayout& L, size_t off)
{
    const size_t vunits = (size_t)s.B * P * s.H;
    const size_t st = vunits * s.dk * s.dv * sizeof(float);
    const size_t esz = s.io == GDN_BF16 ? 2 : 4;
    L.ts_h_off = off;
    off = round_up(off + st, 256);
    L.ts_s_off = off;
    off = round_up(off + st, 256);
    if (s.mode == GDN_DELTA) {
        const size_t sq = vunits * s.dk * s.dk * sizeof(float);
        const size_t tk = (size_t)s.B * s.T * s.H * s.dk * esz;
        L.ts_a_off = off;
        off = round_up(off + sq, 256);
        L.ts_i_off = off;
        off = round_up(off + sq, 256);
        L.ts_zv_off = off;
        off = round_up(off + tk, 256);
        L.ts_so_off = off;
        off = round_up(off + (size_t)s.B * s.T * s.H * s.dk * sizeof(float), 256);
    }
    L.ts_o_off = off;
    off = round_up(off + (size_t)s.B * s.T * s.H * s.dv * sizeof(float), 256);
    if (backward) {
        L.ts_g_off = off;
        off = round_up(off + st, 256);
        L.ts_e_off = off;
        off = round_up(off + st, 256);
    }
    return off;
}

// buffers of the delta forward split in time by walks (see launch_fwd_walks), placed from `off`
static size_t place_fwd_walks(const gdn_shape_t& s, int P, WsLayout& L, size_t off)
{
    const size_t units = (size_t)s.B * s.H, nq = units * (size_t)((s.T + 63) / 64);
    L.ts_h_off = off;
    off = round_up(off + units * P * s.dk * s.dv * sizeof(float), 256);
    L.ts_o_off = off;
    off = round_up(off + (size_t)s.B * s.T * s.H * s.dv * sizeof(float), 256);
    L.fw_res_off = off;
    off = round_up(off + nq * (kSavedStateBytes + saved_solve_bytes(s.mode)), 256);
    L.cb_phi_off = off;
    off = round_up(off + nq * 32768, 256);   // [Phi_hi | Qc_hi | Phi_lo | Qc_lo]
    L.fw_d_off = off;
    off = round_up(off + nq * 16384, 256);
    L.cb_seg_off = off;
    off = round_up(off + units * P * 3 * 16384, 256);
    return off;
}

WsLayout ws_layout_bwd_core(const gdn_shape_t& s, int norm)
{
    WsLayout L;
    L.total = place_bwd_core(s, L, 256, norm);
    return L;
}

int bwd_split(const gdn_shape_t& s, int logits, int norm)
{
    if (s.T <= 0 || chunk_bwd_applies(s, logits, norm)) return 1;
    return tsplit_factor(s, 1);
}

// the chunked backward's per-chunk records, placed from `off`; with the residuals of a saving forward
// (`from_saved`) the entering states and the solve's results are the caller's, not the workspace's
static size_t place_chunk_bwd(const gdn_shape_t& s, WsLayout& L, size_t off, bool from_saved)
{
    const size_t nq = (size_t)s.B * s.H * (size_t)((s.T + 63) / 64);
    const size_t rec = nq * 64 * 64 * sizeof(float);
    if (s.mode == GDN_DELTA) {
        L.cb_phi_off = off;
        off = round_up(off + rec, 256);
        if (!from_saved) {
            L.cb_sv_off = off;
            off = round_up(off + nq * kSavedSolveBytes, 256);
        }
    }
    if (!from_saved) {
        L.cb_dlt_off = off;
        off = round_up(off + rec, 256);
    }
    L.cb_y_off = off;
    off = round_up(off + rec, 256);
    if (!from_saved) {
        L.cb_st_off = off;
        off = round_up(off + rec, 256);
    }
    L.cb_dst_off = off;
    off = round_up(off + rec, 256);
    L.cb_ec_off = off;
    off = round_up(off + nq * 64 * sizeof(float), 256);
    L.cb_da_off = off;
    off = round_up(off + nq * 64 * sizeof(float), 256);
    int seg_len = 0;
    const int dirs = from_saved ? 1 : 2;
    const int nseg = chain_segments(s.mode, (long)s.B * s.H, (s.T + 63) / 64, dirs, &seg_len);
    if (nseg > 1) {
        L.cb_seg_off = off;
        off = round_up(off + (size_t)dirs * s.B * s.H * nseg * 3 * 64 * 64 * sizeof(float), 256);
        if (s.mode == GDN_GATED) {
            L.cb_tvec_off = off;
            off = round_up(off + (size_t)dirs * nq * 64 * sizeof(float), 256);
        }
    }
    return off;
}

// The plain backward of the chunked backward's unsplit shapes runs the saving forward into its workspace and then
// the backward from those residuals when the heads fill most of their waves of one CTA per SM: per chunk the
// forward (one CTA per head, the front and the state chain together) takes about 12 us of its CTA, the chunk-parallel
// prep (the front, Phi, Delta and Y) about 18 us of an SM, and the prep route adds the chain's forward sweep.
static bool bwd_via_forward(const gdn_shape_t& s, int logits, int norm)
{
    if (s.T <= decode_max_tokens() || !chunk_bwd_applies(s, logits, norm)) return false;
    if (fwd_walk_split(s, logits, norm, nullptr) > 1 || tsplit_factor(s, 0) > 1) return false;
    const long units = (long)s.B * s.H, waves = (units + kSplitSMs - 1) / kSplitSMs;
    return 3 * units > 2 * waves * kSplitSMs;
}

WsLayout ws_layout(const gdn_shape_t& s, int backward, int norm, int logits)
{
    WsLayout L;
    size_t off = 256;  // status word
    if (backward && chunk_bwd_applies(s, logits, norm)) {
        if (backward == 1 && bwd_via_forward(s, logits, norm)) {
            // the saving forward's residuals and (unused) outputs, then the backward from the residuals
            const size_t nq = (size_t)s.B * s.H * (size_t)((s.T + 63) / 64);
            L.bf_res_off = off;
            off = round_up(off + nq * (kSavedStateBytes + saved_solve_bytes(s.mode)), 256);
            L.bf_o_off = off;
            off = round_up(off + (size_t)s.B * s.T * s.H * s.dv * 2, 256);
            L.total = place_chunk_bwd(s, L, off, true);
            return L;
        }
        L.total = place_chunk_bwd(s, L, off, backward == 2);
        return L;
    }
    const int walks = backward || s.T <= 0 ? 1 : fwd_walk_split(s, logits, norm, nullptr);
    const int P = s.T > 0 ? (backward ? bwd_split(s, logits, norm) : (walks > 1 ? walks : tsplit_factor(s, 0))) : 1;
    if (backward) {
        gdn_shape_t core = s;
        if (P > 1) {
            core.B = s.B * P;
            core.T = s.T / P;
        }
        off = place_bwd_core(core, L, off, norm);
    }
    if (walks > 1)
        off = place_fwd_walks(s, P, L, off);
    else if (P > 1)
        off = place_tsplit(s, P, backward != 0, L, off);
    L.total = off;
    return L;
}

static int cached_dev_ok[64];  // 0 unknown, 1 ok, 2 not sm_103

gdn_status_t check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return GDN_ERR_DEVICE;
    if (cached_dev_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return GDN_ERR_CUDA;
        cached_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return cached_dev_ok[dev] == 1 ? GDN_OK : GDN_ERR_DEVICE;
}

int test_starve_chunk()
{
    static const int k = [] {
        const char* e = getenv("GDN_TEST_STARVE_CHUNK");
        return e ? atoi(e) : -1;
    }();
    return k;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static gdn_status_t check_common(const gdn_shape_t* s, const void* v, const void* b, const void* c,
                                 const void* g, const void* beta, const float* A_log, const float* h0,
                                 void* ws, size_t ws_bytes, int backward, int norm, int logits)
{
    if (!s) return GDN_ERR_NULL;
    if (s->mode != GDN_GATED && s->mode != GDN_DELTA) return GDN_ERR_MODE;
    if (s->io != GDN_F32 && s->io != GDN_BF16) return GDN_ERR_MODE;
    if (!shape_ok(*s)) return GDN_ERR_SHAPE;
    // with T == 0 there are no tokens: the per-token pointers may be NULL
    const bool tok = s->T > 0;
    if ((tok && (!v || !b || !c || !g)) || !A_log) return GDN_ERR_NULL;
    if (!ws) return GDN_ERR_WORKSPACE;
    if (tok && (s->mode == GDN_DELTA) != (beta != nullptr)) return GDN_ERR_MODE;
    if (s->mode == GDN_GATED && beta) return GDN_ERR_MODE;
    const size_t ioa = s->io == GDN_BF16 ? 16 : 4;
    if (!aligned(v, ioa) || !aligned(b, ioa) || !aligned(c, ioa) || !aligned(g, s->io == GDN_BF16 ? 2 : 4) ||
        (beta && !aligned(beta, s->io == GDN_BF16 ? 2 : 4)))
        return GDN_ERR_ALIGN;
    if (!aligned(A_log, 16) || (h0 && !aligned(h0, 16)) || !aligned(ws, 256)) return GDN_ERR_ALIGN;
    if (ws_bytes < ws_layout(*s, backward, norm, logits).total) return GDN_ERR_WORKSPACE;
    return GDN_OK;
}

// Split the option bits off the mode: `out` gets the plain mode, `logits` the
// GDN_GATE_LOGITS bit, `norm` the GDN_NORM_BC bit, `check` (if not null) the
// GDN_CHECK_FINITE bit.  False if the mode carries an unknown bit.
static bool split_mode(const gdn_shape_t* in, gdn_shape_t* out, int* logits, int* norm, int* check = nullptr)
{
    *out = *in;
    *logits = (in->mode & GDN_GATE_LOGITS) != 0;
    *norm = (in->mode & GDN_NORM_BC) != 0;
    if (check) *check = (in->mode & GDN_CHECK_FINITE) != 0;
    out->mode = in->mode & ~(GDN_GATE_LOGITS | GDN_NORM_BC | GDN_CHECK_FINITE);
    return (out->mode & ~0xff) == 0;
}

static Args make_args(const gdn_shape_t* s)
{
    Args a;
    memset(&a, 0, sizeof(a));
    a.B = s->B; a.H = s->H; a.T = s->T; a.dk = s->dk; a.dv = s->dv; a.mode = s->mode; a.io = s->io;
    return a;
}

// One forward over the whole shape: few tokens -> decode kernel; bf16 ->
// tcgen05 chunked kernel; fp32 -> token-serial kernel.
// Delta heads at most 32 wide in more than two waves of the tensor-core forward (one CTA per SM) take the
// token-serial kernel, which keeps several CTAs on an SM: at 8 x 40 heads x 4096 tokens x 32 it finishes in
// 1.80 ms against 2.00 ms (gated heads, and 160 heads or fewer, are faster on the tensor cores).
static bool serial_first(const Args& a)
{
    return a.mode == GDN_DELTA && a.dk <= 32 && a.dv <= 32 && (long)a.B * a.H > 2 * kSplitSMs;
}

// the forward kernel for a (view) shape: fwd_core dispatches on it and gdn_plan reports it
static gdn_kernel_t fwd_kernel_of(const Args& a)
{
    if (a.T <= 0) return GDN_KERNEL_NONE;
    if (a.T <= decode_max_tokens()) return GDN_KERNEL_DECODE;
    if (a.io == GDN_BF16 && !serial_first(a) && a.dk <= 64) return GDN_KERNEL_TENSOR_CORE;
    return GDN_KERNEL_SERIAL;
}

// the one place that picks a forward kernel; gdn_plan reports the same choice
static cudaError_t fwd_core(const Args& a, cudaStream_t st)
{
    switch (fwd_kernel_of(a)) {
    case GDN_KERNEL_DECODE:
        return launch_decode(a, st);
    case GDN_KERNEL_TENSOR_CORE: {
        bool handled = false;
        const cudaError_t e = launch_fwd_tc(a, st, &handled);
        return (e != cudaSuccess || handled) ? e : cudaErrorInvalidValue;   // the kernel refused a shape it takes
    }
    default:
        return launch_serial_fwd(a, st);
    }
}

// Shapes whose forward can keep the chunked backward's residuals (gdn_fwd_save): the chunked backward's shapes whose
// forward is a split by walks, or unsplit and longer than the decode kernel's reach.  The saving forward always runs
// the tcgen05 kernel, also where gdn_fwd prefers the token-serial one (narrow delta heads over many units): the
// residuals spare the backward far more than that costs.
static bool saved_applies(const gdn_shape_t& s, int logits, int norm)
{
    if (!chunk_bwd_applies(s, logits, norm)) return false;
    if (fwd_walk_split(s, logits, norm, nullptr) > 1) return true;
    if (tsplit_factor(s, 0) > 1) return false;
    return s.T > decode_max_tokens();
}

static size_t saved_bytes_of(const gdn_shape_t& s)
{
    return (size_t)s.B * s.H * (size_t)((s.T + 63) / 64) * (kSavedStateBytes + saved_solve_bytes(s.mode));
}

}  // namespace gdn

using namespace gdn;

extern "C" gdn_status_t gdn_plan(const gdn_shape_t* shape_in, int backward, gdn_plan_t* plan)
{
    gdn_shape_t sh;
    int logits = 0, norm = 0;
    if (!shape_in || !plan) return GDN_ERR_NULL;
    if (!split_mode(shape_in, &sh, &logits, &norm)) return GDN_ERR_MODE;
    if ((sh.mode != GDN_GATED && sh.mode != GDN_DELTA) || (sh.io != GDN_F32 && sh.io != GDN_BF16))
        return GDN_ERR_MODE;
    if (!shape_ok(sh)) return GDN_ERR_SHAPE;
    const int walks = backward || sh.T <= 0 ? 1 : fwd_walk_split(sh, logits, norm, nullptr);
    const int P = sh.T > 0 ? (backward ? bwd_split(sh, logits, norm) : (walks > 1 ? walks : tsplit_factor(sh, 0))) : 1;
    Args a = make_args(&sh);   // the runs' view: P segments of one sequence are P batch rows
    a.B = sh.B * P;
    a.T = sh.T / P;
    plan->segments = P;
    plan->fwd_kernel = (backward && P == 1) ? GDN_KERNEL_NONE
                       : walks > 1 ? GDN_KERNEL_TENSOR_CORE   // the split by walks runs the tcgen05 forward
                                   : fwd_kernel_of(a);
    plan->bwd_kernel = !backward || sh.T <= 0 ? GDN_BWD_NONE
                       : chunk_bwd_applies(sh, logits, norm) ? GDN_BWD_TENSOR_CORE : GDN_BWD_SERIAL;
    if (plan->bwd_kernel == GDN_BWD_TENSOR_CORE)   // the chunked backward's chain, split in time for few heads
        plan->segments = chain_segments(sh.mode, (long)sh.B * sh.H, (sh.T + 63) / 64, backward == 2 ? 1 : 2,
                                        nullptr);
    return GDN_OK;
}

extern "C" size_t gdn_workspace_bytes(const gdn_shape_t* shape_in, int backward)
{
    gdn_shape_t sh;
    int logits = 0, norm = 0;
    if (!shape_in || !split_mode(shape_in, &sh, &logits, &norm)) return 0;
    const gdn_shape_t* shape = &sh;
    if (!shape_ok(*shape)) return 0;
    if ((shape->mode != GDN_GATED && shape->mode != GDN_DELTA) || (shape->io != GDN_F32 && shape->io != GDN_BF16))
        return 0;
    if (backward == 2 && !saved_applies(sh, logits, norm)) return 0;
    return ws_layout(*shape, backward == 2 ? 2 : (backward ? 1 : 0), norm, logits).total;
}

extern "C" size_t gdn_saved_bytes(const gdn_shape_t* shape_in)
{
    gdn_shape_t sh;
    int logits = 0, norm = 0;
    if (!shape_in || !split_mode(shape_in, &sh, &logits, &norm)) return 0;
    if (!shape_ok(sh) || sh.io != GDN_BF16 || !saved_applies(sh, logits, norm)) return 0;
    return saved_bytes_of(sh);
}

static gdn_status_t fwd_impl(const gdn_shape_t* shape_in, const void* v, const void* b, const void* c,
                             const void* g, const void* beta, const float* A_log, const float* h0, void* o,
                             float* hT, void* saved, size_t saved_bytes, bool saving, void* ws, size_t ws_bytes,
                             gdn_stream_t stream)
{
    gdn_shape_t sh;
    int logits = 0, norm = 0, check = 0;
    if (!shape_in) return GDN_ERR_NULL;
    if (!split_mode(shape_in, &sh, &logits, &norm, &check)) return GDN_ERR_MODE;
    const gdn_shape_t* shape = &sh;
    gdn_status_t r = check_common(shape, v, b, c, g, beta, A_log, h0, ws, ws_bytes, 0, norm, logits);
    if (r != GDN_OK) return r;
    if (!o && shape->T > 0) return GDN_ERR_NULL;
    const size_t ioa = shape->io == GDN_BF16 ? 16 : 4;
    if (!aligned(o, ioa) || (hT && !aligned(hT, 16))) return GDN_ERR_ALIGN;
    if (saving) {
        if (!saved) return GDN_ERR_NULL;
        if (!saved_applies(sh, logits, norm)) return GDN_ERR_MODE;
        if (!aligned(saved, 256)) return GDN_ERR_ALIGN;
        if (saved_bytes < saved_bytes_of(sh)) return GDN_ERR_WORKSPACE;
    }
    if ((r = check_device()) != GDN_OK) return r;

    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return GDN_ERR_CUDA;
    Args a = make_args(shape);
    a.v = v; a.b = b; a.c = c; a.g = g; a.beta = beta; a.A_log = A_log; a.h0 = h0; a.o = o; a.hT = hT;
    a.ws = ws; a.ws_bytes = ws_bytes; a.logits = logits; a.norm = norm;
    a.saved = saving ? saved : nullptr;
    const size_t state_bytes = (size_t)a.B * a.H * a.dk * a.dv * sizeof(float);
    if (a.T == 0) {
        if (hT && hT != h0) {
            cudaError_t e = h0 ? cudaMemcpyAsync(hT, h0, state_bytes, cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(hT, 0, state_bytes, st);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    const int P = tsplit_factor(*shape, 0);
    cudaError_t e;
    if (fwd_walk_split(*shape, logits, norm, nullptr) > 1) {
        e = launch_fwd_walks(a, ws_layout(*shape, 0, norm, logits), st);
    } else if (P > 1) {
        e = launch_fwd_tsplit(a, ws_layout(*shape, 0, norm, logits), P, st, fwd_core);
    } else if (saving) {
        bool handled = false;   // the tcgen05 kernel keeps the residuals (saved_applies)
        e = launch_fwd_tc(a, st, &handled);
        if (e == cudaSuccess && !handled) e = cudaErrorInvalidValue;
    } else {
        e = fwd_core(a, st);
    }
    if (e == cudaSuccess && check) {
        e = launch_check_finite(o, (size_t)a.B * a.T * a.H * a.dv, a.io, ws, st);
        if (e == cudaSuccess && hT) e = launch_check_finite(hT, state_bytes / sizeof(float), GDN_F32, ws, st);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status_t gdn_fwd(const gdn_shape_t* shape, const void* v, const void* b, const void* c,
                                const void* g, const void* beta, const float* A_log, const float* h0,
                                void* o, float* hT, void* ws, size_t ws_bytes, gdn_stream_t stream)
{
    return fwd_impl(shape, v, b, c, g, beta, A_log, h0, o, hT, nullptr, 0, false, ws, ws_bytes, stream);
}

extern "C" gdn_status_t gdn_fwd_save(const gdn_shape_t* shape, const void* v, const void* b, const void* c,
                                     const void* g, const void* beta, const float* A_log, const float* h0,
                                     void* o, float* hT, void* saved, size_t saved_bytes, void* ws,
                                     size_t ws_bytes, gdn_stream_t stream)
{
    return fwd_impl(shape, v, b, c, g, beta, A_log, h0, o, hT, saved, saved_bytes, true, ws, ws_bytes, stream);
}

static gdn_status_t bwd_impl(const gdn_shape_t* shape_in, const void* v, const void* b, const void* c,
                             const void* g, const void* beta, const float* A_log, const float* h0,
                             const void* saved, size_t saved_bytes, bool from_saved, const void* dO,
                             const float* dhT, void* dv, void* db, void* dc, void* dg, void* dbeta, float* dA_log,
                             float* dh0, void* ws, size_t ws_bytes, gdn_stream_t stream)
{
    gdn_shape_t sh;
    int logits = 0, norm = 0, check = 0;
    if (!shape_in) return GDN_ERR_NULL;
    if (!split_mode(shape_in, &sh, &logits, &norm, &check)) return GDN_ERR_MODE;
    const gdn_shape_t* shape = &sh;
    if (from_saved) {
        if (!saved) return GDN_ERR_NULL;
        if (!shape_ok(sh)) return GDN_ERR_SHAPE;
        if (!saved_applies(sh, logits, norm)) return GDN_ERR_MODE;
        if (!aligned(saved, 256)) return GDN_ERR_ALIGN;
        if (saved_bytes < saved_bytes_of(sh)) return GDN_ERR_WORKSPACE;
    }
    gdn_status_t r = check_common(shape, v, b, c, g, beta, A_log, h0, ws, ws_bytes, from_saved ? 2 : 1, norm,
                                  logits);
    if (r != GDN_OK) return r;
    const bool tok = shape->T > 0;
    if ((tok && (!dO || !dv || !db || !dc || !dg)) || !dA_log) return GDN_ERR_NULL;
    if (tok && (shape->mode == GDN_DELTA) != (dbeta != nullptr)) return GDN_ERR_MODE;
    if (shape->mode == GDN_GATED && dbeta) return GDN_ERR_MODE;
    const size_t ioa = shape->io == GDN_BF16 ? 16 : 4;
    const size_t sca = shape->io == GDN_BF16 ? 2 : 4;
    if (!aligned(dO, ioa) || !aligned(dv, ioa) || !aligned(db, ioa) || !aligned(dc, ioa) || !aligned(dg, sca) ||
        (dbeta && !aligned(dbeta, sca)) || !aligned(dA_log, 16) || (dhT && !aligned(dhT, 16)) ||
        (dh0 && !aligned(dh0, 16)))
        return GDN_ERR_ALIGN;
    if ((r = check_device()) != GDN_OK) return r;

    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return GDN_ERR_CUDA;
    Args a = make_args(shape);
    a.v = v; a.b = b; a.c = c; a.g = g; a.beta = beta; a.A_log = A_log; a.h0 = h0;
    a.dO = dO; a.dhT = dhT; a.dv_ = dv; a.db = db; a.dc = dc; a.dg = dg; a.dbeta = dbeta;
    a.dA_log = dA_log; a.dh0 = dh0; a.ws = ws; a.ws_bytes = ws_bytes; a.logits = logits; a.norm = norm;
    a.saved = from_saved ? const_cast<void*>(saved) : nullptr;
    cudaError_t e;
    if (a.T > 0 && chunk_bwd_applies(*shape, logits, norm) && !from_saved && bwd_via_forward(*shape, logits, norm)) {
        // the saving forward recomputes the residuals (outputs to the workspace), then the backward from them
        const WsLayout L = ws_layout(*shape, 1, norm, logits);
        Args f = a;
        f.o = (unsigned char*)ws + L.bf_o_off;
        f.hT = nullptr;
        f.saved = (unsigned char*)ws + L.bf_res_off;
        bool handled = false;
        e = launch_fwd_tc(f, st, &handled);
        if (e == cudaSuccess && !handled) e = cudaErrorInvalidValue;
        if (e == cudaSuccess) {
            a.saved = f.saved;
            e = launch_chunk_bwd(a, L, st);
        }
    } else if (a.T > 0 && chunk_bwd_applies(*shape, logits, norm)) {
        e = launch_chunk_bwd(a, ws_layout(*shape, from_saved ? 2 : 1, norm, logits), st);
    } else {
        const int P = bwd_split(*shape, logits, norm);
        e = P > 1 ? launch_bwd_tsplit(a, ws_layout(*shape, 1, norm, logits), P, st, fwd_core)
                  : launch_serial_bwd(a, st);
    }
    if (e == cudaSuccess && check) {
        const size_t ntok = (size_t)a.B * a.T * a.H, st_n = (size_t)a.B * a.H * a.dk * a.dv;
        const struct { const void* p; size_t n; int io; } outs[] = {
            {dv, ntok * a.dv, a.io}, {db, ntok * a.dk, a.io}, {dc, ntok * a.dk, a.io}, {dg, ntok, a.io},
            {dbeta, ntok, a.io}, {dA_log, (size_t)a.H * a.dk, GDN_F32}, {dh0, st_n, GDN_F32}};
        for (const auto& x : outs)
            if (e == cudaSuccess && x.p && x.n) e = launch_check_finite(x.p, x.n, x.io, ws, st);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status_t gdn_bwd(const gdn_shape_t* shape, const void* v, const void* b, const void* c,
                                const void* g, const void* beta, const float* A_log, const float* h0,
                                const void* dO, const float* dhT, void* dv, void* db, void* dc, void* dg,
                                void* dbeta, float* dA_log, float* dh0, void* ws, size_t ws_bytes,
                                gdn_stream_t stream)
{
    return bwd_impl(shape, v, b, c, g, beta, A_log, h0, nullptr, 0, false, dO, dhT, dv, db, dc, dg, dbeta, dA_log,
                    dh0, ws, ws_bytes, stream);
}

extern "C" gdn_status_t gdn_bwd_saved(const gdn_shape_t* shape, const void* v, const void* b, const void* c,
                                      const void* g, const void* beta, const float* A_log, const void* saved,
                                      size_t saved_bytes, const void* dO, const float* dhT, void* dv, void* db,
                                      void* dc, void* dg, void* dbeta, float* dA_log, float* dh0, void* ws,
                                      size_t ws_bytes, gdn_stream_t stream)
{
    return bwd_impl(shape, v, b, c, g, beta, A_log, nullptr, saved, saved_bytes, true, dO, dhT, dv, db, dc, dg,
                    dbeta, dA_log, dh0, ws, ws_bytes, stream);
}

extern "C" gdn_status_t gdn_last_device_status(const void* ws, gdn_stream_t stream)
{
    if (!ws) return GDN_ERR_NULL;
    uint32_t word[2] = {0, 0};
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemcpy(word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    if (word[0] != kDevOk) return GDN_ERR_TIMEOUT;
    return word[1] != 0 ? GDN_ERR_NONFINITE : GDN_OK;
}

extern "C" const char* gdn_status_string(gdn_status_t s)
{
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_NULL: return "GDN_ERR_NULL: a required pointer is NULL";
        case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE: a size is out of range";
        case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: a pointer is misaligned";
        case GDN_ERR_MODE: return "GDN_ERR_MODE: bad mode/dtype or beta presence";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA call failed";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait expired";
        case GDN_ERR_DEVICE: return "GDN_ERR_DEVICE: the current device is not sm_103";
        case GDN_ERR_NONFINITE: return "GDN_ERR_NONFINITE: an output holds NaN or Inf";
    }
    return "unknown gdn status";
}
