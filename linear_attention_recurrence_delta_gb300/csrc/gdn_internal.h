// gdn_internal.h -- shared host-side declarations of libgdn (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

// Everything one gdn_fwd / gdn_bwd call needs, already validated.
struct Args {
    int B, H, T, dk, dv, mode, io;
    int logits;            // g, beta arrive before their sigmoid (GDN_GATE_LOGITS)
    int norm;              // b, c arrive before their L2 normalisation (GDN_NORM_BC)
    const void *v, *b, *c, *g, *beta;
    const float* A_log;
    const float* h0;
    void* o;
    float* o32;            // forward, bf16 I/O: write o in fp32 here instead of `o` (intermediate runs of the
                           // time split; the tcgen05 kernel honours it, the other bf16 paths are never asked)
    float* hT;
    // backward only
    const void* dO;
    const float* dhT;
    void *dv_, *db, *dc, *dg, *dbeta;
    float* dA_log;
    float* dh0;
    // residuals of the chunked backward (delta): a saving forward writes them, the backward reads them
    void* saved;
    int seg, seg_len;      // a saving run over a time split: segments per sequence (else 0 or 1), chunks each
    int save_lite;         // a saving run for the time split's walks alone: P and -W only
    // workspace
    void* ws;
    size_t ws_bytes;
};

// Workspace carve-up.  The first 256 bytes always hold the device status word.
struct WsLayout {
    size_t status_off = 0;        // uint32 status code, uint32 detail
    size_t snap_off = 0;          // serial backward: state entering every kSerialSnap tokens
    size_t xvr_off = 0;           // serial backward, delta: x and v - h'^T b of every token
    size_t dalog_off = 0;         // per-(b,h) dA_log partials, float [B*H, slabs, d_k]
    size_t slab_off = 0;          // serial backward over several column slabs: fp32 partial sums
                                  // db, dc [slabs][B,T,H,d_k]; dg, dbeta [slabs][B,T,H]
    // forward split in time (long sequences over few heads), see gdn_tsplit.cu
    size_t ts_h_off = 0;          // leaving states from a zero start   [B*P, H, d_k, d_v]
    size_t ts_s_off = 0;          // entering states of the segments    [B*P, H, d_k, d_v]
    size_t ts_a_off = 0;          // delta: segment transitions          [B*P, H, d_k, d_k]
    size_t ts_i_off = 0;          // delta: identity starting states     [B*P, H, d_k, d_k]
    size_t ts_zv_off = 0;         // delta: zero values                  [B, T, H, d_k] (I/O dtype)
    size_t ts_so_off = 0;         // delta: outputs of the transition run [B, T, H, d_k] fp32
    // backward split in time
    size_t ts_o_off = 0;          // outputs of the zero-start runs      [B, T, H, d_v] fp32
    size_t ts_g_off = 0;          // segment adjoints from a zero end gradient [B*P, H, d_k, d_v]
    size_t ts_e_off = 0;          // end gradients of the segments       [B*P, H, d_k, d_v]
    // chunked backward (gdn_chunk_bwd.cu): per chunk of 64 tokens, [B*H*chunks][64][64] fp32 records
    size_t cb_phi_off = 0;        // delta: the chunk's state transition Phi
    size_t cb_sv_off = 0;         // delta: the front's results saved for the gradient pass (64 KB per chunk)
    size_t cb_dlt_off = 0;        // the state the chunk leaves from a zero start
    size_t cb_y_off = 0;          // the chunk's share of the entering state's adjoint
    size_t cb_st_off = 0;         // the state entering the chunk
    size_t cb_dst_off = 0;        // the adjoint of the state leaving the chunk
    size_t cb_ec_off = 0;         // gated: the chunk's decay [B*H*chunks][64]
    size_t cb_da_off = 0;         // per-chunk dA partials [B*H*chunks][64]
    size_t cb_seg_off = 0;        // chain split in time: per (direction, unit, segment) three 64 x 64 fp32 records
    size_t cb_tvec_off = 0;       // gated chain split in time: per (direction, chunk) 64 decay products
    // forward split in time by walks (delta, bf16): also ts_h_off (the zero-start run's final states), ts_o_off
    // (its fp32 outputs), cb_phi_off (Phi per chunk) and cb_seg_off (per segment X, Pi, true start)
    size_t fw_res_off = 0;        // the residuals when the caller keeps none (states, then the solve's results)
    size_t fw_d_off = 0;          // D = T_k S_s per chunk, fp32 [B*H*chunks][64][64]
    // chunked backward through the saving forward (bwd_via_forward in gdn_api.cu)
    size_t bf_res_off = 0;        // the residuals (states, then the solve's results)
    size_t bf_o_off = 0;          // the forward's outputs, bf16 [B, T, H, d_v] (not used)
    size_t total = 0;
};

constexpr long kSplitSMs = 152;                // a forward is split in time only while B*H*P <= this (also
                                               // the wave size of the one-CTA-per-SM tensor-core forward)
constexpr int kSplitMinTokens = 512;           // and every segment keeps at least this many tokens
constexpr int kSerialBlock = 32;               // tokens per backward block
constexpr int kSerialSnap = 8;                 // tokens between backward state snapshots
constexpr size_t kStateSlot = 16 * 256 * 4;    // one state snapshot (256 threads x 16 floats)

// The serial backward covers d_k <= 64 with 64 value columns per CTA and
// d_k <= 128 with 32; wider values take several column slabs.
inline int bwd_cols(int dk) { return dk <= 64 ? 64 : 32; }
inline int bwd_slabs(int dk, int dv) { return (dv + bwd_cols(dk) - 1) / bwd_cols(dk); }

// `norm`: GDN_NORM_BC is set (the backward then routes db, dc through fp32 partials); `logits`: GDN_GATE_LOGITS.
// backward: 0 forward, 1 backward, 2 backward from a saving forward's residuals (no state or solve records)
WsLayout ws_layout(const gdn_shape_t& s, int backward, int norm = 0, int logits = 0);

// The chunked tensor-core backward takes bf16 heads up to 64 wide without the option bits; other backward
// calls take the token-serial one (with its time split for long sequences over few heads).
// Residuals a saving forward keeps for it, per chunk of 64 tokens: the entering state (fp32 64 x 64) and the
// delta solve's results (layout in gdn_chunk_bwd.cu, namespace sv), or in gated mode the scores P.
constexpr size_t kSavedStateBytes = 16384, kSavedSolveBytes = 81920, kSavedGatedBytes = 16384;
inline size_t saved_solve_bytes(int mode) { return mode == GDN_DELTA ? kSavedSolveBytes : kSavedGatedBytes; }
inline bool chunk_bwd_applies(const gdn_shape_t& s, int logits, int norm)
{
    return s.io == GDN_BF16 && s.T > 0 && s.dk <= 64 && s.dv <= 64 && !logits && !norm;
}
// The forward split in time by walks (launch_fwd_walks): bf16, heads up to 64 wide, no option bits, at most 76
// (batch, head) units.  P segments of *seg_len chunks of 64 tokens (the last one may be shorter, its last chunk
// ragged) for any length: B * H * P <= 152, at least 8 chunks each, P >= 2.  Returns P (1: no split by walks).
inline int fwd_walk_split(const gdn_shape_t& s, int logits, int norm, int* seg_len)
{
    if (!chunk_bwd_applies(s, logits, norm)) return 1;
    const long units = (long)s.B * s.H, nk = (s.T + 63) / 64;
    long P = kSplitSMs / units;
    if (P > nk / 8) P = nk / 8;
    if (P < 2) return 1;
    const long L = (nk + P - 1) / P;
    if (seg_len) *seg_len = (int)L;
    return (int)((nk + L - 1) / L);
}
// The chunked backward's chain split in time: its `dirs` sweeps (2, or 1 from the forward's residuals) over `units`
// (batch, head) units run as dirs * units * nseg walks side by side (at most 152), each over a segment of *seg_len
// chunks (at least 16).  Splits when that gives at least 2 segments of a sequence of at least 32 chunks.  Returns
// nseg (1 = no split).
inline int chain_segments(int mode, long units, int nchunks, int dirs, int* seg_len)
{
    int P = 1;
    (void)mode;
    if (units > 0 && nchunks >= 32) {
        const long fit = kSplitSMs / (dirs * units);
        P = fit < nchunks / 16 ? (int)fit : nchunks / 16;
        if (P < 2) P = 1;
    }
    const int L = (nchunks + P - 1) / P;
    if (seg_len) *seg_len = L;
    return L > 0 ? (nchunks + L - 1) / L : 1;
}

// segments of the backward's time split (1 = none; never with the chunked backward)
int bwd_split(const gdn_shape_t& s, int logits, int norm);
WsLayout ws_layout_bwd_core(const gdn_shape_t& s, int norm = 0);   // the serial backward's own buffers only

// the serial backward writes fp32 partial sums of db, dc, dg, dbeta (rather than its outputs) when
// it has several column slabs or must still apply the normalisation's Jacobian
inline bool bwd_partials(int dk, int dv, int norm) { return bwd_slabs(dk, dv) > 1 || norm; }

// Launchers (enqueue on `st`, return cudaGetLastError()).
cudaError_t launch_serial_fwd(const Args& a, cudaStream_t st);
cudaError_t launch_serial_bwd(const Args& a, cudaStream_t st);
cudaError_t launch_fwd_tc(const Args& a, cudaStream_t st, bool* handled);
cudaError_t launch_decode(const Args& a, cudaStream_t st);   // 1 <= T <= decode_max_tokens()
cudaError_t launch_chunk_bwd(const Args& a, const WsLayout& L, cudaStream_t st);   // chunk_bwd_applies()
cudaError_t launch_fwd_walks(const Args& a, const WsLayout& L, cudaStream_t st);   // fwd_walk_split() > 1
int tsplit_factor(const gdn_shape_t& s, int backward);   // segments P of a time split, 1 = no split
cudaError_t launch_fwd_tsplit(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                              cudaError_t (*fwd_core)(const Args&, cudaStream_t));
cudaError_t launch_bwd_tsplit(const Args& a, const WsLayout& L, int P, cudaStream_t st,
                              cudaError_t (*fwd_core)(const Args&, cudaStream_t));
int decode_max_tokens();

// Failure-path test hook, for the library's own tests only: the value of the environment variable
// GDN_TEST_STARVE_CHUNK, read once per process (-1 when it is not set).  With it set to k, the tensor-core
// forward never issues the loads of chunk k, so that chunk's bounded wait expires, the kernel winds down and the
// status word reads GDN_ERR_TIMEOUT.  Set it before the process's first forward call.
int test_starve_chunk();

// GDN_OK if the current device is an sm_103 GPU, GDN_ERR_DEVICE if not, GDN_ERR_CUDA if it cannot be queried
gdn_status_t check_device();

constexpr float kNormFloor = 1e-12f;   // L2 normalisation: x / max(||x||, kNormFloor)

// Device status word helpers.
// word 0: a bounded wait expired; word 1: GDN_CHECK_FINITE found NaN or Inf in an output
enum : uint32_t { kDevOk = 0, kDevTimeout = 1 };

// GDN_CHECK_FINITE: flag word 1 of the status block if any of the n elements is NaN or Inf
// (io: GDN_BF16 or GDN_F32 element type)
cudaError_t launch_check_finite(const void* p, size_t n, int io, void* ws, cudaStream_t st);

}  // namespace gdn
