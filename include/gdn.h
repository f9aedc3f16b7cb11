/*
 * gdn.h -- C ABI of libgdn, the GB300 (sm_103a) gated delta rule library.
 *
 * The operation (per batch index b and head h, one independent recurrence
 * over t = 0 .. T-1 on a state h of shape [d_k, d_v], rows indexed by the
 * key/state index i):
 *
 *   "GDN & MLA Mechanism Deep-Dive", Step 4 (Gated delta rule):
 *     alpha_t[i] = exp(g_t * A[i]),  A[i] = -exp(A_log[h, i])
 *     GDN_GATED:  h_t = alpha_t (.)rows h_{t-1} + b_t v_t^T
 *   "HyMo-434M -- documentation portal", card 01 (GDN recurrence, delta rule):
 *     GDN_DELTA:  h_t = alpha_t (.)rows h_{t-1}
 *                       + beta_t b_t (v_t - (alpha_t (.)rows h_{t-1})^T b_t)^T
 *   both modes:  o_t = h_t^T c_t       (the read sees token t's own write)
 *
 * "GDN & MLA Mechanism Deep-Dive", Step 5 (Chunked recurrence) is how the
 * kernels evaluate it: chunks of 64 tokens solved in closed form, with the
 * state carried serially from chunk to chunk.
 *
 * Inputs arrive already transformed: g and beta after their sigmoid (values
 * in [0, 1]), and in delta mode b already L2-normalised by the caller --
 * unless the option bits below ask the kernels to apply those steps.  The
 * library applies no 1/sqrt(d) scale, no output norm and no state clamp
 * ("Signed-state caveat": HyMo does not bound the state norm).
 *
 * Layouts (all contiguous, row-major, element strides implied by the shape):
 *   v, o, dO, dv              [B, T, H, d_v]   dtype `io`
 *   b, c, db, dc              [B, T, H, d_k]   dtype `io`
 *   g, beta, dg, dbeta        [B, T, H]        dtype `io`
 *   A_log, dA_log             [H, d_k]         float32
 *   h0, hT, dhT, dh0          [B, H, d_k, d_v] float32
 *
 * Ownership: the caller allocates and owns every buffer, including the
 * workspace; the library allocates no memory, never synchronises inside
 * gdn_fwd / gdn_bwd, and enqueues all work on the caller's stream.  All data
 * pointers are device pointers.
 *
 * Errors: argument problems are reported synchronously, before anything is
 * enqueued.  A failed launch returns GDN_ERR_CUDA.  Conditions the kernels
 * detect on the device (an expired bounded wait) are written to a status
 * word at the start of the workspace, which gdn_last_device_status reads.
 *
 * Test hook: the library's own failure-path tests set the environment
 * variable GDN_TEST_STARVE_CHUNK=k before a process's first call; the
 * tensor-core forward then never loads chunk k, its bounded wait expires and
 * the device status reads GDN_ERR_TIMEOUT.  It is read once per process and
 * must not be set in production.
 *
 * Limits: B, H >= 1 and B * H <= 2^26; T >= 0 (with T = 0 the per-token pointers may be NULL:
 * the forward copies h0, or zeros, to hT; the backward writes dh0 = dhT and
 * dA_log = 0); 1 <= d_k, d_v <= 128 (the tensor-core forward takes
 * d_k <= 64, wider keys the token-serial kernels).  With io = GDN_BF16, d_k
 * and d_v must be multiples of 8 and every bf16 pointer 16-byte aligned;
 * with io = GDN_F32, every pointer 4-byte aligned.  float32 state and A_log
 * pointers must be 16-byte aligned.  Outputs must not alias inputs.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                      /* same type as cudaStream_t's target */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
    GDN_GATED = 0,   /* h_t = alpha_t h_{t-1} + b_t v_t^T            */
    GDN_DELTA = 1    /* decay, then erase-and-write with key b_t     */
} gdn_mode_t;

/* Option bits OR'ed into gdn_shape_t.mode. */
enum {
    /* g (and, in delta mode, beta) arrive as logits, before their sigmoid
     * ("GDN & MLA Mechanism Deep-Dive", Gated delta rule: g_t is the sigmoid
     * of a projection; beta follows the same convention here).  The kernels
     * apply sigmoid() as they load them, and gdn_bwd returns dg and dbeta
     * with respect to the logits.  Without the bit both arrive already in
     * [0, 1] and the gradients are with respect to those values. */
    GDN_GATE_LOGITS = 0x100,
    /* b and c arrive before their L2 normalisation: every kernel divides
     * b_t and c_t by their Euclidean norm over d_k (floored at 1e-12, so an
     * all-zero vector stays zero) before the rule uses them, and gdn_bwd
     * returns db and dc with respect to the vectors as given.  The pages do
     * not spell out this step; it is the plain L2 normalisation of a key and
     * a read vector, fused so that no separate pass over b and c is needed.
     * Without the bit b and c are used as given. */
    GDN_NORM_BC = 0x200,
    /* After the kernels, scan every output (forward: o and hT; backward:
     * every gradient) for NaN and Inf; gdn_last_device_status then reports
     * GDN_ERR_NONFINITE if one was found.  A diagnostic for training runs:
     * it costs one read of the outputs and changes no result. */
    GDN_CHECK_FINITE = 0x400
};

typedef enum {
    GDN_F32 = 0,     /* float32 I/O (computed in fp32 on CUDA cores) */
    GDN_BF16 = 1     /* bfloat16 I/O, fp32 accumulation              */
} gdn_dtype_t;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_NULL = 1,        /* a required pointer is NULL                  */
    GDN_ERR_SHAPE = 2,       /* a size is out of range                      */
    GDN_ERR_ALIGN = 3,       /* a pointer is not aligned as required        */
    GDN_ERR_MODE = 4,        /* unknown mode/dtype, or beta given/missing   */
    GDN_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than required     */
    GDN_ERR_CUDA = 6,        /* a CUDA call or kernel launch failed         */
    GDN_ERR_TIMEOUT = 7,     /* a bounded device-side wait expired          */
    GDN_ERR_DEVICE = 8,      /* the current device is not an sm_103 GPU     */
    GDN_ERR_NONFINITE = 9    /* an output holds NaN or Inf (checked only
                                with GDN_CHECK_FINITE)                      */
} gdn_status_t;

typedef struct {
    int B, H, T;     /* batch, heads, tokens                               */
    int dk, dv;      /* key (state-row) and value (state-column) widths    */
    int mode;        /* gdn_mode_t                                         */
    int io;          /* gdn_dtype_t of v, b, c, g, beta, o and the grads   */
} gdn_shape_t;

/* Bytes of workspace gdn_fwd (backward = 0), gdn_bwd (backward = 1) or
 * gdn_bwd_saved (backward = 2) needs for this shape; 0 if the shape is invalid
 * (for backward = 2: if gdn_saved_bytes(shape) is 0).  Always a multiple of
 * 256 and at least 256 (the device status word lives in the first bytes). */
size_t gdn_workspace_bytes(const gdn_shape_t* shape, int backward);

/* How the library runs a shape.  Host only: it touches no device and is
 * answered from the shape alone, by the rules the calls themselves follow.
 *   segments    gdn_fwd (backward = 0), gdn_bwd (backward = 1) or
 *               gdn_bwd_saved (backward = 2) cuts the sequence into this many
 *               segments that run side by side (the state a segment passes on
 *               is an affine map of the state it receives, "GDN & MLA
 *               Mechanism Deep-Dive", Step 5: chunked recurrence; a scan over
 *               the segments joins them); 1 = no split.  Long sequences over
 *               few heads are split: the delta bf16 forward (heads up to 64
 *               wide, no option bits) into segments of whole chunks of 64
 *               tokens for any T (the last segment may be shorter), other
 *               forwards into equal segments (T divisible by them).  With the
 *               chunked backward only its
 *               chain over the chunk boundaries is (both modes): its sweeps
 *               (two, or the reverse one alone from the forward's residuals)
 *               times heads x batch rows times segments stay within 152
 *               walks, each segment at least 16 chunks of 64 tokens (the last
 *               one may be shorter).
 *   fwd_kernel  the kernel of the forward runs the call makes (gdn_kernel_t):
 *               gdn_fwd's own runs; gdn_bwd's forward runs over the segments
 *               under a split, GDN_KERNEL_NONE otherwise (both backward
 *               kernels recompute the forward themselves).  NONE for T = 0.
 *   bwd_kernel  (backward = 1 or 2) the backward kernel (gdn_bwd_kernel_t):
 *               GDN_BWD_TENSOR_CORE, the chunked reverse recurrence on tcgen05
 *               (bf16, d_k and d_v <= 64, no option bits: three passes over
 *               the chunks, a chain over the chunk boundaries between them);
 *               GDN_BWD_SERIAL, the token-serial reverse walk (every other
 *               shape); GDN_BWD_NONE for backward = 0 or T = 0.
 * Returns GDN_OK, or the error the call would return for the shape alone
 * (GDN_ERR_NULL, GDN_ERR_MODE, GDN_ERR_SHAPE). */
typedef enum {
    GDN_KERNEL_NONE = 0,
    GDN_KERNEL_DECODE = 1,        /* T <= 8: state-streaming decode kernel      */
    GDN_KERNEL_TENSOR_CORE = 2,   /* chunked tcgen05 forward (bf16, d_k <= 64)  */
    GDN_KERNEL_SERIAL = 3         /* token-serial forward on the CUDA cores     */
} gdn_kernel_t;

typedef enum {
    GDN_BWD_NONE = 0,
    GDN_BWD_SERIAL = 1,           /* token-serial reverse walk (CUDA cores)     */
    GDN_BWD_TENSOR_CORE = 2       /* chunked reverse recurrence on tcgen05      */
} gdn_bwd_kernel_t;

typedef struct {
    int segments;
    int fwd_kernel;   /* gdn_kernel_t */
    int bwd_kernel;   /* gdn_bwd_kernel_t */
} gdn_plan_t;

gdn_status_t gdn_plan(const gdn_shape_t* shape, int backward, gdn_plan_t* plan);

/* Forward pass.  Reads v, b, c, g, beta (NULL iff mode == GDN_GATED), A_log,
 * h0 (NULL => zero initial state); writes o and hT (NULL => not written).
 * hT may be the same buffer as h0: the state is then updated in place, as in
 * token-by-token decoding ("GDN & MLA Mechanism Deep-Dive", Step 4: the
 * state is all a head carries from one token to the next).  Sequences of at
 * most 8 tokens take a kernel laid out for that case.
 * ws must be device memory of at least gdn_workspace_bytes(shape, 0) bytes,
 * 256-byte aligned.  Returns GDN_OK once the work is enqueued on `stream`. */
gdn_status_t gdn_fwd(const gdn_shape_t* shape,
                     const void* v, const void* b, const void* c,
                     const void* g, const void* beta, const float* A_log,
                     const float* h0, void* o, float* hT,
                     void* ws, size_t ws_bytes, gdn_stream_t stream);

/* Backward pass: gradients of L(o, h_T) given dL/do = dO and dL/dh_T = dhT
 * (NULL => zero).  Takes the forward's inputs again (the forward is
 * recomputed inside; nothing from gdn_fwd is kept).  gdn_plan tells which
 * backward kernel a shape takes; both give the same gradients within the
 * tolerance of the I/O dtype, and each is deterministic (fixed-order sums).  Writes dv, db, dc, dg,
 * dbeta (NULL iff mode == GDN_GATED) in dtype `io`, dA_log [H, d_k] float32
 * (overwritten, summed over the batch) and dh0 (NULL => not written).
 * dg and dbeta are gradients with respect to the post-sigmoid g and beta.
 * ws must hold at least gdn_workspace_bytes(shape, 1) bytes. */
gdn_status_t gdn_bwd(const gdn_shape_t* shape,
                     const void* v, const void* b, const void* c,
                     const void* g, const void* beta, const float* A_log,
                     const float* h0, const void* dO, const float* dhT,
                     void* dv, void* db, void* dc, void* dg, void* dbeta,
                     float* dA_log, float* dh0,
                     void* ws, size_t ws_bytes, gdn_stream_t stream);

/* Forward pass that also keeps what the chunked backward would otherwise
 * recompute ("GDN & MLA Mechanism Deep-Dive", Step 5: each chunk's closed form
 * is a function of its inputs and the state entering it).  Per chunk of 64
 * tokens `saved` receives the entering state (fp32 64 x 64, 16 KB) and the
 * results of the chunk's delta solve that the backward reuses (80 KB: the
 * decay-weighted scores P, K, the block inverse D^-1 and N, W and
 * U = Util - W S; in gated mode the scores P, 16 KB; layout private to the
 * library).  gdn_bwd_saved then takes them instead of running
 * the forward sweep again.  Arguments and results are those of gdn_fwd, plus
 * `saved`: device memory of at least gdn_saved_bytes(shape) bytes, 256-byte
 * aligned, written completely by the call.  o and hT equal gdn_fwd's within
 * the bf16 tolerance (the level products form K without beta, M = beta K
 * after them, so the rounding differs).  Shapes: bf16, d_k and d_v <= 64, no
 * option bits but GDN_CHECK_FINITE, and a forward that runs unsplit over
 * more than 8 tokens (the saving call always takes the tensor-core kernel,
 * also where gdn_plan reports the token-serial one for gdn_fwd)
 * or, in delta mode, a split in time (gdn_plan(shape, 0): segments > 1); that
 * split runs every segment from a zero state, keeping the residuals, then
 * walks the segments' transitions on the tensor cores and corrects outputs
 * and residuals by the true entering states (the saving call writes the true
 * ones).  gdn_saved_bytes is 0 for
 * any other shape, and both calls return GDN_ERR_MODE for it.  GDN_ERR_NULL if saved is NULL, GDN_ERR_ALIGN if it is
 * misaligned, GDN_ERR_WORKSPACE if saved_bytes is too small. */
size_t gdn_saved_bytes(const gdn_shape_t* shape);

gdn_status_t gdn_fwd_save(const gdn_shape_t* shape,
                          const void* v, const void* b, const void* c,
                          const void* g, const void* beta, const float* A_log,
                          const float* h0, void* o, float* hT,
                          void* saved, size_t saved_bytes,
                          void* ws, size_t ws_bytes, gdn_stream_t stream);

/* Backward pass from gdn_fwd_save's residuals: gdn_bwd's gradients, for the
 * same shape and the same v, b, c, g, beta, A_log (h0 is not needed: the
 * residuals hold the entering states).  `saved` is read only.  ws must hold at
 * least gdn_workspace_bytes(shape, 2) bytes (smaller than the plain backward's:
 * the states and solve results live in `saved`).  Errors as gdn_bwd, plus
 * those of gdn_fwd_save for `saved`. */
gdn_status_t gdn_bwd_saved(const gdn_shape_t* shape,
                           const void* v, const void* b, const void* c,
                           const void* g, const void* beta, const float* A_log,
                           const void* saved, size_t saved_bytes,
                           const void* dO, const float* dhT,
                           void* dv, void* db, void* dc, void* dg, void* dbeta,
                           float* dA_log, float* dh0,
                           void* ws, size_t ws_bytes, gdn_stream_t stream);

/* Backward pass that allocates nothing and needs no workspace argument.  The
 * pages describe no counterpart; this is a convenience of the library.  It is
 * for callers that cannot call cudaMalloc: latency-critical code that cannot
 * afford cudaMalloc's implicit device synchronisation, plugins inside a host
 * framework that owns all device memory and offers them no allocator, and
 * processes that reserve their memory at start-up and forbid later
 * allocations.  Arguments and results are those of gdn_bwd; the workspace is
 * a 32 MiB array inside the library (one per GPU that loads it, held until
 * the process exits).  Errors: the shape's own errors as gdn_bwd returns them
 * (GDN_ERR_NULL, GDN_ERR_MODE, GDN_ERR_SHAPE), then GDN_ERR_WORKSPACE if
 * gdn_workspace_bytes(shape, 1) exceeds 32 MiB, GDN_ERR_DEVICE on a GPU that
 * is not sm_103, then gdn_bwd's own checks; nothing is enqueued on an error.
 * The status the kernels leave on the device (an expired wait, or with
 * GDN_CHECK_FINITE a non-finite gradient) is read by gdn_bwd_noalloc_status.
 * All calls on a device share the array: calls that may overlap on the GPU
 * race and must be ordered by the caller.  Each call looks up the array's
 * device address (cudaGetSymbolAddress) on the current device; the first
 * lookup on a device may load the library's device code, so make the first
 * call before any stream capture on that device. */
gdn_status_t gdn_bwd_noalloc(const gdn_shape_t* shape,
                             const void* v, const void* b, const void* c,
                             const void* g, const void* beta, const float* A_log,
                             const float* h0, const void* dO, const float* dhT,
                             void* dv, void* db, void* dc, void* dg, void* dbeta,
                             float* dA_log, float* dh0, gdn_stream_t stream);

/* gdn_last_device_status for the array gdn_bwd_noalloc uses as its workspace
 * on the current device: synchronises `stream`, then returns GDN_OK,
 * GDN_ERR_TIMEOUT or GDN_ERR_NONFINITE as left by the last gdn_bwd_noalloc
 * call on this device (GDN_ERR_CUDA if a CUDA call fails, GDN_ERR_DEVICE on a
 * GPU that is not sm_103).  Allocates nothing. */
gdn_status_t gdn_bwd_noalloc_status(gdn_stream_t stream);

/* Synchronises `stream` and returns the status the kernels of the last call
 * that used `ws` left in it (GDN_OK, GDN_ERR_TIMEOUT), or GDN_ERR_CUDA if the
 * synchronisation itself failed. */
gdn_status_t gdn_last_device_status(const void* ws, gdn_stream_t stream);

/* A static, human-readable name for a status code. */
const char* gdn_status_string(gdn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
