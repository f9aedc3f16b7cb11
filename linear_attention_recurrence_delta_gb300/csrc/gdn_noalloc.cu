// gdn_noalloc.cu -- gdn_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory, and gdn_bwd_noalloc_status, which reads the device
// status those calls leave behind.
//
// gdn_bwd needs a caller-provided workspace.  Some callers cannot obtain one:
// code running where cudaMalloc is off limits because it implicitly
// synchronises the device (latency-critical loops), a plugin inside a host
// framework that owns the whole memory pool and exposes no allocator, or a
// process that reserves all memory at start-up and forbids later allocations.
// For them this file keeps the workspace in a file-scope __device__ array of
// fixed size, kNoAllocBytes (32 MiB).  Every GPU that loads the library
// reserves that array until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents; gdn_bwd clears the status word at the start of each call and
// writes every other byte it reads before reading it.  Calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array: serialise them.
//
// In host code the array's name stands for a host-side shadow, not for device
// memory, so every call looks up the array's device address with
// cudaGetSymbolAddress on the current device (a host-side query; the first one
// on a device may load the library's device code, so make the first call
// before any stream capture on that device).
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

#define GDN_NOALLOC_BYTES ((size_t)32 << 20)

static __device__ __align__(256) unsigned char g_bwd_scratch[GDN_NOALLOC_BYTES];

namespace gdn {
namespace {

constexpr size_t kNoAllocBytes = GDN_NOALLOC_BYTES;

// device address of g_bwd_scratch on the current device
gdn_status_t scratch_address(void** out)
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) {
        (void)cudaGetLastError();   // leave no error pending for the caller's next launch check
        return GDN_ERR_CUDA;
    }
    *out = p;
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status_t gdn_bwd_noalloc(const gdn_shape_t* shape, const void* v, const void* b, const void* c,
                                        const void* g, const void* beta, const float* A_log, const float* h0,
                                        const void* dO, const float* dhT, void* dv, void* db, void* dc,
                                        void* dg, void* dbeta, float* dA_log, float* dh0, gdn_stream_t stream)
{
    // the shape's own errors first, as gdn_bwd reports them (NULL, unknown mode or dtype, sizes out of range)
    gdn_plan_t plan;
    gdn_status_t r = gdn_plan(shape, 1, &plan);
    if (r != GDN_OK) return r;
    if (gdn_workspace_bytes(shape, 1) > gdn::kNoAllocBytes) return GDN_ERR_WORKSPACE;
    if ((r = gdn::check_device()) != GDN_OK) return r;
    void* ws = nullptr;
    if ((r = gdn::scratch_address(&ws)) != GDN_OK) return r;
    return gdn_bwd(shape, v, b, c, g, beta, A_log, h0, dO, dhT, dv, db, dc, dg, dbeta, dA_log, dh0, ws,
                   gdn::kNoAllocBytes, stream);
}

extern "C" gdn_status_t gdn_bwd_noalloc_status(gdn_stream_t stream)
{
    gdn_status_t r = gdn::check_device();
    if (r != GDN_OK) return r;
    void* ws = nullptr;
    if ((r = gdn::scratch_address(&ws)) != GDN_OK) return r;
    return gdn_last_device_status(ws, stream);
}
