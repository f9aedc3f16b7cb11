// gdn_noalloc.cu -- gdn_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// gdn_bwd needs a caller-provided workspace (state checkpoints, one segment of
// recomputed states, per-head dA_log partials and a status word).  Some
// callers cannot obtain one: code running where cudaMalloc is off limits
// because it implicitly synchronises the device (latency-critical loops), a
// plugin inside a host framework that owns the whole memory pool and exposes no
// allocator, or a process that reserves all memory at start-up and forbids
// later allocations.  For them this file keeps the workspace in a file-scope
// __device__ array of fixed size, kNoAllocBytes (32 MiB).  Every GPU that loads
// the library reserves that array until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents; gdn_bwd clears the status word at the start of each call and
// writes every other byte it reads before reading it.  Calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// the array: serialise them.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress, with that device current, and caches it.  Make
// that first call before any stream capture on that device.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

#define GDN_NOALLOC_BYTES ((size_t)32 << 20)

static __device__ __align__(256) unsigned char g_bwd_scratch[GDN_NOALLOC_BYTES];

namespace gdn {
namespace {

constexpr size_t kNoAllocBytes = GDN_NOALLOC_BYTES;
constexpr int kMaxDevices = 64;

void* g_scratch_ptr[kMaxDevices];   // device address of g_bwd_scratch per device (NULL = not set up)

gdn_status_t scratch_for_current_device(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_DEVICE;
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status_t gdn_bwd_noalloc(const gdn_shape_t* shape, const void* v, const void* b, const void* c,
                                        const void* g, const void* beta, const float* A_log, const float* h0,
                                        const void* dO, const float* dhT, void* dv, void* db, void* dc,
                                        void* dg, void* dbeta, float* dA_log, float* dh0, gdn_stream_t stream)
{
    if (!shape) return GDN_ERR_NULL;
    const size_t need = gdn_workspace_bytes(shape, 1);
    if (need == 0) return GDN_ERR_SHAPE;
    if (need > gdn::kNoAllocBytes) return GDN_ERR_WORKSPACE;
    void* ws = nullptr;
    gdn_status_t r = gdn::scratch_for_current_device(&ws);
    if (r != GDN_OK) return r;
    return gdn_bwd(shape, v, b, c, g, beta, A_log, h0, dO, dhT, dv, db, dc, dg, dbeta, dA_log, dh0, ws,
                   gdn::kNoAllocBytes, stream);
}
