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
    const void *v, *b, *c, *g, *beta;
    const float* A_log;
    const float* h0;
    void* o;
    float* hT;
    // backward only
    const void* dO;
    const float* dhT;
    void *dv_, *db, *dc, *dg, *dbeta;
    float* dA_log;
    float* dh0;
    // workspace
    void* ws;
    size_t ws_bytes;
};

// Workspace carve-up.  The first 256 bytes always hold the device status word.
struct WsLayout {
    size_t status_off = 0;        // uint32 status code, uint32 detail
    size_t snap_off = 0;          // serial backward: state entering every kSerialSnap tokens
    size_t xvr_off = 0;           // serial backward, delta: x and v - h'^T b of every token
    size_t dalog_off = 0;         // per-(b,h) dA_log partials, float [B*H, d_k]
    size_t total = 0;
};

constexpr int kSerialBlock = 32;               // tokens per backward block
constexpr int kSerialSnap = 8;                 // tokens between backward state snapshots
constexpr size_t kStateSlot = 16 * 256 * 4;    // one state snapshot (256 threads x 16 floats)

WsLayout ws_layout(const gdn_shape_t& s, int backward);

// Launchers (enqueue on `st`, return cudaGetLastError()).
cudaError_t launch_serial_fwd(const Args& a, cudaStream_t st);
cudaError_t launch_serial_bwd(const Args& a, cudaStream_t st);
cudaError_t launch_fwd_tc(const Args& a, cudaStream_t st, bool* handled);
cudaError_t launch_decode(const Args& a, cudaStream_t st);   // 1 <= T <= decode_max_tokens()
int decode_max_tokens();

// Device status word helpers.
enum : uint32_t { kDevOk = 0, kDevTimeout = 1 };

}  // namespace gdn
