"""Helpers shared by the GPU tests: move seeded inputs to the device, call the
library through its C ABI binding, and measure max |gpu - oracle| / max |oracle|."""
import numpy as np
import torch

import linear_attention_recurrence_delta_gb300 as gdn

TOL = {"f32": 1e-5, "bf16": 5e-3}


def tdtype(io):
    return torch.float32 if io == "f32" else torch.bfloat16


def dev(x, io, device="cuda"):
    """float64 numpy array of exactly representable values -> device tensor."""
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=tdtype(io)).contiguous()


def dev32(x, device="cuda"):
    if x is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=torch.float32).contiguous()


def shape_of(w):
    return gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype, gate_logits=w.gate_logits,
                          norm_bc=w.norm_bc)


def run_fwd(w, x, want_hT=True, stream=None):
    s = shape_of(w)
    io = w.dtype
    t = {k: dev(x[k], io) for k in ("v", "b", "c", "g", "beta")}
    A_log, h0 = dev32(x["A_log"]), dev32(x["h0"])
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=tdtype(io), device="cuda")
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda") if want_hT else None
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_fwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, o, hT, ws, stream=stream),
              "gdn_fwd")
    gdn.check(gdn.gdn_last_device_status(ws, stream=stream), "device status")
    return o.double().cpu().numpy(), (hT.double().cpu().numpy() if hT is not None else None)


def run_bwd(w, x, dhT=None, want_dh0=True):
    s = shape_of(w)
    io = w.dtype
    t = {k: dev(x[k], io) for k in ("v", "b", "c", "g", "beta", "dO")}
    A_log, h0, dhT_t = dev32(x["A_log"]), dev32(x["h0"]), dev32(dhT)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    dt = tdtype(io)
    out = {
        "dv": torch.empty((B, T, H, dv), dtype=dt, device="cuda"),
        "db": torch.empty((B, T, H, dk), dtype=dt, device="cuda"),
        "dc": torch.empty((B, T, H, dk), dtype=dt, device="cuda"),
        "dg": torch.empty((B, T, H), dtype=dt, device="cuda"),
        "dbeta": torch.empty((B, T, H), dtype=dt, device="cuda") if w.mode == "delta" else None,
        "dA_log": torch.empty((H, dk), dtype=torch.float32, device="cuda"),
        "dh0": torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda") if want_dh0 else None,
    }
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_bwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, t["dO"], dhT_t,
                          out["dv"], out["db"], out["dc"], out["dg"], out["dbeta"], out["dA_log"], out["dh0"], ws),
              "gdn_bwd")
    gdn.check(gdn.gdn_last_device_status(ws), "device status")
    return {k: (None if v is None else v.double().cpu().numpy()) for k, v in out.items()}


def run_saved(w, x, dhT):
    """gdn_fwd_save then gdn_bwd_saved (bf16): o, h_T and the gradients as float64 arrays."""
    s = shape_of(w)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    delta = w.mode == "delta"
    t = {k: dev(x[k], "bf16") for k in ("v", "b", "c", "g", "beta", "dO")}
    A_log, h0 = dev32(x["A_log"]), dev32(x["h0"])
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda")
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    nbytes = gdn.gdn_saved_bytes(s)
    assert nbytes == B * H * -(-T // 64) * (16384 + (81920 if delta else 16384))
    saved = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN patterns: all must be written
    ws0 = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_fwd_save(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, o, hT, saved, ws0),
              "gdn_fwd_save")
    gdn.check(gdn.gdn_last_device_status(ws0), "forward device status")
    dt = torch.bfloat16
    out = {
        "dv": torch.empty((B, T, H, dv), dtype=dt, device="cuda"),
        "db": torch.empty((B, T, H, dk), dtype=dt, device="cuda"),
        "dc": torch.empty((B, T, H, dk), dtype=dt, device="cuda"),
        "dg": torch.empty((B, T, H), dtype=dt, device="cuda"),
        "dbeta": torch.empty((B, T, H), dtype=dt, device="cuda") if delta else None,
        "dA_log": torch.empty((H, dk), dtype=torch.float32, device="cuda"),
        "dh0": torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda"),
    }
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 2), dtype=torch.uint8, device="cuda")
    assert 0 < ws.numel() < gdn.gdn_workspace_bytes(s, 1)
    gdn.check(gdn.gdn_bwd_saved(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, saved, t["dO"], dev32(dhT),
                                *out.values(), ws), "gdn_bwd_saved")
    gdn.check(gdn.gdn_last_device_status(ws), "backward device status")
    got = {k: (None if v is None else v.double().cpu().numpy()) for k, v in out.items()}
    return o.double().cpu().numpy(), hT.double().cpu().numpy(), got


def rel_err(got, ref):
    den = np.abs(ref).max()
    num = np.abs(got - ref).max()
    if den == 0:
        return float(num)
    return float(num / den)


def assert_close(got, ref, tol, name):
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    e = rel_err(got, ref)
    assert e <= tol, f"{name}: max|d|/max|ref| = {e:.3e} > {tol:.1e}"
    return e
