"""gdn_fwd_save / gdn_bwd_saved through the C ABI: the forward keeps what the chunked backward would recompute
(the state entering every chunk of 64 tokens and the results of the chunk's delta solve, or in gated mode the
scores P), and the backward reads it.  Output, final state and every gradient against the fp64 oracle, on shapes with several chunks, ragged last
chunks and the widths the tensor-core path takes, with and without h0 and dh_T, and on chunks whose decay factors
would overflow (the exact elementwise path).  The gradients are also compared with gdn_bwd's, which recomputes
everything: the two must agree to within the bf16 tolerance of each other."""
import math

import numpy as np
import pytest
import torch

import linear_attention_recurrence_delta_gb300 as gdn
import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, dev, dev32, run_bwd, shape_of

pytestmark = pytest.mark.gpu

KEYS = ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0")


def run_saved(w, x, dhT):
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


def check_saved(w, with_dhT=True):
    x = I.make_inputs(w)
    dhT = None
    if with_dhT:
        dhT = I.round_to(0.5 * I.normal(w.seed + 7, 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv),
                         "f32")
    o, hT, got = run_saved(w, x, dhT)
    tol = TOL["bf16"]
    ro, rhT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)
    assert_close(o, ro, tol, f"{w.name} o")
    assert_close(hT, rhT, tol, f"{w.name} hT")
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=w.mode)
    plain = run_bwd(w, x, dhT=dhT)
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], tol, f"{w.name} {k} vs oracle")
        assert_close(got[k], plain[k], tol, f"{w.name} {k} vs gdn_bwd")


@pytest.mark.parametrize("mode", ["delta", "gated"])
@pytest.mark.parametrize("B,H,T,d", [(1, 2, 64, 64), (2, 3, 300, 64), (2, 2, 100, 56), (2, 2, 37, 16),
                                     (1, 3, 129, 32), (4, 16, 1024, 64)])
@pytest.mark.parametrize("h0_std", [0.0, 0.3])
def test_saved_matches_oracle(mode, B, H, T, d, h0_std):
    w = I.custom(name=f"saved_{mode}_{B}x{H}x{T}x{d}_{h0_std}", mode=mode, dtype="bf16", B=B, H=H, T=T, dk=d, dv=d,
                 seed=3 + T + d, h0_std=h0_std, backward=True)
    check_saved(w, with_dhT=h0_std > 0)


@pytest.mark.parametrize("mode", ["delta", "gated"])
@pytest.mark.parametrize("g_mu", [0.0, 3.0])
def test_saved_steep_decay(mode, g_mu):
    """|A| up to 64 and g near 1: the forward evaluates those chunks' decay factors elementwise."""
    w = I.custom(name=f"saved_steep_{mode}_{g_mu}", mode=mode, dtype="bf16", B=1, H=4, T=192, dk=64, dv=64, seed=8,
                 g_mu=g_mu, alog_max=math.log(64.0), h0_std=0.2, backward=True)
    check_saved(w)


@pytest.mark.parametrize("name", ["delta_bf16_8x16x4096x64", "gated_bf16_8x16x4096x56_bwd"])
def test_saved_full_size(name):
    """The bench's shape (8 x 16 x 4096 x 64, delta) and the gated 8 x 16 x 4096 x 56 workload: forward and
    backward from the residuals on every unit, against gdn_fwd and gdn_bwd (which the full-size oracle tests pin)
    within the bf16 tolerance."""
    w = I.WORKLOADS[name].with_(backward=True)
    x = I.make_inputs(w)
    o, hT, got = run_saved(w, x, None)
    from tests.gdn_testlib import run_fwd
    ro, rhT = run_fwd(w, x)
    tol = TOL["bf16"]
    assert_close(o, ro, tol, "o vs gdn_fwd")
    assert_close(hT, rhT, tol, "hT vs gdn_fwd")
    plain = run_bwd(w, x, dhT=None)
    for k in KEYS:
        if plain[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], plain[k], tol, f"{k} vs gdn_bwd")
