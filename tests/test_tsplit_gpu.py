"""Forward split in time (long sequences over few heads) against the fp64 oracle.

When B*H*P fits the GPU for some P >= 4 (delta) or 3 (gated) dividing T with
at least 512 tokens per segment, gdn_fwd runs every segment from a zero
state, (delta) every segment's transition from the identity with v = 0, a
scan over segments and every segment again from its true entering state.
These shapes take that path; the 1 x 16 x 32768 workload test covers it too.
"""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_delta_gb300 as gdn
import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, dev, dev32, run_fwd, tdtype

pytestmark = pytest.mark.gpu


def oracle_fwd(w, x):
    return oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io,B,H,T,d", [("bf16", 1, 4, 4096, 64), ("bf16", 2, 3, 3072, 56), ("f32", 1, 2, 2048, 32)])
def test_tsplit_parity(mode, io, B, H, T, d):
    w = I.custom(name=f"ts_{mode}_{io}_{B}x{H}x{T}x{d}", mode=mode, dtype=io, B=B, H=H, T=T, dk=d, dv=d,
                 seed=T + d, h0_std=0.3, b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm",
                 g_mu=-1.0)
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle_fwd(w, x)
    assert_close(o, ro, TOL[io], f"{w.name} o")
    assert_close(hT, rhT, TOL[io], f"{w.name} hT")


def test_tsplit_in_place_state():
    """hT may alias h0 on the split path as well."""
    w = I.custom(name="ts_inplace", mode="delta", dtype="bf16", B=1, H=4, T=4096, dk=64, dv=64, seed=12,
                 h0_std=0.3, b_dist="l2norm", c_dist="l2norm", g_mu=-2.0)
    x = I.make_inputs(w)
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype)
    t = {k: dev(x[k], "bf16") for k in ("v", "b", "c", "g", "beta")}
    state = dev32(x["h0"])
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_fwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], dev32(x["A_log"]), state, o, state, ws))
    ro, rhT = oracle_fwd(w, x)
    assert_close(o.double().cpu().numpy(), ro, TOL["bf16"], "o")
    assert_close(state.double().cpu().numpy(), rhT, TOL["bf16"], "state")


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io,B,H,T,d", [("bf16", 1, 4, 4096, 64), ("bf16", 2, 3, 3072, 56), ("f32", 1, 2, 2048, 32)])
def test_tsplit_backward_parity(mode, io, B, H, T, d):
    """The split backward: segment adjoints G_p = sum_t (Phi_t^T c_t) do_t^T, a reverse scan of the end
    gradients, then every segment's backward from its entering state; every gradient against the oracle, with h0
    and dh_T given."""
    from tests.gdn_testlib import run_bwd
    w = I.custom(name=f"tsb_{mode}_{io}_{B}x{H}x{T}x{d}", mode=mode, dtype=io, B=B, H=H, T=T, dk=d, dv=d,
                 seed=3 * T + d, h0_std=0.3, b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm",
                 g_mu=-1.0, backward=True)
    x = I.make_inputs(w)
    dhT = I.round_to(0.4 * I.normal(91, 1, w.B * w.H * d * d).reshape(w.B, w.H, d, d), "f32")
    got = run_bwd(w, x, dhT=dhT)
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=w.mode)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], TOL[io], f"{w.name} {k}")


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_tsplit_ragged_segments(mode):
    """T = 3000 over 4 heads splits into 5 segments of 600 tokens: every segment ends inside a chunk."""
    from tests.gdn_testlib import run_bwd
    w = I.custom(name=f"tsr_{mode}", mode=mode, dtype="bf16", B=1, H=4, T=3000, dk=64, dv=64, seed=21,
                 h0_std=0.3, b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm", g_mu=-1.5,
                 backward=True)
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle_fwd(w, x)
    assert_close(o, ro, TOL["bf16"], "o")
    assert_close(hT, rhT, TOL["bf16"], "hT")
    got = run_bwd(w, x)
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None, mode=w.mode)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is not None:
            assert_close(got[k], ref[k], TOL["bf16"], k)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_tsplit_backward_two_segments(mode):
    """40 heads over 1024 tokens: the forward stays whole, the backward splits into two segments of 512."""
    from tests.gdn_testlib import run_bwd
    w = I.custom(name=f"tsb2_{mode}", mode=mode, dtype="f32", B=1, H=40, T=1024, dk=32, dv=32, seed=33,
                 h0_std=0.3, b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm", g_mu=-1.0,
                 backward=True)
    x = I.make_inputs(w)
    dhT = I.round_to(0.4 * I.normal(92, 1, w.H * 32 * 32).reshape(1, w.H, 32, 32), "f32")
    got = run_bwd(w, x, dhT=dhT)
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=w.mode)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is not None:
            assert_close(got[k], ref[k], TOL["f32"], k)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_tsplit_backward_dO_offset(mode):
    """fp32 dO need only be 4-byte aligned: an upstream gradient starting 4 bytes into its buffer takes the split
    backward's element-wise staging instead of 16-byte copies.  T = 3000 over two heads: five segments of 600
    tokens, each summed in two runs."""
    w = I.custom(name=f"tso_{mode}", mode=mode, dtype="f32", B=1, H=2, T=3000, dk=32, dv=32, seed=57, h0_std=0.3,
                 b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm", g_mu=-1.0, backward=True)
    x = I.make_inputs(w)
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype)
    t = {k: dev(x[k], "f32") for k in ("v", "b", "c", "g", "beta")}
    n = w.B * w.T * w.H * w.dv
    raw = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    dO = raw[1:].view(w.B, w.T, w.H, w.dv)
    dO.copy_(dev(x["dO"], "f32"))
    assert dO.data_ptr() % 16 != 0
    out = {k: torch.empty_like(t[k]) for k in ("v", "b", "c", "g")}
    dbeta = torch.empty_like(t["beta"]) if mode == "delta" else None
    dA = torch.empty((w.H, w.dk), dtype=torch.float32, device="cuda")
    dh0 = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_bwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"] if mode == "delta" else None,
                          dev32(x["A_log"]), dev32(x["h0"]), dO, None, out["v"], out["b"], out["c"], out["g"], dbeta,
                          dA, dh0, ws))
    gdn.check(gdn.gdn_last_device_status(ws), "device status")
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None, mode=w.mode)
    got = {"dv": out["v"], "db": out["b"], "dc": out["c"], "dg": out["g"], "dbeta": dbeta, "dA_log": dA, "dh0": dh0}
    for k, v in got.items():
        if ref[k] is not None:
            assert_close(v.double().cpu().numpy(), ref[k], TOL["f32"], k)
