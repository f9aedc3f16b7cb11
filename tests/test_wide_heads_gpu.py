"""Heads wider than 64 (up to d_k = d_v = 128) against the fp64 oracle.

Value columns past 64 go to further column slabs (the state's columns never
mix); keys past 64 take the token-serial kernels' 128-row layouts, and the
backward adds the slabs' partial sums of db, dc, dg, dbeta and dA_log in a
fixed order.  Bar: the parity tolerance of the other tests (1e-5 of max|ref|
for f32 I/O, 5e-3 for bf16).
"""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

WIDE = [(128, 128), (64, 128), (128, 64), (96, 80), (128, 8), (8, 128), (72, 120)]


def oracle_fwd(w, x):
    return oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)


def check_fwd(w):
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle_fwd(w, x)
    assert_close(o, ro, TOL[w.dtype], f"{w.name} o")
    assert_close(hT, rhT, TOL[w.dtype], f"{w.name} hT")


def check_bwd(w, with_dhT=True, units=None):
    x = I.make_inputs(w)
    dhT = None
    if with_dhT:
        dhT = I.round_to(0.5 * I.normal(91, 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv), "f32")
    got = run_bwd(w, x, dhT=dhT)
    if units is not None:
        x = {k: (None if v is None else (v[:, :, units] if k in ("v", "b", "c", "g", "beta", "dO")
                                         else v[units] if k == "A_log" else v[:, units]))
             for k, v in x.items()}
        got = {k: (None if v is None else (v[:, :, units] if k in ("dv", "db", "dc", "dg", "dbeta")
                                           else v[units] if k == "dA_log" else v[:, units]))
               for k, v in got.items()}
        dhT = None if dhT is None else dhT[:, units]
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=w.mode)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], TOL[w.dtype], f"{w.name} {k}")


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", WIDE)
def test_fwd_wide(mode, io, dk, dv):
    """Several chunks and a ragged tail (T = 130), initial state given."""
    w = I.custom(name=f"wide_{mode}_{io}_{dk}_{dv}", mode=mode, dtype=io, B=2, H=2, T=130, dk=dk, dv=dv,
                 seed=dk * 3 + dv, h0_std=0.2)
    check_fwd(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv,T", [(128, 128, 37), (64, 128, 100), (128, 32, 65), (96, 80, 70),
                                     (40, 104, 33), (128, 64, 1)])
def test_bwd_wide(mode, io, dk, dv, T):
    w = I.custom(name=f"wbwd_{mode}_{io}_{dk}_{dv}_{T}", mode=mode, dtype=io, B=2, H=2, T=T, dk=dk, dv=dv,
                 seed=dk + 7 * dv + T, h0_std=0.3, backward=True)
    check_bwd(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 5])
@pytest.mark.parametrize("dk,dv", [(128, 128), (128, 64), (64, 128), (96, 80)])
def test_decode_wide(mode, io, T, dk, dv):
    w = I.custom(name=f"wdec_{mode}_{io}_{T}_{dk}_{dv}", mode=mode, dtype=io, B=3, H=3, T=T, dk=dk, dv=dv,
                 seed=300 + T + dk + dv, h0_std=0.3)
    check_fwd(w)


def test_wide_gate_logits():
    """g and beta as logits with 128-wide heads: forward and backward."""
    w = I.custom(name="wide_logits", mode="delta", dtype="bf16", B=1, H=2, T=90, dk=128, dv=128, seed=55,
                 h0_std=0.2, gate_logits=True, backward=True)
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle.gdn_fwd_logits(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)
    assert_close(o, ro, TOL["bf16"], "o")
    assert_close(hT, rhT, TOL["bf16"], "hT")
    got = run_bwd(w, x)
    ref = oracle.gdn_bwd_logits(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None,
                                mode=w.mode)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        assert_close(got[k], ref[k], TOL["bf16"], f"logits {k}")


def test_wide_repeatable_backward():
    """The slab partial sums are added in a fixed order: two backward runs agree bit for bit."""
    w = I.custom(name="wide_rep", mode="delta", dtype="bf16", B=2, H=2, T=150, dk=128, dv=128, seed=12,
                 backward=True)
    x = I.make_inputs(w)
    a = run_bwd(w, x)
    b = run_bwd(w, x)
    for k in a:
        if a[k] is not None:
            np.testing.assert_array_equal(a[k], b[k])


def test_workload_delta_bf16_8x16x4096x128_fwd_bwd():
    """The 128-wide workload at full size, in the launch configuration the bench times: forward and backward on
    every unit."""
    w = I.WORKLOADS["delta_bf16_8x16x4096x128"]
    check_fwd(w)
    check_bwd(w, with_dhT=False)
