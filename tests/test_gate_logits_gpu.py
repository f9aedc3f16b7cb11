"""g and beta given as logits (GDN_GATE_LOGITS): every kernel applies the sigmoid
as it loads them and the backward returns dg, dbeta with respect to the logits.
Checked against the fp64 oracle's composition (the rule on the sigmoids, the
chain rule through them), with the tolerance of the other parity tests."""
import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def _check(w, bwd=True):
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle.gdn_fwd_logits(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)
    assert_close(o, ro, TOL[w.dtype], f"{w.name} o")
    assert_close(hT, rhT, TOL[w.dtype], f"{w.name} hT")
    if bwd:
        got = run_bwd(w, x)
        ref = oracle.gdn_bwd_logits(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None,
                                    mode=w.mode)
        for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
            if ref[k] is not None:
                assert_close(got[k], ref[k], TOL[w.dtype], f"{w.name} {k}")


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io,T", [("bf16", 200), ("f32", 100)])
def test_logits_chunked_and_serial(mode, io, T):
    """bf16: the tcgen05 forward; f32: the token-serial forward; both through the serial backward."""
    w = I.custom(name=f"lg_{mode}_{io}", mode=mode, dtype=io, B=2, H=3, T=T, dk=64, dv=64, seed=41, h0_std=0.3,
                 b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm", gate_logits=True,
                 backward=True)
    _check(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_logits_decode(mode):
    w = I.custom(name=f"lgd_{mode}", mode=mode, dtype="bf16", B=3, H=5, T=3, dk=64, dv=64, seed=42, h0_std=0.3,
                 b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm", gate_logits=True,
                 backward=True)
    _check(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_logits_time_split(mode):
    """The split's scans sum the gates of whole segments (gated) from the logits too."""
    w = I.custom(name=f"lgs_{mode}", mode=mode, dtype="bf16", B=1, H=4, T=4096, dk=64, dv=64, seed=43, h0_std=0.3,
                 b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm", gate_logits=True, g_mu=-2.0,
                 backward=True)
    _check(w)
