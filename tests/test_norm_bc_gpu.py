"""b and c given before their L2 normalisation (GDN_NORM_BC) against the fp64 oracle.

Every kernel divides b_t and c_t by their norm over d_k before the rule uses them,
and the backward returns db, dc with respect to the vectors as given.  The oracle
side is oracle.gdn_fwd_opts / gdn_bwd_opts (normalisation in fp64, its gradient by
the vector-Jacobian product pinned by finite differences).  Inputs: b, c ~ N(0, 1)
entries (norm about sqrt(d_k)), so the normalisation changes them.  Bar: the
tolerance of the other parity tests (1e-5 of max|ref| for f32 I/O, 5e-3 for bf16).
"""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def wl(name, mode, io, B, H, T, dk, dv, seed, **kw):
    return I.custom(name=name, mode=mode, dtype=io, B=B, H=H, T=T, dk=dk, dv=dv, seed=seed, norm_bc=True,
                    b_dist="normal", c_dist="normal", **kw)


def ref_fwd(w, x):
    return oracle.gdn_fwd_opts(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode,
                               gate_logits=w.gate_logits, norm_bc=True)


def check_fwd(w, x=None):
    x = x or I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = ref_fwd(w, x)
    assert_close(o, ro, TOL[w.dtype], f"{w.name} o")
    assert_close(hT, rhT, TOL[w.dtype], f"{w.name} hT")


def check_bwd(w, x=None):
    x = x or I.make_inputs(w)
    dhT = I.round_to(0.5 * I.normal(93, 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv), "f32")
    got = run_bwd(w, x, dhT=dhT)
    ref = oracle.gdn_bwd_opts(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT,
                              mode=w.mode, gate_logits=w.gate_logits, norm_bc=True)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], TOL[w.dtype], f"{w.name} {k}")


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,dk,dv", [(130, 64, 64), (65, 32, 48), (70, 128, 128), (100, 64, 128)])
def test_fwd_norm(mode, io, T, dk, dv):
    check_fwd(wl(f"nf_{mode}_{io}_{T}_{dk}_{dv}", mode, io, 2, 3, T, dk, dv, seed=T + dk + dv, h0_std=0.2))


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_fwd_norm_zero_vectors(mode):
    """All-zero b_t or c_t stay zero after the normalisation (the norm is floored, not divided by)."""
    w = wl(f"nz_{mode}", mode, "bf16", 1, 2, 96, 64, 64, seed=31)
    x = I.make_inputs(w)
    x["b"][:, 5] = 0.0
    x["c"][:, 40] = 0.0
    x["b"][:, 90, 1] = 0.0
    check_fwd(w, x)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,dk,dv", [(37, 64, 64), (100, 56, 56), (40, 64, 128), (33, 128, 128)])
def test_bwd_norm(mode, io, T, dk, dv):
    check_bwd(wl(f"nb_{mode}_{io}_{T}_{dk}_{dv}", mode, io, 2, 2, T, dk, dv, seed=7 * T + dk, h0_std=0.3,
                 backward=True))


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,dk,dv", [(1, 64, 64), (4, 128, 96)])
def test_decode_norm(mode, io, T, dk, dv):
    check_fwd(wl(f"nd_{mode}_{io}_{T}_{dk}_{dv}", mode, io, 3, 4, T, dk, dv, seed=400 + T + dk, h0_std=0.3))


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_time_split_norm(mode):
    """Two heads over 2048 tokens take the time-split forward and backward (four segments)."""
    w = wl(f"nts_{mode}", mode, "bf16", 1, 2, 2048, 64, 64, seed=77, h0_std=0.2, backward=True)
    x = I.make_inputs(w)
    check_fwd(w, x)
    check_bwd(w, x)


def test_norm_with_logit_gates():
    """Both option bits at once: logit gates and unnormalised b, c."""
    w = wl("n_logits", "delta", "bf16", 2, 2, 90, 64, 64, seed=44, h0_std=0.2, gate_logits=True, backward=True)
    x = I.make_inputs(w)
    check_fwd(w, x)
    check_bwd(w, x)


def test_norm_is_scale_invariant():
    """Scaling b and c by a positive factor per token does not change the outputs with the bit set."""
    w = wl("n_scale", "delta", "bf16", 1, 2, 130, 64, 64, seed=5)
    x = I.make_inputs(w)
    o1, h1 = run_fwd(w, x)
    y = dict(x)
    y["b"] = I.round_to(x["b"] * 4.0, "bf16")     # powers of two: exact in bf16
    y["c"] = I.round_to(x["c"] * 0.25, "bf16")
    o2, h2 = run_fwd(w, y)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=2e-2 * np.abs(o1).max())
    np.testing.assert_allclose(h1, h2, rtol=0, atol=2e-2 * np.abs(h1).max())
