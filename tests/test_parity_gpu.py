"""GPU parity: libgdn (through its C ABI) against the fp64 oracle.

Bar: max |gpu - oracle| <= tol * max |oracle| per output tensor (o, h_T and
every gradient), tol = 1e-5 for float32 I/O and 5e-3 for bf16 I/O with fp32
accumulation.  The oracle runs on the same seeded inputs, rounded to the I/O
dtype, upcast exactly to fp64.
"""
import functools
import math

import numpy as np
import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def cached_inputs(w):
    return I.make_inputs(w)


def oracle_fwd(w, x):
    return oracle.gdn_fwd_opts(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode,
                               gate_logits=w.gate_logits, norm_bc=w.norm_bc)


def check_fwd(w, x=None, want_hT=True):
    x = x or cached_inputs(w)
    o, hT = run_fwd(w, x, want_hT=want_hT)
    ro, rhT = oracle_fwd(w, x)
    tol = TOL[w.dtype]
    e = assert_close(o, ro, tol, f"{w.name} o")
    if want_hT:
        assert_close(hT, rhT, tol, f"{w.name} hT")
    return e


def check_bwd(w, x=None, dhT=None, units=None):
    """Backward parity.  `units` = list of heads to check (all batches of each
    head, so dA_log rows of those heads are complete); None = every unit (what
    every full-size workload uses)."""
    x = x or cached_inputs(w)
    got = run_bwd(w, x, dhT=dhT)
    if units is not None:
        sub = {k: (None if x[k] is None else (x[k][:, :, units] if k in ("v", "b", "c", "g", "beta", "dO")
                                               else x[k][units] if k == "A_log" else x[k][:, units]))
               for k in x}
        got_sub = {k: (None if v is None else (v[:, :, units] if k in ("dv", "db", "dc", "dg", "dbeta")
                                                else v[units] if k == "dA_log" else v[:, units]))
                   for k, v in got.items()}
        dhT_sub = None if dhT is None else dhT[:, units]
        x, got, dhT = sub, got_sub, dhT_sub
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=w.mode)
    tol = TOL[w.dtype]
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], tol, f"{w.name} {k}")


# ---------------------------------------------------------------------------
# small cases: several chunks, ragged tails, every width class, both modes
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 63, 65, 100, 256])
def test_fwd_small(mode, io, T):
    w = I.custom(name=f"small_{mode}_{io}_{T}", mode=mode, dtype=io, B=2, H=3, T=T, dk=64, dv=64, seed=T,
                 h0_std=0.3)
    check_fwd(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(8, 8), (16, 16), (56, 56), (64, 32), (32, 64), (24, 40)])
def test_fwd_widths(mode, io, dk, dv):
    w = I.custom(name=f"w_{mode}_{io}_{dk}_{dv}", mode=mode, dtype=io, B=1, H=2, T=130, dk=dk, dv=dv, seed=dk + dv)
    check_fwd(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_fwd_no_h0_no_hT_single_unit(mode):
    w = I.custom(name=f"bh1_{mode}", mode=mode, dtype="bf16", B=1, H=1, T=200, dk=64, dv=64, seed=9)
    check_fwd(w, want_hT=False)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_fwd_slow_decay(mode):
    """g ~ sigmoid(N(-4,1)): mean log-decay ~ -0.15/token, long memory."""
    w = I.custom(name=f"slow_{mode}", mode=mode, dtype="bf16", B=2, H=2, T=700, dk=64, dv=64, seed=3, g_mu=-4.0)
    check_fwd(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("g_mu", [0.0, 3.0])
def test_fwd_steep_decay(mode, g_mu):
    """|A| up to 64 and g near 1: the 8-token decay factors would overflow, so
    the kernels take their exact elementwise evaluation for those chunks."""
    w = I.custom(name=f"steep_{mode}_{g_mu}", mode=mode, dtype="bf16", B=1, H=4, T=192, dk=64, dv=64, seed=8,
                 g_mu=g_mu, alog_max=math.log(64.0), h0_std=0.2)
    check_fwd(w)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_fwd_zero_tokens(mode):
    w = I.custom(name=f"t0_{mode}", mode=mode, dtype="bf16", B=2, H=2, T=0, dk=16, dv=16, seed=1, h0_std=0.5)
    x = cached_inputs(w)
    o, hT = run_fwd(w, x)
    assert o.size == 0
    np.testing.assert_array_equal(hT, x["h0"])


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,d", [(1, 16), (37, 16), (100, 64), (129, 56)])
def test_bwd_small(mode, io, T, d):
    w = I.custom(name=f"bs_{mode}_{io}_{T}_{d}", mode=mode, dtype=io, B=2, H=2, T=T, dk=d, dv=d, seed=T + d,
                 h0_std=0.3, backward=True)
    x = cached_inputs(w)
    dhT = 0.5 * I.normal(77, 1, w.B * w.H * d * d).reshape(w.B, w.H, d, d)
    dhT = I.round_to(dhT, "f32")
    check_bwd(w, x, dhT=dhT)


def test_repeatable():
    w = I.custom(name="rep", mode="delta", dtype="bf16", B=2, H=4, T=300, dk=64, dv=64, seed=4)
    x = cached_inputs(w)
    a = run_fwd(w, x)
    b = run_fwd(w, x)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------------------
# the five workloads at full size (the launch configuration bench.py times)
# ---------------------------------------------------------------------------

def test_workload_gated_f32_1x2x128x16():
    check_fwd(I.WORKLOADS["gated_f32_1x2x128x16"])


def test_workload_gated_bf16_4x16x1024x64_h0():
    check_fwd(I.WORKLOADS["gated_bf16_4x16x1024x64_h0"])


def test_workload_delta_bf16_8x16x4096x64():
    check_fwd(I.WORKLOADS["delta_bf16_8x16x4096x64"])


def test_workload_gated_bf16_8x16x4096x64():
    check_fwd(I.WORKLOADS["gated_bf16_8x16x4096x64"])


def test_workload_gated_bf16_8x16x4096x56_fwd_bwd():
    w = I.WORKLOADS["gated_bf16_8x16x4096x56_bwd"]
    check_fwd(w)
    check_bwd(w)


def test_workload_delta_bf16_1x16x32768x64_fwd_bwd():
    w = I.WORKLOADS["delta_bf16_1x16x32768x64_bwd"]
    check_fwd(w)
    check_bwd(w)


def test_shape_40_heads_d32_fwd_bwd():
    """The production head shape (40 heads, d_k = d_v = 32) at two batch rows of 4096 tokens: forward and
    backward on every unit."""
    base = I.WORKLOADS["delta_bf16_8x40x4096x32"]
    w = base.with_(name="delta_bf16_2x40x4096x32", B=2, backward=True)
    check_fwd(w)
    check_bwd(w)


@pytest.mark.parametrize("mode,opts", [("delta", {}), ("delta", {"norm_bc": True, "gate_logits": True}),
                                       ("gated", {})])
@pytest.mark.parametrize("B,H,T,dk,dv", [(8, 40, 300, 32, 32), (4, 80, 150, 24, 16)])
def test_fwd_narrow_many_heads(mode, opts, B, H, T, dk, dv):
    """More than 304 (batch, head) units of heads at most 32 wide: delta takes the token-serial forward in bf16
    (several CTAs per SM beat three waves of the one-CTA-per-SM tensor-core kernel), gated stays on the tensor
    cores; both against the oracle on every unit."""
    w = I.custom(name=f"narrow_{mode}_{B}x{H}x{T}x{dk}x{dv}", mode=mode, dtype="bf16", B=B, H=H, T=T, dk=dk, dv=dv,
                 seed=B + H + dk, h0_std=0.3, **opts)
    check_fwd(w)


def test_fwd_40_heads_full_size():
    """The 8 x 40 x 4096 x 32 delta forward at full size (the token-serial path), every unit against the
    oracle."""
    check_fwd(I.WORKLOADS["delta_bf16_8x40x4096x32"])


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_fwd_many_units_serial(mode):
    """More (batch, head) units than a grid's y dimension holds (65535): the token-serial forward (fp32 I/O)
    indexes them on one flat grid."""
    w = I.custom(name=f"many_{mode}", mode=mode, dtype="f32", B=35000, H=2, T=11, dk=8, dv=8, seed=12, h0_std=0.3)
    check_fwd(w)
