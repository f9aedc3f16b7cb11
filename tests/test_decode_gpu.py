"""Short-sequence forward (1 <= T <= 8, the decoding case) against the fp64 oracle.

The library sends these lengths to a kernel of their own; the state comes in
through h0 and goes out through hT, which may be the same buffer.  Bar: the
parity tolerance of the other forward tests (1e-5 for f32 I/O, 5e-3 for bf16).
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
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 3, 8])
@pytest.mark.parametrize("dk,dv", [(64, 64), (56, 56), (24, 40)])
def test_decode_parity(mode, io, T, dk, dv):
    w = I.custom(name=f"dec_{mode}_{io}_{T}_{dk}_{dv}", mode=mode, dtype=io, B=3, H=5, T=T, dk=dk, dv=dv,
                 seed=100 + T + dk, h0_std=0.3, b_dist="l2norm" if mode == "delta" else "normal/8",
                 c_dist="l2norm")
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle_fwd(w, x)
    assert_close(o, ro, TOL[io], f"{w.name} o")
    assert_close(hT, rhT, TOL[io], f"{w.name} hT")


@pytest.mark.parametrize("dk,dv", [(5, 7), (13, 3)])
def test_decode_odd_widths_f32(dk, dv):
    """f32 rows whose width is no multiple of four take the element-wise state path."""
    w = I.custom(name=f"dec_odd_{dk}_{dv}", mode="delta", dtype="f32", B=2, H=3, T=2, dk=dk, dv=dv, seed=dk * dv,
                 h0_std=0.5, b_dist="l2norm", c_dist="l2norm")
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle_fwd(w, x)
    assert_close(o, ro, TOL["f32"], "o")
    assert_close(hT, rhT, TOL["f32"], "hT")


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_decode_loop_in_place(mode, io):
    """Twenty one-token calls on one state buffer (hT is h0) reproduce the oracle's
    twenty-token sequence: every output and the final state."""
    steps = 20
    w = I.custom(name=f"loop_{mode}_{io}", mode=mode, dtype=io, B=2, H=4, T=steps, dk=64, dv=64, seed=77,
                 h0_std=0.2, b_dist="l2norm" if mode == "delta" else "normal/8", c_dist="l2norm")
    x = I.make_inputs(w)
    ro, rhT = oracle_fwd(w, x)
    s1 = gdn.make_shape(w.B, w.H, 1, w.dk, w.dv, w.mode, w.dtype)
    state = dev32(x["h0"])
    A_log = dev32(x["A_log"])
    ws = torch.empty(gdn.gdn_workspace_bytes(s1, 0), dtype=torch.uint8, device="cuda")
    outs = []
    for t in range(steps):
        step = {k: (None if x[k] is None else dev(np.ascontiguousarray(x[k][:, t:t + 1]), io))
                for k in ("v", "b", "c", "g", "beta")}
        o = torch.empty((w.B, 1, w.H, w.dv), dtype=tdtype(io), device="cuda")
        gdn.check(gdn.gdn_fwd(s1, step["v"], step["b"], step["c"], step["g"], step["beta"], A_log, state, o, state,
                              ws), "gdn_fwd step")
        outs.append(o.double().cpu().numpy())
    got = np.concatenate(outs, axis=1)
    assert_close(got, ro, TOL[io], "o over the loop")
    assert_close(state.double().cpu().numpy(), rhT, TOL[io], "state after the loop")


def test_decode_workload_sample():
    """The bench's decode workload (512 x 16 heads, one token, bf16): every output
    and the states of a sample of heads."""
    w = I.WORKLOADS["delta_bf16_decode_512x16x1x64"]
    x = I.make_inputs(w)
    o, hT = run_fwd(w, x)
    ro, rhT = oracle_fwd(w, x)
    assert_close(o, ro, TOL["bf16"], "o")
    assert_close(hT, rhT, TOL["bf16"], "hT")
