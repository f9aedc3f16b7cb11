"""Seeded random shapes and options, forward and backward, against the fp64 oracle.

The hand-written cases cover each feature; these draw combinations of them: both modes and I/O dtypes, widths up
to 128 (any width for fp32 I/O, multiples of 8 for bf16), equal or not, ragged sequence lengths from 1 to 300 and
some long ones (1536, 2048 tokens over few heads: the time split, when the widths allow it), with or without an
initial state and an end gradient, with or without the option bits GDN_GATE_LOGITS and
GDN_NORM_BC.  The draws come from a fixed seed, so every run checks the same cases.  Bar: the tolerance of the
other parity tests (1e-5 of max|ref| for fp32 I/O, 5e-3 for bf16).
"""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_fwd

pytestmark = pytest.mark.gpu


def draw_cases(n, seed=20261203):
    rng = np.random.RandomState(seed)
    cases = []
    for k in range(n):
        io = ["f32", "bf16"][rng.randint(2)]
        mode = ["gated", "delta"][rng.randint(2)]
        step = 8 if io == "bf16" else 1
        dk = int(step * rng.randint(1, 128 // step + 1))
        dv = int(step * rng.randint(1, 128 // step + 1))
        T = int(rng.choice([1, 2, 7, 8, 9, 63, 64, 65, 100, 129, 200, 300, 1536, 2048]))
        if T >= 1536:   # few heads and at most 64 wide, so that the time split can take it
            dk, dv = min(dk, 64), min(dv, 64)
        cases.append(dict(k=k, io=io, mode=mode, B=int(rng.randint(1, 4)), H=int(rng.randint(1, 5)), T=T, dk=dk,
                          dv=dv, h0=bool(rng.randint(2)), dhT=bool(rng.randint(2)), logits=bool(rng.randint(2)),
                          norm=bool(rng.randint(2))))
    return cases


CASES = draw_cases(96)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['k']}-{c['mode']}-{c['io']}-T{c['T']}-{c['dk']}x{c['dv']}")
def test_fuzz_fwd_bwd(case):
    c = case
    w = I.custom(name=f"fuzz{c['k']}", mode=c["mode"], dtype=c["io"], B=c["B"], H=c["H"], T=c["T"], dk=c["dk"],
                 dv=c["dv"], seed=1000 + c["k"], h0_std=0.3 if c["h0"] else 0.0, backward=True,
                 gate_logits=c["logits"], norm_bc=c["norm"],
                 b_dist="normal" if c["norm"] else ("l2norm" if c["mode"] == "delta" else "normal/8"),
                 c_dist="normal" if c["norm"] else "l2norm")
    x = I.make_inputs(w)
    tol = TOL[c["io"]]
    kw = dict(mode=w.mode, gate_logits=c["logits"], norm_bc=c["norm"])
    o, hT = run_fwd(w, x)
    ro, rhT = oracle.gdn_fwd_opts(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], **kw)
    assert_close(o, ro, tol, "o")
    assert_close(hT, rhT, tol, "hT")
    dhT = None
    if c["dhT"]:
        dhT = I.round_to(0.5 * I.normal(2000 + c["k"], 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv),
                         "f32")
    got = run_bwd(w, x, dhT=dhT)
    ref = oracle.gdn_bwd_opts(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, **kw)
    for key in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[key] is None:
            assert got[key] is None
            continue
        assert_close(got[key], ref[key], tol, key)
