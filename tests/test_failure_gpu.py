"""The failure path of the bounded device waits, exercised without faulting the GPU.

Every wait of the tcgen05 forward (a chunk's loads, the tensor-core products) has a
time limit; on expiry the kernel records GDN_ERR_TIMEOUT in the workspace status
word, lets the copies it issued land, frees its tensor memory and returns.  The
test makes a wait run out by the library's test hook GDN_TEST_STARVE_CHUNK=k (the
loads of chunk k are never issued, so nothing ever completes that stage; the
library reads the variable once per process, so the case runs in a child process)
and checks the status the host reads, the time it took, and that the same
context then runs a normal forward to parity.
"""
import time

import numpy as np
import pytest
import torch

import linear_attention_recurrence_delta_gb300 as gdn
import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, dev, dev32, run_fwd, shape_of, tdtype

pytestmark = pytest.mark.gpu

GDN_ERR_TIMEOUT = 7


def fwd_raw(w, x):
    """gdn_fwd without the status check: returns (call status, device status, seconds)."""
    s = shape_of(w)
    t = {k: dev(x[k], w.dtype) for k in ("v", "b", "c", "g", "beta")}
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=tdtype(w.dtype), device="cuda")
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = gdn.gdn_fwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], dev32(x["A_log"]), None, o, hT, ws)
    st = gdn.gdn_last_device_status(ws)
    return rc, st, time.perf_counter() - t0


_STARVE_CHILD = r"""
import json, sys, time
import torch
import linear_attention_recurrence_delta_gb300 as gdn
import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, rel_err, run_fwd
from tests.test_failure_gpu import fwd_raw
mode, chunk = sys.argv[1], int(sys.argv[2])
w = I.custom(name=f"starve_{mode}_{chunk}", mode=mode, dtype="bf16", B=2, H=4, T=256, dk=64, dv=64, seed=3)
x = I.make_inputs(w)
rc, st, secs = fwd_raw(w, x)
# chunk `chunk` of every tensor-core forward in this process starves; a one-chunk sequence never reaches it
w1 = w.with_(name="after", T=64)
x1 = I.make_inputs(w1)
o, hT = run_fwd(w1, x1)
ro, rhT = oracle.gdn_fwd(x1["v"], x1["b"], x1["c"], x1["g"], x1["beta"], x1["A_log"], None, mode=mode)
print(json.dumps({"rc": rc, "st": st, "secs": secs, "o": rel_err(o, ro), "hT": rel_err(hT, rhT)}))
"""


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("chunk", [1, 3])
def test_starved_load_times_out_and_context_survives(mode, chunk):
    """The hook is read once per process, so each case runs in a child process started with it set."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GDN_TEST_STARVE_CHUNK=str(chunk), PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", _STARVE_CHILD, mode, str(chunk)], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["rc"] == gdn.GDN_OK               # the launch itself succeeded
    assert res["st"] == GDN_ERR_TIMEOUT          # the device reported the expired wait
    assert res["secs"] < 10.0
    assert res["o"] <= TOL["bf16"] and res["hT"] <= TOL["bf16"]   # the context is still usable


def test_stale_status_word_is_cleared():
    """A status word left poisoned in the workspace by an earlier call does not leak into the next one."""
    w = I.custom(name="poison", mode="delta", dtype="bf16", B=1, H=2, T=130, dk=64, dv=64, seed=8)
    x = I.make_inputs(w)
    s = shape_of(w)
    t = {k: dev(x[k], w.dtype) for k in ("v", "b", "c", "g", "beta")}
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")
    ws[:8].view(torch.int32)[0] = GDN_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert gdn.gdn_last_device_status(ws) != gdn.GDN_OK
    rc = gdn.gdn_fwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], dev32(x["A_log"]), None, o, None, ws)
    assert rc == gdn.GDN_OK
    assert gdn.gdn_last_device_status(ws) == gdn.GDN_OK
    ro, _ = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], None, mode="delta")
    assert_close(o.double().cpu().numpy(), ro, TOL["bf16"], "o")


GDN_ERR_NONFINITE = 9


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_check_finite_flags_nan_outputs(mode, io):
    """GDN_CHECK_FINITE: a NaN in one value element reaches the outputs, and the status word says so; clean
    inputs leave it GDN_OK; without the bit nothing is checked."""
    w = I.custom(name=f"fin_{mode}_{io}", mode=mode, dtype=io, B=1, H=2, T=100, dk=64, dv=64, seed=21)
    x = I.make_inputs(w)
    bad = dict(x)
    bad["v"] = x["v"].copy()
    bad["v"][0, 37, 1, 5] = np.nan

    def status(inputs, check):
        s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, mode, io, check_finite=check)
        t = {k: dev(inputs[k], io) for k in ("v", "b", "c", "g", "beta")}
        o = torch.empty((w.B, w.T, w.H, w.dv), dtype=tdtype(io), device="cuda")
        hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
        ws = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")
        gdn.check(gdn.gdn_fwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], dev32(inputs["A_log"]), None, o, hT, ws))
        return gdn.gdn_last_device_status(ws)

    assert status(x, True) == gdn.GDN_OK
    assert status(bad, True) == GDN_ERR_NONFINITE
    assert status(bad, False) == gdn.GDN_OK


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_check_finite_backward(mode):
    """The backward's check covers every gradient: a NaN in one output-gradient element is reported."""
    w = I.custom(name=f"finb_{mode}", mode=mode, dtype="bf16", B=1, H=2, T=70, dk=32, dv=32, seed=22,
                 backward=True)
    x = I.make_inputs(w)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv

    def status(dO):
        s = gdn.make_shape(B, H, T, dk, dv, mode, "bf16", check_finite=True)
        t = {k: dev(x[k], "bf16") for k in ("v", "b", "c", "g", "beta")}
        g = {k: torch.empty(sh, dtype=torch.bfloat16, device="cuda") for k, sh in
             (("dv", (B, T, H, dv)), ("db", (B, T, H, dk)), ("dc", (B, T, H, dk)), ("dg", (B, T, H)))}
        dbeta = torch.empty((B, T, H), dtype=torch.bfloat16, device="cuda") if mode == "delta" else None
        dA = torch.empty((H, dk), dtype=torch.float32, device="cuda")
        ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
        gdn.check(gdn.gdn_bwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], dev32(x["A_log"]), None,
                              dev(dO, "bf16"), None, g["dv"], g["db"], g["dc"], g["dg"], dbeta, dA, None, ws))
        return gdn.gdn_last_device_status(ws)

    assert status(x["dO"]) == gdn.GDN_OK
    bad = x["dO"].copy()
    bad[0, 50, 1, 3] = np.inf
    assert status(bad) == GDN_ERR_NONFINITE
