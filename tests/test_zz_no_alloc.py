"""gdn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (latency-critical code that cannot pay for cudaMalloc's implicit
synchronisation, plugins inside a framework that owns all device memory,
processes that forbid allocations after start-up) get a backward whose
workspace is a fixed array inside the library, shared by every call on the
device.  These tests call it through the C ABI: first on another shape so the
array holds other data, then twice in a row on a shape the chunked tensor-core
backward takes and on one the token-serial backward splits in time (logit
gates), each result bit for bit equal to gdn_bwd with a caller-allocated
workspace (the same kernels run) and within the bf16 tolerance of the fp64
oracle.  They also check its error codes and
the status query that reads the array's status word.  The file is collected
last, so a run that stops at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_delta_gb300 as gdn
import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, dev, dev32

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 32 << 20
GDN_ERR_NULL, GDN_ERR_SHAPE, GDN_ERR_MODE, GDN_ERR_WORKSPACE, GDN_ERR_NONFINITE = 1, 2, 4, 5, 9
KEYS = ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0")


def _grads(w):
    dt = torch.bfloat16
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv
    return {
        "dv": torch.full((B, T, H, dv), float("nan"), dtype=dt, device="cuda"),
        "db": torch.full((B, T, H, dk), float("nan"), dtype=dt, device="cuda"),
        "dc": torch.full((B, T, H, dk), float("nan"), dtype=dt, device="cuda"),
        "dg": torch.full((B, T, H), float("nan"), dtype=dt, device="cuda"),
        "dbeta": torch.full((B, T, H), float("nan"), dtype=dt, device="cuda") if w.mode == "delta" else None,
        "dA_log": torch.full((H, dk), float("nan"), dtype=torch.float32, device="cuda"),
        "dh0": torch.full((B, H, dk, dv), float("nan"), dtype=torch.float32, device="cuda"),
    }


def _case(w):
    x = I.make_inputs(w)
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype, gate_logits=w.gate_logits)
    t = {k: dev(x[k], "bf16") for k in ("v", "b", "c", "g", "beta", "dO")}
    A_log, h0 = dev32(x["A_log"]), dev32(x["h0"])
    dhT_np = I.round_to(0.3 * I.normal(w.seed + 5, 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv),
                        "f32")
    return x, s, t, A_log, h0, dhT_np


def _noalloc(s, t, A_log, h0, dhT, got):
    return gdn.gdn_bwd_noalloc(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, t["dO"], dhT,
                               *got.values())


def _split_shape(mode):
    """A shape (with logit gates, so the token-serial backward runs) that the library splits in time and whose
    workspace fits the fixed array."""
    for B, H, T in ((1, 4, 2048), (1, 2, 2048), (1, 2, 1024), (1, 1, 2048)):
        s = gdn.make_shape(B, H, T, 64, 64, mode, "bf16", gate_logits=True)
        if gdn.gdn_plan(s, 1).segments > 1 and gdn.gdn_workspace_bytes(s, 1) <= NOALLOC_BYTES:
            return B, H, T
    return None


@pytest.mark.parametrize("mode", ["delta", "gated"])
def test_bwd_noalloc_matches_bwd_and_oracle(mode):
    # another shape and seed first, so that the shared array holds the leftovers of a different call
    wd = I.custom(name=f"noalloc_dirty_{mode}", mode=mode, dtype="bf16", B=3, H=3, T=200, dk=64, dv=64, seed=77,
                  h0_std=0.5, backward=True)
    _, sd, td, Ad, hd, dhd = _case(wd)
    gdn.check(_noalloc(sd, td, Ad, hd, dev32(dhd), _grads(wd)), "gdn_bwd_noalloc (other shape)")
    torch.cuda.synchronize()

    split = _split_shape(mode)
    assert split is not None, "no split shape fits the fixed array"
    for (B, H, T), logits in (((2, 4, 300), False), (split, True)):
        w = I.custom(name=f"noalloc_{mode}_{B}x{H}x{T}", mode=mode, dtype="bf16", B=B, H=H, T=T, dk=64, dv=64,
                     seed=31 + T, h0_std=0.2, backward=True, gate_logits=logits)
        x, s, t, A_log, h0, dhT_np = _case(w)
        assert gdn.gdn_workspace_bytes(s, 1) <= NOALLOC_BYTES
        want_kernel = gdn.GDN_BWD_SERIAL if logits else gdn.GDN_BWD_TENSOR_CORE
        assert gdn.gdn_plan(s, 1).bwd_kernel == want_kernel
        dhT = dev32(dhT_np)
        ref = _grads(w)
        ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
        gdn.check(gdn.gdn_bwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, t["dO"], dhT,
                              *ref.values(), ws), "gdn_bwd")
        torch.cuda.synchronize()
        want = oracle.gdn_bwd_opts(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT_np,
                                   mode=mode, gate_logits=logits)
        for call in range(2):
            got = _grads(w)
            gdn.check(_noalloc(s, t, A_log, h0, dhT, got), "gdn_bwd_noalloc")
            assert gdn.gdn_bwd_noalloc_status() == gdn.GDN_OK
            for k in KEYS:
                if ref[k] is None:
                    assert got[k] is None
                    continue
                a = got[k].double().cpu().numpy()
                r = ref[k].double().cpu().numpy()
                np.testing.assert_array_equal(a, r, err_msg=f"{(B, H, T)} call {call} {k}")
                assert_close(a, want[k], TOL["bf16"], f"{(B, H, T)} call {call} {k} vs oracle")


def test_bwd_noalloc_error_codes():
    fake = 1 << 20
    args = (fake, fake, fake, fake, fake, fake, None, fake, None, fake, fake, fake, fake, fake, fake, None)
    # 16 heads x 65536 tokens needs far more than the fixed array
    s = gdn.make_shape(1, 16, 65536, 64, 64, "delta", "bf16")
    assert gdn.gdn_workspace_bytes(s, 1) > NOALLOC_BYTES
    assert gdn.gdn_bwd_noalloc(s, *args) == GDN_ERR_WORKSPACE
    # the shape's own errors come first and match gdn_bwd's
    bad_mode = gdn.make_shape(1, 2, 64, 64, 64, 7, "bf16")
    assert gdn.gdn_bwd_noalloc(bad_mode, *args) == GDN_ERR_MODE
    unknown_bit = gdn.make_shape(1, 2, 64, 64, 64, gdn.GDN_DELTA | 0x800, "bf16")
    assert gdn.gdn_bwd_noalloc(unknown_bit, *args) == GDN_ERR_MODE
    bad_io = gdn.make_shape(1, 2, 64, 64, 64, "delta", 5)
    assert gdn.gdn_bwd_noalloc(bad_io, *args) == GDN_ERR_MODE
    bad_shape = gdn.make_shape(0, 2, 64, 64, 64, "delta", "bf16")
    assert gdn.gdn_bwd_noalloc(bad_shape, *args) == GDN_ERR_SHAPE
    odd_width = gdn.make_shape(1, 2, 64, 60, 64, "delta", "bf16")
    assert gdn.gdn_bwd_noalloc(odd_width, *args) == GDN_ERR_SHAPE
    # nothing was enqueued and no CUDA error is left pending
    torch.cuda.synchronize()
    torch.zeros(4, device="cuda").add_(1)
    torch.cuda.synchronize()


def test_bwd_noalloc_status_reports_nonfinite():
    """With GDN_CHECK_FINITE the non-finite flag lands in the fixed array; the status query reads it."""
    w = I.custom(name="noalloc_fin", mode="delta", dtype="bf16", B=1, H=2, T=70, dk=32, dv=32, seed=22,
                 backward=True)
    x = I.make_inputs(w)
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, "delta", "bf16", check_finite=True)
    t = {k: dev(x[k], "bf16") for k in ("v", "b", "c", "g", "beta", "dO")}
    A_log = dev32(x["A_log"])
    gdn.check(_noalloc(s, t, A_log, None, None, _grads(w)))
    assert gdn.gdn_bwd_noalloc_status() == gdn.GDN_OK
    bad = x["dO"].copy()
    bad[0, 50, 1, 3] = np.inf
    t["dO"] = dev(bad, "bf16")
    gdn.check(_noalloc(s, t, A_log, None, None, _grads(w)))
    assert gdn.gdn_bwd_noalloc_status() == GDN_ERR_NONFINITE
    # the next clean call clears it
    t["dO"] = dev(x["dO"], "bf16")
    gdn.check(_noalloc(s, t, A_log, None, None, _grads(w)))
    assert gdn.gdn_bwd_noalloc_status() == gdn.GDN_OK
