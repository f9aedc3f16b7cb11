"""gdn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (latency-critical code that cannot pay for cudaMalloc's implicit
synchronisation, plugins inside a framework that owns all device memory,
processes that forbid allocations after start-up) get a backward whose
workspace is a fixed array inside the library.  This test calls it through
the C ABI twice in a row and checks each result against gdn_bwd with a
caller-allocated workspace, within the bf16 tolerance the parity tests use.
It sits in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

import linear_attention_recurrence_delta_gb300 as gdn
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, dev, dev32, rel_err

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("mode", ["delta", "gated"])
def test_bwd_noalloc_matches_bwd_twice(mode):
    w = I.custom(name=f"noalloc_{mode}", mode=mode, dtype="bf16", B=2, H=4, T=300, dk=64, dv=64, seed=31,
                 h0_std=0.2, backward=True)
    x = I.make_inputs(w)
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype)
    t = {k: dev(x[k], "bf16") for k in ("v", "b", "c", "g", "beta", "dO")}
    A_log, h0 = dev32(x["A_log"]), dev32(x["h0"])
    dhT = dev32(0.3 * I.normal(5, 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv))

    ref = _grads(w)
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_bwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, t["dO"], dhT, *ref.values(), ws),
              "gdn_bwd")
    torch.cuda.synchronize()
    for call in range(2):
        got = _grads(w)
        gdn.check(gdn.gdn_bwd_noalloc(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, t["dO"], dhT,
                                      *got.values()), "gdn_bwd_noalloc")
        torch.cuda.synchronize()
        for k in ref:
            if ref[k] is None:
                assert got[k] is None
                continue
            a = got[k].double().cpu().numpy()
            r = ref[k].double().cpu().numpy()
            assert np.isfinite(a).all(), (call, k)
            assert rel_err(a, r) <= TOL["bf16"], (call, k, rel_err(a, r))


def test_bwd_noalloc_rejects_oversized_shape():
    # 16 heads x 65536 tokens needs far more than the fixed 32 MiB array
    s = gdn.make_shape(1, 16, 65536, 64, 64, "delta", "bf16")
    assert gdn.gdn_workspace_bytes(s, 1) > (32 << 20)
    fake = 1 << 20
    st = gdn.gdn_bwd_noalloc(s, fake, fake, fake, fake, fake, fake, None, fake, None, fake, fake, fake, fake, fake,
                             fake, None)
    assert st == 5  # GDN_ERR_WORKSPACE, nothing enqueued
