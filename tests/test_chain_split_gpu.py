"""The chunked backward's chain split in time (few (batch, head) units, at least 32 chunks), both modes.

The chunk map S' = Phi S + Delta is affine ("GDN & MLA Mechanism Deep-Dive", Step 5: chunked recurrence), so the
chain over the chunk boundaries runs as segments side by side (gated: Phi = diag(E), all elementwise, the records
fixed up by the segment's decay products; delta as follows): a first walk per segment from zero, carrying its own
transition, then a second from the segment's true start, writing the per-chunk records; the two are joined by
a scan over the segments; the forward and reverse sweeps run side by side.  These shapes make 1 to 4 segments, with a
last segment shorter than the others and a ragged last chunk; every gradient (dh0 included, which the reverse walk
over the first segment writes) against the fp64 oracle, through gdn_bwd and, where the forward is one tensor-core
pass, through gdn_fwd_save + gdn_bwd_saved (the reverse sweep alone)."""
import pytest

import linear_attention_recurrence_delta_gb300 as gdn
import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_saved, shape_of

pytestmark = pytest.mark.gpu

KEYS = ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0")


@pytest.mark.parametrize("mode", ["delta", "gated"])
@pytest.mark.parametrize("B,H,T,d,nseg,saved", [
    (1, 2, 4096, 64, 4, False),     # 64 chunks: 4 x 16
    (1, 1, 3150, 64, 3, False),     # 50 chunks, the last 14 tokens: 17, 17, 16
    (2, 3, 2100, 56, 2, False),     # 33 chunks: 17, 16
    (1, 16, 9000, 32, 4, False),    # 141 chunks over 16 heads: 36, 36, 36, 33
    # residuals exist where the forward is one pass (39 units or more); the reverse sweep alone splits
    (1, 40, 2048, 64, 2, True),     # 32 chunks: 16, 16
    (1, 48, 4050, 32, 3, True),     # 64 chunks, the last 18 tokens: 22, 22, 20
    # no split, the two sweeps side by side
    (1, 40, 2048, 64, 1, False), (2, 5, 1000, 64, 1, False),
])
def test_split_chain_matches_oracle(mode, B, H, T, d, nseg, saved):
    w = I.custom(name=f"chain_split_{mode}_{B}x{H}x{T}x{d}", mode=mode, dtype="bf16", B=B, H=H, T=T, dk=d, dv=d,
                 seed=11 + T, h0_std=0.3, backward=True)
    assert gdn.gdn_plan(shape_of(w), 2 if saved else 1).segments == nseg
    x = I.make_inputs(w)
    dhT = I.round_to(0.5 * I.normal(w.seed + 7, 1, B * H * d * d).reshape(B, H, d, d), "f32")
    tol = TOL["bf16"]
    if saved:
        assert gdn.gdn_saved_bytes(shape_of(w)) > 0
        o, hT, got = run_saved(w, x, dhT)
        ro, rhT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode)
        assert_close(o, ro, tol, "o")
        assert_close(hT, rhT, tol, "hT")
    else:
        got = run_bwd(w, x, dhT=dhT)
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=mode)
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], tol, f"{w.name} {k}")
