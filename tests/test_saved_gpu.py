"""gdn_fwd_save / gdn_bwd_saved through the C ABI: the forward keeps what the chunked backward would recompute
(the state entering every chunk of 64 tokens and the results of the chunk's delta solve, or in gated mode the
scores P), and the backward reads it.  Output, final state and every gradient against the fp64 oracle, on shapes
with several chunks, ragged last chunks and the widths the tensor-core path takes, with and without h0 and dh_T,
and on chunks whose decay factors would overflow (the exact elementwise path).  The gradients are also compared with gdn_bwd's, which recomputes
everything: the two must agree to within the bf16 tolerance of each other."""
import math

import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I
import linear_attention_recurrence_delta_gb300 as gdn
from tests.gdn_testlib import TOL, assert_close, run_bwd, run_saved, shape_of

pytestmark = pytest.mark.gpu

KEYS = ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0")


def check_saved(w, with_dhT=True):
    x = I.make_inputs(w)
    dhT = None
    if with_dhT:
        dhT = I.round_to(0.5 * I.normal(w.seed + 7, 1, w.B * w.H * w.dk * w.dv).reshape(w.B, w.H, w.dk, w.dv),
                         "f32")
    o, hT, got = run_saved(w, x, dhT)
    tol = TOL["bf16"]
    ro, rhT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)
    assert_close(o, ro, tol, f"{w.name} o")
    assert_close(hT, rhT, tol, f"{w.name} hT")
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=w.mode)
    plain = run_bwd(w, x, dhT=dhT)
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_close(got[k], ref[k], tol, f"{w.name} {k} vs oracle")
        assert_close(got[k], plain[k], tol, f"{w.name} {k} vs gdn_bwd")


@pytest.mark.parametrize("mode", ["delta", "gated"])
@pytest.mark.parametrize("B,H,T,d", [(1, 2, 64, 64), (2, 3, 300, 64), (2, 2, 100, 56), (2, 2, 37, 16),
                                     (1, 3, 129, 32), (4, 16, 1024, 64)])
@pytest.mark.parametrize("h0_std", [0.0, 0.3])
def test_saved_matches_oracle(mode, B, H, T, d, h0_std):
    w = I.custom(name=f"saved_{mode}_{B}x{H}x{T}x{d}_{h0_std}", mode=mode, dtype="bf16", B=B, H=H, T=T, dk=d, dv=d,
                 seed=3 + T + d, h0_std=h0_std, backward=True)
    check_saved(w, with_dhT=h0_std > 0)


def test_saved_narrow_heads_many_units():
    """320 narrow delta heads (d = 32, the 40-head production shape at 8 batch rows): gdn_fwd takes the token-serial
    kernel there, but the saving forward runs the tensor-core one and keeps the residuals."""
    w = I.custom(name="saved_narrow_8x40x512x32", mode="delta", dtype="bf16", B=8, H=40, T=512, dk=32, dv=32, seed=41,
                 h0_std=0.2, backward=True)
    assert gdn.gdn_plan(shape_of(w), 0).fwd_kernel == gdn.GDN_KERNEL_SERIAL
    assert gdn.gdn_saved_bytes(shape_of(w)) > 0
    check_saved(w)


@pytest.mark.parametrize("mode", ["delta", "gated"])
@pytest.mark.parametrize("g_mu", [0.0, 3.0])
def test_saved_steep_decay(mode, g_mu):
    """|A| up to 64 and g near 1: the forward evaluates those chunks' decay factors elementwise."""
    w = I.custom(name=f"saved_steep_{mode}_{g_mu}", mode=mode, dtype="bf16", B=1, H=4, T=192, dk=64, dv=64, seed=8,
                 g_mu=g_mu, alog_max=math.log(64.0), h0_std=0.2, backward=True)
    check_saved(w)


@pytest.mark.parametrize("mode", ["delta", "gated"])
@pytest.mark.parametrize("B,H,T,d", [(1, 4, 2048, 64), (2, 3, 3072, 56), (1, 2, 4096, 32),
                                     (1, 3, 2496, 64),     # 39 chunks: segments of 10, the last of 9
                                     (2, 5, 3001, 48)])    # 47 chunks, the last of 57 tokens: 10, 10, 10, 10, 7
def test_saved_split_forward(mode, B, H, T, d):
    """Long sequences over few heads: the forward splits in time into segments of whole chunks (any length: the
    last segment may be shorter and its last chunk ragged) and runs them by walks (zero-start runs keeping their
    residuals, the segments' transitions, a scan, the walks of T_k S_s writing the outputs, and a fix-up that makes
    the residuals true; gated heads' transitions are diagonal); gdn_bwd_saved then reads those residuals."""
    w = I.custom(name=f"saved_split_{mode}_{B}x{H}x{T}x{d}", mode=mode, dtype="bf16", B=B, H=H, T=T, dk=d, dv=d,
                 seed=5 + T + d, h0_std=0.3, backward=True)
    assert gdn.gdn_plan(shape_of(w), 0).segments > 1 and gdn.gdn_saved_bytes(shape_of(w)) > 0
    check_saved(w)


@pytest.mark.parametrize("name", ["delta_bf16_8x16x4096x64", "gated_bf16_8x16x4096x56_bwd",
                                  "delta_bf16_1x16x32768x64_bwd"])
def test_saved_full_size(name):
    """The bench's training step (8 x 16 x 4096 x 64, delta), the gated 8 x 16 x 4096 x 56 workload and the
    long-context 1 x 16 x 32768 x 64 one (forward split in time by walks) at full size, every unit: o, h_T and every gradient from the residuals against the fp64 oracle, and the gradients against
    gdn_bwd's, within the bf16 tolerance."""
    w = I.WORKLOADS[name].with_(backward=True)
    x = I.make_inputs(w)
    o, hT, got = run_saved(w, x, None)
    tol = TOL["bf16"]
    ro, rhT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=w.mode)
    assert_close(o, ro, tol, "o vs oracle")
    assert_close(hT, rhT, tol, "hT vs oracle")
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None, mode=w.mode)
    plain = run_bwd(w, x, dhT=None)
    for k in KEYS:
        if ref[k] is None:
            assert got[k] is None and plain[k] is None
            continue
        assert_close(got[k], ref[k], tol, f"{k} from residuals vs oracle")
        assert_close(plain[k], ref[k], tol, f"{k} (gdn_bwd) vs oracle")
        assert_close(got[k], plain[k], tol, f"{k} from residuals vs gdn_bwd")
