"""CPU-side checks of the C ABI: the library loads, exports every function
include/gdn.h declares, sizes workspaces, and rejects bad arguments before
touching any device (no compute call is made without a GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

import linear_attention_recurrence_delta_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", txt))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(gdn.LIB_PATH):
        from linear_attention_recurrence_delta_gb300 import _build
        _build.build()
    return gdn.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gdn_fwd", "gdn_bwd", "gdn_workspace_bytes", "gdn_last_device_status", "gdn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code, name in gdn.STATUS_NAMES.items():
        assert gdn.gdn_status_string(code).startswith(name)


def test_workspace_sizes(lib):
    s = gdn.make_shape(8, 16, 4096, 64, 64, "delta", "bf16")
    f = gdn.gdn_workspace_bytes(s, 0)
    b = gdn.gdn_workspace_bytes(s, 1)
    assert f >= 256 and f % 256 == 0
    assert b > f and b % 256 == 0
    assert gdn.gdn_workspace_bytes(gdn.make_shape(1, 1, 0, 8, 8), 1) >= 256
    for bad in (gdn.make_shape(0, 1, 8, 8, 8), gdn.make_shape(1, 1, 8, 129, 8), gdn.make_shape(1, 1, 8, 8, 0),
                gdn.make_shape(1, 1, 8, 8, 136, "delta", "bf16"), gdn.make_shape(1 << 14, 1 << 13, 1, 8, 8),
                gdn.make_shape(1, 1, -1, 8, 8), gdn.make_shape(1, 1, 8, 12, 8, "gated", "bf16"),
                gdn.make_shape(1, 1, 8, 8, 8, 7, "bf16"), gdn.make_shape(1, 1, 8, 8, 8, "gated", 5)):
        assert gdn.gdn_workspace_bytes(bad, 0) == 0


FAKE = 1 << 20   # a 256-byte aligned non-null address; never dereferenced


def fwd_args(**kw):
    a = dict(v=FAKE, b=FAKE, c=FAKE, g=FAKE, beta=None, A_log=FAKE, h0=None, o=FAKE, hT=None, ws=FAKE,
             ws_bytes=1 << 30)
    a.update(kw)
    return a


def call_fwd(shape, a):
    return gdn.gdn_fwd(shape, a["v"], a["b"], a["c"], a["g"], a["beta"], a["A_log"], a["h0"], a["o"], a["hT"],
                       a["ws"], ws_bytes=a["ws_bytes"], stream=0)


def test_fwd_rejects_bad_arguments_before_any_device_work(lib):
    s = gdn.make_shape(2, 2, 64, 16, 16, "gated", "bf16")
    assert call_fwd(s, fwd_args(v=None)) == 1                     # NULL input
    assert call_fwd(s, fwd_args(o=None)) == 1                     # NULL output
    assert call_fwd(s, fwd_args(ws=None)) == 5                    # no workspace
    assert call_fwd(s, fwd_args(ws_bytes=16)) == 5                # workspace too small
    assert call_fwd(s, fwd_args(beta=FAKE)) == 4                  # beta in gated mode
    sd = gdn.make_shape(2, 2, 64, 16, 16, "delta", "bf16")
    assert call_fwd(sd, fwd_args()) == 4                          # beta missing in delta mode
    assert call_fwd(s, fwd_args(v=FAKE + 2)) == 3                 # misaligned bf16 tensor
    assert call_fwd(s, fwd_args(ws=FAKE + 16)) == 3               # misaligned workspace
    assert call_fwd(gdn.make_shape(2, 2, 64, 12, 16, "gated", "bf16"), fwd_args()) == 2
    assert call_fwd(gdn.make_shape(2, 2, 64, 16, 132, "gated", "f32"), fwd_args()) == 2
    assert call_fwd(gdn.make_shape(0, 2, 64, 16, 16, "gated", "f32"), fwd_args()) == 2
    assert call_fwd(gdn.make_shape(2, 2, 64, 16, 16, 3, "f32"), fwd_args()) == 4


def test_bwd_rejects_bad_arguments_before_any_device_work(lib):
    s = gdn.make_shape(2, 2, 64, 16, 16, "delta", "f32")

    def call(**kw):
        a = dict(v=FAKE, b=FAKE, c=FAKE, g=FAKE, beta=FAKE, A_log=FAKE, h0=None, dO=FAKE, dhT=None, dv=FAKE,
                 db=FAKE, dc=FAKE, dg=FAKE, dbeta=FAKE, dA_log=FAKE, dh0=None, ws=FAKE, ws_bytes=1 << 40)
        a.update(kw)
        ws_bytes = a.pop("ws_bytes")
        return gdn.gdn_bwd(s, *a.values(), ws_bytes=ws_bytes, stream=0)

    assert call(dO=None) == 1
    assert call(dA_log=None) == 1
    assert call(dbeta=None) == 4
    assert call(ws_bytes=256) == 5
    assert call(dA_log=FAKE + 4) == 3
    assert call(b=FAKE + 2) == 3


def test_wide_head_workspace(lib):
    """Heads up to 128 wide: the forward needs no workspace; the backward's buffers grow with its column slabs
    (64 value columns per CTA up to d_k = 64, 32 above), and with more than one slab it adds fp32 partial sums
    of db, dc [slabs, B, T, H, d_k] and dg, dbeta [slabs, B, T, H]."""
    B, H, T = 2, 4, 256
    assert gdn.gdn_workspace_bytes(gdn.make_shape(B, H, T, 128, 128, "delta", "bf16"), 0) == 256
    # (logit gates keep the 64-wide head on the token-serial backward, whose buffers this compares)
    one = gdn.gdn_workspace_bytes(gdn.make_shape(B, H, T, 64, 64, "delta", "bf16", gate_logits=True), 1)
    two = gdn.gdn_workspace_bytes(gdn.make_shape(B, H, T, 64, 128, "delta", "bf16"), 1)
    four = gdn.gdn_workspace_bytes(gdn.make_shape(B, H, T, 128, 128, "delta", "bf16"), 1)
    ntok = B * T * H
    assert two >= 2 * (one - 256) + 2 * ntok * (2 * 64 + 2) * 4
    assert four >= 4 * ntok * (2 * 128 + 2) * 4 + 4 * B * H * (T // 32) * 4 * 16384
    # d_k = 128 with d_v = 32: one slab, no partial sums -- status word, snapshots every 8 tokens (16 KB),
    # x and v - h'^T b of every token on 32 columns, dA_log partials
    narrow = gdn.gdn_workspace_bytes(gdn.make_shape(B, H, T, 128, 32, "delta", "bf16"), 1)
    assert narrow == 256 + B * H * (T // 8) * 16384 + B * H * T * 2 * 32 * 4 + B * H * 128 * 4


def test_time_split_workspace():
    """Long sequences over few heads take the time-split forward, whose workspace holds per-segment states; many
    heads or short sequences need none.  bf16 heads up to 64 wide without option bits run the split by walks
    (segments of whole chunks, of any length): the zero-start run's final states and fp32 outputs, its residuals (a
    16 KB state and 80 KB of solve results per chunk of 64 tokens, gated the 16 KB scores), Phi with Qc (32 KB) and
    D = T_k S_s (16 KB) per chunk, three 16 KB records per (head, segment).  Other splits (option bits, fp32) keep
    the transition run's buffers (delta: transitions, a zero-value tensor and the transition run's fp32 outputs);
    those need T divisible by P."""
    lib = gdn
    few = lib.gdn_workspace_bytes(lib.make_shape(1, 16, 32768, 64, 64, "delta", "bf16"), 0)
    many = lib.gdn_workspace_bytes(lib.make_shape(8, 16, 4096, 64, 64, "delta", "bf16"), 0)
    gated = lib.gdn_workspace_bytes(lib.make_shape(1, 16, 32768, 64, 64, "gated", "bf16"), 0)
    short = lib.gdn_workspace_bytes(lib.make_shape(1, 16, 500, 64, 64, "delta", "bf16"), 0)   # 8 chunks
    logits = lib.gdn_workspace_bytes(lib.make_shape(1, 16, 32768, 64, 64, "delta", "bf16", gate_logits=True), 0)
    glogits = lib.gdn_workspace_bytes(lib.make_shape(1, 16, 32768, 64, 64, "gated", "bf16", gate_logits=True), 0)
    assert many == 256 and short == 256
    nq, P = 16 * 512, 9   # segments of 57 chunks (the last 56): 16 x 9 <= 152
    assert lib.gdn_plan(lib.make_shape(1, 16, 32768, 64, 64, "delta", "bf16"), 0).segments == P
    assert lib.gdn_plan(lib.make_shape(1, 16, 32768, 64, 64, "gated", "bf16"), 0).segments == P
    walks = 256 + 16 * P * 16384 + 32768 * 16 * 64 * 4 + nq * (32768 + 16384) + 16 * P * 3 * 16384
    assert few == walks + nq * (16384 + 81920)
    assert gated == walks + nq * (16384 + 16384)
    # the transition run's buffers: 2 x 128 states (16 KB) + 2 x 128 transitions + zero values (bf16) and the fp32
    # outputs of the zero-start and transition runs; gated without the transitions
    assert logits >= 256 + 4 * 128 * 16384 + 32768 * 16 * 64 * 2 + 2 * 32768 * 16 * 64 * 4
    assert 256 + 2 * 128 * 16384 <= glogits < logits


def test_time_split_backward_workspace():
    """The token-serial backward splits long sequences over few heads too (shapes the chunked backward does not
    take, e.g. with logit gates): its workspace adds the forward split's buffers (which hold the zero-start runs'
    fp32 outputs) and two sets of per-segment adjoints to its own."""
    kw = dict(gate_logits=True)
    few = gdn.gdn_workspace_bytes(gdn.make_shape(1, 16, 32768, 64, 64, "delta", "bf16", **kw), 1)
    many = gdn.gdn_workspace_bytes(gdn.make_shape(16, 8, 4096, 64, 64, "delta", "bf16", **kw), 1)
    fwd_split = gdn.gdn_workspace_bytes(gdn.make_shape(1, 16, 32768, 64, 64, "delta", "bf16", **kw), 0)
    # same tokens and heads: the backward's own buffers are equal, the split adds at least the forward's
    assert few >= many + fwd_split - 256 + 2 * 128 * 16384


def test_chunked_backward_workspace():
    """The chunked backward (bf16, heads up to 64 wide, no option bits) keeps per chunk of 64 tokens five 16 KB
    64 x 64 records in delta mode (transition as bf16 hi/lo tiles, zero-start state, adjoint share, entering state,
    leaving adjoint) plus the 80 KB of the front's results that the gradient pass reuses, four fp32 records in
    gated mode, and two rows of 64 floats (decay, dA partial), after the 256-byte status word.  Where the heads fill
    most of a wave of one CTA per SM, gdn_bwd runs the saving forward instead of the prep front: its workspace is
    the backward-from-residuals one plus the residuals and the forward's outputs."""
    for mode, per_chunk in (("delta", 5 * 16384 + 81920), ("gated", 4 * 16384)):
        for B, H, T, d in ((8, 16, 4096, 64), (1, 16, 32768, 64), (2, 3, 100, 56), (1, 1, 1, 8), (1, 3, 2500, 64)):
            s = gdn.make_shape(B, H, T, d, d, mode, "bf16")
            nk = -(-T // 64)
            nq = B * H * nk
            # chains over few heads split in time: segments of >= 16 chunks, 2 sweeps x heads x segments <= 152;
            # each (sweep, head, segment) then keeps three 16 KB records, and gated each (sweep, chunk) the rows'
            # 64 decay products
            units, nseg = B * H, 1
            P = min(152 // (2 * units), nk // 16)
            if nk >= 32 and P >= 2:
                L = -(-nk // P)
                nseg = -(-nk // L)
            want = 256 + per_chunk * nq + 2 * -(-(nq * 256) // 256) * 256
            if nseg > 1:
                want += 2 * units * nseg * 3 * 16384
                if mode == "gated":
                    want += 2 * nq * 256
            if units == 128 and T == 4096:
                # heads filling most of a wave: the saving forward recomputes the residuals (a 16 KB state and the
                # solve's 80 KB, gated the 16 KB scores) and outputs into the workspace, then the backward from them
                res = nq * (16384 + (81920 if mode == "delta" else 16384))
                want = gdn.gdn_workspace_bytes(s, 2) + res + B * T * H * d * 2
            assert gdn.gdn_workspace_bytes(s, 1) == want, (mode, B, H, T, d)
            p = gdn.gdn_plan(s, 1)
            assert (p.segments, p.fwd_kernel, p.bwd_kernel) == (nseg, gdn.GDN_KERNEL_NONE, gdn.GDN_BWD_TENSOR_CORE)
            if (mode, B, H, T) == ("delta", 1, 16, 32768):
                assert nseg == 4


def test_gate_logits_option_bit():
    """GDN_GATE_LOGITS rides in the mode field: the forward's workspace is the same with or without it, the
    backward takes the token-serial kernel with it (and the chunked one without), and a mode with an unknown bit
    is rejected (size 0)."""
    plain = gdn.make_shape(2, 4, 300, 64, 64, "delta", "bf16")
    logit = gdn.make_shape(2, 4, 300, 64, 64, "delta", "bf16", gate_logits=True)
    assert logit.mode == gdn.GDN_DELTA | gdn.GDN_GATE_LOGITS
    assert gdn.gdn_workspace_bytes(logit, 0) == gdn.gdn_workspace_bytes(plain, 0) > 0
    assert gdn.gdn_workspace_bytes(logit, 1) > 0 and gdn.gdn_workspace_bytes(plain, 1) > 0
    assert gdn.gdn_plan(logit, 1).bwd_kernel == gdn.GDN_BWD_SERIAL
    assert gdn.gdn_plan(plain, 1).bwd_kernel == gdn.GDN_BWD_TENSOR_CORE
    bad = gdn.make_shape(2, 4, 300, 64, 64, gdn.GDN_DELTA | 0x800, "bf16")
    assert gdn.gdn_workspace_bytes(bad, 0) == 0


def test_norm_bc_option_bit():
    """GDN_NORM_BC rides in the mode field too (alone or with GDN_GATE_LOGITS).  The forward's workspace is
    unchanged; the backward adds fp32 partials of db, dc [B, T, H, d_k] and dg, dbeta [B, T, H] even with a
    single column slab, because the normalisation's Jacobian is applied after the column sums."""
    B, H, T, d = 2, 4, 300, 64
    plain = gdn.make_shape(B, H, T, d, d, "delta", "bf16", gate_logits=True)   # the token-serial backward too
    norm = gdn.make_shape(B, H, T, d, d, "delta", "bf16", norm_bc=True)
    both = gdn.make_shape(B, H, T, d, d, "delta", "bf16", gate_logits=True, norm_bc=True)
    assert norm.mode == gdn.GDN_DELTA | gdn.GDN_NORM_BC
    assert both.mode == gdn.GDN_DELTA | gdn.GDN_NORM_BC | gdn.GDN_GATE_LOGITS
    assert gdn.gdn_workspace_bytes(norm, 0) == gdn.gdn_workspace_bytes(plain, 0) == 256
    assert gdn.gdn_plan(norm, 1).bwd_kernel == gdn.GDN_BWD_SERIAL
    extra = B * T * H * (2 * d + 2) * 4
    assert gdn.gdn_workspace_bytes(norm, 1) >= gdn.gdn_workspace_bytes(plain, 1) + extra
    assert gdn.gdn_workspace_bytes(both, 1) == gdn.gdn_workspace_bytes(norm, 1)


def test_check_finite_option_bit():
    """GDN_CHECK_FINITE changes no workspace size and combines with the other bits."""
    plain = gdn.make_shape(2, 4, 300, 64, 64, "delta", "bf16", gate_logits=True)
    chk = gdn.make_shape(2, 4, 300, 64, 64, "delta", "bf16", gate_logits=True, check_finite=True)
    assert chk.mode == gdn.GDN_DELTA | gdn.GDN_GATE_LOGITS | gdn.GDN_CHECK_FINITE
    for bwd in (0, 1):
        assert gdn.gdn_workspace_bytes(chk, bwd) == gdn.gdn_workspace_bytes(plain, bwd) > 0
    assert gdn.gdn_status_string(9).startswith("GDN_ERR_NONFINITE")


def test_plan_reports_split_and_kernel():
    """gdn_plan answers from the shape alone, by the rules the calls dispatch with: the time split for long
    sequences over few heads (the delta bf16 forward split by walks into at least 2 segments of at least 8 whole
    chunks for any length; other forwards into at least 4 equal segments in delta mode, 3 in gated mode; token-serial
    backward at
    least 2, the chunked backward's chain in delta mode segments of at least 16 chunks),
    the decode kernel up to 8 tokens, the tensor-core forward for bf16 keys up to 64 wide except delta heads up to
    32 wide over more than 304 units, the token-serial forward otherwise."""
    K = gdn

    def plan(*a, bw=0, **kw):
        p = gdn.gdn_plan(gdn.make_shape(*a, **kw), bw)
        return p.segments, p.fwd_kernel

    assert plan(1, 16, 32768, 64, 64, "delta", "bf16") == (9, K.GDN_KERNEL_TENSOR_CORE)   # split by walks
    assert plan(1, 16, 32749, 64, 64, "delta", "bf16") == (9, K.GDN_KERNEL_TENSOR_CORE)   # any length
    assert plan(1, 16, 32768, 64, 64, "delta", "bf16", gate_logits=True) == (8, K.GDN_KERNEL_TENSOR_CORE)
    # chunked backward: its chain over the 512 chunk boundaries split into 4 segments of 128 chunks (2 sweeps x 16
    # heads x 4 <= 152), from the forward's residuals (the reverse sweep alone) into 9 of 57 (16 x 9 <= 152)
    assert plan(1, 16, 32768, 64, 64, "delta", "bf16", bw=1) == (4, K.GDN_KERNEL_NONE)
    assert plan(1, 16, 32768, 64, 64, "delta", "bf16", bw=2) == (9, K.GDN_KERNEL_NONE)
    assert plan(1, 16, 32768, 64, 64, "gated", "bf16", bw=1) == (4, K.GDN_KERNEL_NONE)   # gated chain split too
    assert plan(1, 16, 1024, 64, 64, "delta", "bf16", bw=1) == (1, K.GDN_KERNEL_NONE)    # 16 chunks: too short
    assert plan(1, 16, 32768, 64, 64, "delta", "bf16", bw=1, gate_logits=True) == (8, K.GDN_KERNEL_TENSOR_CORE)
    assert plan(8, 16, 4096, 64, 64, "delta", "bf16") == (1, K.GDN_KERNEL_TENSOR_CORE)
    assert plan(8, 16, 4096, 64, 64, "delta", "bf16", bw=1) == (1, K.GDN_KERNEL_NONE)
    assert plan(1, 40, 1024, 32, 32, "delta", "f32") == (1, K.GDN_KERNEL_SERIAL)   # 152 / 40: 3 < 4 segments
    assert plan(1, 40, 1024, 32, 32, "delta", "f32", bw=1) == (2, K.GDN_KERNEL_SERIAL)
    assert plan(8, 40, 4096, 32, 32, "delta", "bf16") == (1, K.GDN_KERNEL_SERIAL)
    assert plan(8, 40, 4096, 32, 32, "gated", "bf16") == (1, K.GDN_KERNEL_TENSOR_CORE)
    assert plan(4, 40, 4096, 32, 32, "delta", "bf16") == (1, K.GDN_KERNEL_TENSOR_CORE)  # 160 units
    assert plan(512, 16, 1, 64, 64, "delta", "bf16") == (1, K.GDN_KERNEL_DECODE)
    assert plan(8, 16, 4096, 128, 128, "delta", "bf16") == (1, K.GDN_KERNEL_SERIAL)
    assert plan(1, 16, 0, 64, 64, "gated", "bf16") == (1, K.GDN_KERNEL_NONE)
    assert plan(1, 4, 3000, 64, 64, "gated", "bf16", gate_logits=True) == (5, K.GDN_KERNEL_TENSOR_CORE)
    # a split forward is exactly one whose workspace holds more than the 256-byte status word
    for a in [(1, 16, 32768, 64, 64, "delta", "bf16"), (1, 16, 32768, 64, 64, "gated", "bf16"),
              (2, 3, 3072, 56, 56, "gated", "bf16"), (1, 16, 1000, 64, 64, "delta", "bf16"),
              (8, 16, 4096, 64, 64, "delta", "bf16"), (1, 2, 4096, 128, 128, "delta", "bf16")]:
        s = gdn.make_shape(*a)
        assert (gdn.gdn_plan(s, 0).segments > 1) == (gdn.gdn_workspace_bytes(s, 0) > 256), a
    # the errors the calls return for the shape alone
    for bad, status in [(gdn.make_shape(1, 1, 10, 12, 8, "delta", "bf16"), 2),
                        (gdn.make_shape(1, 1, 10, 8, 8, gdn.GDN_DELTA | 0x800, "bf16"), 4)]:
        with pytest.raises(gdn.GdnError) as e:
            gdn.gdn_plan(bad, 0)
        assert e.value.status == status


def test_plan_and_workspace_agree_on_random_shapes():
    """Over random shapes, valid or not: gdn_plan succeeds exactly when both workspace sizes are non-zero; a split
    has T divisible by its segments, at least 512 tokens per segment, heads at most 64 wide and at most 152
    (batch, head, segment) units (forward: at least 4 segments in delta mode, 3 in gated mode; the chunked
    backward's chain: delta mode, segments of at least 16 chunks); a forward splits
    exactly when its workspace holds more than the status word; the forward kernel is NONE only without tokens."""
    rng = np.random.default_rng(7)
    for _ in range(3000):
        B = int(rng.choice([1, 2, 3, 8, 64, 512]))
        H = int(rng.choice([1, 2, 4, 16, 40, 100]))
        T = int(rng.choice([0, 1, 5, 8, 9, 100, 1024, 3000, 4096, 32768]))
        dk = int(rng.choice([8, 16, 24, 32, 56, 64, 72, 128, 130, 12]))
        dv = int(rng.choice([8, 16, 32, 64, 96, 128, 20]))
        mode = str(rng.choice(["gated", "delta"]))
        io = str(rng.choice(["bf16", "f32"]))
        s = gdn.make_shape(B, H, T, dk, dv, mode, io)
        w0, w1 = gdn.gdn_workspace_bytes(s, 0), gdn.gdn_workspace_bytes(s, 1)
        for bw in (0, 1):
            try:
                p = gdn.gdn_plan(s, bw)
            except gdn.GdnError:
                assert w0 == 0 and w1 == 0, (B, H, T, dk, dv, mode, io)
                continue
            assert w0 > 0 and w1 > 0
            P = p.segments
            chunked = io == "bf16" and dk <= 64 and dv <= 64 and T > 0
            assert P >= 1
            if bw and chunked:
                # the chunked backward splits only its chain, into segments of >= 16 whole chunks
                # (the last one may be shorter), at most 152 (sweep, unit, segment) walks
                nk = -(-T // 64)
                assert P == 1 or (2 * B * H * P <= 152 and -(-nk // P) >= 16
                                  and (P - 1) * -(-nk // P) < nk), (B, H, T, P)
            elif not bw and chunked:
                # the split by walks: segments of at least 8 whole chunks (the last may be shorter), any length
                nk = -(-T // 64)
                assert P == 1 or (P >= 2 and B * H * P <= 152 and -(-nk // P) >= 8
                                  and (P - 1) * -(-nk // P) < nk), (B, H, T, P)
            else:
                assert T % P == 0 if T else P == 1
                if P > 1:
                    assert T // P >= 512 and dk <= 64 and dv <= 64 and B * H * P <= 152
                    if not bw:
                        assert P >= (4 if mode == "delta" else 3)
            if bw:
                want = gdn.GDN_BWD_NONE if T == 0 else (gdn.GDN_BWD_TENSOR_CORE if chunked else gdn.GDN_BWD_SERIAL)
                assert p.bwd_kernel == want
                if chunked:
                    assert p.fwd_kernel == gdn.GDN_KERNEL_NONE
            else:
                assert p.bwd_kernel == gdn.GDN_BWD_NONE
            if not bw:
                assert (P > 1) == (w0 > 256)
                assert (p.fwd_kernel == gdn.GDN_KERNEL_NONE) == (T == 0)
                if 0 < T <= 8:
                    assert p.fwd_kernel == gdn.GDN_KERNEL_DECODE
                if p.fwd_kernel == gdn.GDN_KERNEL_TENSOR_CORE:
                    assert io == "bf16" and dk <= 64


def test_saved_residuals_sizes_and_argument_errors(lib):
    """gdn_saved_bytes: per chunk of 64 tokens a 16 KB state and 80 KB of solve results (gated mode: the 16 KB
    scores P), for bf16 shapes whose backward is the chunked one and whose forward is one tensor-core pass or a
    split in time into whole-chunk segments run by walks; 0 for every other shape.  The
    backward from the residuals needs a smaller workspace (backward = 2).  gdn_fwd_save and gdn_bwd_saved reject
    bad arguments before any device work."""
    for B, H, T, d in ((8, 16, 4096, 64), (2, 3, 100, 56), (1, 1, 9, 8), (1, 16, 32768, 64), (1, 3, 2496, 64)):
        s = gdn.make_shape(B, H, T, d, d, "delta", "bf16")
        nq = B * H * -(-T // 64)
        assert gdn.gdn_saved_bytes(s) == nq * (16384 + 81920)
        assert 0 < gdn.gdn_workspace_bytes(s, 2) < gdn.gdn_workspace_bytes(s, 1)
        sg = gdn.make_shape(B, H, T, d, d, "gated", "bf16")
        assert gdn.gdn_saved_bytes(sg) == nq * (16384 + 16384)
        assert 0 < gdn.gdn_workspace_bytes(sg, 2) < gdn.gdn_workspace_bytes(sg, 1)
    none = [gdn.make_shape(2, 2, 256, 64, 64, "delta", "f32"),               # fp32 I/O
            gdn.make_shape(2, 2, 256, 128, 128, "delta", "bf16"),            # wider than 64
            gdn.make_shape(2, 2, 256, 64, 64, "delta", "bf16", gate_logits=True),
            gdn.make_shape(2, 2, 256, 64, 64, "delta", "bf16", norm_bc=True),
            gdn.make_shape(1, 16, 32768, 64, 64, "delta", "bf16", gate_logits=True),   # option bits
            gdn.make_shape(2, 2, 4, 64, 64, "delta", "bf16"),                # the decode kernel's length
            gdn.make_shape(2, 2, 0, 64, 64, "delta", "bf16")]
    for s in none:
        assert gdn.gdn_saved_bytes(s) == 0
        assert gdn.gdn_workspace_bytes(s, 2) == 0
    s = gdn.make_shape(2, 2, 256, 64, 64, "delta", "bf16")
    need = gdn.gdn_saved_bytes(s)

    def fwd_save(shape, saved=FAKE, saved_bytes=need):
        return gdn.gdn_fwd_save(shape, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, saved, FAKE,
                                saved_bytes=saved_bytes, ws_bytes=1 << 30, stream=0)

    def bwd_saved(shape, saved=FAKE, saved_bytes=need, beta=FAKE):
        return gdn.gdn_bwd_saved(shape, FAKE, FAKE, FAKE, FAKE, beta, FAKE, saved, FAKE, None, FAKE, FAKE, FAKE,
                                 FAKE, beta, FAKE, None, FAKE, saved_bytes=saved_bytes, ws_bytes=1 << 30, stream=0)

    assert fwd_save(s, saved=None) == 1
    assert fwd_save(s, saved_bytes=need - 1) == 5
    assert fwd_save(s, saved=FAKE + 16) == 3
    assert fwd_save(gdn.make_shape(2, 2, 256, 64, 64, "delta", "f32")) == 4
    assert fwd_save(gdn.make_shape(2, 2, 256, 64, 64, "gated", "bf16")) == 4   # beta given in gated mode
    assert fwd_save(gdn.make_shape(1, 16, 32768, 64, 64, "delta", "bf16", gate_logits=True), saved_bytes=1 << 40) == 4
    assert bwd_saved(s, saved=None) == 1
    assert bwd_saved(s, saved_bytes=need - 1) == 5
    assert bwd_saved(s, saved=FAKE + 16) == 3
    assert bwd_saved(gdn.make_shape(2, 2, 256, 128, 128, "delta", "bf16")) == 4
    assert bwd_saved(s, beta=None) == 4   # delta mode needs beta (and dbeta)
