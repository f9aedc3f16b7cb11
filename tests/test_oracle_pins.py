"""Pins for the fp64 oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a brute-force
quadratic form, closed forms of special cases, invariants, an independent
matrix-product form, its own chunked restatement, and central finite
differences for the backward.  The inputs are tiny so the whole file runs in
seconds on CPU.
"""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_delta_gb300 import inputs as I


def draw(mode, B=1, H=2, T=9, dk=3, dv=4, seed=11, h0_std=0.7, dtype="f32", backward=False):
    w = I.custom(mode=mode, dtype=dtype, B=B, H=H, T=T, dk=dk, dv=dv, seed=seed, h0_std=h0_std,
                 backward=backward)
    return I.make_inputs(w)


def A_of(x):
    return -np.exp(x["A_log"])


# ---------------------------------------------------------------------------
# gated mode: "GDN & MLA Mechanism Deep-Dive", Step 4
# ---------------------------------------------------------------------------

def test_gated_bruteforce_quadratic_form():
    """o_t = sum_{s<=t} sum_i c_t[i] b_s[i] prod_{r=s+1..t} alpha_r[i] v_s
            + sum_i c_t[i] prod_{r=0..t} alpha_r[i] h0[i,:]."""
    x = draw("gated", B=2, H=2, T=9, dk=3, dv=4)
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], None, x["A_log"], x["h0"], mode="gated")
    B, T, H, dv = x["v"].shape
    dk = x["b"].shape[3]
    A = A_of(x)
    ref = np.zeros_like(o)
    for b in range(B):
        for h in range(H):
            alpha = np.exp(x["g"][b, :, h][:, None] * A[h][None, :])  # [T, dk]
            for t in range(T):
                acc = np.zeros(dv)
                for s in range(t + 1):
                    for i in range(dk):
                        dec = 1.0
                        for r in range(s + 1, t + 1):
                            dec *= alpha[r, i]
                        acc += x["c"][b, t, h, i] * x["b"][b, s, h, i] * dec * x["v"][b, s, h, :]
                for i in range(dk):
                    dec = 1.0
                    for r in range(0, t + 1):
                        dec *= alpha[r, i]
                    acc += x["c"][b, t, h, i] * dec * x["h0"][b, h, i, :]
                ref[b, t, h] = acc
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12 * np.abs(ref).max())


def test_gated_g_zero_is_cumulative_linear_attention():
    """g = 0 => alpha = 1 => o_t = sum_{s<=t} (c_t . b_s) v_s + c_t^T h0
    ("GDN & MLA Mechanism Deep-Dive", Step 2: S_N = sum_j phi(k_j) v_j^T)."""
    x = draw("gated", B=1, H=3, T=17, dk=5, dv=6)
    g0 = np.zeros_like(x["g"])
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], g0, None, x["A_log"], x["h0"], mode="gated")
    for h in range(3):
        Cm, Bm, Vm = x["c"][0, :, h], x["b"][0, :, h], x["v"][0, :, h]
        ref = np.tril(Cm @ Bm.T) @ Vm + Cm @ x["h0"][0, h]
        np.testing.assert_allclose(o[0, :, h], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(hT[0, h], x["h0"][0, h] + Bm.T @ Vm, rtol=0, atol=1e-12)


def test_gated_linear_in_v_and_h0():
    x = draw("gated", B=1, H=2, T=12, dk=4, dv=3)
    y = draw("gated", B=1, H=2, T=12, dk=4, dv=3, seed=99)
    a = 1.7
    f = lambda v, h0: oracle.gdn_fwd(v, x["b"], x["c"], x["g"], None, x["A_log"], h0, mode="gated")
    o_mix, hT_mix = f(a * x["v"] + y["v"], a * x["h0"] + y["h0"])
    o_x, hT_x = f(x["v"], x["h0"])
    o_y, hT_y = f(y["v"], y["h0"])
    np.testing.assert_allclose(o_mix, a * o_x + o_y, rtol=0, atol=1e-12)
    np.testing.assert_allclose(hT_mix, a * hT_x + hT_y, rtol=0, atol=1e-12)


def test_gated_scalar_worked_example():
    """d_k = d_v = 1, T = 3, closed form written out by hand:
    h1 = a1 h0 + b1 v1, h2 = a2 h1 + b2 v2, h3 = a3 h2 + b3 v3, o_t = c_t h_t."""
    v = np.array([0.5, -1.0, 2.0]).reshape(1, 3, 1, 1)
    b = np.array([1.0, 0.25, -0.5]).reshape(1, 3, 1, 1)
    c = np.array([2.0, -1.0, 0.5]).reshape(1, 3, 1, 1)
    g = np.array([0.5, 1.0, 0.25]).reshape(1, 3, 1)
    A_log = np.array([[np.log(2.0)]])  # A = -2
    h0 = np.array([3.0]).reshape(1, 1, 1, 1)
    a = np.exp(-2.0 * np.array([0.5, 1.0, 0.25]))
    h1 = a[0] * 3.0 + 1.0 * 0.5
    h2 = a[1] * h1 + 0.25 * -1.0
    h3 = a[2] * h2 + -0.5 * 2.0
    o, hT = oracle.gdn_fwd(v, b, c, g, None, A_log, h0, mode="gated")
    np.testing.assert_allclose(o.ravel(), [2.0 * h1, -1.0 * h2, 0.5 * h3], rtol=1e-14)
    np.testing.assert_allclose(hT.ravel(), [h3], rtol=1e-14)


# ---------------------------------------------------------------------------
# delta mode: delta-rule card of "HyMo-434M -- documentation portal"
# ---------------------------------------------------------------------------

def test_delta_matrix_product_form():
    """h_t = (I - beta_t b_t b_t^T) diag(alpha_t) h_{t-1} + beta_t b_t v_t^T,
    the page's "(1 - beta q k^T) h + beta v k^T" in [d_k, d_v] orientation."""
    x = draw("delta", B=2, H=2, T=11, dk=4, dv=3)
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode="delta")
    A = A_of(x)
    for bb in range(2):
        for h in range(2):
            S = x["h0"][bb, h].copy()
            for t in range(11):
                bt = x["b"][bb, t, h]
                be = x["beta"][bb, t, h]
                D = np.diag(np.exp(x["g"][bb, t, h] * A[h]))
                S = (np.eye(4) - be * np.outer(bt, bt)) @ D @ S + be * np.outer(bt, x["v"][bb, t, h])
                np.testing.assert_allclose(o[bb, t, h], S.T @ x["c"][bb, t, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(hT[bb, h], S, rtol=0, atol=1e-12)


def test_delta_replace_invariant():
    """beta = 1 and ||b_t|| = 1: the write replaces the value stored under b_t,
    so h_t^T b_t = v_t for any decay ("replace the old contribution with the
    new one", Step 3).  Reading with c = b returns v exactly."""
    x = draw("delta", B=1, H=2, T=23, dk=6, dv=5, dtype="f32")
    bvec = np.random.default_rng(0).normal(size=x["b"].shape)
    bvec /= np.linalg.norm(bvec, axis=-1, keepdims=True)
    ones = np.ones_like(x["beta"])
    o, _ = oracle.gdn_fwd(x["v"], bvec, bvec, x["g"], ones, x["A_log"], x["h0"], mode="delta")
    np.testing.assert_allclose(o, x["v"], rtol=0, atol=1e-12)


def test_delta_beta_zero_is_pure_decay():
    x = draw("delta", B=1, H=2, T=15, dk=4, dv=3)
    zeros = np.zeros_like(x["beta"])
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], zeros, x["A_log"], x["h0"], mode="delta")
    A = A_of(x)
    for h in range(2):
        G = np.cumsum(x["g"][0, :, h])
        for t in range(15):
            St = np.exp(A[h] * G[t])[:, None] * x["h0"][0, h]
            np.testing.assert_allclose(o[0, t, h], St.T @ x["c"][0, t, h], rtol=0, atol=1e-12)
        np.testing.assert_allclose(hT[0, h], np.exp(A[h] * G[-1])[:, None] * x["h0"][0, h], rtol=0, atol=1e-12)


def test_delta_orthonormal_keys_no_decay():
    """alpha = 1 and orthonormal keys (d_k >= T): every erase term vanishes,
    h_T = sum_s beta_s b_s v_s^T and o_t = sum_{s<=t} beta_s (c_t . b_s) v_s."""
    T, dk, dv = 7, 9, 4
    x = draw("delta", B=1, H=1, T=T, dk=dk, dv=dv, h0_std=0.0)
    Q, _ = np.linalg.qr(np.random.default_rng(3).normal(size=(dk, dk)))
    bvec = Q[:T].reshape(1, T, 1, dk)
    g0 = np.zeros_like(x["g"])
    o, hT = oracle.gdn_fwd(x["v"], bvec, x["c"], g0, x["beta"], x["A_log"], None, mode="delta")
    Bm, Vm, Cm, be = bvec[0, :, 0], x["v"][0, :, 0], x["c"][0, :, 0], x["beta"][0, :, 0]
    np.testing.assert_allclose(hT[0, 0], (Bm * be[:, None]).T @ Vm, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o[0, :, 0], np.tril(Cm @ Bm.T) @ (be[:, None] * Vm), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# both modes: chunked form (Step 5), resume, backward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("T,chunk", [(100, 64), (100, 16), (100, 7), (1, 64), (63, 64), (65, 64), (64, 64), (9, 1)])
def test_chunked_equals_serial(mode, T, chunk):
    x = draw(mode, B=2, H=2, T=T, dk=5, dv=3)
    a = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode)
    b = oracle.gdn_fwd_chunked(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode,
                               chunk=chunk)
    scale = max(1.0, np.abs(a[0]).max())
    np.testing.assert_allclose(b[0], a[0], rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(b[1], a[1], rtol=0, atol=1e-12 * max(1.0, np.abs(a[1]).max()))


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_resume_from_state(mode):
    x = draw(mode, B=2, H=1, T=40, dk=4, dv=4)
    full_o, full_hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode)
    T1 = 17
    sl = lambda a, lo, hi: None if a is None else a[:, lo:hi]
    o1, h1 = oracle.gdn_fwd(sl(x["v"], 0, T1), sl(x["b"], 0, T1), sl(x["c"], 0, T1), sl(x["g"], 0, T1),
                            sl(x["beta"], 0, T1), x["A_log"], x["h0"], mode=mode)
    o2, h2 = oracle.gdn_fwd(sl(x["v"], T1, 40), sl(x["b"], T1, 40), sl(x["c"], T1, 40), sl(x["g"], T1, 40),
                            sl(x["beta"], T1, 40), x["A_log"], h1, mode=mode)
    np.testing.assert_allclose(np.concatenate([o1, o2], axis=1), full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(h2, full_hT, rtol=0, atol=1e-12)


def _loss(x, mode, dO, dhT, **over):
    y = dict(x)
    y.update(over)
    o, hT = oracle.gdn_fwd(y["v"], y["b"], y["c"], y["g"], y["beta"], y["A_log"], y["h0"], mode=mode, threads=1)
    return float((o * dO).sum() + (hT * dhT).sum())


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("T,d", [(5, 3), (70, 5)])
def test_backward_finite_differences(mode, T, d):
    """Central differences (eps = 1e-6) of L = <o, dO> + <h_T, dh_T> against
    every gradient the backward returns; segment length 4 exercises the
    checkpoint-and-recompute walk."""
    x = draw(mode, B=1, H=1, T=T, dk=d, dv=d + 1, seed=5, h0_std=0.5)
    rng = np.random.default_rng(7)
    dO = rng.normal(size=x["v"].shape)
    dhT = rng.normal(size=(1, 1, d, d + 1))
    gr = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], dO, dhT, mode=mode, seg=4)
    names = ["v", "b", "c", "g", "A_log", "h0"] + (["beta"] if mode == "delta" else [])
    key = {"A_log": "dA_log", "h0": "dh0"}
    eps = 1e-6
    for name in names:
        base = x[name]
        grad = gr[key.get(name, "d" + name)]
        flat = base.reshape(-1)
        idx = range(flat.size) if flat.size <= 40 else rng.choice(flat.size, 40, replace=False)
        for k in idx:
            p = flat.copy(); p[k] += eps
            m = flat.copy(); m[k] -= eps
            fd = (_loss(x, mode, dO, dhT, **{name: p.reshape(base.shape)}) -
                  _loss(x, mode, dO, dhT, **{name: m.reshape(base.shape)})) / (2 * eps)
            an = grad.reshape(-1)[k]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, k, fd, an)


def test_backward_segment_length_irrelevant():
    x = draw("delta", B=1, H=2, T=37, dk=4, dv=4, backward=True)
    args = (x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None)
    a = oracle.gdn_bwd(*args, mode="delta", seg=64)
    b = oracle.gdn_bwd(*args, mode="delta", seg=5)
    for k in a:
        if a[k] is not None:
            np.testing.assert_allclose(a[k], b[k], rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_logit_gates_finite_differences(mode):
    """g and beta given as logits: the forward is the rule on their sigmoids (the
    logistic function written out here, not the oracle's), and the logit
    gradients match central differences of L = <o, dO> + <h_T, dh_T>."""
    x = draw(mode, B=1, H=1, T=30, dk=4, dv=5, seed=9, h0_std=0.5)
    rng = np.random.default_rng(11)
    zg = rng.normal(size=x["g"].shape)
    zb = rng.normal(size=x["g"].shape) if mode == "delta" else None
    logistic = lambda z: None if z is None else np.exp(z) / (np.exp(z) + 1.0)
    o_l, h_l = oracle.gdn_fwd_logits(x["v"], x["b"], x["c"], zg, zb, x["A_log"], x["h0"], mode=mode)
    o_p, h_p = oracle.gdn_fwd(x["v"], x["b"], x["c"], logistic(zg), logistic(zb), x["A_log"], x["h0"], mode=mode)
    np.testing.assert_allclose(o_l, o_p, rtol=0, atol=1e-13)
    np.testing.assert_allclose(h_l, h_p, rtol=0, atol=1e-13)
    dO = rng.normal(size=x["v"].shape)
    dhT = rng.normal(size=(1, 1, 4, 5))
    gr = oracle.gdn_bwd_logits(x["v"], x["b"], x["c"], zg, zb, x["A_log"], x["h0"], dO, dhT, mode=mode)

    def loss(zg_, zb_):
        o, hT = oracle.gdn_fwd_logits(x["v"], x["b"], x["c"], zg_, zb_, x["A_log"], x["h0"], mode=mode, threads=1)
        return float((o * dO).sum() + (hT * dhT).sum())

    eps = 1e-6
    for name, z, grad in [("dg", zg, gr["dg"])] + ([("dbeta", zb, gr["dbeta"])] if mode == "delta" else []):
        for k in range(z.size):
            p = z.reshape(-1).copy(); p[k] += eps
            m = z.reshape(-1).copy(); m[k] -= eps
            if name == "dg":
                fd = (loss(p.reshape(z.shape), zb) - loss(m.reshape(z.shape), zb)) / (2 * eps)
            else:
                fd = (loss(zg, p.reshape(z.shape)) - loss(zg, m.reshape(z.shape))) / (2 * eps)
            an = grad.reshape(-1)[k]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, k, fd, an)


def test_l2_normalize_closed_forms():
    """Unit length, unchanged direction, invariance to positive scaling, zero stays zero, and a
    3-4-5 vector by hand."""
    rng = np.random.default_rng(5)
    x = rng.normal(size=(3, 7, 2, 9))
    y = oracle.l2_normalize(x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(y * np.linalg.norm(x, axis=-1, keepdims=True), x, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(oracle.l2_normalize(3.5 * x), y, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(oracle.l2_normalize(np.zeros((2, 4))), np.zeros((2, 4)))
    np.testing.assert_allclose(oracle.l2_normalize(np.array([3.0, -4.0])), [0.6, -0.8], rtol=0, atol=1e-16)
    # the gradient is orthogonal to the vector (moving along x does not change x / ||x||)
    d = rng.normal(size=x.shape)
    gx = oracle.l2_normalize_vjp(x, d)
    np.testing.assert_allclose((gx * x).sum(axis=-1), 0.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("logits", [False, True])
def test_norm_bc_finite_differences(mode, logits):
    """b and c given before their L2 normalisation (with and without logit gates): the forward equals the
    rule on b / ||b||, c / ||c|| computed here with numpy, and the gradients with respect to the raw b, c
    (and the gates) match central differences of L = <o, dO> + <h_T, dh_T>."""
    x = draw(mode, B=1, H=1, T=12, dk=4, dv=3, seed=13, h0_std=0.5)
    rng = np.random.default_rng(17)
    b = 2.0 * rng.normal(size=x["b"].shape)
    c = 0.7 * rng.normal(size=x["c"].shape)
    g, be = x["g"], x["beta"]
    if logits:
        g = rng.normal(size=g.shape)
        be = rng.normal(size=g.shape) if mode == "delta" else None
    kw = dict(mode=mode, gate_logits=logits, norm_bc=True)
    o_n, h_n = oracle.gdn_fwd_opts(x["v"], b, c, g, be, x["A_log"], x["h0"], **kw)
    unit = lambda a: a / np.sqrt((a ** 2).sum(axis=-1, keepdims=True))
    o_p, h_p = oracle.gdn_fwd_opts(x["v"], unit(b), unit(c), g, be, x["A_log"], x["h0"], mode=mode,
                                   gate_logits=logits)
    np.testing.assert_allclose(o_n, o_p, rtol=0, atol=1e-13)
    np.testing.assert_allclose(h_n, h_p, rtol=0, atol=1e-13)
    dO = rng.normal(size=x["v"].shape)
    dhT = rng.normal(size=(1, 1, 4, 3))
    gr = oracle.gdn_bwd_opts(x["v"], b, c, g, be, x["A_log"], x["h0"], dO, dhT, **kw)

    def loss(**over):
        a = dict(b=b, c=c, g=g, beta=be)
        a.update(over)
        o, hT = oracle.gdn_fwd_opts(x["v"], a["b"], a["c"], a["g"], a["beta"], x["A_log"], x["h0"], threads=1,
                                    **kw)
        return float((o * dO).sum() + (hT * dhT).sum())

    eps = 1e-6
    checks = [("db", "b", b), ("dc", "c", c)]
    if logits:
        checks += [("dg", "g", g)] + ([("dbeta", "beta", be)] if mode == "delta" else [])
    for name, arg, z in checks:
        for k in range(z.size):
            p = z.reshape(-1).copy(); p[k] += eps
            m = z.reshape(-1).copy(); m[k] -= eps
            fd = (loss(**{arg: p.reshape(z.shape)}) - loss(**{arg: m.reshape(z.shape)})) / (2 * eps)
            an = gr[name].reshape(-1)[k]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, k, fd, an)


# ---------------------------------------------------------------------------
# the affine segment map behind the time split ("GDN & MLA Mechanism Deep-Dive", Step 5: the state is carried
# from chunk to chunk by a closed-form map of the state entering it)
# ---------------------------------------------------------------------------

def _transition_run(x, mode):
    """The same tokens with v = 0 from the identity state: (q_t = Phi_t^T c_t, Phi_T)."""
    B, T, H, dk = x["b"].shape
    eye = np.broadcast_to(np.eye(dk), (B, H, dk, dk)).copy()
    return oracle.gdn_fwd(np.zeros((B, T, H, dk)), x["b"], x["c"], x["g"], x["beta"], x["A_log"], eye, mode=mode)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_segment_map_is_affine(mode):
    """From h0 the state after the tokens is Phi_T h0 + H and every output is o0_t + h0^T q_t, where (o0, H) is
    the run from a zero state and (q, Phi_T) the run with v = 0 from the identity; in gated mode Phi_T is
    diag(exp(A sum_t g_t)) and q_t = c_t (.) exp(A G_t).  Non-square states (d_k = 4, d_v = 5) catch a
    transposed operand."""
    x = draw(mode, B=2, H=2, T=37, dk=4, dv=5, h0_std=0.7)
    o, hT = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], mode=mode)
    o0, Hs = oracle.gdn_fwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], None, mode=mode)
    q, Phi = _transition_run(x, mode)
    np.testing.assert_allclose(hT, Phi @ x["h0"] + Hs, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, o0 + np.einsum("bhkv,bthk->bthv", x["h0"], q), rtol=0, atol=1e-12)
    if mode == "gated":
        A = A_of(x)                                              # [H, d_k]
        G = np.cumsum(x["g"], axis=1)                            # [B, T, H]
        np.testing.assert_allclose(Phi, np.einsum("bhk,kl->bhkl", np.exp(A[None] * G[:, -1, :, None]),
                                                  np.eye(4)), rtol=0, atol=1e-14)
        np.testing.assert_allclose(q, x["c"] * np.exp(A[None, None] * G[..., None]), rtol=0, atol=1e-14)


@pytest.mark.parametrize("mode", ["gated", "delta"])
def test_entering_state_adjoint(mode):
    """The adjoint of the entering state is sum_t q_t do_t^T + Phi_T^T dh_T (q_t = Phi_t^T c_t as above): with
    no end gradient this is the segment adjoint G_p of the split backward, and the second term is the step of its
    reverse scan over segments."""
    x = draw(mode, B=2, H=2, T=29, dk=4, dv=5, h0_std=0.7, backward=True)
    q, Phi = _transition_run(x, mode)
    G = np.einsum("bthk,bthv->bhkv", q, x["dO"])
    ref = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], None, mode=mode)
    scale = np.abs(G).max()
    np.testing.assert_allclose(ref["dh0"], G, rtol=0, atol=1e-12 * scale)
    dhT = 0.5 * I.normal(77, 1, 2 * 2 * 4 * 5).reshape(2, 2, 4, 5)
    ref2 = oracle.gdn_bwd(x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT, mode=mode)
    np.testing.assert_allclose(ref2["dh0"], G + np.swapaxes(Phi, -1, -2) @ dhT, rtol=0, atol=1e-12 * scale)


@pytest.mark.parametrize("mode", ["gated", "delta"])
@pytest.mark.parametrize("T,chunk,dk,dv", [(37, 16, 4, 5), (130, 64, 8, 6), (64, 64, 5, 5), (9, 1, 3, 4)])
def test_chunked_backward_equals_serial(mode, T, chunk, dk, dv):
    """The reverse mode of the chunked form ("GDN & MLA Mechanism Deep-Dive", Step 5), walked chunk by chunk
    backwards, gives the serial backward's gradients: ragged last chunks, non-square states, h0 and dh_T given,
    and chunk = 1 (the chunked form reduces to the token recurrence)."""
    w = I.custom(mode=mode, dtype="f32", B=2, H=2, T=T, dk=dk, dv=dv, seed=T + dk, h0_std=0.5, backward=True)
    x = I.make_inputs(w)
    dhT = 0.3 * I.normal(5, 1, 2 * 2 * dk * dv).reshape(2, 2, dk, dv)
    args = (x["v"], x["b"], x["c"], x["g"], x["beta"], x["A_log"], x["h0"], x["dO"], dhT)
    ref = oracle.gdn_bwd(*args, mode=mode)
    got = oracle.gdn_bwd_chunked(*args, mode=mode, chunk=chunk)
    for k in ("dv", "db", "dc", "dg", "dbeta", "dA_log", "dh0"):
        if ref[k] is None:
            assert got[k] is None
            continue
        np.testing.assert_allclose(got[k], ref[k], rtol=0, atol=1e-12 * np.abs(ref[k]).max(), err_msg=k)
