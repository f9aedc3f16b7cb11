"""Chunked reverse-mode restatement of the gated delta rule, fp64 (test infrastructure).

Only ``tests/`` may use this module; the product path never loads it.

"GDN & MLA Mechanism Deep-Dive", Step 5 (Chunked recurrence) cuts the sequence
into chunks of C tokens, solves each in closed form with C x C matrices and
carries the state from chunk to chunk.  This module writes out the reverse
mode of that chunked form: one forward walk keeps the state entering every
chunk, then the chunks are walked backwards, each taking the adjoint of the
state it hands on and returning the adjoint of the state it received.  It is
the chunk-level counterpart of the serial backward in ``gdn_oracle.c`` and is
held to it by ``tests/test_oracle_pins.py``.

Per (batch, head) and chunk of L tokens t = 0..L-1 entering with state S
(rows i over d_k, columns j over d_v), with A = -exp(A_log):
  G_t = g_0 + ... + g_t,  Gam_t[i] = A[i] G_t,  E_t = exp(Gam_t)
  Ct_t = c_t (.) E_t,  Bt_t = b_t (.) E_t,  Bh_t = b_t (.) exp(Gam_{L-1} - Gam_t)
  Q[t,s] = sum_i c_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])   (s <= t, else 0)
  K[t,s] = sum_i b_t[i] b_s[i] exp(Gam_t[i] - Gam_s[i])   (s <  t, else 0)
  gated ("GDN & MLA Mechanism Deep-Dive", Step 4): U = V
  delta (delta-rule card of "HyMo-434M -- documentation portal"):
        (I + diag(beta) K) U = diag(beta) (V - Bt S)
  O = Ct S + Q U,   S' = diag(E_{L-1}) S + Bh^T U.
Every row of U is the value written at its token (x_t of the serial form).
The reverse mode below takes these steps backwards; the exponentials' share
of the gradient is gathered per (token, channel) in dGam, then
dG_t = sum_i A[i] dGam_t[i], dA[i] = sum_t G_t dGam_t[i] and
dg_r = sum_{t >= r} dG_t within the chunk.
"""
from __future__ import annotations

import numpy as np


def _chunk_fwd(S, v, b, c, g, beta, A, delta):
    """The chunk's closed form: everything the reverse step reuses."""
    L = v.shape[0]
    G = np.cumsum(g)
    Gam = G[:, None] * A[None, :]                    # [L, d_k]
    E = np.exp(Gam)
    D = np.exp(Gam[:, None, :] - Gam[None, :, :])    # D[t, s, i] = exp(Gam_t[i] - Gam_s[i])
    Ct, Bt = c * E, b * E
    Bh = b * np.exp(Gam[-1][None, :] - Gam)
    low = np.tril(np.ones((L, L)))
    strict = np.tril(np.ones((L, L)), -1)
    Tq = c[:, None, :] * b[None, :, :] * D * low[:, :, None]       # terms of Q
    Tk = b[:, None, :] * b[None, :, :] * D * strict[:, :, None]    # terms of K
    Q, K = Tq.sum(axis=2), Tk.sum(axis=2)
    if delta:
        R0 = v - Bt @ S                               # V - Bt S
        Mmat = np.eye(L) + beta[:, None] * K
        U = np.linalg.solve(Mmat, beta[:, None] * R0)
    else:
        R0, Mmat, U = None, None, v
    O = Ct @ S + Q @ U
    S_next = E[-1][:, None] * S + Bh.T @ U
    return dict(G=G, Gam=Gam, E=E, D=D, Ct=Ct, Bt=Bt, Bh=Bh, Tq=Tq, Tk=Tk, Q=Q, K=K, R0=R0, Mmat=Mmat, U=U,
                O=O, S_next=S_next)


def _chunk_bwd(S, f, dO, dSn, v, b, c, beta, A, delta):
    """Adjoints of one chunk given dL/dO and dL/dS'; returns (dS, dv, db, dc, dg, dbeta, dA)."""
    L = v.shape[0]
    E, U = f["E"], f["U"]
    # O = Ct S + Q U
    dCt = dO @ S.T
    dS = f["Ct"].T @ dO
    dQ = (dO @ U.T) * np.tril(np.ones((L, L)))
    dU = f["Q"].T @ dO
    # S' = diag(E_{L-1}) S + Bh^T U
    dS += E[-1][:, None] * dSn
    dGam = np.zeros_like(f["Gam"])
    dGam[-1] += (dSn * S).sum(axis=1) * E[-1]
    dBh = U @ dSn.T
    dU += f["Bh"] @ dSn
    dv = np.zeros_like(v)
    dbeta = np.zeros(L)
    dBt = np.zeros_like(b)
    dK = np.zeros((L, L))
    if delta:
        # (I + diag(beta) K) U = diag(beta) R0,  R0 = V - Bt S
        dR = np.linalg.solve(f["Mmat"].T, dU)        # adjoint of the right-hand side diag(beta) R0
        dMm = -dR @ U.T                              # adjoint of the matrix I + diag(beta) K
        dv = beta[:, None] * dR
        dbeta = (dR * f["R0"]).sum(axis=1) + (dMm * f["K"]).sum(axis=1)
        dR0 = beta[:, None] * dR
        dBt = -dR0 @ S.T
        dS += -f["Bt"].T @ dR0
        dK = (beta[:, None] * dMm) * np.tril(np.ones((L, L)), -1)
    else:
        dv = dU
    # exponential-carrying terms: Ct, Bt, Bh and the entries of Q and K
    dc = dCt * E
    dGam += dCt * f["Ct"]
    db = dBt * E
    dGam += dBt * f["Bt"]
    db += dBh * np.exp(f["Gam"][-1][None, :] - f["Gam"])
    dGam -= dBh * f["Bh"]
    dGam[-1] += (dBh * f["Bh"]).sum(axis=0)
    # entry [t, s] = sum_i left_t[i] b_s[i] D[t, s, i] on its mask (Q: left = c, s <= t; K: left = b, s < t)
    for terms, dM, left, is_q in ((f["Tq"], dQ, c, True), (f["Tk"], dK, b, False)):
        mask = np.tril(np.ones((L, L)), 0 if is_q else -1)
        w = (dM * mask)[:, :, None] * f["D"]         # dM[t,s] D[t,s,i] on the mask
        dleft = (w * b[None, :, :]).sum(axis=1)      # d left_t[i]
        db += (w * left[:, None, :]).sum(axis=0)     # d b_s[i]
        if is_q:
            dc += dleft
        else:
            db += dleft
        wt = dM[:, :, None] * terms                  # the terms carry exp(Gam_t - Gam_s)
        dGam += wt.sum(axis=1) - wt.sum(axis=0)
    dG = dGam @ A
    dA = f["G"] @ dGam
    dg = np.cumsum(dG[::-1])[::-1]
    return dS, dv, db, dc, dg, dbeta, dA


def gdn_bwd_chunked(v, b, c, g, beta, A_log, h0, dO, dhT=None, mode="gated", chunk=64):
    """Gradients of the forward by its chunked form walked in reverse (same returns as oracle.gdn_bwd)."""
    delta = mode in ("delta", 1)
    f64 = lambda x: None if x is None else np.asarray(x, dtype=np.float64)
    v, b, c, g, A_log, dO = map(f64, (v, b, c, g, A_log, dO))
    beta, h0, dhT = f64(beta), f64(h0), f64(dhT)
    B, T, H, dv_ = v.shape
    dk = b.shape[3]
    out = {"dv": np.zeros_like(v), "db": np.zeros_like(b), "dc": np.zeros_like(c), "dg": np.zeros_like(g),
           "dbeta": np.zeros_like(g) if delta else None, "dh0": np.zeros((B, H, dk, dv_)),
           "dA_log": np.zeros((H, dk))}
    for bb in range(B):
        for h in range(H):
            A = -np.exp(A_log[h])
            S = np.zeros((dk, dv_)) if h0 is None else h0[bb, h].copy()
            starts = list(range(0, T, chunk))
            saved = []
            for t0 in starts:
                sl = slice(t0, min(T, t0 + chunk))
                f = _chunk_fwd(S, v[bb, sl, h], b[bb, sl, h], c[bb, sl, h], g[bb, sl, h],
                               beta[bb, sl, h] if delta else None, A, delta)
                saved.append((S, f))
                S = f["S_next"]
            dS = np.zeros((dk, dv_)) if dhT is None else dhT[bb, h].copy()
            dA = np.zeros(dk)
            for t0, (S0, f) in zip(reversed(starts), reversed(saved)):
                sl = slice(t0, min(T, t0 + chunk))
                dS, dvv, dbb, dcc, dgg, dbe, dAc = _chunk_bwd(S0, f, dO[bb, sl, h], dS, v[bb, sl, h],
                                                             b[bb, sl, h], c[bb, sl, h],
                                                             beta[bb, sl, h] if delta else None, A, delta)
                out["dv"][bb, sl, h] = dvv
                out["db"][bb, sl, h] = dbb
                out["dc"][bb, sl, h] = dcc
                out["dg"][bb, sl, h] = dgg
                if delta:
                    out["dbeta"][bb, sl, h] = dbe
                dA += dAc
            out["dh0"][bb, h] = dS
            out["dA_log"][h] += dA * A            # A = -exp(A_log): dA/dA_log = A
    return out
