"""fp64 CPU oracle for the gated delta rule (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never loads it, and the oracle shares no code with that path.

The arithmetic lives in ``gdn_oracle.c`` (plain loops, fp64); this module only
builds it with gcc, marshals numpy arrays through ``ctypes`` and spreads the
independent (batch, head) recurrences over host threads (ctypes releases the
GIL during each call).  See the C file's header for the equations followed:
"GDN & MLA Mechanism Deep-Dive", Step 4 (gated rule) and Step 5 (chunked
recurrence), and the delta-rule card of "HyMo-434M -- documentation portal".

Arguments use the library's layouts: v, b, c as [B, T, H, d]; g and beta as
[B, T, H]; A_log as [H, d_k]; states as [B, H, d_k, d_v].  Every input is
upcast exactly to float64 before the call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()

GATED = 0
DELTA = 1


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into a shared library next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        compile_source(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """The compiled oracle at `path` (the default build, or a planted-bug
    mutant that a test compiled from a modified copy of the source)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.oracle_gdn_fwd.argtypes = [i, i, i, i, i, i, dp, dp, dp, dp, dp, dp, dp, dp, dp, i, i]
        lib.oracle_gdn_bwd.argtypes = [i, i, i, i, i, i, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                       dp, dp, dp, dp, dp, dp, dp, i, i, i]
        lib.oracle_gdn_fwd_chunked.argtypes = [i, i, i, i, i, i, dp, dp, dp, dp, dp, dp, dp, dp, dp, i, i, i]
        for f in (lib.oracle_gdn_fwd, lib.oracle_gdn_bwd, lib.oracle_gdn_fwd_chunked):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def gdn_fwd(self, *a, **k):
        return gdn_fwd(*a, _lib=self.lib, **k)

    def gdn_fwd_chunked(self, *a, **k):
        return gdn_fwd_chunked(*a, _lib=self.lib, **k)

    def gdn_bwd(self, *a, **k):
        return gdn_bwd(*a, _lib=self.lib, **k)


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle source file (the real one or a mutant) to out_path."""
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", out_path, src_path, "-lm"])
    return out_path


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build()).lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # a CPU torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(x):
    if x is None:
        return ctypes.POINTER(ctypes.c_double)()
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _mode(mode) -> int:
    if mode in (GATED, "gated"):
        return GATED
    if mode in (DELTA, "delta"):
        return DELTA
    raise ValueError(f"unknown mode {mode!r}")


def _units(B, H, threads):
    n = B * H
    if threads is None:
        threads = os.cpu_count() or 1
    threads = max(1, min(int(threads), n))
    step = (n + threads - 1) // threads
    return [(u, min(n, u + step)) for u in range(0, n, step)], threads


def _run(fn, B, H, threads):
    ranges, nthr = _units(B, H, threads)
    if nthr == 1:
        rcs = [fn(a, b) for a, b in ranges]
    else:
        with ThreadPoolExecutor(max_workers=nthr) as ex:
            rcs = list(ex.map(lambda r: fn(*r), ranges))
    if any(rc != 0 for rc in rcs):
        raise ValueError("oracle rejected its arguments")


def _shape(v, b):
    B, T, H, dv = v.shape
    dk = b.shape[3]
    return B, H, T, dk, dv


def gdn_fwd(v, b, c, g, beta, A_log, h0=None, mode="gated", threads=None, _lib=None):
    """Serial fp64 forward.  Returns (o [B,T,H,d_v], h_T [B,H,d_k,d_v])."""
    m = _mode(mode)
    v, b, c, g, A_log = map(_f64, (v, b, c, g, A_log))
    beta, h0 = _f64(beta), _f64(h0)
    B, H, T, dk, dv = _shape(v, b)
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    lib = _lib or _load()
    _run(lambda a, e: lib.oracle_gdn_fwd(B, H, T, dk, dv, m, _p(v), _p(b), _p(c), _p(g), _p(beta),
                                         _p(A_log), _p(h0), _p(o), _p(hT), a, e), B, H, threads)
    return o, hT


def gdn_fwd_chunked(v, b, c, g, beta, A_log, h0=None, mode="gated", chunk=64, threads=None, _lib=None):
    """Chunked fp64 restatement of the forward (closed form per chunk)."""
    m = _mode(mode)
    v, b, c, g, A_log = map(_f64, (v, b, c, g, A_log))
    beta, h0 = _f64(beta), _f64(h0)
    B, H, T, dk, dv = _shape(v, b)
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    lib = _lib or _load()
    _run(lambda a, e: lib.oracle_gdn_fwd_chunked(B, H, T, dk, dv, m, _p(v), _p(b), _p(c), _p(g), _p(beta),
                                                 _p(A_log), _p(h0), _p(o), _p(hT), int(chunk), a, e),
         B, H, threads)
    return o, hT


def gdn_bwd(v, b, c, g, beta, A_log, h0, dO, dhT=None, mode="gated", seg=64, threads=None, _lib=None):
    """fp64 reverse-mode gradients of gdn_fwd.

    Returns a dict with dv, db, dc, dg (same shapes as the inputs), dbeta
    (None in gated mode), dA_log [H, d_k] (summed over the batch) and dh0.
    """
    m = _mode(mode)
    v, b, c, g, A_log, dO = map(_f64, (v, b, c, g, A_log, dO))
    beta, h0, dhT = _f64(beta), _f64(h0), _f64(dhT)
    B, H, T, dk, dv = _shape(v, b)
    out = {
        "dv": np.zeros((B, T, H, dv)),
        "db": np.zeros((B, T, H, dk)),
        "dc": np.zeros((B, T, H, dk)),
        "dg": np.zeros((B, T, H)),
        "dbeta": np.zeros((B, T, H)) if m == DELTA else None,
        "dh0": np.zeros((B, H, dk, dv)),
    }
    dA_unit = np.zeros((B * H, dk))
    lib = _lib or _load()
    _run(lambda a, e: lib.oracle_gdn_bwd(B, H, T, dk, dv, m, _p(v), _p(b), _p(c), _p(g), _p(beta),
                                         _p(A_log), _p(h0), _p(dO), _p(dhT), _p(out["dv"]), _p(out["db"]),
                                         _p(out["dc"]), _p(out["dg"]), _p(out["dbeta"]), _p(dA_unit),
                                         _p(out["dh0"]), int(seg), a, e), B, H, threads)
    out["dA_log"] = dA_unit.reshape(B, H, dk).sum(axis=0)
    return out


def sigmoid(z):
    """The logistic function in fp64: g as the rule uses it, from its logit
    ("GDN & MLA Mechanism Deep-Dive", Gated delta rule: g is the sigmoid of a
    projection); beta takes the same form here."""
    z = _f64(z)
    return None if z is None else 1.0 / (1.0 + np.exp(-z))


def gdn_fwd_logits(v, b, c, zg, zbeta, A_log, h0=None, mode="gated", **kw):
    """gdn_fwd with g (and beta) given as logits: the rule on sigmoid(zg), sigmoid(zbeta)."""
    return gdn_fwd(v, b, c, sigmoid(zg), sigmoid(zbeta), A_log, h0, mode=mode, **kw)


def gdn_bwd_logits(v, b, c, zg, zbeta, A_log, h0, dO, dhT=None, mode="gated", **kw):
    """gdn_bwd with g (and beta) given as logits; dg and dbeta are with respect to the logits
    (the chain rule through the sigmoid: d sigmoid(z)/dz = sigmoid(z) (1 - sigmoid(z)))."""
    g, be = sigmoid(zg), sigmoid(zbeta)
    out = gdn_bwd(v, b, c, g, be, A_log, h0, dO, dhT, mode=mode, **kw)
    out["dg"] = out["dg"] * g * (1.0 - g)
    if be is not None:
        out["dbeta"] = out["dbeta"] * be * (1.0 - be)
    return out


NORM_EPS = 1e-12


def l2_normalize(x):
    """Each vector of the last axis divided by its Euclidean norm, in fp64: x / max(||x||, 1e-12).

    The pages do not spell out a normalisation of b and c; this is the plain reading of an L2
    normalisation of a key vector (the floor of 1e-12 keeps an all-zero vector, such as a padded
    token, at zero)."""
    x = _f64(x)
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    return x / np.maximum(n, NORM_EPS)


def l2_normalize_vjp(x, d):
    """Gradient through l2_normalize: for y = x / n with n = ||x|| > 1e-12, dL/dx = (d - y <y, d>) / n;
    below the floor y = x / 1e-12 and dL/dx = d / 1e-12."""
    x, d = _f64(x), _f64(d)
    n = np.sqrt((x * x).sum(axis=-1, keepdims=True))
    big = n > NORM_EPS
    ns = np.where(big, n, NORM_EPS)
    y = x / ns
    return np.where(big, (d - y * (y * d).sum(axis=-1, keepdims=True)) / ns, d / NORM_EPS)


def gdn_fwd_opts(v, b, c, g, beta, A_log, h0=None, mode="gated", gate_logits=False, norm_bc=False, **kw):
    """gdn_fwd with the library's option bits: g (and beta) as logits, and/or b and c given before their
    L2 normalisation (the rule then runs on l2_normalize(b), l2_normalize(c))."""
    if gate_logits:
        g, beta = sigmoid(g), sigmoid(beta)
    if norm_bc:
        b, c = l2_normalize(b), l2_normalize(c)
    return gdn_fwd(v, b, c, g, beta, A_log, h0, mode=mode, **kw)


def gdn_bwd_opts(v, b, c, g, beta, A_log, h0, dO, dhT=None, mode="gated", gate_logits=False, norm_bc=False,
                 **kw):
    """gdn_bwd with the option bits of gdn_fwd_opts; gradients are with respect to the inputs as given
    (logits, and b and c before normalisation)."""
    if gate_logits:
        return _logit_grads(gdn_bwd_opts(v, b, c, sigmoid(g), sigmoid(beta), A_log, h0, dO, dhT, mode=mode,
                                         norm_bc=norm_bc, **kw), sigmoid(g), sigmoid(beta))
    if not norm_bc:
        return gdn_bwd(v, b, c, g, beta, A_log, h0, dO, dhT, mode=mode, **kw)
    out = gdn_bwd(v, l2_normalize(b), l2_normalize(c), g, beta, A_log, h0, dO, dhT, mode=mode, **kw)
    out["db"] = l2_normalize_vjp(b, out["db"])
    out["dc"] = l2_normalize_vjp(c, out["dc"])
    return out


def _logit_grads(out, g, be):
    out["dg"] = out["dg"] * g * (1.0 - g)
    if be is not None:
        out["dbeta"] = out["dbeta"] * be * (1.0 - be)
    return out


from .chunked_bwd import gdn_bwd_chunked  # noqa: E402  (the chunked reverse mode, numpy)
