"""GB300 (sm_103a) gated delta rule: Python binding of libgdn's C ABI.

The functions below carry the C names (``gdn_fwd``, ``gdn_bwd``,
``gdn_bwd_noalloc``, ``gdn_bwd_noalloc_status``, ``gdn_workspace_bytes``, ``gdn_plan``,
``gdn_last_device_status``, ``gdn_status_string``)
and only marshal arguments: torch tensors become device pointers, ``None``
becomes NULL, and the stream defaults to torch's current stream.  Every step
of the computation runs in libgdn's CUDA kernels.  There is no fallback: if
the library is missing or cannot be loaded, the first call raises.

The operation ("GDN & MLA Mechanism Deep-Dive", Step 4 and Step 5; delta rule
from the card "01 GDN recurrence" of "HyMo-434M -- documentation portal"),
layouts and limits are documented in ``include/gdn.h``.

A forward and backward on torch tensors (v, b, c [B, T, H, d] bf16; g, beta
[B, T, H] bf16; A_log [H, d_k] fp32; states [B, H, d_k, d_v] fp32)::

    import linear_attention_recurrence_delta_gb300 as gdn
    s = gdn.make_shape(B, H, T, dk, dv, "delta", "bf16")          # or "gated" (beta = None)
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
    gdn.check(gdn.gdn_fwd(s, v, b, c, g, beta, A_log, h0, o, hT, ws))
    gdn.check(gdn.gdn_bwd(s, v, b, c, g, beta, A_log, h0, dO, dhT,
                          dv, db, dc, dg, dbeta, dA_log, dh0, ws))
    gdn.check(gdn.gdn_last_device_status(ws))                      # synchronises; GDN_OK or the kernels' error

``h0``, ``hT``, ``dhT``, ``dh0`` may be None; ``make_shape(..., gate_logits=True,
norm_bc=True)`` moves the gates' sigmoid and the L2 normalisation of b and c
into the kernels, and ``gdn_plan(s, backward)`` tells which kernels a call
will use.
"""
from __future__ import annotations

import ctypes
import os
import threading

GDN_GATED, GDN_DELTA = 0, 1
GDN_GATE_LOGITS = 0x100      # option bit: g and beta arrive before their sigmoid
GDN_NORM_BC = 0x200          # option bit: b and c arrive before their L2 normalisation
GDN_CHECK_FINITE = 0x400     # option bit: scan the outputs for NaN / Inf (status GDN_ERR_NONFINITE)
GDN_F32, GDN_BF16 = 0, 1
GDN_OK = 0
GDN_KERNEL_NONE, GDN_KERNEL_DECODE, GDN_KERNEL_TENSOR_CORE, GDN_KERNEL_SERIAL = 0, 1, 2, 3
KERNEL_NAMES = {0: "none", 1: "decode", 2: "tensor_core", 3: "serial"}
GDN_BWD_NONE, GDN_BWD_SERIAL, GDN_BWD_TENSOR_CORE = 0, 1, 2
BWD_KERNEL_NAMES = {0: "none", 1: "serial", 2: "tensor_core"}
STATUS_NAMES = {
    0: "GDN_OK", 1: "GDN_ERR_NULL", 2: "GDN_ERR_SHAPE", 3: "GDN_ERR_ALIGN", 4: "GDN_ERR_MODE",
    5: "GDN_ERR_WORKSPACE", 6: "GDN_ERR_CUDA", 7: "GDN_ERR_TIMEOUT", 8: "GDN_ERR_DEVICE",
    9: "GDN_ERR_NONFINITE",
}

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")
_lib = None
_lock = threading.Lock()


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}{': ' if what else ''}{gdn_status_string(status)}")


class gdn_shape_t(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int), ("dk", ctypes.c_int),
                ("dv", ctypes.c_int), ("mode", ctypes.c_int), ("io", ctypes.c_int)]

    def __repr__(self):
        return (f"gdn_shape_t(B={self.B}, H={self.H}, T={self.T}, dk={self.dk}, dv={self.dv}, "
                f"mode={self.mode}, io={self.io})")


class gdn_plan_t(ctypes.Structure):
    _fields_ = [("segments", ctypes.c_int), ("fwd_kernel", ctypes.c_int), ("bwd_kernel", ctypes.c_int)]


def make_shape(B, H, T, dk, dv, mode="gated", io="bf16", gate_logits=False, norm_bc=False,
               check_finite=False) -> gdn_shape_t:
    m = {"gated": GDN_GATED, "delta": GDN_DELTA}.get(mode, mode)
    d = {"f32": GDN_F32, "bf16": GDN_BF16}.get(io, io)
    if gate_logits:
        m = int(m) | GDN_GATE_LOGITS
    if norm_bc:
        m = int(m) | GDN_NORM_BC
    if check_finite:
        m = int(m) | GDN_CHECK_FINITE
    return gdn_shape_t(int(B), int(H), int(T), int(dk), int(dv), int(m), int(d))


def load(path: str | None = None):
    """Load libgdn.so (once).  Raises if it is missing: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libgdn.so not built ({p}); run __graft_entry__.build() first")
            lib = ctypes.CDLL(p)
            vp, sz, sp = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(gdn_shape_t)
            lib.gdn_workspace_bytes.argtypes = [sp, ctypes.c_int]
            lib.gdn_workspace_bytes.restype = sz
            lib.gdn_plan.argtypes = [sp, ctypes.c_int, ctypes.POINTER(gdn_plan_t)]
            lib.gdn_plan.restype = ctypes.c_int
            lib.gdn_fwd.argtypes = [sp] + [vp] * 9 + [vp, sz, vp]
            lib.gdn_fwd.restype = ctypes.c_int
            lib.gdn_bwd.argtypes = [sp] + [vp] * 16 + [vp, sz, vp]
            lib.gdn_bwd.restype = ctypes.c_int
            lib.gdn_saved_bytes.argtypes = [sp]
            lib.gdn_saved_bytes.restype = sz
            lib.gdn_fwd_save.argtypes = [sp] + [vp] * 9 + [vp, sz, vp, sz, vp]
            lib.gdn_fwd_save.restype = ctypes.c_int
            lib.gdn_bwd_saved.argtypes = [sp] + [vp] * 6 + [vp, sz] + [vp] * 9 + [vp, sz, vp]
            lib.gdn_bwd_saved.restype = ctypes.c_int
            lib.gdn_bwd_noalloc.argtypes = [sp] + [vp] * 16 + [vp]
            lib.gdn_bwd_noalloc.restype = ctypes.c_int
            lib.gdn_bwd_noalloc_status.argtypes = [vp]
            lib.gdn_bwd_noalloc_status.restype = ctypes.c_int
            lib.gdn_last_device_status.argtypes = [vp, vp]
            lib.gdn_last_device_status.restype = ctypes.c_int
            lib.gdn_status_string.argtypes = [ctypes.c_int]
            lib.gdn_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def gdn_workspace_bytes(shape: gdn_shape_t, backward: int) -> int:
    return int(load().gdn_workspace_bytes(ctypes.byref(shape), int(backward)))


def gdn_plan(shape: gdn_shape_t, backward: int) -> gdn_plan_t:
    """How the library runs the shape (host only): time segments and forward kernel; raises GdnError."""
    plan = gdn_plan_t()
    check(int(load().gdn_plan(ctypes.byref(shape), int(backward), ctypes.byref(plan))), "gdn_plan")
    return plan


def gdn_fwd(shape, v, b, c, g, beta, A_log, h0, o, hT, ws, ws_bytes=None, stream=None) -> int:
    """Enqueue the forward; returns the gdn_status_t code (0 = GDN_OK)."""
    wsb = _nbytes(ws) if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return int(load().gdn_fwd(ctypes.byref(shape), _ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(beta), _ptr(A_log),
                              _ptr(h0), _ptr(o), _ptr(hT), _ptr(ws), wsb, _stream(stream)))


def gdn_bwd(shape, v, b, c, g, beta, A_log, h0, dO, dhT, dv, db, dc, dg, dbeta, dA_log, dh0, ws,
            ws_bytes=None, stream=None) -> int:
    """Enqueue the backward; returns the gdn_status_t code (0 = GDN_OK)."""
    wsb = _nbytes(ws) if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return int(load().gdn_bwd(ctypes.byref(shape), _ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(beta), _ptr(A_log),
                              _ptr(h0), _ptr(dO), _ptr(dhT), _ptr(dv), _ptr(db), _ptr(dc), _ptr(dg), _ptr(dbeta),
                              _ptr(dA_log), _ptr(dh0), _ptr(ws), wsb, _stream(stream)))


def gdn_saved_bytes(shape: gdn_shape_t) -> int:
    """Bytes of the residuals gdn_fwd_save keeps for gdn_bwd_saved (0: the shape has none)."""
    return int(load().gdn_saved_bytes(ctypes.byref(shape)))


def gdn_fwd_save(shape, v, b, c, g, beta, A_log, h0, o, hT, saved, ws, saved_bytes=None, ws_bytes=None,
                 stream=None) -> int:
    """gdn_fwd that also writes the chunked backward's residuals into `saved`; returns the status code."""
    svb = _nbytes(saved) if saved_bytes is None and saved is not None else (saved_bytes or 0)
    wsb = _nbytes(ws) if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return int(load().gdn_fwd_save(ctypes.byref(shape), _ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(beta),
                                   _ptr(A_log), _ptr(h0), _ptr(o), _ptr(hT), _ptr(saved), svb, _ptr(ws), wsb,
                                   _stream(stream)))


def gdn_bwd_saved(shape, v, b, c, g, beta, A_log, saved, dO, dhT, dv, db, dc, dg, dbeta, dA_log, dh0, ws,
                  saved_bytes=None, ws_bytes=None, stream=None) -> int:
    """The backward from gdn_fwd_save's residuals; returns the status code."""
    svb = _nbytes(saved) if saved_bytes is None and saved is not None else (saved_bytes or 0)
    wsb = _nbytes(ws) if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return int(load().gdn_bwd_saved(ctypes.byref(shape), _ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(beta),
                                    _ptr(A_log), _ptr(saved), svb, _ptr(dO), _ptr(dhT), _ptr(dv), _ptr(db),
                                    _ptr(dc), _ptr(dg), _ptr(dbeta), _ptr(dA_log), _ptr(dh0), _ptr(ws), wsb,
                                    _stream(stream)))


def gdn_bwd_noalloc(shape, v, b, c, g, beta, A_log, h0, dO, dhT, dv, db, dc, dg, dbeta, dA_log, dh0,
                    stream=None) -> int:
    """gdn_bwd without a workspace argument: the library's own fixed 32 MiB
    device array serves as workspace, so the call allocates nothing."""
    return int(load().gdn_bwd_noalloc(ctypes.byref(shape), _ptr(v), _ptr(b), _ptr(c), _ptr(g), _ptr(beta),
                                      _ptr(A_log), _ptr(h0), _ptr(dO), _ptr(dhT), _ptr(dv), _ptr(db), _ptr(dc),
                                      _ptr(dg), _ptr(dbeta), _ptr(dA_log), _ptr(dh0), _stream(stream)))


def gdn_bwd_noalloc_status(stream=None) -> int:
    """gdn_last_device_status of the array gdn_bwd_noalloc uses as its workspace (synchronises)."""
    return int(load().gdn_bwd_noalloc_status(_stream(stream)))


def gdn_last_device_status(ws, stream=None) -> int:
    return int(load().gdn_last_device_status(_ptr(ws), _stream(stream)))


def gdn_status_string(status: int) -> str:
    try:
        return load().gdn_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(status), f"status {status}")


def check(status: int, what: str = "") -> None:
    if status != GDN_OK:
        raise GdnError(status, what)
