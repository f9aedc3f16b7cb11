"""Seeded synthetic inputs for the gated delta rule.

This module holds no arithmetic of the method itself: it only draws random
tensors and rounds them to the I/O precision.  The CUDA path, the fp64 oracle
and the bench all take their inputs from here, so both sides of every parity
check see bit-identical values.

Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) -- value k of a stream is the
SplitMix64 output mixing function applied to ``key + (k + 1) * 0x9E3779B97F4A7C15``
where ``key`` is derived from (seed, stream id).  Uniforms take the top 53
bits, ``(x >> 11) + 0.5`` scaled by 2^-53, so they lie strictly inside (0, 1).
Normals use the Box-Muller transform on consecutive uniform pairs.  Each
tensor has its own stream, so changing one tensor's shape does not move any
other tensor's values.

Values are produced in float64, transformed (L2 normalisation, sigmoid,
scaling) in float64, then rounded once, round-to-nearest-even, to the I/O
dtype (bf16 or fp32).  ``A_log`` and ``h0`` are always fp32.  The returned
float64 arrays are the rounded values, exactly representable in the I/O dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAMS = {"v": 1, "b": 2, "c": 3, "g": 4, "beta": 5, "A_log": 6, "h0": 7, "dO": 8, "dhT": 9}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed & 0xFFFFFFFF) << 32 | (stream & 0xFFFFFFFF)], dtype=np.uint64)
        return _mix(base + _GOLDEN)[0]


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1) from stream `stream` of seed `seed` (float64)."""
    key = _key(seed, stream)
    with np.errstate(over="ignore"):
        idx = np.arange(1, n + 1, dtype=np.uint64)
        x = _mix(key + idx * _GOLDEN)
    return ((x >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (Box-Muller on consecutive uniform pairs)."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = 2.0 * math.pi * u[1::2]
    z = np.empty(2 * m)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return z[:n]


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), as float64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    finite = np.abs(x[np.isfinite(x)])
    if finite.size and (finite.max() > 3.3e38):
        raise ValueError("value outside the bf16 range")
    bits = x.view(np.uint64).copy()
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        bits = bits + (np.uint64((1 << 44) - 1) + lsb)
    bits &= ~np.uint64((1 << 45) - 1)
    y = bits.view(np.float64)
    # values below the bf16 normal range flush the way fp32->bf16 would not;
    # route them through fp32 (exact for the magnitudes drawn here)
    tiny = np.abs(x) < 1.1754943508222875e-38
    if tiny.any():
        y = y.copy()
        y[tiny] = 0.0
    return y


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


@dataclass(frozen=True)
class Workload:
    """Shape, mode, dtype and input distributions of one synthetic workload."""
    name: str
    mode: str            # "gated" | "delta"
    dtype: str           # "bf16" | "f32"  (I/O dtype of v, b, c, g, beta, o)
    B: int
    H: int
    T: int
    dk: int
    dv: int
    seed: int
    backward: bool = False
    b_dist: str = "normal"     # "normal" | "normal/8" | "l2norm"
    c_dist: str = "normal"     # "normal" | "l2norm"
    g_mu: float = 0.0          # g = sigmoid(N(g_mu, 1))
    h0_std: float = 0.0        # h0 = h0_std * N(0, 1) (0 => no h0)
    gate_logits: bool = False  # g (and beta) drawn as logits N(g_mu, 1) (N(0, 1)), not passed through a sigmoid
    norm_bc: bool = False      # the library normalises b and c itself (GDN_NORM_BC); draw them unnormalised
    alog_max: float = math.log(16.0)   # A_log ~ U(0, alog_max)
    notes: str = ""

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the method is checked and measured on, plus two added points.
WORKLOADS = {
    "gated_f32_1x2x128x16": Workload(
        "gated_f32_1x2x128x16", "gated", "f32", 1, 2, 128, 16, 16, seed=0),
    "gated_bf16_4x16x1024x64_h0": Workload(
        "gated_bf16_4x16x1024x64_h0", "gated", "bf16", 4, 16, 1024, 64, 64, seed=1,
        b_dist="normal/8", h0_std=0.1),
    "delta_bf16_8x16x4096x64": Workload(
        "delta_bf16_8x16x4096x64", "delta", "bf16", 8, 16, 4096, 64, 64, seed=2,
        b_dist="l2norm", c_dist="l2norm"),
    "gated_bf16_8x16x4096x56_bwd": Workload(
        "gated_bf16_8x16x4096x56_bwd", "gated", "bf16", 8, 16, 4096, 56, 56, seed=3,
        backward=True, b_dist="normal/8"),
    "delta_bf16_1x16x32768x64_bwd": Workload(
        "delta_bf16_1x16x32768x64_bwd", "delta", "bf16", 1, 16, 32768, 64, 64, seed=4,
        backward=True, b_dist="l2norm", c_dist="l2norm", g_mu=2.0),
    # added: the gated-mode twin of the 8x16x4096x64 delta workload
    "gated_bf16_8x16x4096x64": Workload(
        "gated_bf16_8x16x4096x64", "gated", "bf16", 8, 16, 4096, 64, 64, seed=5,
        b_dist="normal/8", notes="added gated-mode twin"),
    # added: slow decay (g ~ sigmoid(N(-4,1)), mean log-decay ~ -0.15 per token)
    "delta_bf16_1x16x32768x64_slowdecay": Workload(
        "delta_bf16_1x16x32768x64_slowdecay", "delta", "bf16", 1, 16, 32768, 64, 64, seed=6,
        backward=True, b_dist="l2norm", c_dist="l2norm", g_mu=-4.0,
        notes="added slow-decay stress input"),
    # added: the production-scale head shape of "HyMo-434M -- documentation portal", Worked example
    # (40 heads, d_state = headdim = 32) at the 8 x 4096 batch of the delta workload
    "delta_bf16_8x40x4096x32": Workload(
        "delta_bf16_8x40x4096x32", "delta", "bf16", 8, 40, 4096, 32, 32, seed=8,
        b_dist="l2norm", c_dist="l2norm", notes="added 40-head d = 32 shape"),
    # added: heads 128 wide (d_k = d_v = 128) at the 8 x 4096 x 16-head batch of the delta workload
    "delta_bf16_8x16x4096x128": Workload(
        "delta_bf16_8x16x4096x128", "delta", "bf16", 8, 16, 4096, 128, 128, seed=9,
        backward=True, b_dist="l2norm", c_dist="l2norm", notes="added 128-wide heads"),
    # added: one decoding step (T = 1) of a large batch, state in and out
    "delta_bf16_decode_512x16x1x64": Workload(
        "delta_bf16_decode_512x16x1x64", "delta", "bf16", 512, 16, 1, 64, 64, seed=7,
        b_dist="l2norm", c_dist="l2norm", h0_std=0.1, notes="added single-token decode step"),
}


def _draw_keys(seed, stream, shape, dist):
    B, T, H, d = shape
    z = normal(seed, stream, B * T * H * d).reshape(shape)
    if dist == "normal":
        return z
    if dist == "normal/8":
        return z / 8.0
    if dist == "l2norm":
        return z / np.linalg.norm(z, axis=-1, keepdims=True)
    raise ValueError(dist)


def make_inputs(w: Workload) -> dict:
    """Draw every input of workload `w` (float64 arrays of rounded values).

    Keys: v, b, c [B,T,H,d]; g [B,T,H]; beta [B,T,H] (delta mode, else None);
    A_log [H,d_k] (fp32 values); h0 [B,H,d_k,d_v] or None; dO [B,T,H,d_v]
    and dhT (None) when the workload has a backward pass.
    """
    B, H, T, dk, dv, s = w.B, w.H, w.T, w.dk, w.dv, w.seed
    out = {}
    out["v"] = round_to(normal(s, STREAMS["v"], B * T * H * dv).reshape(B, T, H, dv), w.dtype)
    out["b"] = round_to(_draw_keys(s, STREAMS["b"], (B, T, H, dk), w.b_dist), w.dtype)
    out["c"] = round_to(_draw_keys(s, STREAMS["c"], (B, T, H, dk), w.c_dist), w.dtype)
    squash = (lambda z: z) if w.gate_logits else _sigmoid
    out["g"] = round_to(squash(w.g_mu + normal(s, STREAMS["g"], B * T * H)).reshape(B, T, H), w.dtype)
    if w.mode == "delta":
        out["beta"] = round_to(squash(normal(s, STREAMS["beta"], B * T * H)).reshape(B, T, H), w.dtype)
    else:
        out["beta"] = None
    out["A_log"] = round_to(uniform(s, STREAMS["A_log"], H * dk).reshape(H, dk) * w.alog_max, "f32")
    if w.h0_std > 0:
        out["h0"] = round_to(w.h0_std * normal(s, STREAMS["h0"], B * H * dk * dv).reshape(B, H, dk, dv), "f32")
    else:
        out["h0"] = None
    if w.backward:
        out["dO"] = round_to(normal(s, STREAMS["dO"], B * T * H * dv).reshape(B, T, H, dv), w.dtype)
        out["dhT"] = None
    return out


def custom(name="custom", mode="gated", dtype="bf16", B=1, H=1, T=64, dk=64, dv=64, seed=0,
           **kw) -> Workload:
    """A workload of arbitrary shape (used by the edge-case tests)."""
    if mode == "delta" and not kw.get("norm_bc"):
        kw.setdefault("b_dist", "l2norm")
        kw.setdefault("c_dist", "l2norm")
    return Workload(name, mode, dtype, B, H, T, dk, dv, seed, **kw)
