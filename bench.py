"""Throughput of the gated delta rule on GB300 (tokens/s), one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward pass (gdn_fwd, every forward row of the chunked
recurrence) over one batch of the named workload, inputs already resident in
device memory; the line also carries the forward+backward throughput of the
same shape (gdn_fwd_save followed by gdn_bwd_saved where the shape has the
residual hand-off, else gdn_fwd followed by gdn_bwd), the end-to-end throughput through
the C ABI with host buffers (host->device copies of the inputs and the
device->host read of the outputs inside the timed region), the roofline of
the dominant kernel, the clocks seen during the timed region and the fp64
CPU oracle timed on the host cores as a baseline.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and a device synchronise on both sides; CUDA events on the launching stream.
The default workload's inputs (272.6 MB) exceed the 129 MB L2, so no flush is
needed between steps.  Multi-GPU runs (torchrun) are independent replicas, one
batch per rank (weak scaling, no collective on the data path); rank 0 prints
the whole-job tokens/s over the max time across ranks.

--impl reference times the fp64 CPU oracle on the same workload and metric: each
step is a bounded sample of the workload (every head of one batch row).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from linear_attention_recurrence_delta_gb300 import inputs as I  # noqa: E402

DEFAULT_WORKLOAD = "delta_bf16_8x16x4096x64"
METRIC = "GDN fwd / fwd+bwd tokens/sec at H=16,T=4096,d=64 bf16; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one forward launch from an ncu capture, with the
# SHA-256 of the kernel's source files at the time of the capture.  When a source no longer matches, the counters
# describe another kernel and the line reports traffic = null until the capture is retaken.
MEASURED_TRAFFIC = {
    # profiles/fwd_tc_delta_8x16x4096x64.md: dram__bytes_read.sum 203650304 + dram__bytes_write.sum 43600384
    "delta_bf16_8x16x4096x64": {"bytes": 247250688, "files": ["gdn_fwd_tc.cu", "fwd_tc_common.cuh", "tc_ptx.cuh"],
                                "sha256": "7a759f9f630b5aa0044a8d73ada005759034e2d39db730ed384a683bc9361406"},
}


def source_digest(files):
    """SHA-256 over the named files of the library's csrc/ (in the order given)."""
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "linear_attention_recurrence_delta_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(name):
    """Captured DRAM bytes per launch for workload `name`, or None if absent or captured on other sources."""
    rec = MEASURED_TRAFFIC.get(name)
    if rec is None:
        return None
    return rec["bytes"] if source_digest(rec["files"]) == rec["sha256"] else None


def chunk_flops(w, backward=False):
    """Algorithmic tensor FLOPs of the chunked form over workload w (chunks of C = 64, full tiles).

    Per chunk and head, the contractions of the closed form (2 * m * n * k each):
      forward, both modes: P = (c-side) (b-side)^T        2 C^2 d_k
                           O = Ctil S + P U              2 C d_k d_v + 2 C^2 d_v
                           S' = Bhat^T U                 2 C d_k d_v
      forward, delta adds: K (the b b^T scores)          2 C^2 d_k
                           [Util | W] = (I+M)^-1 R       2 C^2 (d_v + d_k)
                           U = Util - W S                2 C d_k d_v
      backward: the forward's products again (recomputed) plus their transposes: every forward product
      X = A B contributes dA = dX B^T and dB = A^T dX, i.e. twice its own FLOPs.
    """
    C, dk, dv = 64, w.dk, w.dv
    f = 2 * C * C * dk + 2 * C * dk * dv + 2 * C * C * dv + 2 * C * dk * dv
    if w.mode == "delta":
        f += 2 * C * C * dk + 2 * C * C * (dv + dk) + 2 * C * dk * dv
    chunks = -(-w.T // C) * w.B * w.H
    return chunks * f * (3 if backward else 1)


def io_bytes(w, backward=False):
    """Algorithmic HBM bytes of one forward (or backward) launch over workload w:
    every input read once, every output written once."""
    e = 2 if w.dtype == "bf16" else 4
    tok = w.B * w.T * w.H
    per_tok = (2 * w.dk + 2 * w.dv) * e + e + (e if w.mode == "delta" else 0)   # v,b,c,o + g (+beta)
    state = w.B * w.H * w.dk * w.dv * 4
    fwd = tok * per_tok + state + w.H * w.dk * 4 + (state if w.h0_std > 0 else 0)
    if not backward:
        return fwd
    # backward: reads v,b,c,g,(beta),dO (+A_log, h0, dhT); writes dv,db,dc,dg,(dbeta) (+dA_log, dh0)
    rd = tok * ((2 * w.dk + 2 * w.dv) * e + e + (e if w.mode == "delta" else 0))
    wr = tok * ((2 * w.dk + w.dv) * e + e + (e if w.mode == "delta" else 0))
    return rd + wr + 2 * state + 2 * w.H * w.dk * 4


def plan(w, backward):
    """The library's own answer (gdn_plan) for workload w: time segments and forward kernel."""
    import linear_attention_recurrence_delta_gb300 as gdn
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype, gate_logits=w.gate_logits, norm_bc=w.norm_bc)
    return gdn.gdn_plan(s, backward)


def tsplit_factor(w, backward):
    """Segments of the library's time split for workload w (1 = none)."""
    return plan(w, backward).segments


def fwd_launches(w, saving=False):
    """Kernels one gdn_fwd call (gdn_fwd_save if saving) launches."""
    if tsplit_factor(w, False) == 1:
        return 1
    if saved_bytes(w) > 0:
        # the split by walks: zero-start run, Phi and Qc, transition walks, scan, output walks (and, saving, the
        # residuals' fix-up)
        return 6 if saving else 5
    return 5 if w.mode == "delta" else 3   # zero-start run, (identity, transition run), scan, output kernel


def saved_bytes(w):
    """gdn_saved_bytes of workload w: the residuals a saving forward keeps (0: it keeps none)."""
    import linear_attention_recurrence_delta_gb300 as gdn
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype, gate_logits=w.gate_logits, norm_bc=w.norm_bc)
    return gdn.gdn_saved_bytes(s)


def bwd_slabs(w):
    """Column slabs of the serial backward (64 value columns per CTA up to d_k = 64, 32 above)."""
    cols = 64 if w.dk <= 64 else 32
    return -(-w.dv // cols)


def bwd_launches(w, saved=False):
    """Kernels one gdn_bwd call (gdn_bwd_saved if saved) launches."""
    p = plan(w, True)
    if p.bwd_kernel == 2:
        # chunked backward: prep, chain, gradients, dA_log sum; a chain split in time runs as first walks over the
        # segments, a scan and second walks
        return 4 if plan(w, 2 if saved else 1).segments == 1 else 6
    if tsplit_factor(w, True) == 1:
        # backward, the slabs' partial sums of db, dc, dg (, dbeta) if several, dA_log reduction
        sums = (4 if w.mode == "delta" else 3) if bwd_slabs(w) > 1 else 0
        return 2 + sums
    P = tsplit_factor(w, True)
    states = 4 if w.mode == "delta" else 2  # zero-start run, (identity, transition run), scan
    runs = -(-(w.T // P) // 512)            # G_p by runs of 512 tokens, their partials summed if several
    return states + 1 + (1 if runs > 1 else 0) + 1 + 2   # G_p (+ sum), reverse scan, backward + dA_log sum


def tc_fwd_ex2_per_launch(w):
    """exp2 evaluations of one tcgen05 forward launch on workload w (overflow-safe chunks), from the kernel:
    per chunk and head, the anchors exp(A (G_t - G_r)) and their inverses (2 per token and channel: 2 * 64 * 64),
    the per-(8-block, reference) constant tables (42 of the 64 (table, 8-block) pairs are live, per channel:
    42 * 64) and the chunk's decay row (64).  None for the other kernels."""
    if plan(w, False).fwd_kernel != 2 or tsplit_factor(w, False) > 1:
        return None
    chunks = -(-w.T // 64) * w.B * w.H * -(-w.dv // 64)
    return chunks * (2 * 64 * 64 + 42 * 64 + 64)


def ex2_rate():
    """exp2 evaluations per second of the special-function units, measured by bench_probes/ex2_rate.cu (built
    here into _build/libgdn_probe.so, outside the library), or None if it cannot be built."""
    import ctypes
    from linear_attention_recurrence_delta_gb300 import _build
    src = os.path.join(ROOT, "bench_probes", "ex2_rate.cu")
    path = os.path.join(ROOT, "_build", "libgdn_probe.so")
    if not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(path), exist_ok=True)
        cmd = [_build.nvcc(), "-std=c++17", "-O3", "-Xcompiler", "-fPIC", *_build.ARCH, "-shared", src, "-o", path,
               "-lcudart"]
        if subprocess.run(cmd, capture_output=True).returncode != 0:
            return None
    lib = ctypes.CDLL(path)
    lib.gdn_probe_ex2_rate.restype = ctypes.c_int
    lib.gdn_probe_ex2_rate.argtypes = [ctypes.POINTER(ctypes.c_double)]
    r = ctypes.c_double(0.0)
    return r.value if lib.gdn_probe_ex2_rate(ctypes.byref(r)) == 0 else None


def host_link(nbytes_in, nbytes_out, reps=5):
    """Host link bandwidth with pinned buffers of the end-to-end step's sizes (copy engines, cudaMemcpyAsync):
    host->device alone, device->host alone, and both directions at once; GB/s, best of `reps`."""
    import torch
    hi = torch.empty(nbytes_in, dtype=torch.uint8).pin_memory()
    di = torch.empty(nbytes_in, dtype=torch.uint8, device="cuda")
    ho = torch.empty(nbytes_out, dtype=torch.uint8).pin_memory()
    do = torch.empty(nbytes_out, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best(fn):
        out = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            out.append(time.perf_counter() - t0)
        return min(out)

    def h2d():
        with torch.cuda.stream(s1):
            di.copy_(hi, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            ho.copy_(do, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = best(h2d), best(d2h), best(both)
    return {"h2d_gbs": nbytes_in / t_in / 1e9, "d2h_gbs": nbytes_out / t_out / 1e9,
            "both_gbs": (nbytes_in + nbytes_out) / t_both / 1e9, "both_ms": t_both * 1e3,
            "how": "pinned host buffers of the step's input and output bytes, cudaMemcpyAsync on two streams, "
                   "best of %d, host wall clock around a device synchronise" % reps}


def fwd_kernel_name(w):
    """The kernel gdn_fwd launches for workload w (one launch per call), as gdn_plan reports it."""
    k = plan(w, False).fwd_kernel
    if k == 1:
        return "decode_kernel (one launch)"
    if k == 2:
        return f"fwd_tc_kernel<{w.mode}> (one launch)"
    return f"serial_fwd_kernel<{w.dtype}, {w.mode}> (one launch)"


def roofline_of(nbytes, flops, ms, peaks, peak_kind):
    """Roofline of a launch (or step) of `ms` milliseconds moving `nbytes` algorithmic bytes and doing `flops`
    algorithmic tensor FLOPs: time = max(bytes / HBM, FLOPs / bf16 dense peak); the bound is the larger term."""
    hbm_ms = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    flop_ms = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    achieved = nbytes / (ms * 1e-3) / 1e9
    r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "frac": achieved / peaks["hbm_gbs"], "peak_kind": peak_kind, "bytes_per_launch": nbytes,
         "launch_ms": ms, "hbm_floor_ms": hbm_ms, "flops_per_launch": flops, "flop_floor_ms": flop_ms,
         "tensor_frac": flops / (ms * 1e-3) / (peaks["bf16_tflops"] * 1e12)}
    if flop_ms > hbm_ms:
        r.update({"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
                  "unit": "TFLOP/s", "frac": flop_ms / ms})
    return r


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle
# ---------------------------------------------------------------------------

def oracle_sample(w, x):
    """Every head of batch row 0: T tokens' worth of work (units = H)."""
    sl = lambda a: None if a is None else a[:1]
    return {k: (sl(v) if k not in ("A_log",) else v) for k, v in x.items()}


def time_oracle(w, x, steps, warmup, min_seconds=0.0):
    """Time the fp64 oracle forward on batch row 0 (all heads, all tokens).
    Repeats the sample until at least `min_seconds` of wall time per step."""
    import oracle
    xs = oracle_sample(w, x)
    threads = os.cpu_count() or 1
    fn = lambda: oracle.gdn_fwd(xs["v"], xs["b"], xs["c"], xs["g"], xs["beta"], xs["A_log"], xs["h0"],
                                mode=w.mode, threads=threads)
    for _ in range(warmup):
        fn()
    reps = 1
    if min_seconds > 0:
        t0 = time.perf_counter()
        fn()
        one = max(time.perf_counter() - t0, 1e-6)
        reps = max(1, int(min_seconds / one + 0.999))
    t0 = time.perf_counter()
    for _ in range(steps * reps):
        fn()
    dt = (time.perf_counter() - t0) / (steps * reps)
    tokens = w.T  # one batch row, all heads
    return tokens / dt, dt, min(threads, w.H), reps


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = I.WORKLOADS[args.workload]
    x = I.make_inputs(w)
    value, dt, cores, reps = time_oracle(w, x, args.steps, args.warmup)
    sample = f"batch row 0 of {w.name}: all {w.H} heads x {w.T} tokens per step, serial fp64"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "pass": "fwd", "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                   "mode": w.mode, "io": w.dtype},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-bwd", action="store_true", help="skip the forward+backward measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch B (profiling captures)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's length T (profiling captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
        return

    import numpy as np
    import torch

    import linear_attention_recurrence_delta_gb300 as gdn
    from linear_attention_recurrence_delta_gb300 import _build, replicas

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    gdn.load()

    base = I.WORKLOADS[args.workload]
    if args.batch or args.tokens:
        B, T = args.batch or base.B, args.tokens or base.T
        base = base.with_(name=f"{base.name}@B{B}T{T}", B=B, T=T)
    w = replicas.rank_workload(base, rank, world)
    wb = w.with_(backward=True)
    x = I.make_inputs(wb)
    s = gdn.make_shape(w.B, w.H, w.T, w.dk, w.dv, w.mode, w.dtype)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = lambda a: None if a is None else torch.from_numpy(a).to("cuda", dt)
    dev32 = lambda a: None if a is None else torch.from_numpy(a).to("cuda", torch.float32)
    t = {k: dev(x[k]) for k in ("v", "b", "c", "g", "beta", "dO")}
    A_log, h0 = dev32(x["A_log"]), dev32(x["h0"])
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=dt, device="cuda")
    hT = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    ws = torch.empty(gdn.gdn_workspace_bytes(s, 1), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def fwd():
        gdn.check(gdn.gdn_fwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, o, hT, ws,
                              stream=stream), "gdn_fwd")

    grads = {
        "dv": torch.empty_like(t["v"]), "db": torch.empty_like(t["b"]), "dc": torch.empty_like(t["c"]),
        "dg": torch.empty_like(t["g"]), "dbeta": torch.empty_like(t["beta"]) if t["beta"] is not None else None,
        "dA_log": torch.empty_like(A_log), "dh0": torch.empty_like(hT),
    }

    def bwd():
        gdn.check(gdn.gdn_bwd(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, t["dO"], None,
                              grads["dv"], grads["db"], grads["dc"], grads["dg"], grads["dbeta"], grads["dA_log"],
                              grads["dh0"], ws, stream=stream), "gdn_bwd")

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return replicas.max_over_ranks(v, dist, device="cuda")

    def timed(step_fn, K, W):
        for _ in range(W):
            step_fn()
        barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(K):
            ev[k][0].record(stream)
            step_fn()
            ev[k][1].record(stream)
        end.record(stream)
        barrier()
        total_ms = start.elapsed_time(end)
        per = [a.elapsed_time(b) for a, b in ev]
        return max_over_ranks(total_ms), statistics.mean(per)

    tokens = w.B * w.T
    with ClockSampler(local) as clk:
        total_ms, launch_ms = timed(fwd, args.steps, args.warmup)
    clocks = clk.summary()
    ms_per_step = total_ms / args.steps
    value = replicas.whole_job_tokens_per_s(tokens, world, ms_per_step)
    gdn.check(gdn.gdn_last_device_status(ws), "device status")

    peaks, peak_kind = load_peaks()
    fwd_bytes = io_bytes(w)
    roofline = roofline_of(fwd_bytes, chunk_flops(w), launch_ms, peaks, peak_kind)
    roofline.update({"traffic": measured_traffic(w.name), "kernel": fwd_kernel_name(w)})
    # launches of our kernels per forward step: the forward kernel itself
    gpu_launches = fwd_launches(w) * args.steps

    # secondary bound: the forward's exponentials on the special-function units (measured rate)
    mufu = None
    n_ex2 = tc_fwd_ex2_per_launch(w)
    rate = ex2_rate() if n_ex2 else None
    if rate:
        floor_ms = n_ex2 / rate * 1e3
        mufu = {"ex2_per_s": rate, "ex2_per_launch": n_ex2, "floor_ms": floor_ms,
                "frac_of_launch": floor_ms / launch_ms}

    # End to end through the C ABI with host buffers.  Every step copies its inputs from pinned host memory,
    # runs gdn_fwd and reads its outputs back; as a serving loop would, step k+1's input copies overlap
    # step k's forward and step k-1's output copies (three streams, two device buffer sets).
    in_keys = [k for k in ("v", "b", "c", "g", "beta") if t[k] is not None]
    hx = {k: t[k].cpu().pin_memory() for k in in_keys}
    hA = A_log.cpu().pin_memory()
    hh0 = h0.cpu().pin_memory() if h0 is not None else None
    dbuf = [{k: torch.empty_like(t[k]) for k in in_keys} for _ in range(2)]
    dA = [torch.empty_like(A_log) for _ in range(2)]
    dh0 = [torch.empty_like(h0) if h0 is not None else None for _ in range(2)]
    dout = [(torch.empty_like(o), torch.empty_like(hT)) for _ in range(2)]
    hout = [(torch.empty(o.shape, dtype=dt).pin_memory(), torch.empty(hT.shape, dtype=torch.float32).pin_memory())
            for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in hx.values()) + hA.numel() * 4 + \
        (hh0.numel() * 4 if hh0 is not None else 0)
    d2h = o.numel() * o.element_size() + hT.numel() * 4
    s_in, s_fw, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_fw = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ws_e2e = torch.empty(gdn.gdn_workspace_bytes(s, 0), dtype=torch.uint8, device="cuda")

    def e2e_run(K):
        for e in ev_fw + ev_out:
            e.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        for k in range(K):
            j = k % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_fw[j])            # the forward that last read this buffer set is done
                for key in in_keys:
                    dbuf[j][key].copy_(hx[key], non_blocking=True)
                dA[j].copy_(hA, non_blocking=True)
                if hh0 is not None:
                    dh0[j].copy_(hh0, non_blocking=True)
                ev_in[j].record(s_in)
            s_fw.wait_event(ev_in[j])
            s_fw.wait_event(ev_out[j])               # its outputs were read back
            d = dbuf[j]
            gdn.check(gdn.gdn_fwd(s, d["v"], d["b"], d["c"], d["g"], d.get("beta"), dA[j], dh0[j], dout[j][0],
                                  dout[j][1], ws_e2e, stream=s_fw), "gdn_fwd")
            ev_fw[j].record(s_fw)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fw[j])
                hout[j][0].copy_(dout[j][0], non_blocking=True)
                hout[j][1].copy_(dout[j][1], non_blocking=True)
                ev_out[j].record(s_out)
        s_out.wait_event(ev_out[(K - 1) % 2])
        end.record(s_out)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    Ke = max(6, args.steps)
    e2e_run(3)
    barrier()
    e2e_total = max_over_ranks(e2e_run(Ke))
    barrier()
    e2e_ms = e2e_total / Ke
    got = hout[(Ke - 1) % 2][0].to(torch.float32)
    ref = o.to(torch.float32).cpu()
    assert torch.equal(got, ref), "end-to-end outputs differ from the device-resident run"
    link = host_link(h2d, d2h)
    e2e = {"value": replicas.whole_job_tokens_per_s(tokens, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "overlap": "step k+1 inputs in, step k forward, step k-1 outputs out on three streams",
           "host_link": link, "link_floor_ms": link["both_ms"], "frac_of_link_floor": link["both_ms"] / e2e_ms}
    gpu_launches += fwd_launches(w) * Ke

    fwdbwd = None
    if not args.no_bwd:
        # training step: the forward keeps the chunked backward's residuals where the shape has them
        n_saved = gdn.gdn_saved_bytes(s)
        if n_saved:
            saved = torch.empty(n_saved, dtype=torch.uint8, device="cuda")
            ws2 = torch.empty(gdn.gdn_workspace_bytes(s, 2), dtype=torch.uint8, device="cuda")

            def fb():
                gdn.check(gdn.gdn_fwd_save(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, h0, o, hT, saved,
                                           ws, stream=stream), "gdn_fwd_save")
                gdn.check(gdn.gdn_bwd_saved(s, t["v"], t["b"], t["c"], t["g"], t["beta"], A_log, saved, t["dO"],
                                            None, grads["dv"], grads["db"], grads["dc"], grads["dg"],
                                            grads["dbeta"], grads["dA_log"], grads["dh0"], ws2, stream=stream),
                          "gdn_bwd_saved")
        else:
            def fb():
                fwd()
                bwd()
        kb = max(3, args.steps // 4)
        fb_total, fb_launch = timed(fb, kb, 3)
        fb_ms = fb_total / kb
        fb_bytes = fwd_bytes + io_bytes(w, backward=True)
        fb_flops = chunk_flops(w) + chunk_flops(w, backward=True)
        fwdbwd = {"value": replicas.whole_job_tokens_per_s(tokens, world, fb_ms), "unit": "tokens/s",
                  "ms_per_step": fb_ms, "bwd_bytes": io_bytes(w, backward=True),
                  "calls": "gdn_fwd_save + gdn_bwd_saved" if n_saved else "gdn_fwd + gdn_bwd",
                  "saved_bytes": n_saved,
                  "roofline": roofline_of(fb_bytes, fb_flops, fb_ms, peaks, peak_kind)}
        gpu_launches += (fwd_launches(w, saving=bool(n_saved)) + bwd_launches(w, saved=bool(n_saved))) * kb

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v_cpu, dt_cpu, cores, reps = time_oracle(w, x, 1, 1, min_seconds=1.5)
        cpu = {"value": v_cpu, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"batch row 0 of {w.name} (all {w.H} heads x {w.T} tokens), serial fp64 forward, "
                         f"repeated {reps}x, {dt_cpu * reps:.2f} s wall on {cores} threads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if w.dtype == "f32" else "bf16", "data": "synthetic",
            "config": {"workload": w.name, "pass": "fwd", "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                       "mode": w.mode, "io": w.dtype, "parallelism": "replicas" if world > 1 else "single",
                       "l2": (f"inputs+outputs {fwd_bytes / 1e6:.1f} MB > 129 MB L2, no flush" if fwd_bytes > 129e6
                              else f"inputs+outputs {fwd_bytes / 1e6:.1f} MB fit the 129 MB L2: L2-warm, no flush")},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "fwd_bwd": fwdbwd, "clocks": clocks,
            "gpu_launches": gpu_launches, "mufu": mufu,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
