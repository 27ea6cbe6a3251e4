"""Benchmark of the GB300 exact-attention library.

``python bench.py --gpus N --steps K --warmup W`` (N > 1 under torchrun) prints
one JSON line. A step is one pass of the measured workload through the
library's C ABI -- by default the largest single-GPU configuration, the long
causal bf16 batch (B=2, H=16, L=16384, d=128, N(0,1) inputs): its forward and
its backward, the whole hot path. Device time is taken with CUDA events on the
launching stream, with L2 flushed (a 256 MiB write) before every timed step;
the library's timing hook records a second pair of events around each main
attention kernel, which gives the roofline of the dominant kernel. ``e2e``
repeats the same steps with the inputs copied in from pinned host memory and
the outputs copied back inside the timed region. Every rank runs its own
replica (the work per GPU is fixed: weak scaling); rank 0 prints the
aggregate.

The same line carries the roofline of the dominant kernel, the fp64 CPU
oracle timed on the host cores (for the largest configuration: one whole
(batch, head) slice), SM clocks sampled during the timed region, the
exponential unit's throughput measured by a probe kernel, and (N = 1,
rank 0) per-workload results for all five workloads (forward and backward
TFLOP/s, microseconds per call, fraction of the measured tensor peak).

``--impl reference`` times the oracle itself on the host cores (each step a
bounded sample of the same workload) and prints the same kind of line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SDPA fwd/bwd TFLOP/s and µs/call at 1 GB300; fraction of dense fp16/bf16 peak"
HEADLINE = "long_causal_bf16_d128"
# The tutorial's own number for the dense fp16 d = 32 batch (flash backend,
# 2262.901 us, hardware not stated) in the same unit: 4*B*H*L*L*d / t. The
# pages time no other configuration.
PAGES_WORKLOAD = "dense_f16_d32"
PAGES_TFLOPS = 4.0 * 32 * 32 * 1024 * 1024 * 32 / 2262.901e-6 / 1e12
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
# Used only when the probe library is missing: the exponential unit's rate
# the probe measured on GB300 (32 ex2 results per clock per SM).
EX2_PER_CLK_SM_DEFAULT = 32.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read only) in a
    background thread; falls back to one nvidia-smi query if NVML is absent."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle",
               0x2: "applications_clocks_setting", 0x10: "sync_boost"}

    def __init__(self, index=0, period=0.005):
        self.index, self.period = index, period
        self.samples, self.reasons = [], 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = mx.value
                    self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                        getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            self._nvml = None

    def _sample_nvml(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
            self.samples.append(clk.value)
        if self._reason_fn(self._h, ctypes.byref(rs)) == 0:
            self.reasons |= rs.value

    def _run(self):
        while not self._stop.is_set():
            try:
                self._sample_nvml()
            except Exception:
                return
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._sample_nvml()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def stop(self):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()
            self._sample_nvml()
        else:
            self._smi_once()
        names = sorted(n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle")
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}

    def _smi_once(self):
        import subprocess
        try:
            out = subprocess.run(["nvidia-smi", f"--id={self.index}", "--query-gpu=clocks.sm,clocks.max.sm",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20).stdout
            a, b = out.strip().split(",")[:2]
            self.samples.append(float(a))
            self.max_mhz = float(b)
        except Exception:
            pass


# --------------------------------------------------------------- helpers
def _code_only(text):
    """C/C++ source with comments and blank space removed (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                   # string literal, escapes included
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(name):
    """Short hash of a kernel's code (its .cu plus the shared device headers,
    comments and blank space left out, so an edit of a comment keeps the
    counters taken on that code)."""
    csrc = os.path.join(ROOT, "exact_attention_softmax_gb300", "csrc")
    h = hashlib.sha256()
    deps = [name, "ptx.cuh", "common.cuh"] + (["bwd_common.cuh"] if name.startswith("bwd") else [])
    for f in sorted(deps):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_file, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    want = kernel_source_hash(kernel_file)
    for fn in sorted(os.listdir(prof)):
        if not fn.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(prof, fn)).read()
        for m in re.finditer(r"traffic_per_launch:\s*workload=(\S+)\s+bytes=(\d+)\s+source=(\w+)", text):
            if m.group(1) == workload and m.group(3) == want:
                return int(m.group(2))
    return None


def _unit_arrays(w, x, unit):
    """fp64 arrays (q, k, v, dO or None) of one (batch|sequence, head) unit."""
    if w.varlen:
        cu = x["cu_seqlens"].numpy()
        s_, h = divmod(unit, w.H)
        lo, hi = int(cu[s_]), int(cu[s_ + 1])
        pick = lambda t: t[lo:hi, h]          # noqa: E731
    else:
        b, h = divmod(unit, w.H)
        pick = lambda t: t[b, h]              # noqa: E731
    arrs = [pick(x[n]).double().numpy() for n in ("q", "k", "v")]
    arrs.append(pick(x["do"]).double().numpy() if "do" in x else None)
    return arrs


def oracle_work(w, x, unit, with_bwd, rows=None):
    """Time the fp64 oracle, as it stands, on one unit of the workload --
    forward, and backward when ``with_bwd`` -- or on the query rows
    ``rows = (r0, r1)`` of that unit (every key they see). Returns
    (algorithmic flops, seconds)."""
    import numpy as np
    from oracle import attn_bwd_unit, attn_fwd_unit
    q, k, v, do = _unit_arrays(w, x, unit)
    vis = None
    if rows is None:
        n = q.shape[0]
        pairs = n * k.shape[0] * (0.5 if w.causal else 1.0)
        causal = w.causal
    else:
        r0, r1 = rows
        kv = r1 if w.causal else k.shape[0]
        q, k, v = q[r0:r1], k[:kv], v[:kv]
        do = None if do is None else do[r0:r1]
        if w.causal:
            # query r0 + i sees keys j <= r0 + i
            vis = np.arange(kv)[None, :] <= (r0 + np.arange(r1 - r0))[:, None]
            pairs = float(vis.sum())
        else:
            pairs = float((r1 - r0) * kv)
        causal = False
    flops = 4.0 * w.d * pairs * (3.5 if with_bwd else 1.0)
    t0 = time.perf_counter()
    attn_fwd_unit(q, k, v, w.scale, causal, visible=vis)
    if with_bwd:
        attn_bwd_unit(q, k, v, do, w.scale, causal, visible=vis)
    return flops, time.perf_counter() - t0


def units_of(w, x):
    return (w.nseq if w.varlen else w.B) * w.H


def oracle_sample(w, x, budget_s, with_bwd, max_units=None):
    """Whole units of the workload through the oracle until ``budget_s``
    seconds of CPU work (or ``max_units``); returns (flops, seconds, text)."""
    import numpy as np
    order = np.random.default_rng(0).permutation(units_of(w, x))
    done_flops, t_total, n = 0.0, 0.0, 0
    for u in order:
        f, t = oracle_work(w, x, int(u), with_bwd)
        done_flops += f
        t_total += t
        n += 1
        if t_total >= budget_s or (max_units and n >= max_units):
            break
    what = "forward + backward" if with_bwd else "forward"
    return done_flops, t_total, f"{n} of {len(order)} whole (unit, head) slices of {w.name}, {what}, fp64 NumPy"


def measure_ex2(dev_index=0):
    """Exponentials per SM per clock of the exponential unit, measured by the
    probe kernel (fp32 ex2, and the packed fp16 / bf16 forms); None if the
    probe library is missing."""
    from exact_attention_softmax_gb300.build import PROBE_PATH
    if not os.path.exists(PROBE_PATH):
        return None
    lib = ctypes.CDLL(PROBE_PATH)
    lib.sdpa_probe_ex2.restype = ctypes.c_int
    lib.sdpa_probe_ex2.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_float), ctypes.c_void_p]
    out = {}
    for kind, name in ((0, "f32"), (1, "f16x2"), (2, "bf16x2")):
        per = (ctypes.c_double * 1024)()
        ms = ctypes.c_float()
        runs = []
        for _ in range(3):
            n = lib.sdpa_probe_ex2(kind, 2000, per, ctypes.byref(ms), None)
            if n <= 0:
                return None
            runs.append((statistics.median(per[:n]), ms.value))
        out[name] = {"per_clk_sm": round(max(r[0] for r in runs), 3), "launch_ms": round(min(r[1] for r in runs), 4)}
    return out


def reduce_max_ms(ms, world, device=None):
    """Largest value of ``ms`` over all ranks (the slowest replica sets the job time)."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_step, steps, max_ms):
    """Aggregate throughput: every rank processes its own replica of the workload."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- our arm
class Runner:
    """Holds device inputs/outputs of one workload and runs its calls."""

    def __init__(self, w, x, dev, with_bwd):
        import torch
        import exact_attention_softmax_gb300 as ops
        self.ops, self.w, self.dev = ops, w, dev
        self.q, self.k, self.v = (x[n].to(dev) for n in ("q", "k", "v"))
        self.kw = {}
        if w.varlen:
            self.kw = dict(cu_seqlens=x["cu_seqlens"].to(dev), max_seqlen=x["max_seqlen"])
        self.o = torch.empty_like(self.q)
        lshape = (w.H, self.q.shape[0]) if w.varlen else tuple(self.q.shape[:-1])
        self.lse = torch.empty(lshape, dtype=torch.float32, device=dev)
        self.with_bwd = with_bwd
        if with_bwd:
            self.do = x["do"].to(dev)
            self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))
            code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[self.q.dtype]
            n = ops.sdpa_bwd_workspace_size(self.q.shape[0], w.H, self.q.shape[2], w.d, code)
            self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)

    def fwd(self):
        self.ops.sdpa_fwd(self.q, self.k, self.v, self.o, self.lse, scale=self.w.scale,
                          is_causal=self.w.causal, **self.kw)

    def bwd(self):
        self.ops.sdpa_bwd(self.q, self.k, self.v, self.o, self.lse, self.do, self.dq, self.dk, self.dv,
                          scale=self.w.scale, is_causal=self.w.causal, workspace=self.ws)


def time_calls(fn, iters, flush, stream):
    """Per-call device times (ms) with an L2 flush before each call."""
    import torch
    ts = []
    for _ in range(iters):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ts]


def exp_ceiling_tflops(d, ex2_rate, sms, clk_mhz):
    """Forward ceiling set by the exponential unit: one ex2 per score element,
    4*d algorithmic flops per score element, ``ex2_rate`` results per clock
    per SM."""
    return 4.0 * d * ex2_rate * sms * clk_mhz * 1e6 / 1e12


def per_workload_results(dev, flush, peaks, peak_kind, ex2_rate=EX2_PER_CLK_SM_DEFAULT, clk_mhz=2070):
    """Forward (and backward) timings of all five workloads (N = 1 only)."""
    import torch
    from exact_attention_softmax_gb300 import workloads as wl
    out = {}
    stream = torch.cuda.current_stream(dev)
    for name, w in wl.WORKLOADS.items():
        x = wl.workload_inputs(w, seed=0)
        r = Runner(w, x, dev, w.bwd)
        lengths = x.get("lengths")
        ff = wl.fwd_flops(w, lengths)
        iters = 5 if name == "long_causal_bf16_d128" else 20
        for _ in range(3):
            r.fwd()
            if w.bwd:
                r.bwd()
        torch.cuda.synchronize()
        tf = time_calls(r.fwd, iters, flush, stream)
        res = {"fwd_us": 1e3 * statistics.median(tf), "fwd_us_min": 1e3 * min(tf)}
        res["fwd_tflops"] = ff / (res["fwd_us"] * 1e-6) / 1e12
        res["fwd_frac_of_peak"] = res["fwd_tflops"] / peaks["bf16_tflops"] if w.dtype != "f32" else None
        if name == "dense_f16_d32":
            min_bytes = 2 * 4 * w.B * w.H * w.Lq * w.d + 4 * w.B * w.H * w.Lq
            res["fwd_hbm_gbs"] = min_bytes / (res["fwd_us"] * 1e-6) / 1e9
            res["fwd_frac_of_hbm"] = res["fwd_hbm_gbs"] / peaks["hbm_gbs"]
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            res["fwd_frac_of_exp_ceiling"] = res["fwd_tflops"] / exp_ceiling_tflops(w.d, ex2_rate, sms, clk_mhz)
        if w.bwd:
            tb = time_calls(r.bwd, iters, flush, stream)
            bf = wl.bwd_flops(w, lengths)
            res["bwd_us"] = 1e3 * statistics.median(tb)
            res["bwd_tflops"] = bf / (res["bwd_us"] * 1e-6) / 1e12
            res["bwd_frac_of_peak"] = res["bwd_tflops"] / peaks["bf16_tflops"] if w.dtype != "f32" else None
        res["fwd_gflop"] = ff / 1e9
        res["peak"] = f"{peak_kind} bf16 dense {peaks['bf16_tflops']:.1f} TFLOP/s"
        out[name] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in res.items()}
        del r, x
        torch.cuda.empty_cache()
    return out


def extra_results(dev, flush, peaks):
    """Timings of the layouts and masks added beyond the five workloads:
    block-sparse attention and packed cross-attention (N = 1 only)."""
    import torch
    import exact_attention_softmax_gb300 as ops
    from exact_attention_softmax_gb300 import workloads as wl
    out = {}
    stream = torch.cuda.current_stream(dev)

    def timed(name, fwd, bwd, ff, bf, desc):
        for _ in range(3):
            fwd()
            bwd()
        torch.cuda.synchronize()
        tf = time_calls(fwd, 20, flush, stream)
        tb = time_calls(bwd, 20, flush, stream)
        res = {"config": desc, "fwd_us": 1e3 * statistics.median(tf), "bwd_us": 1e3 * statistics.median(tb)}
        res["fwd_tflops"] = ff / (res["fwd_us"] * 1e-6) / 1e12
        res["bwd_tflops"] = bf / (res["bwd_us"] * 1e-6) / 1e12
        res["fwd_frac_of_peak"] = res["fwd_tflops"] / peaks["bf16_tflops"]
        out[name] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in res.items()}

    # block-sparse: half of the 128 x 128 score tiles kept (seeded), flops counted on kept tiles
    B, H, L, d = 4, 16, 4096, 64
    x = wl.dense_inputs(B, H, L, L, d, "f16", "normal", seed=0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    mask = wl.block_mask((B, H, L // 128, L // 128), 0.5, seed=0).to(dev)
    kept = float(mask.sum().item()) * 128 * 128
    o, lse = ops.sdpa_fwd_blocksparse(q, k, v, mask)
    ws = torch.empty(ops.sdpa_bwd_workspace_size(B, H, L, d, 1), dtype=torch.uint8, device=dev)
    g = [torch.empty_like(t) for t in (q, k, v)]
    timed("blocksparse_f16_d64", lambda: ops.sdpa_fwd_blocksparse(q, k, v, mask, o, lse),
          lambda: ops.sdpa_bwd_blocksparse(q, k, v, o, lse, do, mask, *g, workspace=ws),
          4 * d * kept, 2.5 * 4 * d * kept,
          f"B={B} H={H} L={L} d={d} f16 non-causal, 50 % of 128x128 tiles kept (seeded)")
    # the dense calls on the same shape, for the block-sparse saving
    od, ld = torch.empty_like(q), torch.empty(B, H, L, dtype=torch.float32, device=dev)
    for _ in range(3):
        ops.sdpa_fwd(q, k, v, od, ld)
        ops.sdpa_bwd(q, k, v, od, ld, do, *g, workspace=ws)
    torch.cuda.synchronize()
    dense_f = statistics.median(time_calls(lambda: ops.sdpa_fwd(q, k, v, od, ld), 20, flush, stream)) * 1e3
    dense_b = statistics.median(time_calls(lambda: ops.sdpa_bwd(q, k, v, od, ld, do, *g, workspace=ws), 20, flush,
                                           stream)) * 1e3
    e = out["blocksparse_f16_d64"]
    e["dense_fwd_us"], e["dense_bwd_us"] = round(dense_f, 3), round(dense_b, 3)
    e["fwd_time_vs_dense"] = round(e["fwd_us"] / dense_f, 4)
    e["bwd_time_vs_dense"] = round(e["bwd_us"] / dense_b, 4)
    del od, ld
    del q, k, v, do, o, lse, g, ws, x

    # additive mask: one [L, L] mask per head (about 10 % -inf), shared over the batch
    x = wl.dense_inputs(B, H, L, L, d, "f16", "normal", seed=0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    am = wl.attn_mask((1, H, L, L), "f16", seed=0).to(dev)[..., :L]
    o, lse = ops.sdpa_fwd_masked(q, k, v, am)
    ws = torch.empty(ops.sdpa_bwd_workspace_size(B, H, L, d, 1), dtype=torch.uint8, device=dev)
    g = [torch.empty_like(t) for t in (q, k, v)]
    timed("masked_f16_d64", lambda: ops.sdpa_fwd_masked(q, k, v, am, o, lse),
          lambda: ops.sdpa_bwd_masked(q, k, v, o, lse, do, am, *g, workspace=ws),
          4.0 * d * B * H * L * L, 2.5 * 4.0 * d * B * H * L * L,
          f"B={B} H={H} L={L} d={d} f16 non-causal, additive mask [1, {H}, {L}, {L}] f16 (N(0,1), 10 % -inf)")
    del q, k, v, do, o, lse, g, ws, x, am

    # dropout on the probabilities, p = 0.1 (Philox keep pattern from a fixed seed)
    x = wl.dense_inputs(B, H, L, L, d, "f16", "normal", seed=0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = ops.sdpa_fwd_dropout(q, k, v, 0.1, 1234)
    ws = torch.empty(ops.sdpa_bwd_workspace_size(B, H, L, d, 1), dtype=torch.uint8, device=dev)
    g = [torch.empty_like(t) for t in (q, k, v)]
    timed("dropout_f16_d64", lambda: ops.sdpa_fwd_dropout(q, k, v, 0.1, 1234, o, lse),
          lambda: ops.sdpa_bwd_dropout(q, k, v, o, lse, do, 0.1, 1234, *g, workspace=ws),
          4.0 * d * B * H * L * L, 2.5 * 4.0 * d * B * H * L * L,
          f"B={B} H={H} L={L} d={d} f16 non-causal, dropout p = 0.1")
    del q, k, v, do, o, lse, g, ws, x

    # strided: the SDPA tutorial module's [B, L, 3E] projection viewed as
    # [B, H, L, d] (the causal d = 64 workload's shape), outputs written into
    # [B, L, E] / [B, L, 3E] views, no copy
    B, L, H, d = 32, 1024, 8, 64
    E = H * d
    g = torch.Generator("cpu").manual_seed(0)
    qkv = torch.randn(B, L, 3 * E, generator=g).half().to(dev)
    q, k, v = (t.view(B, L, H, d).transpose(1, 2) for t in qkv.split(E, dim=2))
    do = torch.randn(B, L, E, generator=g).half().to(dev).view(B, L, H, d).transpose(1, 2)
    o = torch.empty(B, L, E, dtype=torch.half, device=dev).view(B, L, H, d).transpose(1, 2)
    dqkv = torch.empty(B, L, 3 * E, dtype=torch.half, device=dev)
    g3 = [t.view(B, L, H, d).transpose(1, 2) for t in dqkv.split(E, dim=2)]
    _, lse = ops.sdpa_fwd(q, k, v, o, is_causal=True)
    ws = torch.empty(ops.sdpa_bwd_workspace_size(B, H, L, d, 1), dtype=torch.uint8, device=dev)
    timed("strided_module_f16_d64", lambda: ops.sdpa_fwd(q, k, v, o, lse, is_causal=True),
          lambda: ops.sdpa_bwd(q, k, v, o, lse, do, *g3, is_causal=True, workspace=ws),
          2.0 * d * B * H * L * L, 2.5 * 2.0 * d * B * H * L * L,
          f"B={B} H={H} L={L} d={d} f16 causal, q/k/v views of a [B, L, 3E] projection, O and dQ/dK/dV "
          "written into [B, L, E] / [B, L, 3E] views (strided calls, no copy)")
    del qkv, q, k, v, do, o, dqkv, g3, lse, ws

    # the dispatcher example's d = 32 batch, trained: forward and backward
    B, H, L, d = 32, 32, 1024, 32
    x = wl.dense_inputs(B, H, L, L, d, "f16", "normal", seed=0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = ops.sdpa_fwd(q, k, v)
    ws = torch.empty(ops.sdpa_bwd_workspace_size(B, H, L, d, 1), dtype=torch.uint8, device=dev)
    g = [torch.empty_like(t) for t in (q, k, v)]
    timed("dense_f16_d32_train", lambda: ops.sdpa_fwd(q, k, v, o, lse),
          lambda: ops.sdpa_bwd(q, k, v, o, lse, do, *g, workspace=ws),
          4.0 * d * B * H * L * L, 2.5 * 4.0 * d * B * H * L * L,
          f"B={B} H={H} L={L} d={d} f16 non-causal, forward and backward")
    del x, q, k, v, do, o, lse, ws, g

    # packed cross-attention: 32 sequences, queries around 256 long, keys around 512
    lq = wl.varlen_lengths(32, 512, 0.5, 0)
    lk = wl.varlen_lengths(32, 1024, 0.5, 1)
    x = wl.varlen_cross_inputs(lq, lk, 8, 64, "f16", "normal", seed=0)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    cq, ck = x["cu_seqlens_q"].to(dev), x["cu_seqlens_k"].to(dev)
    mq, mk = x["max_seqlen_q"], x["max_seqlen_k"]
    o, lse = ops.sdpa_fwd_varlen(q, k, v, cq, ck, mq, mk)
    ws = torch.empty(ops.sdpa_bwd_workspace_size(1, 8, q.shape[0], 64, 1), dtype=torch.uint8, device=dev)
    g = [torch.empty_like(t) for t in (q, k, v)]
    pairs = float(sum(a * b for a, b in zip(lq, lk)))
    timed("cross_varlen_f16_d64", lambda: ops.sdpa_fwd_varlen(q, k, v, cq, ck, mq, mk, o, lse),
          lambda: ops.sdpa_bwd_varlen(q, k, v, o, lse, do, cq, ck, mq, mk, *g, workspace=ws),
          4 * 8 * 64 * pairs, 2.5 * 4 * 8 * 64 * pairs,
          f"32 sequences, query lengths sum {sum(lq)} (max {mq}), key lengths sum {sum(lk)} (max {mk}), H=8 d=64 f16")
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    from exact_attention_softmax_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import exact_attention_softmax_gb300 as ops
    ops._abi.load()

    peaks, peak_kind = load_peaks()
    w = wl.WORKLOADS[args.workload]
    x = wl.workload_inputs(w, seed=rank)
    lengths = x.get("lengths")
    passes = args.passes if args.passes != "auto" else ("both" if w.bwd else "fwd")
    do_fwd = passes in ("fwd", "both")
    do_bwd = passes in ("bwd", "both")
    if do_bwd and not w.bwd:
        raise SystemExit(f"workload {w.name} has no backward")
    fwd_f = wl.fwd_flops(w, lengths)
    bwd_f = wl.bwd_flops(w, lengths) if w.bwd else 0.0
    flops = (fwd_f if do_fwd else 0.0) + (bwd_f if do_bwd else 0.0)
    r = Runner(w, x, dev, with_bwd=do_bwd)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # kernels of one step: the forward's, and the backward's row-statistic
    # pass, main kernel and dQ conversion
    launches_per_step = (1 if do_fwd else 0) + (3 if do_bwd else 0)
    ex2 = measure_ex2(local)
    ex2_rate = ex2["f32"]["per_clk_sm"] if ex2 else EX2_PER_CLK_SM_DEFAULT

    def step():
        if do_fwd:
            r.fwd()
        if do_bwd:
            r.bwd()

    r.fwd()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    ops.sdpa_device_status()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # one event pair per step around each main kernel (the library records
    # them on the launching stream); created before the timed region
    def pairs(n):
        ps = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a_, b_ in ps:
            a_.record(stream)
            b_.record(stream)
        return ps
    kev = {"fwd": pairs(args.steps) if do_fwd else [], "bwd": pairs(args.steps) if do_bwd else []}

    # ---- device-resident timed region
    clocks = ClockSampler(local).start()
    barrier()
    evs = []
    for i in range(args.steps):
        flush.zero_()
        if do_fwd:
            ops.sdpa_trace_events("fwd", *kev["fwd"][i])
        if do_bwd:
            ops.sdpa_trace_events("bwd", *kev["bwd"][i])
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        evs.append((a, b))
    barrier()
    clk = clocks.stop()
    ops.sdpa_trace_events("fwd")
    ops.sdpa_trace_events("bwd")
    kernel_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = reduce_max_ms(sum(kernel_ms), world, dev)
    main_ms = {k: [a.elapsed_time(b) for a, b in v] for k, v in kev.items() if v}
    ops.sdpa_device_status()

    # ---- end to end: pinned host inputs in, outputs out, inside the timed region
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.empty(r.o.shape, dtype=r.o.dtype).pin_memory()
    hl = torch.empty(r.lse.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    if w.varlen:
        h2d += x["cu_seqlens"].numel() * 4
    d2h = ho.numel() * ho.element_size() + hl.numel() * 4
    if do_bwd:
        hd = x["do"].pin_memory()
        hg = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (r.dq, r.dk, r.dv)]
        h2d += hd.numel() * hd.element_size()
        d2h += sum(t.numel() * t.element_size() for t in hg)
    e2e_steps = max(1, min(args.steps, 20))
    # Steps are pipelined the way a serving loop would run them: two sets of
    # device buffers and three streams, so step k+1's inputs travel to the GPU
    # and step k-1's outputs travel back while step k computes. Every step's
    # copies are inside the timed region.
    rb = [r, Runner(w, x, dev, do_bwd)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer b on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # compute finished with buffer b
    ev_out = [torch.cuda.Event() for _ in range(2)]    # outputs of buffer b copied back

    def e2e_steps_run(n):
        for i in range(n):
            bi, rr = i % 2, rb[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[bi])
                rr.q.copy_(hq, non_blocking=True)
                rr.k.copy_(hk, non_blocking=True)
                rr.v.copy_(hv, non_blocking=True)
                if do_bwd:
                    rr.do.copy_(hd, non_blocking=True)
                ev_in[bi].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[bi])
                if i >= 2:
                    s_cmp.wait_event(ev_out[bi])
                rr.fwd()
                if do_bwd:
                    rr.bwd()
                ev_done[bi].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[bi])
                if do_bwd:
                    for h, g in zip(hg, (rr.dq, rr.dk, rr.dv)):
                        h.copy_(g, non_blocking=True)
                ho.copy_(rr.o, non_blocking=True)
                hl.copy_(rr.lse, non_blocking=True)
                ev_out[bi].record(s_out)

    e2e_steps_run(2)
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    s_cmp.wait_event(a)
    s_out.wait_event(a)
    e2e_steps_run(e2e_steps)
    stream.wait_stream(s_in)
    stream.wait_stream(s_cmp)
    stream.wait_stream(s_out)
    b.record(stream)
    barrier()
    e2e_ms = reduce_max_ms(a.elapsed_time(b), world, dev)

    value = whole_job_tflops(world, flops, args.steps, total_ms)
    # the end-to-end step always runs the forward (the backward needs its O and LSE)
    e2e_flops = flops + (fwd_f if not do_fwd else 0.0)
    e2e_value = whole_job_tflops(world, e2e_flops, e2e_steps, e2e_ms)

    # Rooflines of the main kernels, from their own events. The tensor-core
    # ceiling is the measured dense bf16 peak (fp16 has the same rate); the
    # small-head-dim forward has a lower one, the exponential unit's: one ex2
    # per score element at the rate the probe measured.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_mhz = clk.get("sm_max_mhz") or 2070
    # (the d <= 64 backward of dense batches runs the persistent kernel,
    # packed batches and d = 128 the one-CTA-per-key-block kernel)
    bwd_k = ("bwd_persist_kernel", "bwd_persist.cu") if w.d <= 64 and not w.varlen else ("bwd_tc_kernel", "bwd_tc.cu")
    kinfo = {"fwd": ("fwd_tc_kernel", "fwd_tc.cu", fwd_f), "bwd": (bwd_k[0], bwd_k[1], bwd_f)}
    kernels = {}
    for key, ms in main_ms.items():
        name, src, f = kinfo[key]
        avg_s = statistics.mean(ms) * 1e-3
        achieved = f / avg_s / 1e12
        exp_ceiling = exp_ceiling_tflops(w.d, ex2_rate, sms, clk_mhz)
        if key == "fwd" and exp_ceiling < peaks["bf16_tflops"]:
            roof = {"kernel": name, "bound": "alu", "achieved": round(achieved, 2), "peak": round(exp_ceiling, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / exp_ceiling, 4),
                    "peak_source": f"exponential unit: {ex2_rate:g} ex2/clk/SM (probe, measured in this run) x "
                                   f"{sms} SMs x {clk_mhz} MHz, {4 * w.d} flop per score element",
                    "tensor_peak": peaks["bf16_tflops"], "tensor_frac": round(achieved / peaks["bf16_tflops"], 4)}
        else:
            roof = {"kernel": name, "bound": "tensor", "achieved": round(achieved, 2),
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "peak_source": f"{peak_kind} dense bf16 burst (fp16 has the same tensor rate), of {peak_kind}"}
        roof["us_per_launch"] = round(1e3 * statistics.mean(ms), 2)
        roof["share_of_step"] = round(sum(ms) / sum(kernel_ms), 4)
        roof["traffic"] = profiled_traffic(src, w.name)
        kernels[name] = roof
    dominant = max(kernels.values(), key=lambda k: k["share_of_step"])
    shape = (f"B={w.B} H={w.H} Lq={w.Lq} Lk={w.Lk} d={w.d}" if not w.varlen else
             f"{w.nseq} packed sequences (max {w.max_len}, total {x['q'].shape[0]}) H={w.H} d={w.d}")
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "us_per_call": round(1e3 * total_ms / args.steps, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": (round(value / world / PAGES_TFLOPS, 3)
                        if args.workload == PAGES_WORKLOAD and passes == "fwd" else None),
        "dtype": w.dtype,
        "data": "synthetic (seeded torch.rand / torch.randn of the workload's shape)",
        "config": {"workload": f"{w.name}: {shape} {w.dtype} {w.dist} "
                               f"{'causal' if w.causal else 'non-causal'} {passes}",
                   "flops_per_step": flops, "fwd_flops": fwd_f if do_fwd else 0.0,
                   "bwd_flops": bwd_f if do_bwd else 0.0,
                   "l2": "flushed before every timed step (256 MiB write)",
                   "parallelism": f"replicas x{world} (one independent problem per GPU)"},
        "roofline": dominant,
        "kernels": kernels,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "pipelining": "inputs of step k+1 and outputs of step k-1 copied while step k computes "
                              "(two device buffer sets, three streams)"},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
        "ex2_probe": ex2,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if w.name == HEADLINE:
            # the largest configuration: one whole (batch, head) slice
            f, sec = oracle_work(w, x, 0, do_bwd)
            desc = (f"one whole (batch, head) slice, (0, 0), of {w.name} (1 of {units_of(w, x)}), "
                    f"{'forward + backward' if do_bwd else 'forward'}, fp64 NumPy")
        else:
            f, sec, desc = oracle_sample(w, x, args.cpu_budget, do_bwd)
        line["cpu_baseline"] = {"value": round(f / sec / 1e12, 6), "unit": "TFLOP/s", "cores": host_cores(),
                                "kind": "oracle", "sample": desc + f", {sec:.1f} s"}
    if rank == 0 and world == 1 and not args.no_extras:
        line["per_workload"] = per_workload_results(dev, flush, peaks, peak_kind, ex2_rate, clk_mhz)
        line["extras"] = extra_results(dev, flush, peaks)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 oracle, as it stands, on the host cores; each step is a bounded
    sample of the workload: one whole (batch, head) unit, or for the long
    sequences a block of 1024 query rows of one unit (with every key those
    rows see), the blocks walking over units and positions from step to step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from exact_attention_softmax_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    x = wl.workload_inputs(w, seed=0)
    passes = args.passes if args.passes != "auto" else ("both" if w.bwd else "fwd")
    with_bwd = passes in ("bwd", "both")
    nunits = units_of(w, x)
    blocked = not w.varlen and w.Lq > 4096
    rows = 1024

    def sample(i):
        unit = (7 * i) % nunits
        if blocked:
            nb = w.Lq // rows
            r0 = ((5 * i + 3) % nb) * rows
            return oracle_work(w, x, unit, with_bwd, rows=(r0, r0 + rows))
        return oracle_work(w, x, unit, with_bwd)

    for i in range(args.warmup):
        sample(1000 + i)
    flops = secs = 0.0
    for i in range(args.steps):
        f, t = sample(i)
        flops += f
        secs += t
    value = flops / secs / 1e12
    what = "forward + backward" if with_bwd else "forward"
    desc = (f"per step one block of {rows} query rows of one (batch, head) unit of {w.name} with every key "
            f"they see, {what}, fp64 NumPy" if blocked else
            f"per step one whole (unit, head) slice of {w.name}, {what}, fp64 NumPy")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "passes": passes, "sample_per_step": desc},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": host_cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--pass", dest="passes", choices=["auto", "fwd", "bwd", "both"], default="auto",
                    help="what one step runs (auto: forward and backward where the workload has a backward)")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
