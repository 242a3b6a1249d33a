#!/usr/bin/env python3
"""Throughput benchmark of the SDPA forward library on synthetic workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--headline-only]

One step of the headline workload is one fused prefill launch over the GQA causal
batch (B=2, Hq=32, Hkv=8, Sq=Sk=4096, D=Dv=128, bf16); `value` is its throughput in
TFLOP/s of algorithmic work (2 (D + Dv) per visible query/key pair), inputs resident in
HBM, L2 flushed before every timed step.  The other workloads (tiny fp16 prefill,
unaligned + additive mask, split-KV decode in GB/s, MLA FP8 prefill) are timed the same way
and reported under "workloads".  For N > 1 (torchrun) every rank runs the same workload on
its own GPU (replicas; no collective on the data path) and `value` sums the ranks' work over
the slowest rank's time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload on the
host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s (prefill) & HBM GB/s (decode), % of GB300 roofline"
HEADLINE = "gqa_causal_prefill_bf16_d128"
L2_FLUSH_BYTES = 256 << 20
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor ratio (4.5 / 2.25 PFLOP/s)
# dense e4m3 library GEMM measured on this GPU type with `python bench.py --tensor-peaks`
# (torch._scaled_mm, 16384^3, best of 10): context beside the nominal-ratio FP8 peak
FP8_MEASURED_TFLOPS = 3783.0


# ----------------------------------------------------------------------------- work counts

def visible_pairs(Sq: int, Sk: int, causal: bool) -> int:
    """(i, j) pairs with key j visible to query i (top-left causal: j <= i)."""
    if not causal:
        return Sq * Sk
    m = min(Sq, Sk)
    return m * (m + 1) // 2 + max(0, Sq - Sk) * Sk


def prefill_flops(w) -> float:
    return 2.0 * (w.D + w.Dv) * w.B * w.Hq * visible_pairs(w.Sq, w.Sk, w.causal)


def varlen_flops(w, lengths) -> float:
    return sum(2.0 * (w.D + w.Dv) * w.Hq * visible_pairs(L, L, w.causal) for L in lengths)


def decode_bytes(w, kv_len) -> float:
    esz = 2
    kv = float(np.sum(np.asarray(kv_len, dtype=np.int64))) * w.Hkv * (w.D + w.Dv) * esz
    return kv + w.B * w.Hq * (w.D + w.Dv) * esz


# ----------------------------------------------------------------------------- environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _code_only(text: str) -> str:
    """Source text without // and /* */ comments and with whitespace collapsed, so that edits to
    comments do not count as kernel changes (the kernel sources hold no string literal with //)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_sha() -> str:
    """Hash of the kernel sources' code (comments and whitespace ignored)."""
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "flash_attention_forward_gb300", "csrc", "*"))):
        with open(p, encoding="utf-8") as f:
            h.update(os.path.basename(p).encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu capture, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(workload)
    if not d or d.get("source_sha") != source_sha():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- timing

# The launch queue is primed before the timed steps: a GPU-side sleep (torch's bounded
# clock-count spin) holds the stream while the host enqueues the first steps, so that the events
# around a step measure the device's time for it and not the host's time to prepare its launch.
# The sleep runs before the first event, outside every timed step.
PRIME_US_PER_STEP = 150.0
PRIME_MAX_US = 20000.0
PRIME_CLOCK_HZ = 2.07e9


def prime_queue(steps: int):
    us = min(PRIME_MAX_US, PRIME_US_PER_STEP * max(1, steps))
    torch.cuda._sleep(int(us * 1e-6 * PRIME_CLOCK_HZ))


def time_steps(step, K: int, W: int, flush=None, host_us=None, prime=True):
    """W untimed steps, then K steps each bracketed by CUDA events on the launching stream
    (an optional L2 flush runs before each step, outside the events; unless prime is False the
    queue is primed first).  Returns per-step ms; host_us, if given, receives the host time of
    each step() call in us."""
    stream = torch.cuda.current_stream()
    for _ in range(W):
        if flush:
            flush()
        step(-1)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if prime:
        prime_queue(K)
    for i in range(K):
        if flush:
            flush()
        ev[i][0].record(stream)
        t0 = time.perf_counter()
        step(i)
        if host_us is not None:
            host_us.append((time.perf_counter() - t0) * 1e6)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def step_stats(ms):
    """Mean, median, min, max and 10th / 90th percentiles of per-step times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"mean": float(a.mean()), "median": float(np.median(a)), "min": float(a.min()), "max": float(a.max()),
            "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90)), "n": int(a.size)}


class Flusher:
    def __init__(self, dev):
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.fill_(1)


def prefill_setup(w, dev, rotation=0):
    import flash_attention_forward_gb300 as fa

    x = workloads.prefill_inputs(w, rotation)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    mask = x["mask"].to(dev) if x["mask"] is not None else None
    out_dtype = torch.float16 if w.dtype == "f16" else torch.bfloat16
    o = torch.empty((w.B, w.Sq, w.Hq, w.Dv), dtype=out_dtype, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    ws = None
    need = fa.sdpa_fwd_workspace_size(w.B, w.Hq, w.Sq, w.Sk, w.Dv, w.causal, mask is not None)
    if need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    dq, dk, dv = x["descale"]

    def step(_i=0):
        if w.dtype == "e4m3":
            fa.sdpa_fwd_fp8(q, k, v, dq, dk, dv, scale=w.scale, causal=w.causal, mask=mask, out=o, lse=lse,
                            workspace=ws)
        else:
            fa.sdpa_fwd(q, k, v, scale=w.scale, causal=w.causal, mask=mask, out=o, lse=lse, workspace=ws)

    return x, step


def bench_prefill(w, K, W, dev, peaks, flusher):
    _, step = prefill_setup(w, dev)
    ms = time_steps(step, K, W, flusher)
    flops = prefill_flops(w)
    avg = sum(ms) / len(ms)
    tflops = flops / (avg * 1e-3) / 1e12
    launches = 1 + (1 if w.mask else 0)
    bf16 = peaks["bf16_tflops"]
    r = {"workload": w.name, "value": tflops, "unit": "TFLOP/s", "ms_per_step": avg, "flops_per_step": flops,
         "launches_per_step": launches, "step_ms": step_stats(ms)}
    if w.dtype == "e4m3":
        fp8 = bf16 * FP8_PER_BF16
        qk = 2.0 * w.D * w.B * w.Hq * visible_pairs(w.Sq, w.Sk, w.causal)
        pv = flops - qk
        mixed = flops / (qk / fp8 + pv / bf16)
        r["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": fp8, "unit": "TFLOP/s", "frac": tflops / fp8,
                         "peak_note": "FP8 = measured bf16 burst x 2 (nominal ratio); of measured",
                         "mixed_ceiling": mixed, "frac_of_mixed_ceiling": tflops / mixed,
                         "fp8_measured_peak": FP8_MEASURED_TFLOPS, "frac_of_measured_fp8": tflops / FP8_MEASURED_TFLOPS,
                         "traffic": recorded_traffic(w.name)}
    else:
        r["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": bf16, "unit": "TFLOP/s", "frac": tflops / bf16,
                         "peak_note": "bf16 burst, of " + peaks["source"], "traffic": recorded_traffic(w.name)}
    return r


def varlen_setup(w, dev, rotation=0):
    import flash_attention_forward_gb300 as fa

    x = workloads.varlen_inputs(w, rotation)
    q, k, v, cu_q, cu_k = (x[n].to(dev) for n in ("q", "k", "v", "cu_q", "cu_k"))
    total_q = q.shape[0]
    o = torch.empty((total_q, w.Hq, w.Dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.Hq, total_q), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.sdpa_fwd_varlen_workspace_size(w.B), dtype=torch.uint8, device=dev)
    max_q = max(x["lengths"])

    def step(_i=0):
        fa.sdpa_fwd_varlen(q, k, v, cu_q, cu_k, max_q, scale=w.scale, causal=w.causal, out=o, lse=lse, workspace=ws)

    return x, step


def bench_varlen(w, K, W, dev, peaks, flusher):
    """Packed sequences of the drawn lengths: one tile-prefix scan and one prefill per step."""
    x, step = varlen_setup(w, dev)
    ms = time_steps(step, K, W, flusher)
    flops = varlen_flops(w, x["lengths"])
    avg = sum(ms) / len(ms)
    tflops = flops / (avg * 1e-3) / 1e12
    bf16 = peaks["bf16_tflops"]
    return {"workload": w.name, "value": tflops, "unit": "TFLOP/s", "ms_per_step": avg, "flops_per_step": flops,
            "launches_per_step": 2, "sequences": w.B, "total_tokens": int(sum(x["lengths"])),
            "step_ms": step_stats(ms),
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16, "unit": "TFLOP/s", "frac": tflops / bf16,
                         "peak_note": "bf16 burst, of " + peaks["source"], "traffic": recorded_traffic(w.name)}}


def int8_setup(w, dev, rotation=0):
    import flash_attention_forward_gb300 as fa

    x = workloads.int8_inputs(w, rotation)
    g = {n: (None if t is None else t.to(dev)) for n, t in x.items()}
    out_dtype = workloads.torch_dtype(w.out_dtype)
    o = torch.empty((w.B, w.Sq, w.Hq, w.Dv), dtype=out_dtype, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.sdpa_fwd_int8_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, g["v_scale"] is not None,
                                                     w.causal), dtype=torch.uint8, device=dev)

    def step(_i=0):
        fa.sdpa_fwd_int8(g["q"], g["k"], g["v"], g["q_scale"], g["k_scale"], g["v_scale"], scale=w.scale,
                         causal=w.causal, out_dtype=out_dtype, out=o, lse=lse, workspace=ws)

    return x, step


def bench_int8(w, K, W, dev, peaks, flusher):
    """int8 Q/K codes: the widening copy and the block-scaled prefill per step."""
    _, step = int8_setup(w, dev)
    ms = time_steps(step, K, W, flusher)
    flops = prefill_flops(w)
    avg = sum(ms) / len(ms)
    tflops = flops / (avg * 1e-3) / 1e12
    bf16 = peaks["bf16_tflops"]
    return {"workload": w.name, "value": tflops, "unit": "TFLOP/s", "ms_per_step": avg, "flops_per_step": flops,
            "launches_per_step": 2, "step_ms": step_stats(ms),
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16, "unit": "TFLOP/s", "frac": tflops / bf16,
                         "peak_note": "16-bit MMA (no int8 MMA on sm_103a); bf16 burst, of " + peaks["source"],
                         "traffic": recorded_traffic(w.name)}}


def bench_decode(w, K, W, dev, peaks, page_size: int = 64, n_sets: int = 4, paged: bool = True):
    """The split-KV decode over n_sets rotating input sets (each far larger than L2), then, if
    paged, the same rows in page_size-row pages scattered over a pool (the paged decode).
    Returns (contiguous line, paged line or None)."""
    import flash_attention_forward_gb300 as fa

    sets = []
    for r in range(n_sets):  # rotating buffer sets, every one far larger than L2
        x = workloads.decode_inputs(w, rotation=r, pad_value=0.0)
        d = {n: x[n].to(dev) for n in ("q", "k", "v", "kv_len")}
        d["bytes"] = decode_bytes(w, x["kv_len"].numpy())
        sets.append(d)
        del x
    o = torch.empty((w.B, w.Hq, w.Dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.sdpa_decode_workspace_size(w.B, w.Hq, w.Sk, w.Dv), dtype=torch.uint8, device=dev)
    hbm = peaks["hbm_gbs"]

    def line(name, ms, launches, extra=None):
        by = [sets[i % n_sets]["bytes"] for i in range(K)]
        gbs = [b / (t * 1e-3) / 1e9 for b, t in zip(by, ms)]
        value = sum(by) / (sum(ms) * 1e-3) / 1e9
        r = {"workload": name, "value": value, "unit": "GB/s", "ms_per_step": sum(ms) / K, "bytes_per_step": sum(by) / K,
             "launches_per_step": launches, "per_step_gbs_min": min(gbs), "step_ms": step_stats(ms),
             "roofline": {"bound": "hbm", "achieved": value, "peak": hbm, "unit": "GB/s", "frac": value / hbm,
                          "peak_note": "copy bandwidth, of " + peaks["source"], "traffic": recorded_traffic(name)}}
        if extra:
            r.update(extra)
        return r

    def step(i):
        s = sets[i % n_sets] if i >= 0 else sets[0]
        fa.sdpa_decode(s["q"], s["k"], s["v"], s["kv_len"], scale=w.scale, out=o, lse=lse, workspace=ws)

    contiguous = line(w.name, time_steps(step, K, W), 2)
    if not paged:
        return contiguous, None
    for r, d in enumerate(sets):  # the same rows, paged: every page lands at a seeded random pool slot
        d["kp"], d["vp"], d["table"] = workloads.page_caches(d["k"], d["v"], page_size, seed=100 + r, spare_pages=64)
        del d["k"], d["v"]
    torch.cuda.empty_cache()

    def step_paged(i):
        s = sets[i % n_sets] if i >= 0 else sets[0]
        fa.sdpa_decode_paged(s["q"], s["kp"], s["vp"], s["table"], s["kv_len"], scale=w.scale, out=o, lse=lse,
                             workspace=ws)

    paged = line("paged_" + w.name, time_steps(step_paged, K, W), 2,
                 {"page_size": page_size, "pages": "seeded random placement in a pool with 64 spare pages"})
    return contiguous, paged


def bench_e2e_prefill(w, K, dev):
    """Same metric through the public host-buffer call (sdpa_fwd_host): every step copies the
    inputs from pinned host memory to the device, computes, and copies O and LSE back to pinned
    host memory, the library overlapping the three over chunks of query rows; all of it timed."""
    import flash_attention_forward_gb300 as fa

    x = workloads.prefill_inputs(w)
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.empty((w.B, w.Sq, w.Hq, w.Dv), dtype=hq.dtype).pin_memory()
    hl = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.sdpa_fwd_host_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.Dv, w.causal),
                     dtype=torch.uint8, device=dev)

    def step(_i):
        fa.sdpa_fwd_host(hq, hk, hv, scale=w.scale, causal=w.causal, out=ho, lse=hl, workspace=ws)

    # no queue priming here: the end-to-end time includes the host's work of every call
    ms = time_steps(step, K, 3, prime=False)
    avg = sum(ms) / len(ms)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return {"value": prefill_flops(w) / (avg * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": avg,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "api": "sdpa_fwd_host (pinned host buffers)",
            "link": link_floor((hq, hk, hv), (ho, hl), dev)}


def link_floor(ups, downs, dev, reps: int = 5):
    """The host link alone on the same pinned buffers: the upward copies, the downward copies,
    and both at once on two streams (median of reps, CUDA events).  The last is the floor of any
    end-to-end step that moves these bytes."""
    dups = [torch.empty_like(t, device=dev) for t in ups]
    ddowns = [torch.empty_like(t, device=dev) for t in downs]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_up = sum(t.numel() * t.element_size() for t in ups)
    n_down = sum(t.numel() * t.element_size() for t in downs)

    def timed(up: bool, down: bool) -> float:
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            main = torch.cuda.current_stream()
            a.record(main)
            for st, go, pairs in ((s_up, up, zip(dups, ups)), (s_down, down, zip(downs, ddowns))):
                if not go:
                    continue
                st.wait_event(a)
                with torch.cuda.stream(st):
                    for dst, src in pairs:
                        dst.copy_(src, non_blocking=True)
                main.wait_stream(st)
            b.record(main)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return float(np.median(ts))

    t_up, t_down, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_ms": t_up, "h2d_gbs": n_up / (t_up * 1e-3) / 1e9, "d2h_ms": t_down,
            "d2h_gbs": n_down / (t_down * 1e-3) / 1e9, "both_concurrent_ms": t_both,
            "note": "plain copies of the step's bytes on two streams: the floor of an end-to-end step"}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(w, target_s: float, seed: int = 0):
    """Rows of the workload for a bounded oracle run: (inputs, rows, flops of those rows)."""
    import oracle

    x = workloads.prefill_inputs(w)
    g = np.random.default_rng(seed)

    def flops_of(rows):
        vis = [min(i + 1, w.Sk) if w.causal else w.Sk for (_, _, i) in rows]
        return 2.0 * (w.D + w.Dv) * float(sum(vis))

    def pick(n):
        b = g.integers(w.B, size=n)
        h = g.integers(w.Hq, size=n)
        i = g.integers(w.Sq, size=n)
        return np.stack([b, h, i], axis=1).astype(np.int64)

    probe = pick(256)
    t0 = time.perf_counter()
    oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"], scale=w.scale, causal=w.causal, rows=probe,
                    descale=x["descale"])
    dt = max(time.perf_counter() - t0, 1e-3)
    # rows are drawn with replacement, up to four times the workload's rows
    n = int(max(256, min(4 * w.B * w.Hq * w.Sq, 256 * target_s / dt)))
    rows = pick(n)
    return x, rows, flops_of(rows)


def run_oracle(w, x, rows):
    import oracle

    t0 = time.perf_counter()
    oracle.sdpa_fwd(x["q"], x["k"], x["v"], x["mask"], scale=w.scale, causal=w.causal, rows=rows,
                    descale=x["descale"])
    return time.perf_counter() - t0


def cpu_baseline(w, target_s=15.0):
    import oracle

    x, rows, flops = oracle_sample(w, target_s)
    t = run_oracle(w, x, rows)
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{len(rows)} random query rows (b, h, i), drawn with replacement, of {w.name}, fp64, "
                      f"{t:.1f} s on the host cores",
            "seconds": t}


# ----------------------------------------------------------------------------- main

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 0, 1
    import torch.distributed as dist

    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest x over all ranks (the slowest rank's time); x itself on a single process."""
    if world <= 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank_step: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time (per second)."""
    return world * work_per_rank_step * steps / (max_ms * 1e-3)


def config_of(w):
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D, "Dv": w.Dv,
         "dtype": w.dtype, "causal": w.causal, "mask": w.mask}
    return c


def main_reference(args, rank, world):
    if rank != 0:
        return
    import oracle

    oracle.build()
    w = workloads.WORKLOADS[HEADLINE]
    # about 150 s of oracle work for the whole run, whatever --steps and --warmup are
    per_step_s = max(0.01, 150.0 / max(1, args.steps + args.warmup))
    x, rows, flops = oracle_sample(w, per_step_s)
    for _ in range(args.warmup):
        run_oracle(w, x, rows)
    ts = [run_oracle(w, x, rows) for _ in range(args.steps)]
    total = sum(ts)
    value = flops * len(ts) / total / 1e12
    cfg = config_of(w)
    cfg["l2"] = "n/a (host CPU)"
    cfg["parallelism"] = f"replicas x{world}"  # the same key as the GPU arm's line
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / len(ts) * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg, "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"each step: {len(rows)} random query rows of {w.name} in fp64"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def profile_run(args):
    """Launch one workload's kernels warmup + steps times and print their mean time (no L2 flush,
    no e2e, no CPU baseline): a small, self-contained command for ncu captures."""
    import flash_attention_forward_gb300 as fa

    fa.library()
    w = workloads.WORKLOADS[args.profile]
    if args.batch:
        w = w.with_shape(B=args.batch)
    dev = torch.device("cuda", torch.cuda.current_device())
    if w.kind == "decode":
        x = workloads.decode_inputs(w, pad_value=0.0)
        q, k, v, kvl = (x[n].to(dev) for n in ("q", "k", "v", "kv_len"))
        ws = torch.empty(fa.sdpa_decode_workspace_size(w.B, w.Hq, w.Sk, w.Dv), dtype=torch.uint8, device=dev)
        if args.page_size:
            kp, vp, table = workloads.page_caches(k, v, args.page_size, seed=100, spare_pages=64)
            del k, v

            def step(_i=0):
                fa.sdpa_decode_paged(q, kp, vp, table, kvl, scale=w.scale, workspace=ws)
        else:
            def step(_i=0):
                fa.sdpa_decode(q, k, v, kvl, scale=w.scale, workspace=ws)
    elif w.kind == "varlen":
        _, step = varlen_setup(w, dev)
    elif w.dtype == "i8":
        _, step = int8_setup(w, dev)
    else:
        _, step = prefill_setup(w, dev)
    ms = time_steps(step, max(args.steps, 1), max(args.warmup, 1))
    status = fa.sdpa_status_string(fa.sdpa_check_device_status())
    print(json.dumps({"profile": w.name, "B": w.B, "page_size": args.page_size or None, "ms_per_step": sum(ms) / len(ms),
                      "device_status": status}))


def tensor_peaks(dev, n: int = 8192, reps: int = 10, sustain_s: float = 4.0):
    """Dense GEMM throughput of the library GEMMs on this GPU, measured like the bf16 figure the
    roofline uses: torch.matmul bf16 and torch._scaled_mm e4m3 (per-tensor scales, bf16 out) at
    n^3, best of reps (burst) and back to back for sustain_s (sustained), CUDA events."""
    out = {"n": n, "method": f"best of {reps} (burst) and back to back for {sustain_s} s (sustained), CUDA events"}
    a16 = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    b16 = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    one = torch.ones((), device=dev, dtype=torch.float32)
    a8 = a16.to(torch.float8_e4m3fn)
    b8t = b16.to(torch.float8_e4m3fn).t()  # column-major second operand
    fns = {"bf16": lambda: torch.matmul(a16, b16),
           "e4m3": lambda: torch._scaled_mm(a8, b8t, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)}
    flops = 2.0 * n ** 3
    for name, fn in fns.items():
        try:
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1))
            count, t_end = 0, time.perf_counter() + sustain_s
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            while time.perf_counter() < t_end:
                for _ in range(20):
                    fn()
                count += 20
                torch.cuda.synchronize()
            e1.record()
            torch.cuda.synchronize()
            out[name] = {"burst_tflops": flops / (best * 1e-3) / 1e12,
                         "sustained_tflops": flops * count / (e0.elapsed_time(e1) * 1e-3) / 1e12}
        except Exception as exc:  # noqa: BLE001 - a library without this GEMM is reported, not fatal
            out[name] = {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}
    if "burst_tflops" in out.get("bf16", {}) and "burst_tflops" in out.get("e4m3", {}):
        out["e4m3_per_bf16_burst"] = out["e4m3"]["burst_tflops"] / out["bf16"]["burst_tflops"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", metavar="WORKLOAD", help="only run WORKLOAD's launches (for ncu captures)")
    ap.add_argument("--batch", type=int, default=0, help="with --profile: override the batch size")
    ap.add_argument("--page-size", type=int, default=0, help="with --profile on the decode: a paged cache of this page size")
    ap.add_argument("--tensor-peaks", action="store_true",
                    help="only measure the dense bf16 and e4m3 library GEMM throughput (with clocks) and exit")
    args = ap.parse_args()
    if args.profile:
        profile_run(args)
        return
    if args.tensor_peaks:
        dev = torch.device("cuda", torch.cuda.current_device())
        for n in (8192, 16384):
            sampler = ClockSampler(dev.index or 0)
            sampler.start()
            res = tensor_peaks(dev, n=n)
            res["clocks"] = sampler.stop()
            print(json.dumps({"tensor_peaks": res}), flush=True)
            torch.cuda.empty_cache()
        return
    args.warmup = max(args.warmup, 3)
    rank, local, world = dist_setup()
    if args.impl == "reference":
        main_reference(args, rank, world)
        return

    import flash_attention_forward_gb300 as fa

    fa.library()  # fails loudly if the CUDA library was not built
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flusher = Flusher(dev)
    w = workloads.WORKLOADS[HEADLINE]

    # ---- headline: timed region bracketed by barrier + synchronize, max over ranks
    _, step = prefill_setup(w, dev)
    for _ in range(args.warmup):
        flusher()
        step()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    host_us = []
    ms = time_steps(step, args.steps, 0, flusher, host_us=host_us)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if rank == 0 else None
    ok_status = fa.sdpa_check_device_status()
    total_ms = max_over_ranks(sum(ms), world)
    flops = prefill_flops(w)
    value = whole_job_rate(flops, args.steps, total_ms, world) / 1e12
    avg_kernel_ms = sum(ms) / len(ms)
    achieved = flops / (avg_kernel_ms * 1e-3) / 1e12
    bf16 = peaks["bf16_tflops"]

    e2e = bench_e2e_prefill(w, min(args.steps, 20), dev)
    e2e_ms = max_over_ranks(e2e["ms_per_step"], world)
    e2e_value = whole_job_rate(flops, 1, e2e_ms, world) / 1e12

    others = {}
    if not args.headline_only and rank == 0:
        k2 = min(args.steps, 100)
        for name in ("tiny_prefill_f16_d64", "unaligned_mask_prefill_bf16_d128", "mla_fp8_causal_prefill_d192"):
            others[name] = bench_prefill(workloads.WORKLOADS[name], k2, args.warmup, dev, peaks, flusher)
            torch.cuda.empty_cache()
        iw = workloads.WORKLOADS["int8_qk_causal_prefill_d128"]
        others[iw.name] = bench_int8(iw, k2, args.warmup, dev, peaks, flusher)
        torch.cuda.empty_cache()
        vw = workloads.WORKLOADS["varlen_causal_prefill_bf16_d128"]
        others[vw.name] = bench_varlen(vw, k2, args.warmup, dev, peaks, flusher)
        torch.cuda.empty_cache()
        dec, dec_paged = bench_decode(workloads.WORKLOADS["splitkv_decode_bf16_d128"], k2, args.warmup, dev, peaks)
        others[dec["workload"]] = dec
        others[dec_paged["workload"]] = dec_paged
        del dec_paged
        torch.cuda.empty_cache()
        mla, _ = bench_decode(workloads.WORKLOADS["mla_decode_bf16_d192_g16"], k2, args.warmup, dev, peaks, n_sets=2,
                              paged=False)
        others[mla["workload"]] = mla
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, target_s=45.0)  # the 256-row probe overestimates the time per row ~2x

    if rank == 0:
        cfg = config_of(w)
        cfg["l2"] = "flushed before every timed step (256 MiB write, outside the events)"
        cfg["parallelism"] = f"replicas x{world}"
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                         "frac": achieved / bf16, "traffic": recorded_traffic(w.name),
                         "kernel": "prefill_kernel<bf16, D=128, Dv=128, causal>",
                         "peak_note": "bf16 dense burst, of " + peaks["source"]},
            "cpu_baseline": None if cpu is None else {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                    "d2h_bytes_per_step": e2e["d2h_bytes_per_step"], "api": e2e["api"], "ms_per_step": e2e_ms,
                    "link": e2e["link"]},
            "step_ms": step_stats(ms),
            "host_us_per_call": {"median": float(np.median(host_us)), "max": float(np.max(host_us))},
            "timing": "CUDA events around each step on the launching stream; the launch queue is primed by a "
                      "GPU-side sleep before the first step (outside every event), so the events measure the "
                      "device's time per step",
            "gpu_launches": args.steps,
            "clocks": clocks,
            "device_status": fa.sdpa_status_string(ok_status),
            "workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
