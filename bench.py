"""Throughput bench for the GB300 exact-attention library.

One step = one pass of the whole hot path on synthetic inputs:
  * the training-shaped sweep: hidden 2048 as (D=64, H=32) and (D=128, H=16),
    seqlen S in {512, 1k, 2k, 4k, 8k, 16k}, batch 16384/S, causal off and on,
    each point a forward (fa_fwd) and a backward (fa_bwd);
  * split-KV decode (fa_decode_splitkv): B=16, H=32, D=128, one query row,
    KV caches of 4k, 32k and 128k keys;
  * the other workload shapes: the mask variants (B=2, H=16, D=128: causal
    with Sq=2048, Sk=8192; window (4096, 0) at 16k; causal + ALiBi at 4k),
    each a forward and a backward, and the long head dim (B=1, H=8, D=256,
    16k, forward only, causal off and on).
The headline value is the sweep's forward+backward TFLOP/s (4*B*H*S*S*D for
the forward, halved for causal, and 2.5x that for the backward); the forward
alone, decode HBM GB/s and each other workload (with both the convention
flops and the exact count over the live (query, key) pairs) are reported
beside it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs the same per-GPU workload on its own GPU
(replicas; each (batch, head) is independent, so no collective is involved)
and the value is the sum over ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SWEEP_S = (512, 1024, 2048, 4096, 8192, 16384)
# The other workload shapes, timed in every step beside the sweep: the mask
# variants (fwd + bwd, B2 H16 D128) and the long head dim (forward only).
WORKLOADS = (
    dict(name="causal 2048x8192 (bottom-right)", B=2, Sq=2048, Sk=8192, H=16, D=128, causal=True, window=(-1, -1),
         alibi=False, bwd=True),
    dict(name="window (4096, 0) at 16k", B=2, Sq=16384, Sk=16384, H=16, D=128, causal=False, window=(4096, 0),
         alibi=False, bwd=True),
    dict(name="causal + ALiBi at 4k", B=2, Sq=4096, Sk=4096, H=16, D=128, causal=True, window=(-1, -1), alibi=True,
         bwd=True),
    dict(name="long head dim D256 16k", B=1, Sq=16384, Sk=16384, H=8, D=256, causal=False, window=(-1, -1),
         alibi=False, bwd=False),
    dict(name="long head dim D256 16k causal", B=1, Sq=16384, Sk=16384, H=8, D=256, causal=True, window=(-1, -1),
         alibi=False, bwd=False),
)
SWEEP_DH = ((64, 32), (128, 16))
DECODE_SK = (4096, 32768, 131072)
DECODE_B, DECODE_H, DECODE_D = 16, 32, 128
TOKENS = 16384

PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(PEAK_FALLBACK), "fallback"


def sweep_points():
    pts = []
    for D, H in SWEEP_DH:
        for S in SWEEP_S:
            for causal in (False, True):
                pts.append(dict(B=TOKENS // S, S=S, H=H, D=D, causal=causal))
    return pts


def fwd_flops(pt):
    f = 4.0 * pt["B"] * pt["H"] * pt["S"] * pt["S"] * pt["D"]
    return f / 2 if pt["causal"] else f


def live_pairs(Sq, Sk, causal, window):
    """Exact (query row, key) pairs the mask keeps, per (batch, head): row i keeps
    keys [c - left, c + right] of its bottom-right diagonal c = i + Sk - Sq,
    clipped to [0, Sk - 1] (causal: right = 0; -1: unbounded)."""
    import numpy as np

    wl, wr = window
    if causal:
        wr = 0
    c = np.arange(Sq, dtype=np.int64) + Sk - Sq
    lo = np.maximum(c - wl, 0) if wl >= 0 else np.zeros(Sq, np.int64)
    hi = np.minimum(c + wr, Sk - 1) if wr >= 0 else np.full(Sq, Sk - 1, np.int64)
    return int(np.maximum(hi - lo + 1, 0).sum())


def workload_flops(w):
    """Forward flops of a workload: the convention (4 B H Sq Sk D, halved when
    causal) and the exact count over the live pairs (4 D per pair)."""
    conv = 4.0 * w["B"] * w["H"] * w["Sq"] * w["Sk"] * w["D"] / (2 if w["causal"] else 1)
    exact = 4.0 * w["B"] * w["H"] * w["D"] * live_pairs(w["Sq"], w["Sk"], w["causal"], w["window"])
    return conv, exact


def decode_bytes(Sk):
    # K and V read once, plus q, out and lse (split partials are a few MB and not counted)
    return 2 * DECODE_B * Sk * DECODE_H * DECODE_D * 2 + 2 * DECODE_B * DECODE_H * DECODE_D * 2 + DECODE_B * DECODE_H * 4


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def _read(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.lines.append(ln)
                self._first.set()

    def __enter__(self):
        import threading

        self.lines = []
        self._first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()
        # the timed region starts once the sampler is running
        self._first.wait(timeout=3.0)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        # median over samples taken under load (clock above idle)
        load = [x for x in sm if x > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _cpu_cores_used():
    try:
        import threadpoolctl  # noqa: F401

        info = threadpoolctl.threadpool_info()
        n = [d.get("num_threads") for d in info if d.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def _traffic_per_launch(group, steps, launches_per_step):
    """DRAM bytes per launch of a kernel group, from the committed ncu summary
    (profiles/traffic.json), or None once the kernel source has changed since
    the capture."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[group]
        with open(os.path.join(ROOT, t["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != t["source_sha256"]:
                return None
    except Exception:
        return None
    if "bytes_per_launch" in t:
        return float(t["bytes_per_launch"])
    if "bytes_per_key" in t:  # decode: per launch over the decode cache sizes
        keys = sum(DECODE_B * DECODE_H * Sk for Sk in DECODE_SK) / len(DECODE_SK)
        return float(t["bytes_per_key"]) * keys
    return None


def oracle_sample(budget_s=12.0, points=None):
    """Time the fp64 oracle (fwd + bwd of single heads) on a bounded sample of the sweep.

    Returns (TFLOP/s, description, seconds). Heads are drawn from the sweep
    points with S <= 4096, one (b, h) each, cycling until the budget is spent.
    """
    import numpy as np

    import oracle
    from fa_inputs import attention_inputs, bf16_bits_to_f64

    pts = [p for p in (points or sweep_points()) if p["S"] <= 4096]
    flops, t_used, n = 0.0, 0.0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        pt = pts[n % len(pts)]
        inp = attention_inputs(1, pt["S"], pt["S"], 1, pt["D"], seed=n, with_dout=True)
        q, k, v, do = (bf16_bits_to_f64(inp[x])[0, :, 0, :] for x in ("q", "k", "v", "dout"))
        s0 = time.perf_counter()
        scale = 1.0 / math.sqrt(pt["D"])
        oracle.head_fwd(q, k, v, scale, pt["causal"])
        oracle.head_bwd(do, q, k, v, scale, pt["causal"])
        t_used += time.perf_counter() - s0
        f = 4.0 * pt["S"] * pt["S"] * pt["D"] / (2 if pt["causal"] else 1)
        flops += 3.5 * f
        n += 1
    desc = f"{n} single (b,h) heads fwd+bwd cycling over sweep points with S<=4096 (fp64 NumPy oracle)"
    return flops / t_used / 1e12, desc, t_used


def oracle_tiny_single_core(repeats=5):
    """The fp64 oracle's fwd+bwd on the tiny workload (B1 H2 S128 D64, causal off
    and on) in a child process whose BLAS runs one thread: the median seconds of
    a pass and the TFLOP/s by the same flop convention."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-tiny", str(repeats)], env=env,
                       capture_output=True, text=True, timeout=120)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["seconds"], d["tflops"]


def _oracle_tiny_pass(repeats):
    import numpy as np

    import oracle
    from fa_inputs import attention_inputs, bf16_bits_to_f64

    inp = attention_inputs(1, 128, 128, 2, 64, seed=1, with_dout=True)
    q, k, v, do = (bf16_bits_to_f64(inp[x]) for x in ("q", "k", "v", "dout"))
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        for causal in (False, True):
            oracle.attention_fwd(q, k, v, None, causal)
            oracle.attention_bwd(do, q, k, v, None, causal)
        times.append(time.perf_counter() - t0)
    sec = float(np.median(times))
    flops = 3.5 * 4.0 * 1 * 2 * 128 * 128 * 64 * 1.5  # non-causal + causal (half)
    print(json.dumps({"seconds": sec, "tflops": flops / sec / 1e12}), flush=True)
    return 0


def bench_config(ws):
    """The workload both arms report on."""
    return {"workload": "training-shaped sweep: hidden 2048 as D64/H32 and D128/H16, S 512..16k, "
                        "B=16384/S, causal off+on, fwd+bwd; plus split-KV decode B16 H32 D128 Sk 4k/32k/128k; "
                        "plus the mask variants (B2 H16 D128: causal 2048x8192, window (4096,0) at 16k, causal+ALiBi "
                        "at 4k; fwd+bwd) and the long head dim (B1 H8 D256 16k, forward, causal off+on), reported "
                        "beside the headline",
            "global_batch_tokens": TOKENS * ws, "parallelism": f"replicas x{ws}",
            "l2": "inputs larger than L2 (each sweep pass reads >= 320 MiB; decode caches >= 1 GiB)"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample(budget_s=0.5)
    vals, secs = [], 0.0
    desc = ""
    per_step = min(8.0, 150.0 / max(args.steps, 1))
    for _ in range(args.steps):
        v, desc, t = oracle_sample(budget_s=per_step)
        vals.append(v)
        secs += t
    value = statistics.median(vals)
    cores = _cpu_cores_used()
    line = {
        "impl": "reference",
        "metric": "attention fwd+bwd TFLOP/s (bf16 training-shaped sweep)",
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * secs / max(args.steps, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(ws),
        "impl_note": "fp64 CPU oracle (test infrastructure) on the host cores; each step a bounded sample of "
                     "single (b, h) heads of this workload",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import exact_attention_56_gb300 as fa
    from fa_inputs import device_normal_bf16

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = _peaks()

    # ---------------------------------------------------------------- inputs (resident in HBM)
    pts = sweep_points()
    bufs = []
    for n, pt in enumerate(pts):
        B, S, H, D = pt["B"], pt["S"], pt["H"], pt["D"]
        seed = 2000 + 97 * n + 1000003 * rank
        t = {x: device_normal_bf16((B, S, H, D), seed + i, dev) for i, x in enumerate(("q", "k", "v", "do"))}
        t["out"] = torch.empty_like(t["q"])
        t["lse"] = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        t["dq"] = torch.empty_like(t["q"])
        t["dk"] = torch.empty_like(t["q"])
        t["dv"] = torch.empty_like(t["q"])
        t["ws"] = torch.empty(fa.fa_bwd_workspace_size(B, S, S, H, D, False), dtype=torch.uint8, device=dev)
        bufs.append(t)
    dec = []
    for n, Sk in enumerate(DECODE_SK):
        seed = 5000 + n + 1000003 * rank
        B, H, D = DECODE_B, DECODE_H, DECODE_D
        d = {"q": device_normal_bf16((B, 1, H, D), seed, dev),
             "k": device_normal_bf16((B, Sk, H, D), seed + 1, dev),
             "v": device_normal_bf16((B, Sk, H, D), seed + 2, dev)}
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty((B, H, 1), dtype=torch.float32, device=dev)
        d["n"] = fa.fa_decode_num_splits(B, 1, Sk, H, D)
        d["ws"] = torch.empty(fa.fa_decode_workspace_size(B, 1, Sk, H, D, d["n"]), dtype=torch.uint8, device=dev)
        dec.append(d)
    wls = []
    for n, w in enumerate(WORKLOADS):
        B, Sq, Sk, H, D = w["B"], w["Sq"], w["Sk"], w["H"], w["D"]
        seed = 7000 + 11 * n + 1000003 * rank
        t = {"q": device_normal_bf16((B, Sq, H, D), seed, dev), "k": device_normal_bf16((B, Sk, H, D), seed + 1, dev),
             "v": device_normal_bf16((B, Sk, H, D), seed + 2, dev)}
        t["out"] = torch.empty_like(t["q"])
        t["lse"] = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
        t["alibi"] = (torch.exp2(-8.0 * torch.arange(1, H + 1, dtype=torch.float32) / H).to(dev)
                      if w["alibi"] else None)
        if w["bwd"]:
            t["do"] = device_normal_bf16((B, Sq, H, D), seed + 3, dev)
            t["dq"] = torch.empty_like(t["q"])
            t["dk"] = torch.empty_like(t["k"])
            t["dv"] = torch.empty_like(t["v"])
            t["ws"] = torch.empty(fa.fa_bwd_workspace_size(B, Sq, Sk, H, D, False), dtype=torch.uint8, device=dev)
        wls.append(t)
    torch.cuda.synchronize()
    n_ev = len(pts) + len(dec) + len(WORKLOADS)

    def run_workload(w, t, e=None):
        kw = dict(causal=w["causal"], window_size=w["window"], alibi_slopes=t["alibi"], stream=stream)
        if e is not None:
            e[0].record(stream)
        fa.fa_fwd(t["q"], t["k"], t["v"], out=t["out"], lse=t["lse"], **kw)
        if e is not None:
            e[1].record(stream)
        if w["bwd"]:
            fa.fa_bwd(t["do"], t["q"], t["k"], t["v"], t["out"], t["lse"], dq=t["dq"], dk=t["dk"], dv=t["dv"],
                      workspace=t["ws"], **kw)
        if e is not None:
            e[2].record(stream)

    def step(ev=None):
        for i, (pt, t) in enumerate(zip(pts, bufs)):
            if ev is not None:
                ev[i][0].record(stream)
            fa.fa_fwd(t["q"], t["k"], t["v"], causal=pt["causal"], out=t["out"], lse=t["lse"], stream=stream)
            if ev is not None:
                ev[i][1].record(stream)
            fa.fa_bwd(t["do"], t["q"], t["k"], t["v"], t["out"], t["lse"], causal=pt["causal"], dq=t["dq"],
                      dk=t["dk"], dv=t["dv"], workspace=t["ws"], stream=stream)
            if ev is not None:
                ev[i][2].record(stream)
        for m, d in enumerate(dec):
            if ev is not None:
                ev[len(pts) + m][0].record(stream)
            fa.fa_decode_splitkv(d["q"], d["k"], d["v"], causal=True, num_splits=d["n"], workspace=d["ws"],
                                 out=d["out"], lse=d["lse"], stream=stream)
            if ev is not None:
                ev[len(pts) + m][1].record(stream)
        for m, (w, t) in enumerate(zip(WORKLOADS, wls)):
            run_workload(w, t, None if ev is None else ev[len(pts) + len(dec) + m])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {word:#x} after warm-up")

    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    evs = [[[mk(), mk(), mk()] for _ in range(n_ev)] for _ in range(args.steps)]
    e_all0, e_all1 = mk(), mk()
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        e_all0.record(stream)
        for s in range(args.steps):
            step(evs[s])
        e_all1.record(stream)
        torch.cuda.synchronize()
    _barrier(ws)
    st, word = fa.fa_device_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {word:#x} after the timed region")

    total_ms = e_all0.elapsed_time(e_all1)
    t_fwd = [0.0] * len(pts)
    t_bwd = [0.0] * len(pts)
    t_dec = [0.0] * len(dec)
    for s in range(args.steps):
        for i in range(len(pts)):
            t_fwd[i] += evs[s][i][0].elapsed_time(evs[s][i][1])
            t_bwd[i] += evs[s][i][1].elapsed_time(evs[s][i][2])
        for m in range(len(dec)):
            t_dec[m] += evs[s][len(pts) + m][0].elapsed_time(evs[s][len(pts) + m][1])
    t_wf = [0.0] * len(WORKLOADS)
    t_wb = [0.0] * len(WORKLOADS)
    for s in range(args.steps):
        for m in range(len(WORKLOADS)):
            e = evs[s][len(pts) + len(dec) + m]
            t_wf[m] += e[0].elapsed_time(e[1])
            t_wb[m] += e[1].elapsed_time(e[2])
    K = args.steps
    f_fwd = sum(fwd_flops(p) for p in pts)
    f_all = 3.5 * f_fwd
    ms_fb = sum(t_fwd) + sum(t_bwd)
    ms_fb = _max_over_ranks(ms_fb, ws, dev)
    value = ws * f_all * K / (ms_fb * 1e-3) / 1e12
    fwd_value = ws * f_fwd * K / (_max_over_ranks(sum(t_fwd), ws, dev) * 1e-3) / 1e12
    dec_bytes = sum(decode_bytes(Sk) for Sk in DECODE_SK)
    dec_gbs = ws * dec_bytes * K / (_max_over_ranks(sum(t_dec), ws, dev) * 1e-3) / 1e9
    total_ms = _max_over_ranks(total_ms, ws, dev)

    # roofline of the dominant kernel group
    groups = {"fa_bwd (pre + dK/dV + dQ launch group)": (sum(t_bwd), 2.5 * f_fwd, "tensor"),
              "fa_fwd_kernel": (sum(t_fwd), f_fwd, "tensor"),
              "fa_decode_split (+combine)": (sum(t_dec), dec_bytes, "hbm")}
    dom = max(groups, key=lambda g: groups[g][0])
    g_ms, g_work, bound = groups[dom]
    launches_per_step = len(pts) if dom == "fa_fwd_kernel" else (len(pts) if dom.startswith("fa_bwd") else len(dec))
    per_launch_ms = g_ms / (K * launches_per_step)
    if bound == "tensor":
        achieved = g_work * K / (g_ms * 1e-3) / 1e12
        peak = float(peaks.get("bf16_tflops_sustained", PEAK_FALLBACK["bf16_tflops_sustained"]))
        unit = "TFLOP/s"
    else:
        achieved = g_work * K / (g_ms * 1e-3) / 1e9
        peak = float(peaks.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"]))
        unit = "GB/s"
    roofline = {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": _traffic_per_launch(dom, K, launches_per_step), "peak_source": f"{peak_src} (sustained bf16)"
                if bound == "tensor" else f"{peak_src} (copy bandwidth)", "per_launch_ms_avg": per_launch_ms}

    sweep = []
    for i, pt in enumerate(pts):
        ff = fwd_flops(pt)
        sweep.append({"S": pt["S"], "D": pt["D"], "H": pt["H"], "B": pt["B"], "causal": pt["causal"],
                      "fwd_tflops": round(ff * K / (t_fwd[i] * 1e-3) / 1e12, 1),
                      "bwd_tflops": round(2.5 * ff * K / (t_bwd[i] * 1e-3) / 1e12, 1),
                      "fwdbwd_tflops": round(3.5 * ff * K / ((t_fwd[i] + t_bwd[i]) * 1e-3) / 1e12, 1)})
    decode = {"gbs": dec_gbs, "unit": "GB/s",
              "frac": dec_gbs / ws / float(peaks.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"])),
              "per_sk": [{"Sk": Sk, "splits": d["n"], "gbs": round(decode_bytes(Sk) * K / (t * 1e-3) / 1e9, 1)}
                         for Sk, d, t in zip(DECODE_SK, dec, t_dec)]}

    peak_sus = float(peaks.get("bf16_tflops_sustained", PEAK_FALLBACK["bf16_tflops_sustained"]))
    workloads = []
    for w, tf, tb in zip(WORKLOADS, t_wf, t_wb):
        conv, exact = workload_flops(w)
        tf_ms, tb_ms = _max_over_ranks(tf, ws, dev) / K, _max_over_ranks(tb, ws, dev) / K
        r = {"name": w["name"], "B": w["B"], "H": w["H"], "Sq": w["Sq"], "Sk": w["Sk"], "D": w["D"],
             "causal": w["causal"], "window": list(w["window"]), "alibi": w["alibi"],
             "fwd_flops_convention": conv, "fwd_flops_exact": exact, "fwd_ms": round(tf_ms, 4),
             "fwd_tflops_exact": round(ws * exact / (tf_ms * 1e-3) / 1e12, 1),
             "fwd_tflops_convention": round(ws * conv / (tf_ms * 1e-3) / 1e12, 1)}
        r["fwd_frac_exact"] = round(r["fwd_tflops_exact"] / ws / peak_sus, 3)
        if w["bwd"]:
            r["bwd_ms"] = round(tb_ms, 4)
            r["bwd_tflops_exact"] = round(ws * 2.5 * exact / (tb_ms * 1e-3) / 1e12, 1)
            r["fwdbwd_tflops_exact"] = round(ws * 3.5 * exact / ((tf_ms + tb_ms) * 1e-3) / 1e12, 1)
            r["fwdbwd_tflops_convention"] = round(ws * 3.5 * conv / ((tf_ms + tb_ms) * 1e-3) / 1e12, 1)
            r["fwdbwd_frac_exact"] = round(r["fwdbwd_tflops_exact"] / ws / peak_sus, 3)
        workloads.append(r)

    # ---------------------------------------------------------------- end to end (pinned host <-> device)
    e2e = None
    if not args.skip_e2e:
        e2e = run_e2e(fa, pts, bufs, dec, stream, dev, args, ws)

    cpu = None
    if rank == 0 and not args.skip_cpu:
        v, desc, _ = oracle_sample(budget_s=args.cpu_budget)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": _cpu_cores_used(), "kind": "oracle", "sample": desc}
        try:
            sec, tfs = oracle_tiny_single_core()
            cpu["tiny_single_core"] = {"seconds": sec, "tflops": tfs, "cores": 1,
                                       "workload": "B1 H2 S128 D64 fwd+bwd, causal off and on"}
        except Exception as e:
            cpu["tiny_single_core"] = {"unavailable": str(e)[:120]}

    if rank == 0:
        line = {
            "metric": "attention fwd+bwd TFLOP/s (bf16 training-shaped sweep)",
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": bench_config(ws),
            "fwd_tflops": fwd_value,
            "fwd_frac": fwd_value / ws / float(peaks.get("bf16_tflops_sustained", 1700.0)),
            "fwdbwd_frac": value / ws / float(peaks.get("bf16_tflops_sustained", 1700.0)),
            "decode": decode,
            "sweep": sweep,
            "workloads": workloads,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            # per sweep point: forward, then pre-pass, rescale, dK/dV and dQ; per
            # decode: split and combine; per other workload: forward (+ the four)
            "gpu_launches": K * (5 * len(pts) + 2 * len(dec) + sum(5 if w["bwd"] else 1 for w in WORKLOADS)),
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_e2e(fa, pts, bufs, dec, stream, dev, args, ws):
    """Same metric through the public API with host buffers: each step copies the
    inputs of every sweep point from pinned host memory, runs fa_fwd + fa_bwd, and
    copies O, dQ, dK, dV back to pinned host memory.

    The copies run on their own streams, so the host->device copy of point i+1
    and the device->host copy of point i-1 overlap the kernels of point i (each
    point has its own device buffers; events order every reuse)."""
    import torch

    # Every sweep point holds 16384 tokens x hidden 2048 per tensor. The pinned
    # inputs are only read, and all device->host copies run in order on one
    # stream, so one set of pinned buffers serves every point.
    numel = bufs[0]["q"].numel()
    assert all(t[x].numel() == numel for t in bufs for x in ("q", "k", "v", "do", "out", "dq", "dk", "dv"))
    pin_in = {x: torch.empty(numel, dtype=torch.bfloat16, pin_memory=True) for x in ("q", "k", "v", "do")}
    pin_out = {x: torch.empty(numel, dtype=torch.bfloat16, pin_memory=True) for x in ("out", "dq", "dk", "dv")}
    for x in pin_in:
        pin_in[x].copy_(bufs[0][x].view(-1))
    host_in = [{x: pin_in[x].view(t[x].shape) for x in pin_in} for t in bufs]
    host_out = [{x: pin_out[x].view(t[x].shape) for x in pin_out} for t in bufs]
    h2d = sum(t[x].numel() * 2 for t in bufs for x in pin_in)
    d2h = sum(t[x].numel() * 2 for t in bufs for x in pin_out)

    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n = len(pts)
    ev_in = [torch.cuda.Event() for _ in range(n)]    # inputs of point i are on the device
    ev_done = [torch.cuda.Event() for _ in range(n)]  # kernels of point i have finished
    ev_out = [torch.cuda.Event() for _ in range(n)]   # outputs of point i are back on the host

    def step():
        for i, (pt, t, hi, ho) in enumerate(zip(pts, bufs, host_in, host_out)):
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[i])  # the previous step's kernels of point i read these inputs
                for x in hi:
                    t[x].copy_(hi[x], non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])  # the previous step's outputs of point i have been read back
            fa.fa_fwd(t["q"], t["k"], t["v"], causal=pt["causal"], out=t["out"], lse=t["lse"], stream=stream)
            fa.fa_bwd(t["do"], t["q"], t["k"], t["v"], t["out"], t["lse"], causal=pt["causal"], dq=t["dq"],
                      dk=t["dk"], dv=t["dv"], workspace=t["ws"], stream=stream)
            ev_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                for x in ho:
                    ho[x].copy_(t[x], non_blocking=True)
                ev_out[i].record(s_out)

    step()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(steps):
        step()
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = _max_over_ranks(e0.elapsed_time(e1), ws, dev)
    f_all = 3.5 * sum(fwd_flops(p) for p in pts)
    return {"value": ws * f_all * steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "fwd+bwd sweep only; host->device and device->host copies on two copy streams, overlapping "
                    "the kernels of the neighbouring sweep points"}


PROFILE_CASES = {
    # small cases (inputs > L2, < 1 GB on the device) for ncu captures of one kernel group
    "fwd128": dict(op="fwd", B=4, S=4096, H=16, D=128, causal=False),
    "fwd64": dict(op="fwd", B=4, S=4096, H=32, D=64, causal=False),
    "fwd64c": dict(op="fwd", B=4, S=4096, H=32, D=64, causal=True),
    "fwd128c": dict(op="fwd", B=4, S=4096, H=16, D=128, causal=True),
    "fwd256": dict(op="fwd", B=1, S=8192, H=8, D=256, causal=False),
    # the causal + ALiBi mask variant's shape (geometric slopes)
    "fwd128a": dict(op="fwd", B=2, S=4096, H=16, D=128, causal=True, alibi=True),
    "bwd128c": dict(op="bwd", B=4, S=4096, H=16, D=128, causal=True),
    "bwd128": dict(op="bwd", B=4, S=4096, H=16, D=128, causal=False),
    "bwd64": dict(op="bwd", B=4, S=4096, H=32, D=64, causal=False),
    # the same with deterministic=True: the two-kernel path (dK/dV, then dQ) at D = 64
    "bwd64d": dict(op="bwd", B=4, S=4096, H=32, D=64, causal=False, deterministic=True),
    # short and long training-sweep points of the backward
    "bwd64_512c": dict(op="bwd", B=32, S=512, H=32, D=64, causal=True),
    "bwd64_16kc": dict(op="bwd", B=1, S=16384, H=32, D=64, causal=True),
    "decode": dict(op="decode", B=16, S=32768, H=32, D=128, causal=True),
    # decode with a 1.07 GB cache: small enough for multi-pass captures
    "decode4k": dict(op="decode", B=16, S=4096, H=32, D=128, causal=True),
    # grouped decode (8 key/value heads, 4 query heads each): the tensor-core split kernel
    "decode_gqa4k": dict(op="decode", B=16, S=4096, H=32, Hk=8, D=128, causal=True),
    # multi-query decode (one key/value head): 268 MB of cache
    "decode_mqa32k": dict(op="decode", B=16, S=32768, H=32, Hk=1, D=128, causal=True),
}


def run_profile(name):
    """Warm-up calls then one timed call of a single op; prints one short line."""
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import exact_attention_56_gb300 as fa
    from fa_inputs import device_normal_bf16

    c = PROFILE_CASES[name]
    dev = torch.device("cuda", 0)
    B, S, H, D = c["B"], c["S"], c["H"], c["D"]
    if c["op"] == "decode":
        Hk = c.get("Hk", H)
        q = device_normal_bf16((B, 1, H, D), 1, dev)
        k = device_normal_bf16((B, S, Hk, D), 2, dev)
        v = device_normal_bf16((B, S, Hk, D), 3, dev)
        n = fa.fa_decode_num_splits(B, 1, S, H, D, Hk=Hk)
        ws = torch.empty(fa.fa_decode_workspace_size(B, 1, S, H, D, n, Hk=Hk), dtype=torch.uint8, device=dev)
        run = lambda: fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=n, workspace=ws)  # noqa: E731
    else:
        q, k, v, do = (device_normal_bf16((B, S, H, D), i, dev) for i in range(4))
        al = (torch.exp2(-8.0 * torch.arange(1, H + 1, dtype=torch.float32) / H).to(dev)
              if c.get("alibi") else None)
        out, lse = fa.fa_fwd(q, k, v, causal=c["causal"], alibi_slopes=al)
        if c["op"] == "fwd":
            run = lambda: fa.fa_fwd(q, k, v, causal=c["causal"], alibi_slopes=al, out=out, lse=lse)  # noqa: E731
        else:
            det = c.get("deterministic", False)
            ws = torch.empty(fa.fa_bwd_workspace_size(B, S, S, H, D, det), dtype=torch.uint8, device=dev)
            run = lambda: fa.fa_bwd(do, q, k, v, out, lse, causal=c["causal"], alibi_slopes=al,  # noqa: E731
                                    deterministic=det, workspace=ws)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run()
    e1.record()
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    print(json.dumps({"profile": name, "ms": e0.elapsed_time(e1), "status": st, "word": word, **c}), flush=True)
    return 0 if st == fa.FA_OK else 1


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES), default=None,
                    help="run one small case of one op (for ncu captures) instead of the bench")
    ap.add_argument("--oracle-tiny", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.oracle_tiny:
        return _oracle_tiny_pass(args.oracle_tiny)
    if args.profile:
        return run_profile(args.profile)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
