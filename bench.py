#!/usr/bin/env python3
"""Benchmark of the fused attention forward on one or more GB300s.

A step is one fmha_fwd call (one kernel launch) over one batch of seeded
synthetic input.  The default workload is causal bf16 grouped-query attention,
B=2, H=32, H_k=8, Sq=Sk=8192, D=128 (the size the 60%-of-peak target is set
at).  Metric: TFLOP/s counting 4*B*H*Sq*Sk*D, halved for causal.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Under torchrun every rank runs the same per-GPU workload on its own GPU
(independent problems, no data exchange: weak scaling); rank 0 prints one
JSON line.  ``--impl reference`` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from head_attention_forward_02_gb300 import workloads as wl  # noqa: E402
from head_attention_forward_02_gb300.metrics import (algorithmic_bytes, attention_flops, gen_bytes,  # noqa: E402
                                                     gen_flops)

DEFAULT_CONFIG = "bf16_causal_gqa_b2_h32_hk8_s8192_d128"
ALL_CONFIGS = {**wl.CONFIGS, **wl.EXTRA_CONFIGS}
DEFAULT_GEN_CONFIG = "gen_bf16_b32_h32_hk8_s8192"
L2_BYTES = 129 * 2 ** 20
KERNEL_SOURCES = ["head_attention_forward_02_gb300/csrc/fmha_sm103.cu",
                  "head_attention_forward_02_gb300/csrc/fmha_common.h"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # short timed bursts by default (20 launches of the headline, ~13 ms), the
    # regime of the measured burst peak they are reported against; 300
    # back-to-back launches (~0.2 s) measured about 5% slower on the same box
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--op", default="fwd", choices=["fwd", "gen", "bwd"],
                    help="fwd: the fused forward (fmha_fwd); gen: generation phase against a "
                         "K/V cache (fmha_gen_fwd); bwd: the backward pass (fmha_bwd)")
    ap.add_argument("--bwd-config", default="bwd_bf16_causal_b2_h16_s8192_d128", choices=list(BWD_SHAPES))
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(ALL_CONFIGS))
    ap.add_argument("--gen-config", default=DEFAULT_GEN_CONFIG, choices=list(wl.GEN_CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernel", default="tc", choices=["tc", "simt"],
                    help="tc: tcgen05 kernel (fmha_fwd); simt: CUDA-core cross-check kernel")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--configs", action=argparse.BooleanOptionalAction, default=True,
                    help="also time every other workload of the config list, after the headline one, "
                         "and report them under 'configs' in the same JSON line")
    ap.add_argument("--config-steps", type=int, default=20,
                    help="timed launches per extra workload (--configs)")
    ap.add_argument("--context", action=argparse.BooleanOptionalAction, default=True,
                    help="also time torch SDPA on the same inputs (reported as context)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (timing only: barrier and max over ranks)
# ----------------------------------------------------------------------------

def dist_setup(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest value over all ranks (the job's time is its slowest rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.rows = []
        self.proc = None
        self.gpu_id = gpu_id
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        window = "timed"
        if not inside:   # timed region shorter than the sampling period
            inside = [r for t, r in self.rows if t <= t1 + 0.2]
            window = "warmup+timed"
        sm = sorted(v for v in (num(r[1]) for r in inside if len(r) > 1) if v is not None)
        mx = [num(r[2]) for r in inside if len(r) > 2 and num(r[2])]
        reasons = set()
        for r in inside:
            for name, val in zip(self.NAMES, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


def gpu_uuid(dev: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        return "0"


# ----------------------------------------------------------------------------
# roofline inputs
# ----------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for s in KERNEL_SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary of this kernel source
    and workload (profiles/*.md lines 'workload:', 'source_sha256:',
    'traffic_bytes_per_launch:'); None if absent or the kernel changed since."""
    want = kernel_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        kv = dict(re.findall(r"^- ?(workload|source_sha256|traffic_bytes_per_launch): *(\S+)",
                             text, flags=re.M))
        if kv.get("workload") == workload and kv.get("source_sha256") == want:
            try:
                return float(kv["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


# ----------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ----------------------------------------------------------------------------

def oracle_rows_flops(inp, rows):
    """Algorithmic FLOPs of the selected oracle rows: 4*D per visible key, with
    the causal half counted as the accounting of the whole call does (x 1/2
    of the dense count), so that rows sum to attention_flops."""
    w = inp.w
    import numpy as np
    rows = np.asarray(rows)
    if inp.cu_seqlens_q is not None:
        cq = inp.cu_seqlens_q.numpy()
        ck = inp.cu_seqlens_k.numpy()
        t = rows % inp.total_length
        b = np.searchsorted(cq, t, side="right") - 1
        sk = (ck[b + 1] - ck[b]).astype(np.float64)
    else:
        sk = np.full(rows.shape, float(w.Sk))
    f = 0.5 if w.mask == "causal" else 1.0
    return float((4.0 * w.D * sk * f).sum())


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(inp, target_s: float, seed: int = 0):
    """Run the oracle on growing seeded row samples until ~target_s of CPU work."""
    import numpy as np
    import oracle
    from tests.helpers import oracle_on
    oracle.build()
    w = inp.w
    rng = np.random.default_rng(seed)
    if inp.cu_seqlens_q is None:
        pool = np.arange(w.B * w.H * w.Sq)
    else:
        T, end = inp.total_length, int(inp.cu_seqlens_q[-1])
        pool = np.array([h * T + t for h in range(w.H) for t in range(end)])
    n, done_t, done_f, done_rows = 512, 0.0, 0.0, 0
    threads = cpu_threads()
    while done_t < target_s:
        rows = rng.choice(pool, size=n)
        t = time.perf_counter()
        oracle_on(oracle, inp, rows=rows, threads=threads)
        dt = time.perf_counter() - t
        done_t += dt
        done_f += oracle_rows_flops(inp, rows)
        done_rows += n
        if dt < target_s / 4:
            n *= 2
    return done_f, done_t, done_rows, threads


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def make_device_set(inp, dev):
    w = inp.w
    s = {"q": inp.q.to(dev), "k": inp.k.to(dev), "v": inp.v.to(dev)}
    if inp.cu_seqlens_q is not None:
        s["cu_q"] = inp.cu_seqlens_q.to(dev)
        s["cu_k"] = inp.cu_seqlens_k.to(dev)
        s["lse"] = torch.empty((w.H, inp.total_length), dtype=torch.float32, device=dev)
    else:
        s["lse"] = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    s["o"] = torch.empty_like(s["q"])
    return s


def e2e_pipelined(dev, steps, sets, h_in, h_out, launch):
    """Milliseconds per step of `steps` end-to-end steps.  Step i copies the
    pinned host inputs `h_in` (name -> tensor) into device set i % len(sets),
    runs `launch(set, stream)` and copies the set's outputs into the pinned
    host tensors h_out[i % len(sets)] (name -> tensor).  Host-to-device copies,
    kernels and device-to-host copies run on three streams, so the copies of
    one step overlap the kernels of its neighbours, as a serving loop would
    run them; a set is refilled only after its previous step's kernel read
    its inputs and its outputs were copied out.  Every step still moves all
    of its own input and output bytes."""
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ran = [None] * len(sets)
    out_done = [None] * len(sets)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    s_run.wait_event(start)
    s_out.wait_event(start)
    for i in range(steps):
        j = i % len(sets)
        d = sets[j]
        if ran[j] is not None:
            s_in.wait_event(ran[j])
        with torch.cuda.stream(s_in):
            for k, t in h_in.items():
                d[k].copy_(t, non_blocking=True)
        copied = torch.cuda.Event()
        copied.record(s_in)
        s_run.wait_event(copied)
        if out_done[j] is not None:
            s_run.wait_event(out_done[j])
        launch(d, s_run)
        ran[j] = torch.cuda.Event()
        ran[j].record(s_run)
        s_out.wait_event(ran[j])
        with torch.cuda.stream(s_out):
            for k, t in h_out[j].items():
                t.copy_(d[k], non_blocking=True)
        out_done[j] = torch.cuda.Event()
        out_done[j].record(s_out)
    end.record(s_out)          # after the last D2H, which follows every earlier step
    torch.cuda.synchronize(dev)
    return start.elapsed_time(end) / steps


def call(fm, inp, s, kernel, stream):
    w = inp.w
    f = fm.fmha_fwd if kernel == "tc" else fm.fmha_fwd_simt
    if inp.cu_seqlens_q is not None:
        rc = f(s["q"], s["k"], s["v"], s["o"], s["lse"], len(inp.seqlens_q), w.H, w.H_k, 0, 0, w.D,
               w.softmax_scale, w.out_scale, wl.MASK_CODE[w.mask], wl.CAUSAL_CODE[w.causal_type],
               s["cu_q"], s["cu_k"], inp.max_len, inp.total_length, stream)
    else:
        rc = f(s["q"], s["k"], s["v"], s["o"], s["lse"], w.B, w.H, w.H_k, w.Sq, w.Sk, w.D,
               w.softmax_scale, w.out_scale, wl.MASK_CODE[w.mask], wl.CAUSAL_CODE[w.causal_type],
               None, None, 0, 0, stream)
    if rc != 0:
        raise RuntimeError(f"fmha call failed: {fm.status_string(rc)}")


def sdpa_context(inputs, sets, w, flops, dev):
    """torch's scaled_dot_product_attention on the same inputs (context only:
    a library kernel, not a target).  None if torch cannot run this case."""
    import torch.nn.functional as F
    if w.dtype == "e4m3" or inputs[0].cu_seqlens_q is not None:
        return None
    try:
        views = [(s["q"].transpose(1, 2), s["k"].transpose(1, 2), s["v"].transpose(1, 2)) for s in sets]
        kw = {"is_causal": w.mask == "causal", "scale": w.softmax_scale}
        if w.H != w.H_k:
            kw["enable_gqa"] = True

        def step(i):
            q, k, v = views[i % len(views)]
            return F.scaled_dot_product_attention(q, k, v, **kw)
        for i in range(3):
            step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 20
        e0.record()
        for i in range(n):
            step(i)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / n
        return {"torch_sdpa_tflops": round(flops / (ms * 1e-3) / 1e12, 2), "torch_sdpa_ms": round(ms, 4),
                "note": "torch.nn.functional.scaled_dot_product_attention, same inputs, same GPU"}
    except Exception as e:   # an unsupported case in this torch build
        return {"torch_sdpa_tflops": None, "note": f"torch SDPA unavailable: {type(e).__name__}"}


def roofline_of(flops, nbytes, launch_ms, dtype, peaks, peak_src):
    """Tensor or HBM roofline of one launch (whichever side of the ridge point
    the workload's arithmetic intensity falls)."""
    peak = float(peaks["bf16_tflops"]) * (2.0 if dtype == "e4m3" else 1.0)
    hbm = float(peaks["hbm_gbs"])
    if flops / nbytes < peak * 1e12 / (hbm * 1e9):
        bw = nbytes / (launch_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(bw, 2), "peak": hbm, "unit": "GB/s",
                "frac": round(bw / hbm, 4), "peak_source": f"hbm_gbs of {peak_src}"}
    achieved = flops / (launch_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{'2 x bf16_tflops' if dtype == 'e4m3' else 'bf16_tflops'} of {peak_src}"}


def work_of(inp):
    w = inp.w
    if inp.cu_seqlens_q is not None:
        flops = attention_flops(0, w.H, 0, 0, w.D, w.mask == "causal", inp.seqlens_q, inp.seqlens_k)
        nbytes = algorithmic_bytes(0, w.H, w.H_k, 0, 0, w.D, inp.q.element_size(), inp.q.element_size(),
                                   True, inp.seqlens_q, inp.seqlens_k)
    else:
        flops = attention_flops(w.B, w.H, w.Sq, w.Sk, w.D, w.mask == "causal")
        nbytes = algorithmic_bytes(w.B, w.H, w.H_k, w.Sq, w.Sk, w.D, inp.q.element_size(),
                                   inp.q.element_size())
    return flops, nbytes


def time_config(fm, name, dev, kernel, warmup, steps, peaks, peak_src):
    """One more workload in the same run: per-launch CUDA-event time with the
    same L2 rule as the headline (a ring of input sets above L2, an L2 flush
    before every launch below it).  A workload far below L2 that one launch
    cannot fill the GPU with (the 128-token fp16 case) is instead timed as a
    CUDA graph of 1000 back-to-back launches, the way a latency-bound call
    runs in a serving loop, with its inputs L2-resident."""
    w = ALL_CONFIGS[name]
    stream = torch.cuda.current_stream(dev)
    inp0 = wl.generate(w)
    flops, nbytes = work_of(inp0)
    set_bytes = 2 * inp0.q.numel() * inp0.q.element_size() + sum(
        t.numel() * t.element_size() for t in (inp0.k, inp0.v))
    rec = {"workload": name, "dtype": w.dtype, "B": w.B, "H": w.H, "H_k": w.H_k, "Sq": w.Sq, "Sk": w.Sk,
           "D": w.D, "mask": w.mask, "algorithmic_flops": flops, "algorithmic_bytes": nbytes}
    if set_bytes < 4 * 2 ** 20:
        s = make_device_set(inp0, dev)
        for _ in range(max(3, warmup)):
            call(fm, inp0, s, kernel, stream)
        torch.cuda.synchronize(dev)
        n = 1000
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cs = torch.cuda.current_stream(dev)
                for _ in range(n):
                    call(fm, inp0, s, kernel, cs)
            g.replay()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            how = f"CUDA graph of {n} launches, inputs L2-resident"
        except Exception as e:        # capture refused: plain back-to-back launches instead
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                call(fm, inp0, s, kernel, stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            how = f"{n} back-to-back launches (graph capture failed: {type(e).__name__})"
        launch_ms = e0.elapsed_time(e1) / n
        rec.update({"l2": how, "us_per_launch": round(launch_ms * 1e3, 3),
                    "hbm_gbs": round(nbytes / (launch_ms * 1e-3) / 1e9, 2)})
    else:
        n_sets = 2 if set_bytes >= L2_BYTES else 1
        inputs = [inp0] * n_sets                # same problem, separate buffers
        sets = [make_device_set(x, dev) for x in inputs]
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if n_sets == 1 else None
        for i in range(max(3, warmup)):
            if flush is not None:
                flush.zero_()
            call(fm, inputs[i % n_sets], sets[i % n_sets], kernel, stream)
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            if flush is not None:
                flush.zero_()
            starts[i].record(stream)
            call(fm, inputs[i % n_sets], sets[i % n_sets], kernel, stream)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        times = sorted(a.elapsed_time(b) for a, b in zip(starts, ends))
        launch_ms = times[len(times) // 2]           # median launch (the mean is reported too)
        rec.update({"l2": (f"ring of {n_sets} input sets of {set_bytes / 2**20:.0f} MiB" if n_sets > 1 else
                           f"L2 flushed (256 MiB write) before each launch; inputs {set_bytes / 2**20:.0f} MiB"),
                    "launch_ms_mean": round(sum(times) / steps, 5)})
        del sets, inputs, flush
    if fm.device_status(reset=True) != 0:
        raise RuntimeError(f"device status reports a timeout ({name})")
    roof = roofline_of(flops, nbytes, launch_ms, w.dtype, peaks, peak_src)
    # DRAM bytes of one launch from the committed ncu summary of this kernel
    # source and workload, as for the headline (None once the kernel changed)
    roof["traffic"] = profiled_traffic(name)
    rec.update({"launch_ms": round(launch_ms, 5), "steps": steps,
                "value": round(flops / (launch_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "roofline": roof})
    return rec


def run_ours(args, rank, world, local):
    from head_attention_forward_02_gb300 import build, fmha as fm
    build.build()
    fm.lib()
    dev = torch.device("cuda", local if world > 1 else 0)
    w = ALL_CONFIGS[args.config]
    stream = torch.cuda.current_stream(dev)

    inp0 = wl.generate(w)
    set_bytes = 2 * inp0.q.numel() * inp0.q.element_size() + sum(
        t.numel() * t.element_size() for t in (inp0.k, inp0.v))          # Q, O, K, V
    # inputs larger than L2: alternate two input sets so that no step finds the
    # previous step's K/V in L2; smaller inputs: flush L2 before every launch
    n_sets = 2 if set_bytes >= L2_BYTES else 1
    # every set holds the same problem (for varlen: the same lengths) in its own
    # device buffers, so that alternating sets defeats L2 without changing the work
    inputs = [inp0] * n_sets
    sets = [make_device_set(x, dev) for x in inputs]
    if n_sets == 1:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    if inp0.cu_seqlens_q is not None:
        flops = attention_flops(0, w.H, 0, 0, w.D, w.mask == "causal",
                                inp0.seqlens_q, inp0.seqlens_k)
        nbytes = algorithmic_bytes(0, w.H, w.H_k, 0, 0, w.D, inp0.q.element_size(),
                                   inp0.q.element_size(), True, inp0.seqlens_q, inp0.seqlens_k)
    else:
        flops = attention_flops(w.B, w.H, w.Sq, w.Sk, w.D, w.mask == "causal")
        nbytes = algorithmic_bytes(w.B, w.H, w.H_k, w.Sq, w.Sk, w.D, inp0.q.element_size(),
                                   inp0.q.element_size())

    sampler = ClockSampler(gpu_uuid(dev.index or 0))
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    for i in range(args.warmup):
        if n_sets == 1:
            flush.zero_()
        call(fm, inputs[i % n_sets], sets[i % n_sets], args.kernel, stream)
    torch.cuda.synchronize(dev)
    if fm.device_status(reset=True) != 0:
        raise RuntimeError("device status reports a timeout")

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(K):
        j = i % n_sets
        if n_sets == 1:
            flush.zero_()
        starts[i].record(stream)
        call(fm, inputs[j], sets[j], args.kernel, stream)
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_host1 = time.time()
    total_ms = ev0.elapsed_time(ev1)
    launch_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K
    if rank == 0:
        sampler.stop()
    if fm.device_status(reset=True) != 0:
        raise RuntimeError("device status reports a timeout")
    total_ms = max_over_ranks(total_ms, world)
    launch_ms = max_over_ranks(launch_ms, world)
    ms_per_step = total_ms / K
    # with a flush buffer the step time includes the flush; report the launch time
    step_ms = launch_ms if n_sets == 1 else ms_per_step
    value = world * flops / (step_ms * 1e-3) / 1e12

    # end to end through the public API: every step copies its inputs in from
    # pinned host memory and its O and LSE out, pipelined over two device sets
    e2e_steps = args.e2e_steps or max(3, min(K, 20))
    h = {"q": inputs[0].q.pin_memory(), "k": inputs[0].k.pin_memory(), "v": inputs[0].v.pin_memory()}
    e2e_sets = sets if len(sets) >= 2 else sets + [make_device_set(inputs[0], dev)]
    h_out = [{"o": torch.empty(d["o"].shape, dtype=d["o"].dtype).pin_memory(),
              "lse": torch.empty(d["lse"].shape, dtype=torch.float32).pin_memory()} for d in e2e_sets[:2]]

    def launch(d, st):
        call(fm, inputs[0], d, args.kernel, st)

    e2e_pipelined(dev, 2, e2e_sets[:2], h, h_out, launch)          # warm-up
    barrier(world)
    e2e_ms = max_over_ranks(e2e_pipelined(dev, e2e_steps, e2e_sets[:2], h, h_out, launch), world)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())

    if rank != 0:
        return
    peaks, peak_src = measured_peaks()
    dtype_name = {"bf16": "bf16", "f16": "f16", "e4m3": "e4m3"}[w.dtype]
    traffic = profiled_traffic(args.config)
    clk_ghz = float(peaks.get("sm_max_mhz", 2070.0)) / 1e3
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    # one exp2 per visible score (flops / 4D); MUFU ex2 rate 32 results/clk/SM
    # (measured on this part), so the softmax ceiling is visible next to the MMA one
    exp2_per_s = flops / (4.0 * w.D) / (launch_ms * 1e-3)
    mufu_peak = 32.0 * n_sm * clk_ghz * 1e9
    # fp8 peak: twice the measured bf16 rate (4.5 vs 2.25 PFLOP/s nominal)
    roofline = roofline_of(flops, nbytes, launch_ms, w.dtype, peaks, peak_src)
    roofline.update({"traffic": traffic, "algorithmic_bytes": nbytes,
                     "algorithmic_flops": flops, "launch_ms": round(launch_ms, 5),
                     "secondary": {"bound": "mufu_ex2", "achieved_per_s": round(exp2_per_s, 1),
                                   "peak_per_s": mufu_peak,
                                   "frac": round(exp2_per_s / mufu_peak, 4),
                                   "peak_source": "32 ex2/clk/SM x SMs x max SM clock"}})
    line = {
        "metric": "FMHA forward TFLOP/s and % of GB300 dense tensor peak (bf16/fp8)",
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name,
        "data": "synthetic (seeded N(0,1); varlen lengths seeded uniform)",
        "config": {"workload": args.config, "B": w.B, "H": w.H, "H_k": w.H_k, "Sq": w.Sq,
                   "Sk": w.Sk, "D": w.D, "mask": w.mask, "causal_type": w.causal_type,
                   "kernel": "fmha_fwd" if args.kernel == "tc" else "fmha_fwd_simt",
                   "l2": (f"ring of {n_sets} input sets of {set_bytes / 2**20:.0f} MiB"
                          if n_sets > 1 else "L2 flushed (256 MiB write) before every launch"),
                   "parallelism": f"replicas x{world} (independent problems)"},
        "roofline": roofline,
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": K,
        "clocks": sampler.summary(t_host0, t_host1),
    }
    sdpa = sdpa_context(inputs, sets, w, flops, dev) if args.context else None
    if sdpa is not None:
        line["context"] = sdpa
    if not args.no_cpu_baseline:
        f, t, nrows, threads = time_oracle(inputs[0], target_s=10.0)
        line["cpu_baseline"] = {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s",
                                "cores": threads, "kind": "oracle",
                                "sample": f"{nrows} seeded random query rows of {args.config} "
                                          f"({f / 1e9:.1f} GFLOP, {t:.1f} s)"}
    if args.configs:
        # the other workloads, timed in the same run after the headline one
        del sets, inputs, e2e_sets
        torch.cuda.empty_cache()
        line["configs"] = [time_config(fm, name, dev, args.kernel, args.warmup, args.config_steps, peaks,
                                       peak_src) for name in ALL_CONFIGS if name != args.config]
    print(json.dumps(line), flush=True)


def gen_source_hash() -> str:
    """Hash of the generation kernel's source (profiles carry it)."""
    h = hashlib.sha256()
    for f in ("fmha_gen.cu", "fmha_common.h"):
        h.update(open(os.path.join(ROOT, "head_attention_forward_02_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def gen_profiled_traffic(workload: str):
    want = gen_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read()
        kv = dict(re.findall(r"^- ?(workload|source_sha256|traffic_bytes_per_launch): *(\S+)",
                             text, flags=re.M))
        if kv.get("workload") == workload and kv.get("source_sha256") == want:
            try:
                return float(kv["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


def time_gen_oracle(inp, target_s: float):
    """The generation oracle on the first sequences of the workload (one more
    each round) until about target_s of CPU work; returns (bytes, seconds,
    sequences, threads)."""
    import oracle
    oracle.build()
    w = inp.w
    odt = {"bf16": oracle.BF16, "f16": oracle.F16, "e4m3": oracle.E4M3}[w.dtype]
    esz = 1 if w.dtype == "e4m3" else 2
    threads = cpu_threads()
    n, total_b, total_t = 1, 0.0, 0.0
    while True:
        sl = inp.seqlen[:n].numpy()
        args = [wl.bits(inp.q[:n]), wl.bits(inp.k_cache[:n]), wl.bits(inp.v_cache[:n]),
                wl.bits(inp.k_new[:n]) if inp.k_new is not None else None,
                wl.bits(inp.v_new[:n]) if inp.v_new is not None else None]
        t = time.perf_counter()
        oracle.gen_fwd(*args, odt, n, w.H, w.H_k, 128, n, w.S_max, sl, None, 128 ** -0.5, 1.0,
                       threads=threads)
        dt = time.perf_counter() - t
        total_b, total_t = gen_bytes(n, w.H, w.H_k, sl.tolist(), w.insert, esz), dt
        if dt >= target_s or n >= w.B:
            return total_b, total_t, n, threads
        n = min(w.B, max(n + 1, int(n * target_s / max(dt, 1e-3))))


def run_gen(args, rank, world, local):
    """Generation phase (fmha_gen_fwd) on a synthetic K/V cache; one JSON line
    on the HBM roofline."""
    from head_attention_forward_02_gb300 import build, fmha as fm
    build.build()
    fm.lib()
    dev = torch.device("cuda", local if world > 1 else 0)
    w = wl.GEN_CONFIGS[args.gen_config]
    stream = torch.cuda.current_stream(dev)
    inp = wl.generate_gen(w)
    d = {"q": inp.q.to(dev), "kc": inp.k_cache.to(dev), "vc": inp.v_cache.to(dev),
         "kn": inp.k_new.to(dev) if inp.k_new is not None else None,
         "vn": inp.v_new.to(dev) if inp.v_new is not None else None,
         "sl": inp.seqlen.to(dev)}
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    nws = fm.fmha_gen_workspace_size(w.B, w.H, w.H_k, 128, w.S_max)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    cache_bytes = 2 * d["kc"].numel() * d["kc"].element_size()
    nbytes = gen_bytes(w.B, w.H, w.H_k, inp.seqlen.tolist(), w.insert, d["q"].element_size())
    flops = gen_flops(w.H, inp.seqlen.tolist(), w.insert)

    def step():
        fm.gen_fwd(d["q"], d["kc"], d["vc"], d["sl"], k_new=d["kn"], v_new=d["vn"], out=d["o"],
                   lse=d["lse"], workspace=ws, stream=stream)

    sampler = ClockSampler(gpu_uuid(dev.index or 0))
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fm.device_status(reset=True) != 0:
        raise RuntimeError("device status reports an error")
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(K):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_host1 = time.time()
    if rank == 0:
        sampler.stop()
    if fm.device_status(reset=True) != 0:
        raise RuntimeError("device status reports an error")
    ms_per_step = max_over_ranks(ev0.elapsed_time(ev1) / K, world)
    launch_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / K, world)
    value = world * nbytes / (ms_per_step * 1e-3) / 1e9

    # end to end: the cache stays resident; every step copies the new token's
    # q (and K/V rows) and the lengths in from pinned memory, and O and LSE out
    h = {k: inp_t.pin_memory() for k, inp_t in (("q", inp.q), ("kn", inp.k_new), ("vn", inp.v_new),
                                                 ("sl", inp.seqlen)) if inp_t is not None}
    ho = torch.empty(d["o"].shape, dtype=d["o"].dtype).pin_memory()
    hl = torch.empty(d["lse"].shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        for k, t in h.items():
            d[k].copy_(t, non_blocking=True)
        step()
        ho.copy_(d["o"], non_blocking=True)
        hl.copy_(d["lse"], non_blocking=True)

    e2e_steps = args.e2e_steps or max(3, min(K, 50))
    e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    d2h = ho.numel() * ho.element_size() + hl.numel() * 4
    if rank != 0:
        return
    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = nbytes / (launch_ms * 1e-3) / 1e9
    line = {
        "metric": "generation-phase attention HBM bandwidth (GB/s) and % of measured copy rate",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1) cache, query and new rows)",
        "config": {"workload": args.gen_config, "op": "fmha_gen_fwd", "B": w.B, "H": w.H, "H_k": w.H_k,
                   "D": 128, "S_max": w.S_max, "lengths": w.lengths, "insert": w.insert,
                   "cached_tokens": int(inp.seqlen.sum()),
                   "l2": f"K/V cache of {cache_bytes / 2**30:.2f} GiB (> L2) read once per step",
                   "parallelism": f"replicas x{world} (independent problems)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": f"hbm_gbs of {peak_src}",
                     "traffic": gen_profiled_traffic(args.gen_config), "algorithmic_bytes": nbytes,
                     "algorithmic_flops": flops, "launch_ms": round(launch_ms, 5)},
        "e2e": {"value": round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * K,
        "clocks": sampler.summary(t_host0, t_host1),
    }
    if not args.no_cpu_baseline:
        b, t, n, threads = time_gen_oracle(inp, target_s=10.0)
        line["cpu_baseline"] = {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"the first {n} of {w.B} sequences, all heads "
                                          f"({b / 1e9:.2f} GB of the workload, {t:.1f} s)"}
    print(json.dumps(line), flush=True)


def run_gen_reference(args, rank, world):
    """The generation oracle as the reference arm: each step one sequence of the
    workload (all heads), on the host cores."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.GEN_CONFIGS[args.gen_config]
    inp = wl.generate_gen(w)
    odt = {"bf16": oracle.BF16, "f16": oracle.F16, "e4m3": oracle.E4M3}[w.dtype]
    esz = 1 if w.dtype == "e4m3" else 2
    threads = cpu_threads()

    def one(b):
        sl = inp.seqlen[b:b + 1].numpy()
        oracle.gen_fwd(wl.bits(inp.q[b:b + 1]), wl.bits(inp.k_cache[b:b + 1]), wl.bits(inp.v_cache[b:b + 1]),
                       wl.bits(inp.k_new[b:b + 1]) if inp.k_new is not None else None,
                       wl.bits(inp.v_new[b:b + 1]) if inp.v_new is not None else None, odt, 1, w.H, w.H_k,
                       128, 1, w.S_max, sl, None, 128 ** -0.5, 1.0, threads=threads)
        return gen_bytes(1, w.H, w.H_k, sl.tolist(), w.insert, esz)

    for i in range(args.warmup):
        one(i % w.B)
    t = time.perf_counter()
    nb = sum(one((args.warmup + i) % w.B) for i in range(args.steps))
    dt = time.perf_counter() - t
    value = nb / dt / 1e9
    print(json.dumps({
        "metric": "generation-phase attention HBM bandwidth (GB/s) and % of measured copy rate",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": args.gen_config}, "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": "one sequence (all heads) per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


BWD_SHAPES = {   # name -> (B, H, S, D, mask[, dtype]); synthetic N(0,1) q, k, v, dO
    "bwd_bf16_causal_b2_h16_s8192_d128": (2, 16, 8192, 128, "causal"),
    "bwd_e4m3_causal_b2_h16_s8192_d128": (2, 16, 8192, 128, "causal", "e4m3"),
    "bwd_bf16_nomask_b2_h16_s8192_d128": (2, 16, 8192, 128, "none"),
    "bwd_bf16_causal_b4_h16_s2048_d128": (4, 16, 2048, 128, "causal"),
    "bwd_bf16_causal_b2_h16_s4096_d128": (2, 16, 4096, 128, "causal"),   # profiling size (7 x 32 MB)
}


def bwd_flops(B, H, S, D, causal):
    """Algorithmic FLOPs of the backward: the five products of the chain rule
    (S, dP, dV, dQ, dK), 2*S*S*D each per head, halved for a causal mask."""
    return 10.0 * B * H * S * S * D * (0.5 if causal else 1.0)


def run_bwd(args, rank, world, local):
    """Backward pass (fmha_bwd) on synthetic inputs; O and LSE come from fmha_fwd."""
    from head_attention_forward_02_gb300 import build, fmha as fm
    build.build()
    fm.lib()
    dev = torch.device("cuda", local if world > 1 else 0)
    B, H, S, D, mask = BWD_SHAPES[args.bwd_config][:5]
    dtype = (BWD_SHAPES[args.bwd_config][5:] or ("bf16",))[0]
    tdt = wl.DTYPES[dtype]
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator().manual_seed(31)
    host = {n: torch.randn(B, S, H, D, generator=g).clamp_(-448, 448).to(tdt) for n in ("q", "k", "v", "do")}
    d = {n: t.to(dev) for n, t in host.items()}
    o, lse = fm.fwd(d["q"], d["k"], d["v"], mask=mask)
    code = {"f16": fm.F16, "bf16": fm.BF16, "e4m3": fm.E4M3}[dtype]
    ws = torch.empty(fm.fmha_bwd_workspace_size_ex(B, H, S, S, D, code), dtype=torch.uint8, device=dev)
    grads = [torch.empty(d["q"].shape, dtype=torch.bfloat16 if dtype == "e4m3" else tdt, device=dev)
             for _ in range(3)]
    flops = bwd_flops(B, H, S, D, mask == "causal")

    def step():
        fm.bwd(d["q"], d["k"], d["v"], o, d["do"], lse, mask=mask, dq=grads[0], dk=grads[1], dv=grads[2],
               workspace=ws, stream=stream)

    sampler = ClockSampler(gpu_uuid(dev.index or 0))
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fm.device_status(reset=True) != 0:
        raise RuntimeError("device status reports an error")
    K = args.steps
    barrier(world)
    torch.cuda.synchronize(dev)
    t_host0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(K):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_host1 = time.time()
    if rank == 0:
        sampler.stop()
    if fm.device_status(reset=True) != 0:
        raise RuntimeError("device status reports an error")
    ms = max_over_ranks(ev0.elapsed_time(ev1) / K, world)
    value = world * flops / (ms * 1e-3) / 1e12
    # end to end: every step copies q, k, v, O, dO and LSE in from pinned
    # memory and dQ, dK, dV out, pipelined over two device sets
    pin = {n: t.pin_memory() for n, t in host.items()}
    pin["o"], pin["lse"] = o.cpu().pin_memory(), lse.cpu().pin_memory()
    e2e_sets = [{n: torch.empty_like(t, device=dev) for n, t in pin.items()} for _ in range(2)]
    for es in e2e_sets:
        es.update({"dq": torch.empty_like(grads[0]), "dk": torch.empty_like(grads[0]),
                   "dv": torch.empty_like(grads[0]), "ws": torch.empty_like(ws)})
    outs = [{n: torch.empty(tuple(host["q"].shape), dtype=torch.bfloat16).pin_memory() for n in ("dq", "dk", "dv")}
            for _ in range(2)]

    def launch(es, st):
        fm.bwd(es["q"], es["k"], es["v"], es["o"], es["do"], es["lse"], mask=mask, dq=es["dq"], dk=es["dk"],
               dv=es["dv"], workspace=es["ws"], stream=st)

    e2e_steps = args.e2e_steps or 6
    e2e_pipelined(dev, 2, e2e_sets, pin, outs, launch)          # warm-up
    barrier(world)
    e2e_ms = max_over_ranks(e2e_pipelined(dev, e2e_steps, e2e_sets, pin, outs, launch), world)
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs[0].values())
    if rank != 0:
        return
    peaks, peak_src = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": "FMHA backward TFLOP/s (5 products of the chain rule) and % of GB300 dense bf16 peak",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype, "data": "synthetic (seeded N(0,1) q, k, v, dO; O and LSE from fmha_fwd)",
        "config": {"workload": args.bwd_config, "op": "fmha_bwd", "B": B, "H": H, "S": S, "D": D, "mask": mask,
                   "gradients": "bf16" if dtype == "e4m3" else dtype,
                   "l2": f"inputs and outputs {7 * B * S * H * D * 2 / 2**20:.0f} MiB (> L2)",
                   "parallelism": f"replicas x{world} (independent problems)"},
        "roofline": {"bound": "tensor", "achieved": round(flops / (ms * 1e-3) / 1e12, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(flops / (ms * 1e-3) / 1e12 / peak, 4),
                     "peak_source": f"bf16_tflops of {peak_src}", "traffic": None,
                     "algorithmic_flops": flops, "executed_flops": flops * 7 / 5,
                     "note": "two-pass design: S and dP are computed in both the dQ and the dK/dV kernel"},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (4 if dtype == "e4m3" else 3) * K,
        "clocks": sampler.summary(t_host0, t_host1),
    }
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        oracle.build()
        n = 384                                   # the first query rows of batch 0, every head, all keys
        dec = lambda t: t.float().numpy().astype(np.float64)
        q1, k1, v1, g1 = (dec(host[x][:1]) for x in ("q", "k", "v", "do"))
        t = time.perf_counter()
        oracle.attn_bwd_f64(q1[:, :n], k1, v1, g1[:, :n], D ** -0.5, oracle.MASK_NONE, oracle.QBEGIN,
                            threads=cpu_threads())
        dt = time.perf_counter() - t
        f = 10.0 * H * n * S * D
        line["cpu_baseline"] = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"{n} query rows x {S} keys x {H} heads, no mask "
                                          f"({f / 1e9:.1f} GFLOP, {dt:.1f} s)"}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded seeded sample
    of query rows of the same workload."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from tests.helpers import oracle_on
    oracle.build()
    w = ALL_CONFIGS[args.config]
    inp = wl.generate(w)
    threads = cpu_threads()
    rng = np.random.default_rng(1)
    if inp.cu_seqlens_q is None:
        pool = np.arange(w.B * w.H * w.Sq)
    else:
        T, end = inp.total_length, int(inp.cu_seqlens_q[-1])
        pool = np.array([h * T + t for h in range(w.H) for t in range(end)])
    rows_per_step = 64
    samples = [rng.choice(pool, size=rows_per_step) for _ in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle_on(oracle, inp, rows=samples[i], threads=threads)
    t = time.perf_counter()
    fl = 0.0
    for i in range(args.steps):
        r = samples[args.warmup + i]
        oracle_on(oracle, inp, rows=r, threads=threads)
        fl += oracle_rows_flops(inp, r)
    dt = time.perf_counter() - t
    value = fl / dt / 1e12
    line = {"metric": "FMHA forward TFLOP/s and % of GB300 dense tensor peak (bf16/fp8)",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded N(0,1))",
            "config": {"workload": args.config}, "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"{rows_per_step} seeded random query rows per step"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        (run_gen_reference if args.op == "gen" else run_reference)(args, rank, world)
        return
    rank, world, local = dist_setup(args.gpus)
    try:
        {"gen": run_gen, "bwd": run_bwd}.get(args.op, run_ours)(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
