"""Benchmark of the attention forward on B300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one attn_fwd call (V -> fp16 pre-pass + the tensor-core attention kernel) over the whole
workload, inputs resident in HBM. Default workload: B=1, H=16, N=8192, d=128, bf16, non-causal,
1% of key rows scaled x8 (the headline N=8192, d=128 point). L2 is flushed (256 MiB write) before
every timed step, outside the timed events. Under torchrun each rank runs the same workload on its
own GPU (independent problems, no collective on the data path) and the max time over ranks counts.

The line also carries ``extras`` (skip with ``--no-extras``): the fp8, backward, bias + dropout and
dropout paths timed on the same workload, the device time of one call of every workload (replayed
from a CUDA graph, so that host launch overhead is not in it), and the oracle on one host core for
the two smallest workloads.

``--impl reference`` times the fp64 CPU oracle instead (the only reference implementation available:
the pages ship no runnable code), on a bounded sample of the workload's query rows per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_tiled_attention_50_b300 import inputs  # noqa: E402

METRIC = "attention fwd TFLOP/s and % of B300 dense-BF16 peak at N=8192, d=128"
METRIC_BWD = "attention bwd TFLOP/s (10 B H N^2 d) and % of B300 dense-BF16 peak at N=8192, d=128"
METRIC_EX = "attention fwd TFLOP/s with additive bias and/or dropout p=0.1 at N=8192, d=128"
METRIC_FP8 = "attention fwd TFLOP/s of the fp8 (E4M3) path and % of B300 dense-FP8 peak at N=8192, d=128"
UNIT = "TFLOP/s"
# query rows of the fp64 oracle: the CPU-baseline leg times CPU_ROWS rows (10-30 s on the host cores);
# the reference arm spreads about REF_BUDGET_ROWS rows over all of its steps
CPU_ROWS = 32768
REF_BUDGET_ROWS = 262144


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(bf16=float(d["bf16_tflops"]), bf16_sustained=float(d["bf16_tflops_sustained"]),
                    hbm=float(d["hbm_gbs"]), source="measured")
    return dict(bf16=1800.0, bf16_sustained=1400.0, hbm=6400.0, source="fallback")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over every rank of the default process group (the slowest
    rank sets a job's time); the values themselves when there is no process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_value(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time (ms), in
    units per second divided by 1e12 (TFLOP/s for FLOP units)."""
    return world * units_per_rank / (ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            self.t0 = time.time()
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(rows), "reasons": reasons,
                "power_w_max": max(num(r[3]) for r in rows)}


def flops_of(w) -> float:
    return w.nominal_flops()


KERNEL_SOURCES = ("exact_tiled_attention_50_b300/csrc/attn_tc.cu", "exact_tiled_attention_50_b300/csrc/sm103_ptx.cuh",
                  "exact_tiled_attention_50_b300/csrc/attn_internal.h")


BWD_SOURCES = ("exact_tiled_attention_50_b300/csrc/attn_bwd.cu", "exact_tiled_attention_50_b300/csrc/sm103_ptx.cuh",
               "exact_tiled_attention_50_b300/csrc/attn_internal.h")


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(w, path_kind="bf16"):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary of this workload,
    or None when there is none or the kernel source changed since it was taken."""
    tag = "" if path_kind == "bf16" else "_" + path_kind
    name = "attn_bwd_q64_kernel" if path_kind == "bwd" else f"attn_fwd_tc_kernel{tag}"
    sources = BWD_SOURCES if path_kind == "bwd" else KERNEL_SOURCES
    path = os.path.join(ROOT, "profiles", f"{name}_b{w.B}h{w.H}_n{w.N}_d{w.d}.md")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            m = re.match(r"^(traffic_bytes_per_launch|kernel_source_sha256_16):\s*(\S+)", line)
            if m:
                kv[m.group(1)] = m.group(2)
    if kv.get("kernel_source_sha256_16") != kernel_source_hash(sources) or "traffic_bytes_per_launch" not in kv:
        return None
    return float(kv["traffic_bytes_per_launch"])


def oracle_sample_rows(w, n_rows, seed=0):
    rng = np.random.default_rng(seed)
    total = w.B * w.H * w.N
    return np.sort(rng.choice(total, size=min(n_rows, total), replace=False)).astype(np.int64)


def time_oracle(x, w, rows_per_step, steps, warmup):
    """The fp64 CPU oracle (as it stands) on `rows_per_step` query rows per step."""
    import oracle
    per_row = 4.0 * w.N * w.d * (0.5 if w.causal else 1.0)  # nominal FLOPs of one query row
    times = []
    for s in range(warmup + steps):
        rows = oracle_sample_rows(w, rows_per_step, seed=s)
        t0 = time.perf_counter()
        oracle.attention_rows(x.q, x.k, x.v, x.scale, rows, causal=w.causal, kv_len=x.kv_len)
        dt = time.perf_counter() - t0
        if s >= warmup:
            times.append(dt)
    sec = sum(times) / len(times)
    return dict(value=per_row * rows_per_step / sec / 1e12, sec_per_step=sec, cores=oracle.num_threads(),
                sample=f"{rows_per_step} query rows (of {w.B * w.H * w.N}) of {w.name} per step, each row over all "
                       f"{w.N} keys in fp64")


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = inputs.make_inputs(w)
    # about REF_BUDGET_ROWS rows over the whole run (a few minutes on 8-16 host cores)
    rows = max(16, min(args.ref_rows, REF_BUDGET_ROWS // (args.steps + args.warmup)))
    r = time_oracle(x, w, rows, args.steps, args.warmup)
    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["sec_per_step"] * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, on the host)",
        "impl": "reference",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d, "causal": w.causal,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
        "e2e": {"value": r["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _path_meta(path):
    """(metric, FLOP multiplier over the forward's nominal FLOPs, peak multiplier over the bf16 peak)."""
    return {"bf16": (METRIC, 1.0, 1.0), "fp8": (METRIC_FP8, 1.0, 2.0), "bias_dropout": (METRIC_EX, 1.0, 1.0),
            "dropout": (METRIC_EX, 1.0, 1.0), "bwd": (METRIC_BWD, 2.5, 1.0)}[path]


PATH_DESC = {"fp8": "fp8: Q, K rotated (random signs) + E4M3 per 128-row tile; E4M3 tensor cores",
             "bias_dropout": "bf16 + additive bf16 bias [B,H,N,N] + dropout p=0.1 (Philox4x32-10)",
             "dropout": "bf16 + dropout p=0.1 (Philox4x32-10)",
             "bwd": "backward: dQ, dK, dV (fp32) from bf16 Q, K, V, dO and the forward's O, LSE",
             "bf16": "bf16 tensor cores (fp16 P, fp16 V)"}


class Problem:
    """Device tensors of one workload and the step of each path over them (every step one call of the
    library's public API on the current stream, inputs resident)."""

    def __init__(self, attn, w, x, dev):
        self.attn, self.w, self.x, self.dev = attn, w, x, dev
        self.q, self.k, self.v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        self.kv = x.kv_len.to(dev) if x.kv_len is not None else None
        B, H, N, d = self.q.shape
        self.out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        wsb = max(attn.workspace_bytes(B, w.H, w.H_kv, N, d, self.q.dtype),
                  int(attn.lib.attn_fwd_fp8_workspace_bytes(B, w.H, w.H_kv, N, d)) if d == 128 else 0)
        self.work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        self.bias = None
        self.dO = None
        self.grads = []

    def prepare(self, path):
        w, attn = self.w, self.attn
        if path == "bias_dropout" and self.bias is None:  # one bf16 bias value per (b, h, i, j), drawn on the device
            gen = torch.Generator(device=self.dev)
            gen.manual_seed(inputs.SEED_BASE + 4000)
            self.bias = torch.randn((w.B, w.H, w.N, w.N), generator=gen, device=self.dev,
                                    dtype=torch.float32).to(torch.bfloat16)
        if path == "fp8":
            self.signs = inputs.random_signs(w.d, seed=0).to(self.dev)
        if path == "bwd" and self.dO is None:  # the forward's O and LSE once, and a seeded upstream gradient
            attn.attn_fwd(self.q, self.k, self.v, scale=self.x.scale, causal=w.causal, kv_len=self.kv, out=self.out,
                          lse=self.lse, workspace=self.work)
            gen = torch.Generator().manual_seed(inputs.SEED_BASE + 5000)
            self.dO = torch.randn(tuple(self.q.shape), generator=gen).to(torch.bfloat16).to(self.dev)

    def step_fn(self, path):
        self.prepare(path)
        attn, x, w = self.attn, self.x, self.w
        q, k, v, kv, out, lse, work = self.q, self.k, self.v, self.kv, self.out, self.lse, self.work
        if path == "bwd":
            def step():
                self.grads[:] = attn.attn_bwd(q, k, v, out, self.dO, lse, scale=x.scale, causal=w.causal, kv_len=kv)
        elif path == "fp8":
            def step():
                attn.attn_fwd_fp8(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, signs=self.signs, out=out,
                                  lse=lse, workspace=work)
        elif path in ("bias_dropout", "dropout"):
            bias = self.bias if path == "bias_dropout" else None

            def step():
                attn.attn_fwd_ex(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, bias=bias, dropout_p=0.1,
                                 seed=1, offset=0, out=out, lse=lse, workspace=work)
        else:
            def step():
                attn.attn_fwd(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, out=out, lse=lse, workspace=work)
        return step


def timed_steps(attn, step, flush, stream, K, warmup, world=1):
    """Per-step device times (ms) of K steps and of the library's main kernel inside each (CUDA events
    on the launching stream; the L2 flush runs before each step, outside the events)."""
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rc = attn.check()
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"warm-up failed: {attn.status_string(rc)}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in kev:  # torch creates the CUDA event on first record: materialise the handles now
        a.record(stream)
        b.record(stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()  # outside the timed events: evicts Q/K/V/O from L2
        attn.set_kernel_events(*kev[i])
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    attn.set_kernel_events(None, None)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    rc = attn.check()
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"timed run failed: {attn.status_string(rc)}")
    return [a.elapsed_time(b) for a, b in ev], [attn.event_elapsed_ms(a, b) for a, b in kev], wall


def graph_call_times(attn, step, flush, stream, reps=20, warmup=3):
    """Device time (ms) of one call replayed from a CUDA graph, so that the host's launch overhead is
    not in it: events before and after each replay, L2 flushed before each (outside the events)."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    cs = torch.cuda.Stream(stream.device)
    cs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        step()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    rc = attn.check()
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"graph replay failed: {attn.status_string(rc)}")
    del g
    return ts


def roofline_of(path, w, kern_ms, prob, peaks):
    metric, fmul, pmul = _path_meta(path)
    flops = flops_of(w) * fmul
    achieved = flops / (kern_ms * 1e-3) / 1e12
    peak = peaks["bf16"] * pmul
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak}
    if path == "bias_dropout":
        # the bias (2 B per score) outweighs the tensor work at these sizes: the kernel is HBM-bound
        nbytes = (prob.bias.numel() * 2 + (prob.q.numel() + prob.k.numel() + prob.v.numel()) * 2 +
                  prob.out.numel() * 4 + prob.lse.numel() * 4)
        gbs = nbytes / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                "algorithmic_bytes": nbytes, "tensor_tflops": achieved}
    return roof


def run_extras(attn, prob, flush, stream, peaks, args):
    """Other numbers on the same box in the same run: the other paths on the headline workload, the
    device time of one call of every workload (graph replay, L2 flushed), and the oracle on one host
    core for the two smallest workloads."""
    extras = {}
    paths = {}
    for path in ("fp8", "bwd", "bias_dropout", "dropout"):
        if path == "fp8" and prob.w.d != 128:
            continue
        step = prob.step_fn(path)
        st, kt, _ = timed_steps(attn, step, flush, stream, args.extra_steps, 3)
        metric, fmul, pmul = _path_meta(path)
        flops = flops_of(prob.w) * fmul
        km = statistics.median(kt)
        roof = roofline_of(path, prob.w, km, prob, peaks)
        paths[path] = {"metric": metric, "path": PATH_DESC[path], "steps": len(st),
                       "ms_per_step_median": statistics.median(st), "ms_per_step_mean": sum(st) / len(st),
                       "value": flops / (statistics.median(st) * 1e-3) / 1e12, "unit": UNIT,
                       "kernel_ms_median": km, "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit",
                                                                                 "frac")}}
    prob.bias = None
    prob.grads[:] = []
    torch.cuda.empty_cache()
    extras["paths"] = paths
    wl = {}
    for name, w in inputs.WORKLOADS.items():
        x = inputs.make_inputs_device(w, prob.dev)
        p2 = Problem(attn, w, x, prob.dev)
        ts = graph_call_times(attn, p2.step_fn("bf16"), flush, stream)
        med = statistics.median(ts)
        lens = None if x.kv_len is None else x.kv_len.cpu().tolist()
        wl[name] = {"us_per_call_median": med * 1e3, "tflops_nominal": w.nominal_flops() / (med * 1e-3) / 1e12,
                    "tflops_effective": inputs.effective_flops(w, lens) / (med * 1e-3) / 1e12,
                    "frac_of_bf16_peak": w.nominal_flops() / (med * 1e-3) / 1e12 / peaks["bf16"]}
        del p2, x
    torch.cuda.empty_cache()
    extras["workloads"] = {"how": "one attn_fwd call (all its launches) captured in a CUDA graph, replayed 20 times, "
                                  "median of the device time between events around each replay, L2 flushed before "
                                  "each; inputs drawn on the device with the workload's recipe",
                           "per_workload": wl}
    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.num_threads()
        oracle.set_num_threads(1)
        one = {}
        for name, frac in (("tiny_b1h1_n256_d64_f32", 1), ("b4h8_n1024_d64", 8)):
            w = inputs.WORKLOADS[name]
            x = inputs.make_inputs(w)
            total = w.B * w.H * w.N
            r = time_oracle(x, w, total // frac, 1, 0)
            one[name] = {"value": r["value"], "unit": UNIT, "cores": 1, "kind": "oracle", "sample": r["sample"]}
        oracle.set_num_threads(threads)
        extras["cpu_baseline_1thread"] = one
    return extras


def run_ours(args, w):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from exact_tiled_attention_50_b300 import attn

    x = inputs.make_inputs(w)
    prob = Problem(attn, w, x, dev)
    q, kv, out, lse = prob.q, prob.kv, prob.out, prob.lse
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    bwd = args.path == "bwd"
    step = prob.step_fn(args.path)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    st, kt, wall = timed_steps(attn, step, flush, stream, K, args.warmup, ws)
    clocks = sampler.stop()
    step_ms, kern_ms = sum(st) / K, sum(kt) / K
    step_med, kern_med = statistics.median(st), statistics.median(kt)
    step_ms, kern_ms, step_med, kern_med = max_over_ranks([step_ms, kern_ms, step_med, kern_med], device=dev)

    # ---- end to end through the public API: pinned host inputs -> device -> the call -> host ----
    hq, hk, hv = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
    hkv = x.kv_len.pin_memory() if x.kv_len is not None else None
    ho = torch.empty_like(out, device="cpu").pin_memory()
    hl = torch.empty_like(lse, device="cpu").pin_memory()
    # the backward's extra inputs (dO, and O, LSE of the forward) and its three gradients
    h_in = [(prob.dO.cpu().pin_memory(), prob.dO), (ho, out), (hl, lse)] if bwd else []
    h_grads = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in prob.grads] if bwd else []
    e2e_steps = max(1, min(K, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    # the bf16 forward's public host-buffer call: copies in, attention and copies back pipelined over
    # groups of heads inside the library (attn_fwd_host)
    e2e_pipe_ms = []
    if args.path == "bf16":
        for i in range(e2e_steps + 1):
            flush.zero_()
            e0.record(stream)
            attn.attn_fwd_host(hq, hk, hv, ho, hl, prob.q, prob.k, prob.v, out, lse, scale=x.scale, causal=w.causal,
                               kv_len_h=hkv, kv_len_d=kv, workspace=prob.work)
            e1.record(stream)
            torch.cuda.synchronize()
            if i > 0:
                e2e_pipe_ms.append(e0.elapsed_time(e1))
        rc = attn.check()
        if rc != attn.ATTN_OK:
            raise RuntimeError(f"attn_fwd_host failed: {attn.status_string(rc)}")
    # the same step with the copies issued one after another on one stream around the device call
    e2e_ms = []
    for i in range(e2e_steps + 1):
        flush.zero_()
        e0.record(stream)
        prob.q.copy_(hq, non_blocking=True)
        prob.k.copy_(hk, non_blocking=True)
        prob.v.copy_(hv, non_blocking=True)
        if hkv is not None:
            kv.copy_(hkv, non_blocking=True)
        for h, dvc in h_in:
            dvc.copy_(h, non_blocking=True)
        step()
        if bwd:
            for h, g in zip(h_grads, prob.grads):
                h.copy_(g, non_blocking=True)
        else:
            ho.copy_(out, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i > 0:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_serial = sum(e2e_ms) / len(e2e_ms)
    e2e = sum(e2e_pipe_ms) / len(e2e_pipe_ms) if e2e_pipe_ms else e2e_serial
    e2e, e2e_serial = max_over_ranks([e2e, e2e_serial], device=dev)
    h2d = sum(t.numel() * t.element_size() for t in [hq, hk, hv] + [h for h, _ in h_in]) + \
        (hkv.numel() * 4 if hkv is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in h_grads) if bwd else ho.numel() * 4 + hl.numel() * 4

    metric, fmul, pmul = _path_meta(args.path)
    flops = flops_of(w) * fmul
    lens = None if x.kv_len is None else x.kv_len.tolist()
    eff = inputs.effective_flops(w, lens) * fmul
    peaks = load_peaks()
    roof = roofline_of(args.path, w, kern_ms, prob, peaks)
    peak_sus = peaks["bf16_sustained"] * pmul
    fp8 = args.path == "fp8"
    ex = args.path in ("bias_dropout", "dropout")
    line = {
        "metric": metric,
        "value": job_value(flops, ws, step_ms),
        "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "ms_per_step_median": step_med,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), 1% of key rows x8)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d, "causal": w.causal,
                   "in": "bf16", "out": "fp32 O + fp32 LSE", "path": PATH_DESC[args.path],
                   "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
                   **({"bias": "bf16 [B,H,N,N] resident on the device (not part of the e2e copies)"}
                      if args.path == "bias_dropout" else {}),
                   "parallelism": f"replicas x{ws} (independent problems per GPU)",
                   "pct_of_peak_bf16": 100.0 * flops / (step_ms * 1e-3) / 1e12 / peaks["bf16"]},
        "effective": {"flops_per_step": eff, "nominal_flops_per_step": flops,
                      "value": job_value(eff, ws, step_ms), "unit": UNIT,
                      "note": "4 d per unmasked (query, key) pair (x2.5 for the backward)"},
        "roofline": {**roof,
                     "traffic": args.traffic if args.traffic is not None else profiled_traffic(w, args.path),
                     "kernel": (("attn_bwd_q64_kernel" if w.d == 128 else f"attn_bwd_tc_kernel<{w.d}>")
                                + " (with its row-statistics pass)") if bwd
                     else f"attn_fwd_tc_kernel<{w.d},false,{1 if fp8 else 2 if ex else 0}>", "kernel_ms": kern_ms,
                     "kernel_ms_median": kern_med,
                     "peak_source": (f"{peaks['source']} bf16 burst (cuBLAS) x 2 (nominal fp8/bf16 dense ratio)"
                                     if fp8 else f"{peaks['source']} " + ("copy bandwidth" if args.path == "bias_dropout"
                                                                          else "bf16 burst (cuBLAS)"))
                                    + f"; tensor frac of sustained {flops / (kern_ms * 1e-3) / 1e12 / peak_sus:.3f}"},
        "e2e": {"value": job_value(flops, ws, e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e,
                "how": ("attn_fwd_host: pinned host Q, K, V (kv_len) in, O, LSE back, copies and compute "
                        "pipelined over groups of heads" if e2e_pipe_ms else
                        "copies to the device, the call, copies back, one after another on one stream"),
                "serial": {"value": job_value(flops, ws, e2e_serial), "ms_per_step": e2e_serial,
                           "how": "the same copies one after another on one stream around the device call"}},
        "gpu_launches": K * (2 if bwd else attn.launches_per_call(q.dtype)),
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        r = time_oracle(x, w, args.cpu_rows, 1, 0)
        line["cpu_baseline"] = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                                "sample": r["sample"]}
    if rank == 0 and ws == 1 and args.path == "bf16" and not args.no_extras:
        line["extras"] = run_extras(attn, prob, flush, stream, peaks, args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_launch_list(args):
    """Three plain attn_fwd calls per workload, every workload in turn (inputs drawn on the device),
    for a profiler's launch list: the kernels appear in workload order, two launches per bf16 call
    (the V pre-pass, then the attention kernel) and one per fp32 call."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    from exact_tiled_attention_50_b300 import attn
    for name, w in inputs.WORKLOADS.items():
        x = inputs.make_inputs_device(w, dev)
        prob = Problem(attn, w, x, dev)
        step = prob.step_fn("bf16")
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        rc = attn.check()
        print(json.dumps({"workload": name, "calls": 3, "launches_per_call": attn.launches_per_call(x.q.dtype),
                          "status": attn.status_string(rc)}), flush=True)
        del prob, x
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--ref-rows", type=int, default=4096, help="max oracle query rows per step (reference arm)")
    ap.add_argument("--cpu-rows", type=int, default=CPU_ROWS, help="oracle query rows of the cpu_baseline leg")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--traffic", type=float, default=None, help="DRAM bytes per launch from an ncu capture")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other paths, the per-workload device times and the one-core oracle timings")
    ap.add_argument("--extra-steps", type=int, default=20, help="timed steps of each other path in the extras")
    ap.add_argument("--launch-list", action="store_true",
                    help="no timing: three calls of every workload in turn, for a profiler's launch list")
    ap.add_argument("--path", choices=["bf16", "fp8", "bias_dropout", "dropout", "bwd"], default="bf16",
                    help="bf16 tensor-core path (the headline) or the fp8 path with incoherent processing")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.launch_list:
        return run_launch_list(args)
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
