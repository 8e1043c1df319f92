"""Benchmark of the attention forward on B300: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one attn_fwd call (V -> fp16 pre-pass + the tensor-core attention kernel) over the whole
workload, inputs resident in HBM. Default workload: B=1, H=16, N=8192, d=128, bf16, non-causal,
1% of key rows scaled x8 (the headline N=8192, d=128 point). L2 is flushed (256 MiB write) before
every timed step, outside the timed events. Under torchrun each rank runs the same workload on its
own GPU (independent problems, no collective on the data path) and the max time over ranks counts.

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


def run_ours(args, w):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from exact_tiled_attention_50_b300 import attn

    x = inputs.make_inputs(w)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    kv = x.kv_len.to(dev) if x.kv_len is not None else None
    B, H, N, d = q.shape
    out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fp8 = args.path == "fp8"
    ex = args.path in ("bias_dropout", "dropout")
    bias = None
    if fp8:
        wsb = int(attn.lib.attn_fwd_fp8_workspace_bytes(B, w.H, w.H_kv, N, d))
        signs = inputs.random_signs(d, seed=0).to(dev)
    else:
        wsb = attn.workspace_bytes(B, w.H, w.H_kv, N, d, q.dtype)
    if args.path == "bias_dropout":  # one bf16 bias value per (b, h, i, j), drawn on the device
        gen = torch.Generator(device=dev)
        gen.manual_seed(inputs.SEED_BASE + 4000)
        bias = torch.randn((B, w.H, N, N), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    bwd = args.path == "bwd"
    if bwd:  # the forward's O and LSE once, and a seeded upstream gradient
        attn.attn_fwd(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, out=out, lse=lse, workspace=work)
        gen = torch.Generator().manual_seed(inputs.SEED_BASE + 5000)
        dO = torch.randn(tuple(q.shape), generator=gen).to(torch.bfloat16).to(dev)
    grads = []

    def step():
        if bwd:
            grads[:] = attn.attn_bwd(q, k, v, out, dO, lse, scale=x.scale, causal=w.causal, kv_len=kv)
        elif fp8:
            attn.attn_fwd_fp8(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, signs=signs, out=out, lse=lse,
                              workspace=work)
        elif ex:
            attn.attn_fwd_ex(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, bias=bias, dropout_p=0.1, seed=1,
                             offset=0, out=out, lse=lse, workspace=work)
        else:
            attn.attn_fwd(q, k, v, scale=x.scale, causal=w.causal, kv_len=kv, out=out, lse=lse, workspace=work)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    rc = attn.check()
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"warm-up failed: {attn.status_string(rc)}")

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in kev:  # torch creates the CUDA event on first record: materialise the handles now
        a.record(stream)
        b.record(stream)
    if ws > 1:
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
    clocks = sampler.stop()
    rc = attn.check()
    if rc != attn.ATTN_OK:
        raise RuntimeError(f"timed run failed: {attn.status_string(rc)}")
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    kern_ms = sum(attn.event_elapsed_ms(a, b) for a, b in kev) / K
    step_ms, kern_ms = max_over_ranks([step_ms, kern_ms], device=dev)

    # ---- end to end through the public API: pinned host inputs -> device -> attn_fwd -> host ----
    hq, hk, hv = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
    hkv = x.kv_len.pin_memory() if x.kv_len is not None else None
    ho = torch.empty_like(out, device="cpu").pin_memory()
    hl = torch.empty_like(lse, device="cpu").pin_memory()
    # the backward's extra inputs (dO, and O, LSE of the forward) and its three gradients
    h_in = [(dO.cpu().pin_memory(), dO), (ho, out), (hl, lse)] if bwd else []
    h_grads = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in grads] if bwd else []
    e2e_steps = max(1, min(K, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(e2e_steps + 1):
        flush.zero_()
        e0.record(stream)
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        if hkv is not None:
            kv.copy_(hkv, non_blocking=True)
        for h, dvc in h_in:
            dvc.copy_(h, non_blocking=True)
        step()
        if bwd:
            for h, g in zip(h_grads, grads):
                h.copy_(g, non_blocking=True)
        else:
            ho.copy_(out, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i > 0:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e = sum(e2e_ms) / len(e2e_ms)
    (e2e,) = max_over_ranks([e2e], device=dev)
    h2d = sum(t.numel() * t.element_size() for t in [hq, hk, hv] + [h for h, _ in h_in]) + \
        (hkv.numel() * 4 if hkv is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in h_grads) if bwd else ho.numel() * 4 + hl.numel() * 4

    # backward: 5 products of the forward's size (recomputed S, dP, dV, dK, dQ) against its 2
    flops = flops_of(w) * (2.5 if bwd else 1.0)
    peaks = load_peaks()
    achieved = flops / (kern_ms * 1e-3) / 1e12
    # the contraction's own dtype: E4M3 takes the measured bf16 peak times the nominal fp8 / bf16 ratio
    # (4.5 / 2.25 PFLOP/s dense)
    peak = peaks["bf16"] * (2.0 if fp8 else 1.0)
    peak_sus = peaks["bf16_sustained"] * (2.0 if fp8 else 1.0)
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak}
    if bias is not None:
        # the bias (2 B per score) outweighs the tensor work at these sizes: the kernel is HBM-bound
        nbytes = (bias.numel() * 2 + (q.numel() + k.numel() + v.numel()) * 2 + out.numel() * 4 + lse.numel() * 4)
        gbs = nbytes / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                "algorithmic_bytes": nbytes, "tensor_tflops": achieved}
    line = {
        "metric": {"fp8": METRIC_FP8, "bias_dropout": METRIC_EX, "dropout": METRIC_EX,
                   "bwd": METRIC_BWD}.get(args.path, METRIC),
        "value": job_value(flops, ws, step_ms),
        "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), 1% of key rows x8)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.H_kv, "N": w.N, "d": w.d, "causal": w.causal,
                   "in": "bf16", "out": "fp32 O + fp32 LSE",
                   "path": {"fp8": "fp8: Q, K rotated (random signs) + E4M3 per 128-row tile; E4M3 tensor cores",
                            "bias_dropout": "bf16 + additive bf16 bias [B,H,N,N] + dropout p=0.1 (Philox4x32-10)",
                            "dropout": "bf16 + dropout p=0.1 (Philox4x32-10)",
                            "bwd": "backward: dQ, dK, dV (fp32) from bf16 Q, K, V, dO and the forward's O, LSE"
                            }.get(args.path,
                                                                                  "bf16 tensor cores (fp16 P, fp16 V)"),
                   "l2": "flushed before every timed step (256 MiB write, outside the timed events)",
                   **({"bias": "bf16 [B,H,N,N] resident on the device (not part of the e2e copies)"}
                      if bias is not None else {}),
                   "parallelism": f"replicas x{ws} (independent problems per GPU)",
                   "pct_of_peak_bf16": 100.0 * flops / (step_ms * 1e-3) / 1e12 / peaks["bf16"]},
        "roofline": {**roof,
                     "traffic": args.traffic if args.traffic is not None else profiled_traffic(w, args.path),
                     "kernel": (("attn_bwd_q64_kernel" if w.d == 128 else f"attn_bwd_tc_kernel<{w.d}>")
                                + " (with its row-statistics pass)") if bwd
                     else f"attn_fwd_tc_kernel<{w.d},false,{1 if fp8 else 2 if ex else 0}>", "kernel_ms": kern_ms,
                     "peak_source": (f"{peaks['source']} bf16 burst (cuBLAS) x 2 (nominal fp8/bf16 dense ratio)"
                                     if fp8 else f"{peaks['source']} " + ("copy bandwidth" if bias is not None
                                                                          else "bf16 burst (cuBLAS)"))
                                    + f"; tensor frac of sustained {achieved / peak_sus:.3f}"},
        "e2e": {"value": job_value(flops, ws, e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e},
        "gpu_launches": K * attn.launches_per_call(q.dtype),
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        r = time_oracle(x, w, args.cpu_rows, 1, 0)
        line["cpu_baseline"] = {"value": r["value"], "unit": UNIT, "cores": r["cores"], "kind": "oracle",
                                "sample": r["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
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
    ap.add_argument("--path", choices=["bf16", "fp8", "bias_dropout", "dropout", "bwd"], default="bf16",
                    help="bf16 tensor-core path (the headline) or the fp8 path with incoherent processing")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
