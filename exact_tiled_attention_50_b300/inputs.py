"""Seeded synthetic inputs for the attention forward, shared by the CUDA path and the oracle.

This module draws random numbers and nothing else: it holds none of the attention arithmetic, so the
oracle and the CUDA kernels can both consume its tensors without sharing any of the method's code.

Recipe (one ``torch.Generator('cpu')`` per workload, seeded ``20261202 + config_index``), drawn in
this order:

1. Q, K, V as fp32 ``randn`` of shapes [B,H,N,d], [B,H_kv,N,d], [B,H_kv,N,d], then rounded to the
   input dtype (round-to-nearest-even for bf16);
2. for key-padded workloads, ``kv_len = randint(N//2, N+1, (B,))`` (int32);
3. for "peaky" workloads, per (b, kv-head) in row-major order, ``randperm(N)[:ceil(0.01*N)]`` picks the
   key rows that are multiplied by 8 (a power of two, so exact in bf16).

The workloads are the ones the attention pages motivate (multi-head attention over long sequences,
with padding masks, grouped/multi-query heads and long-context sweeps): value distribution N(0,1),
layout [B, heads, N, d] row-major.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    H_kv: int
    N: int
    d: int
    dtype: str  # "f32" or "bf16" (input dtype of Q, K, V)
    causal: bool = False
    padded: bool = False  # per-batch key-padding length kv_len ~ U[N/2, N]
    peaky: bool = False  # 1% of K rows scaled x8
    config_index: int = 0  # selects the seed

    @property
    def scale(self) -> float:
        """1/sqrt(head_dim), rounded to fp32 (the value the C ABI receives)."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32).item())

    @property
    def seed(self) -> int:
        return SEED_BASE + self.config_index

    def nominal_flops(self) -> float:
        """4*B*H*N^2*d, halved when causal (the headline FLOP convention)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _sweep(n: int, causal: bool) -> Workload:
    tag = "causal" if causal else "noncausal"
    return Workload(f"sweep_b1h16_d128_n{n}_{tag}_peaky", 1, 16, 16, n, 128, "bf16",
                    causal=causal, peaky=True, config_index=5)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_b1h1_n256_d64_f32", 1, 1, 1, 256, 64, "f32", config_index=1),
        Workload("b4h8_n1024_d64", 4, 8, 8, 1024, 64, "bf16", config_index=2),
        Workload("b8h16_n4096_d128_causal_padded", 8, 16, 16, 4096, 128, "bf16",
                 causal=True, padded=True, config_index=3),
        Workload("gqa_b2h32kv8_n8192_d128_causal", 2, 32, 8, 8192, 128, "bf16",
                 causal=True, config_index=4),
        Workload("mqa_b2h32kv1_n8192_d128_causal", 2, 32, 1, 8192, 128, "bf16",
                 causal=True, config_index=4),
        *[_sweep(n, c) for c in (False, True) for n in (512, 1024, 2048, 4096, 8192, 16384)],
    ]
}

# The workload the headline throughput is quoted on: N=8192, d=128, one GPU.
HEADLINE = "sweep_b1h16_d128_n8192_noncausal_peaky"


@dataclass
class Inputs:
    q: torch.Tensor  # [B,H,N,d] in the input dtype, CPU
    k: torch.Tensor  # [B,H_kv,N,d]
    v: torch.Tensor  # [B,H_kv,N,d]
    kv_len: Optional[torch.Tensor]  # int32 [B] or None (all N keys valid)
    scale: float
    causal: bool


_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_inputs(w: Workload, seed: Optional[int] = None) -> Inputs:
    """Draw the inputs of workload ``w`` on the CPU (see the module docstring for the recipe)."""
    g = torch.Generator("cpu")
    g.manual_seed(w.seed if seed is None else seed)
    dt = _DT[w.dtype]
    q = torch.randn((w.B, w.H, w.N, w.d), generator=g, dtype=torch.float32).to(dt)
    k = torch.randn((w.B, w.H_kv, w.N, w.d), generator=g, dtype=torch.float32).to(dt)
    v = torch.randn((w.B, w.H_kv, w.N, w.d), generator=g, dtype=torch.float32).to(dt)
    kv_len = None
    if w.padded:
        kv_len = torch.randint(w.N // 2, w.N + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
    if w.peaky:
        n_rows = math.ceil(0.01 * w.N)
        for b in range(w.B):
            for hk in range(w.H_kv):
                rows = torch.randperm(w.N, generator=g)[:n_rows]
                k[b, hk, rows] = k[b, hk, rows] * 8
    return Inputs(q.contiguous(), k.contiguous(), v.contiguous(), kv_len, w.scale, w.causal)


def make_inputs_device(w: Workload, device, seed: Optional[int] = None) -> Inputs:
    """The recipe of ``make_inputs`` drawn on the device (a CUDA generator seeded the same way): the same
    shapes, distributions and structure, a different stream of numbers. For timing large workloads
    without drawing them on the host; parity always uses ``make_inputs``."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    dt = _DT[w.dtype]
    q = torch.randn((w.B, w.H, w.N, w.d), generator=g, dtype=torch.float32, device=device).to(dt)
    k = torch.randn((w.B, w.H_kv, w.N, w.d), generator=g, dtype=torch.float32, device=device).to(dt)
    v = torch.randn((w.B, w.H_kv, w.N, w.d), generator=g, dtype=torch.float32, device=device).to(dt)
    kv_len = None
    if w.padded:
        kv_len = torch.randint(w.N // 2, w.N + 1, (w.B,), generator=g, dtype=torch.int64, device=device).to(torch.int32)
    if w.peaky:
        n_rows = math.ceil(0.01 * w.N)
        for b in range(w.B):
            for hk in range(w.H_kv):
                rows = torch.randperm(w.N, generator=g, device=device)[:n_rows]
                k[b, hk, rows] = k[b, hk, rows] * 8
    return Inputs(q.contiguous(), k.contiguous(), v.contiguous(), kv_len, w.scale, w.causal)


def effective_flops(w: Workload, kv_len=None) -> float:
    """4 d per unmasked (query, key) pair, summed over batches and heads: the work the masks leave
    (kv_len given as a host sequence of B lengths, or None)."""
    total = 0
    for b in range(w.B):
        L = w.N if kv_len is None else min(max(int(kv_len[b]), 0), w.N)
        if w.causal:  # row i sees min(L, i + 1) keys
            total += L * (L + 1) // 2 + (w.N - L) * L
        else:
            total += w.N * L
    return 4.0 * w.d * w.H * total


def custom(B: int, H: int, H_kv: int, N: int, d: int, dtype: str = "bf16", *, causal: bool = False,
           padded: bool = False, peaky: bool = False, seed: int = 0, kv_len=None) -> Inputs:
    """Inputs of an arbitrary shape (edge-case tests); ``kv_len`` overrides the drawn lengths."""
    w = Workload("custom", B, H, H_kv, N, d, dtype, causal=causal, padded=padded, peaky=peaky)
    x = make_inputs(w, seed=SEED_BASE + 1000 + seed)
    if kv_len is not None:
        x.kv_len = torch.as_tensor(kv_len, dtype=torch.int32).reshape(B)
    return x


def random_signs(d: int, seed: int = 0) -> torch.Tensor:
    """d random signs (int8, +-1): the random draw of the fp8 path's rotation, passed to it as an input.
    Drawn as ``randint(0, 2, (d,))`` from a generator seeded ``SEED_BASE + 2000 + seed``; 0 -> -1."""
    g = torch.Generator("cpu")
    g.manual_seed(SEED_BASE + 2000 + seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.int8)


def with_outlier_channels(x: Inputs, n_channels: int = 4, factor: float = 16.0, seed: int = 0) -> Inputs:
    """The same inputs with ``n_channels`` channels of Q and K (the same channels in both, drawn as
    ``randperm(d)[:n_channels]`` from a generator seeded ``SEED_BASE + 3000 + seed``) multiplied by
    ``factor`` (a power of two, so exact in bf16): the large-magnitude feature channels that make
    per-tile low-precision scales coarse for every other channel."""
    d = x.q.shape[-1]
    g = torch.Generator("cpu")
    g.manual_seed(SEED_BASE + 3000 + seed)
    ch = torch.randperm(d, generator=g)[:n_channels]
    q, k = x.q.clone(), x.k.clone()
    q[..., ch] = q[..., ch] * factor
    k[..., ch] = k[..., ch] * factor
    return Inputs(q.contiguous(), k.contiguous(), x.v, x.kv_len, x.scale, x.causal)
