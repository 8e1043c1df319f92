"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and compare it with
the oracle on the same seeded inputs.

Tolerances (the attention parity bar): bf16 inputs -> max |dO| <= 2e-3 and mean |dO| <= 2e-4;
fp32 inputs -> max |dO| <= 1e-5; |dLSE| <= 1e-3. bf16 outputs add the output rounding itself: half a
bf16 ulp of the reference value to the max bound, and the mean of those half-ulps to the mean bound.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"bf16": dict(max_abs=2e-3, mean_abs=2e-4), "f32": dict(max_abs=1e-5, mean_abs=1e-5)}
LSE_TOL = 1e-3


def run_gpu(x, out_dtype=torch.float32, device="cuda"):
    from exact_tiled_attention_50_b300 import attn
    q, k, v = x.q.to(device), x.k.to(device), x.v.to(device)
    kv = x.kv_len.to(device) if x.kv_len is not None else None
    O, L = attn.attn_fwd(q, k, v, scale=x.scale, causal=x.causal, kv_len=kv, out_dtype=out_dtype)
    rc = attn.check()
    assert rc == attn.ATTN_OK, f"{attn.status_string(rc)} bits {attn.lib.attn_debug_last_error_bits():#x}"
    return O, L


def sample_rows(B, H, N, kv_len=None, per_head=48, seed=0):
    """Flat row ids (b*H + h)*N + i: tile edges, the last row, kv_len boundaries, and random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(B):
        fixed = {0, 1, 127, 128, 129, 255, 256, 383, 384, N // 2, N - 2, N - 1}
        if kv_len is not None:
            L = int(kv_len[b])
            fixed |= {L - 1, L, L + 1}
        fixed = [i for i in fixed if 0 <= i < N]
        for h in range(H):
            extra = rng.integers(0, N, size=max(0, per_head - len(fixed)))
            for i in sorted(set(fixed) | set(int(e) for e in extra)):
                rows.append((b * H + h) * N + i)
    return np.array(rows, dtype=np.int64)


def compare(O_gpu, L_gpu, O_ref, L_ref, dtype, out_dtype=torch.float32, what=""):
    """Element-wise comparison; returns a dict of error statistics (asserts the bar)."""
    O = O_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(O_ref.shape)
    d = np.abs(O - O_ref)
    tol = TOL[dtype]
    max_bound = tol["max_abs"]
    if out_dtype == torch.bfloat16:
        # half an ulp of bf16 at the reference magnitude (2^-8 relative, times 2^-1)
        ulp_half = np.ldexp(1.0, np.frexp(np.abs(O_ref))[1] - 9)
        bound = max_bound + ulp_half
        assert np.all(d <= bound), f"{what}: bf16-out error above bound, worst {float(np.max(d - bound))}"
    else:
        assert np.isfinite(O).all(), f"{what}: non-finite output"
        assert float(d.max()) <= max_bound, f"{what}: max abs {float(d.max()):.3g} > {max_bound}"
    mean_bound = tol["mean_abs"]
    if out_dtype == torch.bfloat16:
        mean_bound += float(np.mean(ulp_half))  # the output rounding itself, on average at most half an ulp
    assert float(d.mean()) <= mean_bound, f"{what}: mean abs {float(d.mean()):.3g} > {mean_bound:.3g}"
    stats = dict(max_abs=float(d.max()), mean_abs=float(d.mean()))
    if L_gpu is not None:
        L = L_gpu.detach().cpu().numpy().astype(np.float64).reshape(L_ref.shape)
        fin = np.isfinite(L_ref)
        assert np.array_equal(np.isfinite(L), fin), f"{what}: LSE finiteness differs"
        assert np.all(L[~fin] == -np.inf), f"{what}: empty rows must have LSE = -inf"
        if fin.any():
            dl = float(np.abs(L[fin] - L_ref[fin]).max())
            assert dl <= LSE_TOL, f"{what}: LSE max abs {dl:.3g} > {LSE_TOL}"
            stats["lse_max_abs"] = dl
    return stats


def check_full(x, dtype, out_dtype=torch.float32, what=""):
    O, L = run_gpu(x, out_dtype)
    O_ref, L_ref = oracle.attention(x.q, x.k, x.v, x.scale, causal=x.causal, kv_len=x.kv_len)
    return compare(O, L, O_ref, L_ref, dtype, out_dtype, what)


def check_sampled(x, dtype, per_head=48, out_dtype=torch.float32, what="", seed=0):
    O, L = run_gpu(x, out_dtype)
    B, H, N, d = x.q.shape
    rows = sample_rows(B, H, N, x.kv_len, per_head=per_head, seed=seed)
    O_ref, L_ref = oracle.attention_rows(x.q, x.k, x.v, x.scale, rows, causal=x.causal, kv_len=x.kv_len)
    O_s = O.reshape(-1, d)[torch.as_tensor(rows, device=O.device)]
    L_s = L.reshape(-1)[torch.as_tensor(rows, device=L.device)]
    return compare(O_s, L_s, O_ref, L_ref, dtype, out_dtype, what)
