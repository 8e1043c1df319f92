"""GPU backward (attn_bwd, through the C ABI) against the fp64 backward oracle on the same seeded inputs.

The parity cases give attn_bwd the oracle's O and LSE (fp64 rounded to fp32), so that the bar
measures the backward alone; one chained case gives it attn_fwd's own outputs, as a user would.

Tolerance (derived from the arithmetic, not stated by the pages): P and dS enter the tensor-core
products as bf16 (relative rounding 2^-9) with fp32 accumulation. Emulating exactly that rounding in
fp64 on these workloads gives max |error| up to 0.35% of the tensor's max |gradient|; the bar is
|error| <= 1e-2 * max |ref| + F elementwise and mean |error| <= 1e-3 * max |ref| + mean F for each of
dQ, dK, dV. F is the floor for gradients that cancel to (near) zero: dS = P (dP - D) subtracts two
fp32 sums, dP_ij = dO_i . V_j and D_i = dO_i . O_i, and where they cancel (a single key: P = 1,
O = V, D = dP) only their rounding is left. The rounding of dP_ij is at most gamma A_ij with
A_ij = |dO_i| . |V_j| and gamma = 2^-16 (twice the worst case (n - 1) u of a 128-term fp32 sum); that
of D_i at most gamma_D B_i with B_i = |dO_i| . (P |V|)_i, gamma_D = 2^-16 when O is the oracle's and
2^-10 when O comes from attn_fwd (whose fp16 P rounds each term of O by up to 2^-11 relative).
Roundings of different terms are independent and add in quadrature (the probabilistic rounding-error
model); the D error of one row is shared by all keys of that row and adds linearly into dQ_i.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_50_b300 import inputs

pytestmark = pytest.mark.gpu


def _upstream(x, seed):
    B, H, N, d = x.q.shape
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)


def _np64(t):
    return t.double().numpy()


def _run(x, seed=7, gpu_forward=False):
    from exact_tiled_attention_50_b300 import attn
    dO = _upstream(x, seed)
    lens = None if x.kv_len is None else x.kv_len.numpy()
    O64, L64, P = oracle.attention(x.q.float().numpy(), x.k.float().numpy(), x.v.float().numpy(), x.scale,
                                   causal=x.causal, kv_len=lens, return_p=True)
    q, k, v, do = x.q.cuda(), x.k.cuda(), x.v.cuda(), dO.cuda()
    kv = x.kv_len.cuda() if x.kv_len is not None else None
    if gpu_forward:
        O, L = attn.attn_fwd(q, k, v, scale=x.scale, causal=x.causal, kv_len=kv)
    else:
        O = torch.from_numpy(O64.astype(np.float32)).cuda()
        L = torch.from_numpy(L64.astype(np.float32)).cuda()
    dq, dk, dv = attn.attn_bwd(q, k, v, O, do, L, scale=x.scale, causal=x.causal, kv_len=kv)
    rc = attn.check()
    assert rc == attn.ATTN_OK, f"{attn.status_string(rc)} bits {attn.lib.attn_debug_last_error_bits():#x}"
    ref = oracle.attention_bwd_np(_np64(x.q), _np64(x.k), _np64(x.v), _np64(dO), x.scale, causal=x.causal,
                                  kv_len=lens)
    floors = _floors(x, dO, P, gamma_d=2.0 ** -10 if gpu_forward else 2.0 ** -16)
    return (dq, dk, dv), ref, floors


def _floors(x, dO, P, gamma_d, gamma=2.0 ** -16):
    """Elementwise allowance (dQ [B,H,N,1], dK [B,H_kv,N,1], dV 0) for the cancellation in
    dS = P (dP - D), as the module text derives it."""
    B, H, N, d = x.q.shape
    H_kv = x.k.shape[1]
    g = H // H_kv
    dOa = np.abs(_np64(dO))
    Va = np.repeat(np.abs(_np64(x.v)), g, axis=1)
    A = np.einsum("bhic,bhjc->bhij", dOa, Va)
    Bv = np.einsum("bhic,bhic->bhi", dOa, np.einsum("bhij,bhjc->bhic", P, Va))
    kmax = np.repeat(np.abs(_np64(x.k)).max(-1), g, axis=1)[:, :, None, :]  # [B, H, 1, N]
    qmax = np.abs(_np64(x.q)).max(-1)[..., None]                           # [B, H, N, 1]
    fq = x.scale * (gamma * np.sqrt(((P * A * kmax) ** 2).sum(-1)) + gamma_d * Bv * (P * kmax).sum(-1))
    tk = P * (gamma * A + gamma_d * Bv[..., None]) * qmax                  # [B, H, i, j]
    fk = x.scale * np.sqrt((tk ** 2).sum(2).reshape(B, H_kv, g, N).sum(2))
    return fq[..., None], fk[..., None], 0.0


def _check(got, ref, floors, what):
    for name, a, r, f in zip(("dQ", "dK", "dV"), got, ref, floors):
        a = a.double().cpu().numpy()
        assert np.isfinite(a).all(), f"{what} {name}: non-finite"
        top = float(np.abs(r).max())
        e = np.abs(a - r)
        bar = 1e-2 * top + np.broadcast_to(f, e.shape)
        worst = np.unravel_index(int(np.argmax(e - bar)), e.shape)
        assert np.all(e <= bar), f"{what} {name}: err {e[worst]:.3g} at {worst} > bar {bar[worst]:.3g} " \
            f"(max|ref| {top:.3g})"
        assert float(e.mean()) <= 1e-3 * top + float(np.mean(f)), f"{what} {name}: mean err {float(e.mean()):.3g}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_oracle(d, causal):
    x = inputs.custom(2, 4, 2, 300, d, causal=causal, peaky=True, seed=51 + d)
    _check(*_run(x), f"d={d} causal={causal}")


@pytest.mark.parametrize("N", [1, 127, 129, 513])
def test_bwd_ragged_lengths(N):
    x = inputs.custom(1, 2, 1, N, 128, causal=True, seed=N)
    _check(*_run(x), f"N={N}")


def test_bwd_key_padding_and_mqa():
    x = inputs.custom(2, 8, 1, 400, 128, causal=False, kv_len=[1, 257], seed=61)
    _check(*_run(x), "kv_len [1, 257], MQA")


def test_bwd_empty_key_set_and_gqa4():
    # batch 0 has no keys: its rows get no weight, every gradient there is exactly zero
    x = inputs.custom(2, 8, 2, 200, 64, causal=True, kv_len=[0, 131], seed=63)
    got, ref, floors = _run(x)
    _check(got, ref, floors, "kv_len [0, 131], GQA 4")
    for t in got:
        assert torch.count_nonzero(t[0]).item() == 0


def test_bwd_longer_sequence():
    x = inputs.custom(1, 2, 2, 2048, 128, causal=True, peaky=True, seed=71)
    _check(*_run(x), "N=2048 causal")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_after_gpu_forward(d):
    x = inputs.custom(2, 4, 2, 384, d, causal=True, padded=True, peaky=True, seed=81 + d)
    _check(*_run(x, gpu_forward=True), f"chained d={d}")
