"""GPU backward (attn_bwd, through the C ABI) against the fp64 backward oracle on the same seeded inputs.

The parity cases give attn_bwd the oracle's O and LSE (fp64 rounded to fp32), so that the bar
measures the backward alone; the chained cases give it attn_fwd's own outputs, as a user would. The
benchmark's workload (B1 H16 N8192 d128, non-causal and causal) is checked on sampled dQ rows and
dK, dV key rows of two heads, each entry exact over all N in fp64.

Tolerance (derived from the arithmetic, not stated by the pages). The kernel rounds P and dS to
bf16 before its tensor-core products (fp32 accumulation). A value x rounded to bf16 moves by at most
half an ulp, ulp(x) = 2^(floor(log2 |x|) - 7), and, modelled as uniform, by a standard deviation of
ulp(x) / sqrt(12). The errors of different terms are independent, so each gradient entry has a
rounding standard deviation
    sigma(dV_jc)^2 = sum_i ulp(P_ij)^2 / 12 dO_ic^2,
    sigma(dK_jc)^2 = scale^2 sum_i ulp(dS_ij)^2 / 12 Q_ic^2,
    sigma(dQ_ic)^2 = scale^2 sum_j ulp(dS_ij)^2 / 12 K_jc^2
(sums over the query heads of a group for dK, dV), computed from the oracle's P and dS. The bar is
|error| <= 6 sigma + F + 2^-23 |ref| per entry and mean |error| <= 1.25 mean sigma + mean F per
tensor (a sum of independent zero-mean errors has mean |e| = sqrt(2/pi) sigma = 0.8 sigma). An fp64
emulation of that rounding (bf16 P and dS, fp32 products) on peaky N = 1024 and 2048 heads stays
below 4.8 sigma + F per entry and at 0.75-0.85 of the mean bar's sigma term, so the bar has margin
and a kernel whose rounding error doubled would fail the mean check.
F is the floor for gradients that cancel to (near) zero: dS = P (dP - D) subtracts two fp32 sums,
dP_ij = dO_i . V_j and D_i = dO_i . O_i, and where they cancel (a single key: P = 1, O = V, D = dP)
only their rounding is left. The rounding of dP_ij is at most gamma A_ij with A_ij = |dO_i| . |V_j|
and gamma = 2^-16 (twice the worst case (n - 1) u of a 128-term fp32 sum); that of D_i at most
gamma_D B_i with B_i = |dO_i| . (P |V|)_i, gamma_D = 2^-16 when O is the oracle's and 2^-10 when O
comes from attn_fwd (whose fp16 P rounds each term of O by up to 2^-11 relative). Roundings of
different terms add in quadrature; the D error of one row is shared by all keys of that row and adds
linearly into dQ_i. When LSE comes from attn_fwd, its deviation from the oracle's, dL_i, scales row
i of P by e^(-dL_i): the chained cases add that first-order change, sum_i |dL_i| P_ij |dO_i| for dV
and likewise for dK and dQ through dS.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_50_b300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu

K_SIGMA = 6.0        # elementwise bar, in standard deviations of the rounding model
MEAN_FACTOR = 1.25   # mean |error| against the mean standard deviation
GAMMA = 2.0 ** -16


def ulp_bf16(a):
    a = np.abs(a)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 7).astype(np.int64)), 0.0)


def _upstream(x, seed):
    B, H, N, d = x.q.shape
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)


def _np64(t):
    return t.double().numpy()


def _bars_full(x, dO, P, O, scale, gamma_d, dL=None):
    """Per-entry allowances (F + chained-LSE term) and rounding sigmas of dQ, dK, dV for whole
    tensors, from the oracle's P [B,H,N,N] and O."""
    B, H, N, d = x.q.shape
    H_kv = x.k.shape[1]
    g = H // H_kv
    q, k, v, do = _np64(x.q), _np64(x.k), _np64(x.v), _np64(dO)
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    D = np.einsum("bhic,bhic->bhi", do, O)
    dS = P * (np.einsum("bhic,bhjc->bhij", do, vr) - D[..., None])
    uP2, udS2 = ulp_bf16(P) ** 2 / 12, ulp_bf16(dS) ** 2 / 12
    sig_v = np.sqrt(np.einsum("bhij,bhic->bhjc", uP2, do ** 2).reshape(B, H_kv, g, N, d).sum(2))
    sig_k = scale * np.sqrt(np.einsum("bhij,bhic->bhjc", udS2, q ** 2).reshape(B, H_kv, g, N, d).sum(2))
    sig_q = scale * np.sqrt(np.einsum("bhij,bhjc->bhic", udS2, kr ** 2))
    # cancellation floor F
    dOa, Va = np.abs(do), np.abs(vr)
    A = np.einsum("bhic,bhjc->bhij", dOa, Va)
    Bv = np.einsum("bhic,bhic->bhi", dOa, np.einsum("bhij,bhjc->bhic", P, Va))
    kmax = np.abs(kr).max(-1)[:, :, None, :]
    qmax = np.abs(q).max(-1)[..., None]
    fq = scale * (GAMMA * np.sqrt(((P * A * kmax) ** 2).sum(-1)) + gamma_d * Bv * (P * kmax).sum(-1))
    tk = P * (GAMMA * A + gamma_d * Bv[..., None]) * qmax
    fk = scale * np.sqrt((tk ** 2).sum(2).reshape(B, H_kv, g, N).sum(2))
    allow = [fq[..., None], fk[..., None], np.zeros((B, H_kv, N, 1))]
    if dL is not None:  # first-order change of P from the forward's LSE deviation
        w = np.abs(dL)[..., None] * P                                     # [B,H,i,j]
        allow[2] = allow[2] + np.einsum("bhij,bhic->bhjc", w, dOa).reshape(B, H_kv, g, N, d).sum(2)
        wdS = np.abs(dL)[..., None] * np.abs(dS)
        allow[1] = allow[1] + scale * np.einsum("bhij,bhic->bhjc", wdS, np.abs(q)).reshape(B, H_kv, g, N, d).sum(2)
        allow[0] = allow[0] + scale * np.einsum("bhij,bhjc->bhic", wdS, np.abs(kr))
    return allow, (sig_q, sig_k, sig_v)


def _run(x, seed=7, gpu_forward=False):
    from exact_tiled_attention_50_b300 import attn
    dO = _upstream(x, seed)
    lens = None if x.kv_len is None else x.kv_len.numpy()
    O64, L64, P = oracle.attention(x.q.float().numpy(), x.k.float().numpy(), x.v.float().numpy(), x.scale,
                                   causal=x.causal, kv_len=lens, return_p=True)
    q, k, v, do = x.q.cuda(), x.k.cuda(), x.v.cuda(), dO.cuda()
    kv = x.kv_len.cuda() if x.kv_len is not None else None
    dL = None
    if gpu_forward:
        O, L = attn.attn_fwd(q, k, v, scale=x.scale, causal=x.causal, kv_len=kv)
        Lg = L.double().cpu().numpy()
        fin = np.isfinite(L64)
        dL = np.where(fin, Lg - np.where(fin, L64, 0.0), 0.0)
    else:
        O = torch.from_numpy(O64.astype(np.float32)).cuda()
        L = torch.from_numpy(L64.astype(np.float32)).cuda()
    dq, dk, dv = attn.attn_bwd(q, k, v, O, do, L, scale=x.scale, causal=x.causal, kv_len=kv)
    rc = attn.check()
    assert rc == attn.ATTN_OK, f"{attn.status_string(rc)} bits {attn.lib.attn_debug_last_error_bits():#x}"
    ref = oracle.attention_bwd_np(_np64(x.q), _np64(x.k), _np64(x.v), _np64(dO), x.scale, causal=x.causal,
                                  kv_len=lens)
    allow, sig = _bars_full(x, dO, P, O64, x.scale, gamma_d=2.0 ** -10 if gpu_forward else GAMMA, dL=dL)
    got = tuple(t.double().cpu().numpy() for t in (dq, dk, dv))
    return got, ref, allow, sig


def _check(got, ref, allow, sig, what):
    stats = {}
    for name, a, r, f, s in zip(("dQ", "dK", "dV"), got, ref, allow, sig):
        assert np.isfinite(a).all(), f"{what} {name}: non-finite"
        e = np.abs(a - r)
        f = np.broadcast_to(f, e.shape)
        bar = K_SIGMA * s + f + 2.0 ** -23 * np.abs(r)
        worst = np.unravel_index(int(np.argmax(e - bar)), e.shape)
        assert np.all(e <= bar), f"{what} {name}: err {e[worst]:.3g} at {worst} > bar {bar[worst]:.3g} " \
            f"(sigma {s[worst]:.3g}, floor {f[worst]:.3g}, max|ref| {float(np.abs(r).max()):.3g})"
        mean_bar = MEAN_FACTOR * float(s.mean()) + float(f.mean())
        assert float(e.mean()) <= mean_bar, f"{what} {name}: mean err {float(e.mean()):.3g} > {mean_bar:.3g}"
        stats[name] = (float(np.max((e - f) / np.maximum(s, 1e-300))), float(e.mean()) / max(float(s.mean()), 1e-300))
    return stats


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
    got, ref, allow, sig = _run(x)
    _check(got, ref, allow, sig, "kv_len [0, 131], GQA 4")
    for t in got:
        assert np.count_nonzero(t[0]) == 0


def test_bwd_longer_sequence():
    x = inputs.custom(1, 2, 2, 2048, 128, causal=True, peaky=True, seed=71)
    _check(*_run(x), "N=2048 causal")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_after_gpu_forward(d):
    x = inputs.custom(2, 4, 2, 384, d, causal=True, padded=True, peaky=True, seed=81 + d)
    _check(*_run(x, gpu_forward=True), f"chained d={d}")


# ---------------------------------------------------------------- the benchmark's workload, sampled
def _bars_sampled(r, q, k, v, do, scale, rows, keys):
    """Allowances and sigmas at the sampled rows (dQ) and keys (dK, dV) of one head (H_kv = H)."""
    Pr, dSr = r["P_rows"], r["dS_rows"]             # [R, N]
    Pk, dSk = r["P_keys"][0], r["dS_keys"][0]       # [N, C]
    sig_q = scale * np.sqrt((ulp_bf16(dSr) ** 2 / 12) @ (k ** 2))
    sig_k = scale * np.sqrt((ulp_bf16(dSk) ** 2 / 12).T @ (q ** 2))
    sig_v = np.sqrt((ulp_bf16(Pk) ** 2 / 12).T @ (do ** 2))
    dOa, Va = np.abs(do), np.abs(v)
    kmax = np.abs(k).max(-1)[None, :]
    qmax = np.abs(q).max(-1)[:, None]
    A_r = dOa[rows] @ Va.T
    B_r = np.sum(dOa[rows] * (Pr @ Va), axis=1)
    fq = scale * (GAMMA * np.sqrt(((Pr * A_r * kmax) ** 2).sum(-1)) + GAMMA * B_r * (Pr * kmax).sum(-1))
    A_k = dOa @ Va[keys].T
    B_all = dOa @ Va.max(axis=0)                      # >= |dO_i| . (P |V|)_i for every row
    tk = Pk * (GAMMA * A_k + GAMMA * B_all[:, None]) * qmax
    fk = scale * np.sqrt((tk ** 2).sum(0))
    return [fq[:, None], fk[:, None], 0.0], (sig_q, sig_k, sig_v)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_bench_workload_sampled(causal):
    """B1 H16 N8192 d128 with 1% of key rows x8 and the benchmark's seeded upstream gradient: the
    kernel runs on all 16 heads; heads 0 and 11 are checked at 48 query rows (dQ) and 48 key rows
    (dK, dV) each, tile edges and the last rows included, every entry exact over all 8192 keys or
    query rows. Those two heads get the oracle's O and LSE, the others attn_fwd's."""
    from exact_tiled_attention_50_b300 import attn
    tag = "causal" if causal else "noncausal"
    x = inputs.make_inputs(inputs.WORKLOADS[f"sweep_b1h16_d128_n8192_{tag}_peaky"])
    B, H, N, d = x.q.shape
    g = torch.Generator().manual_seed(inputs.SEED_BASE + 5000)  # the benchmark's upstream gradient
    dO = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16)
    q, k, v, do = x.q.cuda(), x.k.cuda(), x.v.cuda(), dO.cuda()
    O, L = attn.attn_fwd(q, k, v, scale=x.scale, causal=causal)
    q64, k64, v64, do64 = _np64(x.q), _np64(x.k), _np64(x.v), _np64(dO)
    rows = parity.sample_rows(1, 1, N, per_head=48, seed=3)
    keys = parity.sample_rows(1, 1, N, per_head=48, seed=4)
    heads = (0, 11)
    refs = {}
    for h in heads:
        r = oracle.attention_bwd_sampled_np(q64, k64, v64, do64, x.scale, 0, h, rows, keys, causal=causal)
        O[0, h] = torch.from_numpy(r["O"][0].astype(np.float32)).cuda()
        L[0, h] = torch.from_numpy(r["LSE"][0].astype(np.float32)).cuda()
        refs[h] = r
    dq, dk, dv = attn.attn_bwd(q, k, v, O, do, L, scale=x.scale, causal=causal)
    rc = attn.check()
    assert rc == attn.ATTN_OK, f"{attn.status_string(rc)} bits {attn.lib.attn_debug_last_error_bits():#x}"
    for h in heads:
        r = refs[h]
        got = (dq[0, h, torch.as_tensor(rows)].double().cpu().numpy(),
               dk[0, h, torch.as_tensor(keys)].double().cpu().numpy(),
               dv[0, h, torch.as_tensor(keys)].double().cpu().numpy())
        allow, sig = _bars_sampled(r, q64[0, h], k64[0, h], v64[0, h], do64[0, h], x.scale, rows, keys)
        _check(got, (r["dq"], r["dk"], r["dv"]), allow, sig, f"N=8192 {tag} head {h}")
