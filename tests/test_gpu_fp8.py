"""GPU fp8 path (attn_fwd_fp8, through the C ABI) against the fp8 oracle on the same seeded inputs.

The oracle takes the method's steps (rotation of Q and K by the random signs, E4M3 rounding per
128-row tile at a power-of-two scale, exact fp64 attention over the rounded values); its rounding
decisions are taken in fp32 in the kernel's butterfly order, so the rounded inputs are the same on
both sides. The kernel additionally rounds the probabilities P to E4M3 before P V. Bound (derived
from that rounding, not stated by the pages), per output element, with P the oracle's probabilities
and V~ its rounded V:
    |O - O_ref|_ic <= 2^-4 (P |V~|)_ic                           (relative 2^-4 of a normal E4M3 value)
                    + 2^-10 sum_j 2^(E_i - e_j) |V~_jc| / l_i     (E4M3 subnormals: absolute 2^-10)
                    + 1e-5 max|O_ref| + 1e-5                      (fp32 arithmetic)
where e_j is the exponent of key j's V tile, E_i the largest over the row's valid keys, and
l_i = sum_j exp(s_ij - max_j s_ij) >= 1. Mean |error| <= 0.1 of the mean bound (an emulation of the
rounding gives at most 0.04). LSE is computed from unrounded probabilities: |LSE - LSE_ref| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_50_b300 import inputs

pytestmark = pytest.mark.gpu


def _gpu(x, signs):
    from exact_tiled_attention_50_b300 import attn
    kv = x.kv_len.cuda() if x.kv_len is not None else None
    s = signs.cuda() if signs is not None else None
    O, L = attn.attn_fwd_fp8(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale, causal=x.causal, kv_len=kv,
                             signs=s)
    rc = attn.check()
    assert rc == attn.ATTN_OK, f"{attn.status_string(rc)} bits {attn.lib.attn_debug_last_error_bits():#x}"
    return O.double().cpu().numpy(), L.double().cpu().numpy()


def _bound(P, parts, O_ref, H, H_kv, N):
    g = H // H_kv
    vd = np.repeat(parts["v"], g, axis=1)
    evk = np.repeat(np.repeat(parts["ev"], g, axis=1), 128, axis=2)[:, :, :N]  # exponent per key
    valid = P > 0
    Emax = np.where(valid, evk[:, :, None, :], -(10 ** 9)).max(-1)
    pmax = P.max(-1)
    l_true = np.where(pmax > 0, 1.0 / np.where(pmax > 0, pmax, 1.0), 1.0)
    w = np.where(valid, 2.0 ** (np.minimum(Emax[..., None] - evk[:, :, None, :], 60)), 0.0)
    sub = 2.0 ** -10 * np.einsum("bhij,bhjc->bhic", w, np.abs(vd)) / l_true[..., None]
    rel = 2.0 ** -4 * np.einsum("bhij,bhjc->bhic", P, np.abs(vd))
    return rel + sub + 1e-5 * np.abs(O_ref).max() + 1e-5


def _check(x, signs, what):
    q, k, v = (t.float().numpy() for t in (x.q, x.k, x.v))
    lens = None if x.kv_len is None else x.kv_len.numpy()
    O_ref, L_ref, P, parts = oracle.attention_fp8_np(q, k, v, x.scale, signs=None if signs is None else signs.numpy(),
                                                     causal=x.causal, kv_len=lens, return_p=True)
    O, L = _gpu(x, signs)
    B, H, N, d = q.shape
    bnd = _bound(P, parts, O_ref, H, k.shape[1], N)
    e = np.abs(O - O_ref)
    assert np.isfinite(O).all(), what
    worst = np.unravel_index(int(np.argmax(e / bnd)), e.shape)
    assert np.all(e <= bnd), f"{what}: err {e[worst]:.3g} > bound {bnd[worst]:.3g} at {worst}"
    assert e.mean() <= 0.1 * bnd.mean(), f"{what}: mean err {e.mean():.3g} vs mean bound {bnd.mean():.3g}"
    fin = np.isfinite(L_ref)
    assert np.array_equal(fin, np.isfinite(L)), what
    assert np.abs(L[fin] - L_ref[fin]).max(initial=0.0) <= 1e-3, what
    return O, O_ref


@pytest.mark.parametrize("rotate", [True, False])
def test_fp8_matches_oracle(rotate):
    x = inputs.custom(2, 4, 2, 300, 128, peaky=True, seed=31)
    _check(x, inputs.random_signs(128, seed=1) if rotate else None, f"rotate={rotate}")


def test_fp8_causal_padded_gqa():
    x = inputs.custom(2, 8, 2, 384, 128, causal=True, padded=True, peaky=True, seed=32)
    _check(x, inputs.random_signs(128, seed=2), "causal padded GQA")


@pytest.mark.parametrize("N", [1, 129, 640])
def test_fp8_ragged_lengths(N):
    x = inputs.custom(1, 2, 1, N, 128, causal=True, seed=33 + N)
    _check(x, inputs.random_signs(128, seed=3), f"N={N}")


def test_fp8_key_padding_with_an_empty_batch():
    x = inputs.custom(2, 4, 1, 256, 128, kv_len=[0, 200], seed=34)
    O, _ = _check(x, inputs.random_signs(128, seed=4), "kv_len [0, 200]")
    assert np.all(O[0] == 0)


def test_fp8_stream_k_split_units():
    # enough work units per CTA that the persistent schedule splits some of them between CTAs
    x = inputs.custom(1, 24, 24, 1536, 128, seed=35)
    _check(x, inputs.random_signs(128, seed=5), "B1 H24 N1536")


def test_fp8_rotation_reduces_the_error_on_outlier_channels():
    """Incoherent processing does what the pages say it is for: against the exact attention of the
    unrounded inputs, the rotated fp8 result has a several times smaller error than the unrotated one
    on inputs with outlier channels."""
    x = inputs.with_outlier_channels(inputs.custom(1, 4, 2, 512, 128, seed=36), seed=2)
    q, k, v = (t.float().numpy() for t in (x.q, x.k, x.v))
    O_exact, _ = oracle.attention(q, k, v, x.scale)
    O_rot, _ = _gpu(x, inputs.random_signs(128, seed=6))
    O_plain, _ = _gpu(x, None)
    rm = lambda a: float(np.sqrt(np.mean((a - O_exact) ** 2)))  # noqa: E731
    assert rm(O_plain) >= 2.5 * rm(O_rot), (rm(O_plain), rm(O_rot))


def test_fp8_full_size_sampled_rows():
    """The bench's fp8 workload (B1 H16 N8192 d128, peaky keys), rows sampled across every head and
    tile (first, last, tile edges): each checked against the oracle's rows with the same bound."""
    x = inputs.make_inputs(inputs.WORKLOADS[inputs.HEADLINE])
    signs = inputs.random_signs(128, seed=0)
    B, H, N, d = x.q.shape
    O, L = _gpu(x, signs)
    q32 = oracle.fwht_f32(x.q.float().numpy() * signs.numpy().astype(np.float32))
    k32 = oracle.fwht_f32(x.k.float().numpy() * signs.numpy().astype(np.float32))
    qd, _ = oracle.quantize_e4m3_tiles(q32)
    kd, _ = oracle.quantize_e4m3_tiles(k32)
    vd, ev = oracle.quantize_e4m3_tiles(x.v.float().numpy())
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 12)]))
    for h in range(H):
        idx = h * N + rows
        Or, Lr = oracle.attention_rows(qd.astype(np.float32), kd.astype(np.float32), vd.astype(np.float32),
                                       x.scale / d, idx)
        s = (x.scale / d) * (qd[0, h, rows] @ kd[0, h].T)
        p = np.exp(s - s.max(-1, keepdims=True))
        l_true = p.sum(-1)
        P = p / l_true[:, None]
        evk = np.repeat(ev[0, h], 128)[:N]
        Emax = evk.max()
        bnd = (2.0 ** -4 * P @ np.abs(vd[0, h]) + 2.0 ** -10 * (2.0 ** (Emax - evk) @ np.abs(vd[0, h]))[None] /
               l_true[:, None] + 1e-5 * np.abs(Or).max() + 1e-5)
        e = np.abs(O[0, h, rows] - Or)
        assert np.all(e <= bnd), f"head {h}: worst {np.max(e / bnd):.3g} of the bound"
        assert np.abs(L[0, h, rows] - Lr).max() <= 1e-3, h
