"""The bias + dropout oracle against what fixes it (CPU only): the generator by its published
known-answer vectors, the drop rate by the binomial law, the bias by torch's fp64 softmax (library
special case), by the softmax's shift invariance and by its equivalence with key padding, dropout by
its expectation (the mean over many offsets tends to the undropped output) and by p = 0, and planted
mistakes in a copy of the oracle."""
import inspect
import math
import os

import numpy as np
import pytest
import torch

from oracle import attn_oracle_np as o
from exact_tiled_attention_50_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        c, k, y = (part.split() for part in line.split("|"))
        rows.append(([int(a, 16) for a in c], [int(a, 16) for a in k], [int(a, 16) for a in y]))
    return rows


def test_philox_known_answers():
    rows = _kat()
    assert len(rows) == 3
    for c, k, y in rows:
        got = o.philox4x32_10(np.array(c, np.uint64), np.array(k, np.uint64))
        assert [int(a) for a in got] == y


def _x(B=2, H=4, H_kv=2, N=150, d=64, causal=False, seed=0, kv_len=None):
    x = inputs.custom(B, H, H_kv, N, d, causal=causal, seed=seed, kv_len=kv_len)
    return x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(), x.scale


def test_drop_rate_is_binomial():
    B, H, N = 2, 4, 300
    for p in (0.1, 0.5, 0.03):
        keep = o.dropout_keep_mask(B, H, N, p, seed=12345, offset=7)
        n = keep.size
        q = o.dropout_threshold(p) / 65536.0
        dropped = n - int(keep.sum())
        assert abs(dropped - n * q) <= 5 * math.sqrt(n * q * (1 - q)), (p, dropped, n * q)
    assert o.dropout_threshold(0.1) == 6553 and o.dropout_threshold(0.0) == 0


def test_masks_differ_across_offsets_seeds_and_heads():
    a = o.dropout_keep_mask(1, 2, 200, 0.5, seed=1, offset=0)
    b = o.dropout_keep_mask(1, 2, 200, 0.5, seed=1, offset=1)
    c = o.dropout_keep_mask(1, 2, 200, 0.5, seed=2, offset=0)
    for other in (b, c):
        frac = np.mean(a != other)
        assert 0.45 < frac < 0.55  # independent masks at p = 0.5 differ in half the places
    assert 0.45 < np.mean(a[0, 0] != a[0, 1]) < 0.55
    np.testing.assert_array_equal(a, o.dropout_keep_mask(1, 2, 200, 0.5, seed=1, offset=0))


def test_mask_layout_as_documented():
    """The documented counter layout (j >> 3, i, b H + h, offset) and word split, for a few entries
    (a consistency check of the layout the C ABI documents, not of the generator)."""
    B, H, N, p, seed, off = 2, 3, 40, 0.3, (7 << 32) | 99, 5
    keep = o.dropout_keep_mask(B, H, N, p, seed, off)
    t = o.dropout_threshold(p)
    for (b, h, i, j) in [(0, 0, 0, 0), (1, 2, 39, 39), (0, 1, 17, 9), (1, 0, 3, 22)]:
        y = o.philox4x32_10(np.array([j >> 3, i, b * H + h, off], np.uint64), np.array([99, 7], np.uint64))
        u = [int(w) & 0xFFFF if s == 0 else int(w) >> 16 for w in y for s in (0, 1)][j & 7]
        assert keep[b, h, i, j] == (u >= t)


@pytest.mark.parametrize("causal", [False, True])
def test_bias_matches_torch_softmax(causal):
    q, k, v, scale = _x(causal=causal, seed=3)
    B, H, N, d = q.shape
    rng = np.random.default_rng(0)
    bias = rng.standard_normal((B, H, N, N)) * 2
    O, L = o.attention_bias_dropout_np(q, k, v, scale, bias=bias, causal=causal)
    kk = torch.from_numpy(np.repeat(k, 2, axis=1))
    vv = torch.from_numpy(np.repeat(v, 2, axis=1))
    S = scale * torch.from_numpy(q) @ kk.transpose(-1, -2) + torch.from_numpy(bias)
    if causal:
        S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(O, (torch.softmax(S, -1) @ vv).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, torch.logsumexp(S, -1).numpy(), rtol=0, atol=1e-12)


def test_bias_shift_and_padding_equivalences():
    q, k, v, scale = _x(seed=4, kv_len=[70, 150])
    B, H, N, d = q.shape
    O0, L0 = o.attention_np(q, k, v, scale, kv_len=[70, 150])
    Ob, Lb = o.attention_bias_dropout_np(q, k, v, scale, bias=None, kv_len=[70, 150])
    np.testing.assert_array_equal(Ob, O0)
    # a constant per row does not change the softmax: O unchanged, LSE shifted by it
    c = np.random.default_rng(1).standard_normal((B, H, N, 1)) * 5
    Oc, Lc = o.attention_bias_dropout_np(q, k, v, scale, bias=c, kv_len=[70, 150])
    np.testing.assert_allclose(Oc, O0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lc, L0 + c[..., 0], rtol=0, atol=1e-12)
    # -inf on the keys past kv_len is the key padding
    pad = np.zeros((B, 1, 1, N))
    pad[0, ..., 70:] = -np.inf
    Op, Lp = o.attention_bias_dropout_np(q, k, v, scale, bias=pad)
    np.testing.assert_allclose(Op, O0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lp, L0, rtol=0, atol=1e-12)


def _mean_over_offsets_ok(fn, q, k, v, scale, n, p=0.1):
    """Inverted dropout is unbiased: the mean of O over n independent masks lies within 5 sigma / sqrt(n)
    of the undropped O, elementwise, with sigma_ic^2 = (q / (1 - q)) sum_j P_ij^2 v_jc^2 (q the drop
    probability) the variance of one masked output; the normaliser (LSE) is untouched."""
    O0, L0, P = o.attention_np(q, k, v, scale, return_p=True)
    qd = o.dropout_threshold(p) / 65536.0
    g = q.shape[1] // k.shape[1]
    vv = np.repeat(v, g, axis=1)
    sigma = np.sqrt(qd / (1 - qd) * np.einsum("bhij,bhjc->bhic", P ** 2, vv ** 2))
    acc = np.zeros_like(O0)
    for off in range(n):
        Od, Ld = fn(q, k, v, scale, p=p, seed=11, offset=off)
        np.testing.assert_array_equal(Ld, L0)
        acc += Od
    assert np.all(np.abs(acc / n - O0) <= 5 * sigma / np.sqrt(n) + 1e-12)


def test_dropout_zero_and_expectation():
    q, k, v, scale = _x(B=1, H=2, H_kv=1, N=64, d=32, seed=5)
    O0, L0 = o.attention_np(q, k, v, scale)
    Oz, Lz = o.attention_bias_dropout_np(q, k, v, scale, p=0.0, seed=3)
    np.testing.assert_array_equal(Oz, O0)
    _mean_over_offsets_ok(o.attention_bias_dropout_np, q, k, v, scale, 400)


def test_dropout_applies_the_mask_to_probabilities():
    q, k, v, scale = _x(B=1, H=2, H_kv=2, N=50, d=16, seed=6)
    p = 0.25
    O, L, P = o.attention_bias_dropout_np(q, k, v, scale, p=p, seed=9, offset=2, return_p=True)
    keep = o.dropout_keep_mask(1, 2, 50, p, 9, 2)
    t = o.dropout_threshold(p)
    ref = torch.from_numpy(P * keep * (65536.0 / (65536 - t))) @ torch.from_numpy(v)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


MUTANTS = {
    "bias_before_scale": ("S = float(scale) * (q[b, h] @ k[b, h // g].T) + bias_full[b, h]",
                          "S = float(scale) * (q[b, h] @ k[b, h // g].T + bias_full[b, h])"),
    "no_inverse_keep": ("inv_keep = 65536.0 / (65536.0 - t)", "inv_keep = 1.0"),
    "keep_reversed": ("keep = u >= t  ", "keep = u < t  "),
    "philox_rotated_output": ("x = [hi1 ^ x[1] ^ k0, lo1, hi0 ^ x[3] ^ k1, lo0]",
                              "x = [hi0 ^ x[1] ^ k0, lo0, hi1 ^ x[3] ^ k1, lo1]"),
    "key_not_advanced": ("k0 = (k0 + np.uint64(PHILOX_W0)) & _U32", "k0 = k0"),
    "nine_rounds": ("for _ in range(10):", "for _ in range(9):"),
    "dropout_in_lse": ("l = E.sum(axis=1)", "l = (E * keep[b, h]).sum(axis=1)"),
}


def _mutant(old, new):
    src = inspect.getsource(o)
    assert old in src, old
    ns = {}
    exec(compile(src.replace(old, new), "<bias-dropout-mutant>", "exec"), ns)
    return ns


def _checks_fail(ns):
    try:
        for c, k, y in _kat():
            assert [int(a) for a in ns["philox4x32_10"](np.array(c, np.uint64), np.array(k, np.uint64))] == y
        keep = ns["dropout_keep_mask"](2, 4, 300, 0.1, 12345, 7)
        q_ = ns["dropout_threshold"](0.1) / 65536.0
        dropped = keep.size - int(keep.sum())
        assert abs(dropped - keep.size * q_) <= 5 * math.sqrt(keep.size * q_ * (1 - q_))
        q, k, v, scale = _x(B=1, H=2, H_kv=1, N=40, d=16, seed=7)
        bias = np.random.default_rng(2).standard_normal((1, 2, 40, 40))
        O, L = ns["attention_bias_dropout_np"](q, k, v, scale, bias=bias)
        kk = torch.from_numpy(np.repeat(k, 2, axis=1))
        S = scale * torch.from_numpy(q) @ kk.transpose(-1, -2) + torch.from_numpy(bias)
        np.testing.assert_allclose(L, torch.logsumexp(S, -1).numpy(), rtol=0, atol=1e-12)
        _mean_over_offsets_ok(ns["attention_bias_dropout_np"], q, k, v, scale, 200)
    except AssertionError:
        return True
    return False


def test_unmutated_copy_passes():
    assert not _checks_fail(_mutant("import numpy as np", "import numpy as np"))


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name):
    assert _checks_fail(_mutant(*MUTANTS[name])), name


@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, [37, 50])])
def test_row_restricted_oracle_equals_the_full_one(causal, kv_len):
    """attention_bias_dropout_rows_np (the full-size tests' per-row oracle) against the whole-matrix
    attention_bias_dropout_np: every row of every head, with a bias, dropout, GQA, causal and padding."""
    rng = np.random.default_rng(11)
    B, H, H_kv, N, d = 2, 4, 2, 50, 16
    q, k, v = rng.standard_normal((B, H, N, d)), rng.standard_normal((B, H_kv, N, d)), rng.standard_normal((B, H_kv, N, d))
    bias = rng.standard_normal((B, H, N, N)) * 2.0
    bias[0, 1, :, 5:9] = -np.inf
    lens = None if kv_len is None else np.array(kv_len)
    O, L = o.attention_bias_dropout_np(q, k, v, 0.3, bias=bias, p=0.3, seed=2 ** 33 + 9, offset=4, causal=causal,
                                       kv_len=lens)
    rows = np.arange(N)
    for b in range(B):
        for h in range(H):
            Or, Lr = o.attention_bias_dropout_rows_np(q, k, v, 0.3, b, h, rows, bias_rows=bias[b, h], p=0.3,
                                                      seed=2 ** 33 + 9, offset=4, causal=causal, kv_len=lens)
            np.testing.assert_allclose(Or, O[b, h], rtol=0, atol=1e-12)
            np.testing.assert_allclose(Lr, L[b, h], rtol=0, atol=1e-12)
