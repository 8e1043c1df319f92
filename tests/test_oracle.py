"""The oracle against its pins (CPU only): closed forms, invariants, library special cases, brute
force, the tiled recurrence against the full definition, the two oracles against each other, and
planted mistakes that the pins must catch."""
import math

import numpy as np
import pytest

import oracle
from oracle import attn_oracle_np
from tests import oracle_pins as pins


def c_attn(q, k, v, scale, causal, kv_len):
    return oracle.attention(q, k, v, scale, causal=causal, kv_len=kv_len)


def np_attn(q, k, v, scale, causal, kv_len):
    return oracle.attention_np(q, k, v, scale, causal=causal, kv_len=kv_len)


def tiled_attn(q, k, v, scale, causal, kv_len):
    return oracle.attention_tiled(q, k, v, scale, causal=causal, kv_len=kv_len, Br=2, Bc=3)


def rows_attn(q, k, v, scale, causal, kv_len):
    B, H, N, d = np.shape(q)
    O, L = oracle.attention_rows(q, k, v, scale, np.arange(B * H * N), causal=causal, kv_len=kv_len)
    return O.reshape(B, H, N, d), L.reshape(B, H, N)


ORACLES = {"c_full": c_attn, "numpy": np_attn, "c_tiled": tiled_attn, "c_rows": rows_attn}


@pytest.mark.parametrize("name", list(ORACLES))
@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pins(name, pin):
    pin(ORACLES[name])


def test_rows_of_p_sum_to_one():
    rng = np.random.default_rng(11)
    B, H, H_kv, N, d = 2, 4, 2, 33, 16
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = rng.standard_normal((B, H_kv, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H_kv, N, d)).astype(np.float32)
    for causal in (False, True):
        O, LSE, P = oracle.attention(q, k, v, 0.25, causal=causal, kv_len=[17, 33], return_p=True)
        np.testing.assert_allclose(P.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert np.all(P >= 0)
        assert np.all(P[0, :, :, 17:] == 0)  # padded keys get no weight
        if causal:
            assert np.all(np.triu(P[1], k=1) == 0)
        # O is P times V (reconstructed from the returned probabilities)
        g = H // H_kv
        np.testing.assert_allclose(O, np.einsum("bhij,bhjd->bhid", P, np.repeat(v, g, 1).astype(np.float64)),
                                   rtol=0, atol=1e-12)
        # exp(LSE) is the sum of exponentiated valid scores (recomputed from the definition)
        s = 0.25 * np.einsum("bhid,bhjd->bhij", q.astype(np.float64), np.repeat(k, g, 1).astype(np.float64))
        valid = P > 0
        np.testing.assert_allclose(np.exp(LSE), np.where(valid, np.exp(s), 0).sum(-1), rtol=1e-12, atol=0)


@pytest.mark.parametrize("N", [1, 7, 64, 130])
@pytest.mark.parametrize("blocks", [(16, 16), (32, 16), (16, 32)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_recurrence_equals_full(N, blocks, causal):
    rng = np.random.default_rng(N)
    B, H, H_kv, d = 2, 4, 2, 16
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = (rng.standard_normal((B, H_kv, N, d)) * np.where(rng.random((B, H_kv, N, 1)) < 0.1, 8, 1)).astype(np.float32)
    v = rng.standard_normal((B, H_kv, N, d)).astype(np.float32)
    lens = [max(1, N // 2), N]
    O1, L1 = oracle.attention(q, k, v, 0.25, causal=causal, kv_len=lens)
    O2, L2 = oracle.attention_tiled(q, k, v, 0.25, causal=causal, kv_len=lens, Br=blocks[0], Bc=blocks[1])
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_c_oracle_equals_numpy_oracle(causal):
    rng = np.random.default_rng(12)
    B, H, H_kv, N, d = 2, 8, 2, 150, 64
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = rng.standard_normal((B, H_kv, N, d)).astype(np.float32)
    v = rng.standard_normal((B, H_kv, N, d)).astype(np.float32)
    lens = [77, 150]
    O1, L1 = oracle.attention(q, k, v, 0.125, causal=causal, kv_len=lens)
    O2, L2 = oracle.attention_np(q, k, v, 0.125, causal=causal, kv_len=lens)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-12)


def test_rows_oracle_equals_full_on_workload_shape():
    from exact_tiled_attention_50_b300 import inputs
    x = inputs.custom(2, 4, 1, 300, 128, causal=True, padded=True, peaky=True, seed=3)
    O, L = oracle.attention(x.q, x.k, x.v, x.scale, causal=True, kv_len=x.kv_len)
    rows = np.array([0, 1, 127, 128, 299, 300 + 5, 3 * 300 + 299, 7 * 300 + 150])
    Or, Lr = oracle.attention_rows(x.q, x.k, x.v, x.scale, rows, causal=True, kv_len=x.kv_len)
    np.testing.assert_array_equal(Or, O.reshape(-1, 128)[rows])
    np.testing.assert_array_equal(Lr, L.reshape(-1)[rows])


# Planted mistakes: each edit to the NumPy oracle's source must make at least one pin fail.
MUTANTS = {
    "no_scale": ("S = float(scale) * (q[b, h] @ k[b, kh].T)", "S = (q[b, h] @ k[b, kh].T)"),
    "gqa_modulo": ("kh = h // g", "kh = h % H_kv"),
    "causal_strict": ("ok = ok & (j <= i)", "ok = ok & (j < i)"),
    "causal_transposed": ("ok = ok & (j <= i)", "ok = ok & (j >= i)"),
    "padding_off_by_one": ("ok = j < max(0, min(int(kv_len), N))", "ok = j <= max(0, min(int(kv_len), N))"),
    "lse_without_max": ("m_safe + np.log(", "np.log("),
    "p_transposed": ("O[b, h] = P @ v[b, kh]", "O[b, h] = P.T @ v[b, kh]"),
    "sum_wrong_axis": ("l = E.sum(axis=1)", "l = E.sum(axis=0)"),
    "scores_transposed": ("(q[b, h] @ k[b, kh].T)", "(k[b, kh] @ q[b, h].T)"),
    "v_from_k": ("O[b, h] = P @ v[b, kh]", "O[b, h] = P @ k[b, kh]"),
    "exp_sign": ("E = np.exp(S - m_safe[:, None])", "E = np.exp(m_safe[:, None] - S)"),
}


def _mutant(src_old, src_new):
    import inspect
    src = inspect.getsource(attn_oracle_np)
    assert src_old in src, src_old
    ns = {}
    exec(compile(src.replace(src_old, src_new), "<mutant>", "exec"), ns)
    return lambda q, k, v, scale, causal, kv_len: ns["attention_np"](q, k, v, scale, causal=causal, kv_len=kv_len)


def test_unmutated_copy_passes_every_pin():
    m = _mutant("import numpy as np", "import numpy as np")
    assert pins.failing_pins(m) == []


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = _mutant(*MUTANTS[name])
    assert pins.failing_pins(m), f"no pin caught the planted mistake {name}"


# ---------------------------------------------------------------- merge over disjoint key sets
def _split_parts(q, k, v, scale, L):
    """Attention over keys [0, L) and over keys [L, N) with the C oracle: the second set is made the
    first N - L keys by rotating K and V (attention without a causal mask does not depend on the
    order of the keys)."""
    N = q.shape[2]
    B = q.shape[0]
    A = oracle.attention(q, k, v, scale, kv_len=[L] * B)
    kr, vr = np.roll(k, -L, axis=2), np.roll(v, -L, axis=2)
    Bp = oracle.attention(q, kr, vr, scale, kv_len=[N - L] * B)
    return A, Bp


@pytest.mark.parametrize("L", [0, 1, 37, 64, 99, 100])
def test_merge_of_split_keys_equals_full_attention(L):
    rng = np.random.default_rng(40 + L)
    B, H, H_kv, N, d = 2, 4, 2, 100, 16
    q = rng.standard_normal((B, H, N, d)).astype(np.float32)
    k = (rng.standard_normal((B, H_kv, N, d)) * np.where(rng.random((B, H_kv, N, 1)) < 0.1, 8, 1)).astype(np.float32)
    v = rng.standard_normal((B, H_kv, N, d)).astype(np.float32)
    O_full, L_full = oracle.attention(q, k, v, 0.25)
    (OA, LA), (OB, LB) = _split_parts(q, k, v, 0.25, L)
    O, LSE = oracle.merge_np(np.stack([OA, OB]), np.stack([LA, LB]))
    np.testing.assert_allclose(O, O_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, L_full, rtol=0, atol=1e-12)


def test_merge_special_cases():
    rng = np.random.default_rng(7)
    O1 = rng.standard_normal((3, 5, 8))
    L1 = rng.standard_normal((3, 5))
    O, L = oracle.merge_np(O1[None], L1[None])  # one part: unchanged
    np.testing.assert_allclose(O, O1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L, L1, rtol=0, atol=1e-15)
    empty = np.full_like(L1, -np.inf)  # a part without keys contributes nothing
    O, L = oracle.merge_np(np.stack([O1, np.zeros_like(O1)]), np.stack([L1, empty]))
    np.testing.assert_allclose(O, O1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(L, L1, rtol=0, atol=1e-15)
    O, L = oracle.merge_np(np.stack([O1, O1]), np.stack([empty, empty]))  # no keys anywhere
    assert np.all(O == 0) and np.all(L == -np.inf)
    # two equal parts: same output, LSE + ln 2
    O, L = oracle.merge_np(np.stack([O1, O1]), np.stack([L1, L1]))
    np.testing.assert_allclose(O, O1, rtol=0, atol=1e-14)
    np.testing.assert_allclose(L, L1 + np.log(2.0), rtol=0, atol=1e-14)
