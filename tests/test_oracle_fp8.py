"""The fp8 oracle steps against what fixes them (CPU only): the E4M3 format by brute force over its
codes and by torch's own E4M3 cast (library special case), the fast Walsh-Hadamard transform by
scipy's Hadamard matrix, the tile exponent by its closed form, the rotation by exactness of the
rotated attention without rounding, the rounding error by the format's spacing, the purpose of the
rotation (a smaller error on inputs with outlier channels), and planted mistakes."""
import inspect

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from oracle import attn_oracle_np
from exact_tiled_attention_50_b300 import inputs


def _all_e4m3_values():
    """Every finite E4M3 value from the format's definition: sign, 4-bit exponent (bias 7), 3-bit
    mantissa; exponent field 0 is subnormal (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN."""
    vals = set()
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            vals.add(v)
            vals.add(-v)
    return np.array(sorted(vals))


def test_e4m3_grid_from_the_format_definition():
    grid = _all_e4m3_values()
    assert grid.max() == 448.0 and grid[grid > 0].min() == 2.0 ** -9
    assert len(grid[grid > 0]) == 126  # 7 subnormals + 14 binades x 8 + 7 in the last binade
    np.testing.assert_array_equal(oracle.e4m3_round(grid), grid)  # representable values are fixed points
    # every other value goes to a nearest grid point (brute force), ties to the even mantissa
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-1, 1, 20000) * 2.0 ** -5,
                        (grid[1:] + grid[:-1]) / 2])  # midpoints: the ties
    r = oracle.e4m3_round(x)
    dist = np.abs(x[:, None] - grid[None, :])
    best = dist.min(axis=1)
    np.testing.assert_array_equal(np.abs(x - r), best)
    # at a tie the chosen value has an even code: an even mantissa field (for 0: +-0)
    ties = (grid[1:] + grid[:-1]) / 2
    rt = oracle.e4m3_round(ties)
    a = np.abs(rt)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.clip(ex - 1, -6, 8)
    code = np.round(a / np.ldexp(1.0, e - 3)).astype(np.int64)
    assert np.all((code % 2 == 0) | (a == 0))


def test_e4m3_matches_torch_cast():
    """torch's float8_e4m3fn conversion (round to nearest even) agrees wherever it is finite."""
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-464, 464, 200000), rng.standard_normal(100000) * 0.01,
                        (rng.integers(-2 ** 15, 2 ** 15, 50000) / 2 ** 12)]).astype(np.float32)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = np.isfinite(t)
    assert ok.mean() > 0.99
    np.testing.assert_array_equal(oracle.e4m3_round(x.astype(np.float64))[ok], t[ok])


def test_e4m3_saturates():
    np.testing.assert_array_equal(oracle.e4m3_round([464.0, 480.0, 1e6, -1e30]), [448.0, 448.0, 448.0, -448.0])


@pytest.mark.parametrize("n", [2, 8, 64, 128])
def test_fwht_is_the_hadamard_matrix(n):
    rng = np.random.default_rng(n)
    x = rng.standard_normal((5, n)).astype(np.float32)
    Hm = scipy.linalg.hadamard(n).astype(np.float64)
    ref = x.astype(np.float64) @ Hm.T
    got = oracle.fwht_f32(x).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.log2(n) * 2.0 ** -23 * np.abs(x).sum(-1, keepdims=True))
    # twice the transform is n times the identity (H H^T = n I)
    np.testing.assert_allclose(oracle.fwht_f32(oracle.fwht_f32(x.astype(np.float64))), n * x, rtol=1e-5, atol=1e-4)


def test_fwht_exact_on_small_integers():
    x = np.arange(8, dtype=np.float32)
    np.testing.assert_array_equal(oracle.fwht_f32(x), scipy.linalg.hadamard(8) @ np.arange(8))


def test_tile_exponent_closed_form():
    rng = np.random.default_rng(3)
    for _ in range(200):
        t = (rng.standard_normal((128, 16)) * 2.0 ** rng.integers(-30, 30)).astype(np.float32)
        e = oracle.tile_exponent(t)
        m = float(np.abs(t).max()) * 2.0 ** -e
        assert 128.0 <= m < 256.0
    assert oracle.tile_exponent(np.zeros((4, 4), np.float32)) == 0
    assert oracle.tile_exponent(np.full((2, 2), 2.0 ** -140, np.float32)) == -100  # clamped


def test_quantisation_error_within_the_format_spacing():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((2, 300, 64)) * np.exp(rng.standard_normal((2, 300, 1)))).astype(np.float32)
    deq, ex = oracle.quantize_e4m3_tiles(x)
    assert ex.shape == (2, 3)
    for b in range(2):
        for t in range(3):
            xt = x[b, 128 * t:128 * (t + 1)].astype(np.float64)
            dt = deq[b, 128 * t:128 * (t + 1)]
            e = ex[b, t]
            # relative 2^-4 in the normal range, absolute 2^-10 * 2^e below it
            assert np.all(np.abs(dt - xt) <= np.maximum(2.0 ** -4 * np.abs(xt), 2.0 ** (e - 10)) + 1e-300)


def _without_rounding(monkeypatch):
    monkeypatch.setattr(attn_oracle_np, "e4m3_round", lambda x: np.asarray(x, dtype=np.float64))


@pytest.mark.parametrize("causal", [False, True])
def test_rotation_leaves_attention_unchanged_without_rounding(monkeypatch, causal):
    """With the rounding step removed, the rotated path is the exact attention: the same rotation on
    Q and K and the factor 1/d in the scale (fp32 transform: close to fp32 accuracy)."""
    _without_rounding(monkeypatch)
    x = inputs.custom(2, 4, 2, 200, 128, causal=causal, kv_len=[150, 200], seed=9)
    s = inputs.random_signs(128, seed=1).numpy()
    q, k, v = (t.float().numpy() for t in (x.q, x.k, x.v))
    O, L = oracle.attention(q, k, v, x.scale, causal=causal, kv_len=[150, 200])
    Or, Lr, _ = oracle.attention_fp8_np(q, k, v, x.scale, signs=s, causal=causal, kv_len=[150, 200])
    np.testing.assert_allclose(Or, O, rtol=0, atol=2e-5)
    np.testing.assert_allclose(Lr, L, rtol=0, atol=2e-5)
    On, Ln, _ = oracle.attention_fp8_np(q, k, v, x.scale, signs=None, causal=causal, kv_len=[150, 200])
    np.testing.assert_allclose(On, O, rtol=0, atol=1e-12)


def test_rotation_reduces_the_error_on_outlier_channels():
    """The purpose the pages give the processing step: a smaller quantisation error. Inputs with four
    x16 channels in Q and K: the rotated path's error against the exact attention is several times
    smaller; on inputs without outliers both are alike."""
    s = inputs.random_signs(128, seed=2).numpy()
    for outl, lo, hi in ((True, 2.5, None), (False, 0.7, 1.4)):
        x = inputs.custom(1, 2, 2, 384, 128, seed=11)
        if outl:
            x = inputs.with_outlier_channels(x, seed=1)
        q, k, v = (t.float().numpy() for t in (x.q, x.k, x.v))
        O, _ = oracle.attention(q, k, v, x.scale)
        Or, _, _ = oracle.attention_fp8_np(q, k, v, x.scale, signs=s)
        On, _, _ = oracle.attention_fp8_np(q, k, v, x.scale, signs=None)
        ratio = np.sqrt(np.mean((On - O) ** 2)) / np.sqrt(np.mean((Or - O) ** 2))
        assert ratio >= lo and (hi is None or ratio <= hi), ratio


# Planted mistakes in a copy of the oracle's source: each must fail one of the checks below.
FP8_MUTANTS = {
    "rotate_q_only": ("k32 = fwht_f32(k32 * s)", "k32 = k32 * s"),
    "scale_not_divided": ("sc = sc / d", "sc = sc"),
    "exponent_off_by_one": ("max(e8 - 134, -100)", "max(e8 - 133, -100)"),
    "round_half_up": ("r = np.round(a / step) * step", "r = np.floor(a / step + 0.5) * step"),
    "no_subnormals": ("e = np.clip(ex - 1, -6, 8)", "e = np.clip(ex - 1, -9, 8)"),
    "v_unquantised": ("vd, ev = quantize_e4m3_tiles(v32)", "vd, ev = v32.astype(np.float64), 0"),
    "signs_ignored": ("q32 = fwht_f32(q32 * s)", "q32 = fwht_f32(q32)"),
}


def _mutant_module(old, new):
    src = inspect.getsource(attn_oracle_np)
    assert old in src, old
    ns = {}
    exec(compile(src.replace(old, new), "<fp8-mutant>", "exec"), ns)
    return ns


def _fp8_checks_fail(ns):
    """True if one of the checks above (rerun against the mutant) fails."""
    try:
        grid = _all_e4m3_values()
        np.testing.assert_array_equal(ns["e4m3_round"](grid), grid)
        rng = np.random.default_rng(2)
        x = np.concatenate([rng.uniform(-464, 464, 20000), (rng.integers(-2 ** 15, 2 ** 15, 5000) / 2 ** 12),
                            rng.standard_normal(5000) * 0.003]).astype(np.float32)
        t = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        ok = np.isfinite(t)
        np.testing.assert_array_equal(ns["e4m3_round"](x.astype(np.float64))[ok], t[ok])
        t2 = (rng.standard_normal((128, 16)) * 3).astype(np.float32)
        m = float(np.abs(t2).max()) * 2.0 ** -ns["tile_exponent"](t2)
        assert 128.0 <= m < 256.0
        # the rotated, rounded path stays close to the exact attention on plain inputs (fp8-size error)
        x = inputs.custom(1, 2, 2, 256, 128, seed=12)
        q, k, v = (a.float().numpy() for a in (x.q, x.k, x.v))
        s = inputs.random_signs(128, seed=3).numpy()
        O, _ = oracle.attention(q, k, v, x.scale)
        Or, _, parts = ns["attention_fp8_np"](q, k, v, x.scale, signs=s)
        assert np.sqrt(np.mean((Or - O) ** 2)) < 0.01
        # the signs matter: the rotated q differs from the unsigned transform
        q_rot = parts["q"]
        q_plain, _ = ns["quantize_e4m3_tiles"](ns["fwht_f32"](q))
        assert not np.allclose(q_rot, q_plain)
        # V is rounded: every dequantised V value sits on its tile's E4M3 grid
        vt = parts["v"][0, 0, :128] * 2.0 ** -int(np.asarray(parts["ev"]).reshape(-1)[0])
        np.testing.assert_array_equal(oracle.e4m3_round(vt), vt)
        assert not np.array_equal(parts["v"], v.astype(np.float64))
    except AssertionError:
        return True
    return False


def test_unmutated_fp8_oracle_passes_the_checks():
    assert not _fp8_checks_fail(_mutant_module("import numpy as np", "import numpy as np"))


@pytest.mark.parametrize("name", list(FP8_MUTANTS))
def test_planted_fp8_mistake_is_caught(name):
    assert _fp8_checks_fail(_mutant_module(*FP8_MUTANTS[name])), name
