"""Pins for an attention oracle: checks that do not rely on the oracle's own formula.

Each check takes ``attn(q, k, v, scale, causal, kv_len) -> (O, LSE)`` (fp64 NumPy outputs) and raises
AssertionError on a mismatch. They are run against both oracles, and against copies of the NumPy
oracle with a planted mistake (which must fail at least one check).

What pins what:
 - golden closed-form cases (tests/golden/closed_form_cases.txt): rational softmax weights, masks,
   grouped heads, the empty row;
 - identical keys => O is the mean of the valid V rows (closed form), per mask;
 - a dominant score => O equals that key's V row and LSE equals that score;
 - one key (N = 1) and causal row 0 => O = V_0, LSE = s_00;
 - special cases that reduce to library routines: torch's fp64 scaled_dot_product_attention (no mask,
   causal, and key padding as truncation of K/V), scipy's logsumexp for the LSE;
 - grouped heads equal the same computation with K/V replicated per query head;
 - a scalar brute-force per-(i, j) loop with math.exp for tiny inputs (mask semantics).
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_form_cases.txt")


def _eval(expr: str):
    return eval(expr, {"math": math, "None": None})  # fixture values are plain math expressions


def load_golden():
    cases, cur = [], {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.rstrip("\n")
            if line.startswith("#"):
                continue
            if not line.strip():
                if cur:
                    cases.append(cur)
                    cur = {}
                continue
            key, val = line.split(":", 1)
            cur[key.strip()] = val.strip()
    if cur:
        cases.append(cur)
    out = []
    for c in cases:
        out.append(dict(
            name=c["name"], scale=float(_eval(c["scale"])), causal=bool(int(c["causal"])),
            kv_len=_eval(c["kv_len"]),
            q=np.array(_eval(c["q"]), np.float64), k=np.array(_eval(c["k"]), np.float64),
            v=np.array(_eval(c["v"]), np.float64), O=np.array(_eval(c["O"]), np.float64),
            LSE=np.array(_eval(c["LSE"]), np.float64)))
    return out


def _rng(seed):
    return np.random.default_rng(seed)


def _f32n(rng, shape):
    # standard normal values rounded to fp32, so both oracles (fp32 input arrays) see them exactly
    return rng.standard_normal(shape).astype(np.float32).astype(np.float64)


def _bf16_like(rng, shape):
    # small-integer-over-power-of-two values, exactly representable in fp32 and bf16
    return rng.integers(-64, 65, size=shape).astype(np.float64) / 32.0


def check_golden(attn):
    for c in load_golden():
        O, LSE = attn(c["q"], c["k"], c["v"], c["scale"], c["causal"], c["kv_len"])
        np.testing.assert_allclose(O, c["O"], rtol=0, atol=1e-12, err_msg=c["name"])
        fin = np.isfinite(c["LSE"])
        assert np.array_equal(np.isfinite(LSE), fin), c["name"]
        np.testing.assert_allclose(LSE[fin], c["LSE"][fin], rtol=0, atol=1e-12, err_msg=c["name"])
        assert np.all(LSE[~fin] == -np.inf), c["name"]


def check_identical_keys(attn):
    rng = _rng(1)
    B, H, N, d = 2, 2, 9, 4
    q = _bf16_like(rng, (B, H, N, d))
    krow = _bf16_like(rng, (d,))
    k = np.broadcast_to(krow, (B, H, N, d)).copy()
    v = _bf16_like(rng, (B, H, N, d))
    for causal in (False, True):
        for kv_len in (None, [5, 9]):
            O, _ = attn(q, k, v, 0.37, causal, kv_len)
            for b in range(B):
                L = N if kv_len is None else kv_len[b]
                for i in range(N):
                    hi = min(L, i + 1) if causal else L
                    np.testing.assert_allclose(O[b, :, i], v[b, :, :hi].mean(axis=1), rtol=0, atol=1e-12)


def check_dominant(attn):
    rng = _rng(2)
    N, d = 11, 8
    q = np.zeros((1, 1, N, d))
    q[..., 0] = 1.0
    k = _bf16_like(rng, (1, 1, N, d)) / 128.0
    j0 = 6
    k[0, 0, j0, :] = 0.0
    k[0, 0, j0, 0] = 2000.0  # score 2000*scale, others ~0: weight of the rest ~ exp(-2000*scale)
    v = _bf16_like(rng, (1, 1, N, d))
    scale = 0.5
    O, LSE = attn(q, k, v, scale, False, None)
    for i in range(N):
        np.testing.assert_allclose(O[0, 0, i], v[0, 0, j0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(LSE[0, 0, i], 2000.0 * scale, rtol=0, atol=1e-9)


def check_single_key_and_causal_row0(attn):
    rng = _rng(3)
    d = 5
    q = _bf16_like(rng, (1, 2, 1, d))
    k = _bf16_like(rng, (1, 2, 1, d))
    v = _bf16_like(rng, (1, 2, 1, d))
    O, LSE = attn(q, k, v, 0.25, False, None)
    np.testing.assert_allclose(O[0, :, 0], v[0, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(LSE[0, :, 0], 0.25 * np.sum(q[0, :, 0] * k[0, :, 0], axis=-1), rtol=0, atol=1e-14)
    N = 7
    q = _bf16_like(rng, (1, 1, N, d))
    k = _bf16_like(rng, (1, 1, N, d))
    v = _bf16_like(rng, (1, 1, N, d))
    O, LSE = attn(q, k, v, 0.25, True, None)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(LSE[0, 0, 0], 0.25 * float(q[0, 0, 0] @ k[0, 0, 0]), rtol=0, atol=1e-14)


def check_library(attn):
    import torch
    import torch.nn.functional as F
    from scipy.special import logsumexp

    rng = _rng(4)
    B, H, N, d = 2, 3, 13, 8
    q = _f32n(rng, (B, H, N, d))
    k = _f32n(rng, (B, H, N, d))
    v = _f32n(rng, (B, H, N, d))
    scale = 1 / math.sqrt(d)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    for causal in (False, True):
        O, LSE = attn(q, k, v, scale, causal, None)
        ref = F.scaled_dot_product_attention(T(q), T(k), T(v), is_causal=causal, scale=scale).numpy()
        np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)
        S = scale * np.einsum("bhid,bhjd->bhij", q, k)
        if causal:
            S = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)
        np.testing.assert_allclose(LSE, logsumexp(S, axis=-1), rtol=0, atol=1e-12)
    # key padding == attention over the truncated key set
    lens = [4, 13]
    O, LSE = attn(q, k, v, scale, False, lens)
    for b, L in enumerate(lens):
        ref = F.scaled_dot_product_attention(T(q[b]), T(k[b, :, :L]), T(v[b, :, :L]), scale=scale).numpy()
        np.testing.assert_allclose(O[b], ref, rtol=0, atol=1e-12)
        S = scale * np.einsum("hid,hjd->hij", q[b], k[b, :, :L])
        np.testing.assert_allclose(LSE[b], logsumexp(S, axis=-1), rtol=0, atol=1e-12)


def check_gqa_replication(attn):
    rng = _rng(5)
    B, H, H_kv, N, d = 2, 6, 2, 10, 4
    q = _f32n(rng, (B, H, N, d))
    k = _f32n(rng, (B, H_kv, N, d))
    v = _f32n(rng, (B, H_kv, N, d))
    g = H // H_kv
    kr = np.repeat(k, g, axis=1)  # query head h reads kv head h // g
    vr = np.repeat(v, g, axis=1)
    for causal in (False, True):
        O1, L1 = attn(q, k, v, 0.3, causal, [7, 10])
        O2, L2 = attn(q, kr, vr, 0.3, causal, [7, 10])
        np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(L1, L2, rtol=0, atol=1e-13)


def brute_force(q, k, v, scale, causal, kv_len):
    """Scalar loops over (b, h, i, j) with math.exp; tiny inputs only."""
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    O = np.zeros((B, H, N, d))
    LSE = np.full((B, H, N), -np.inf)
    for b in range(B):
        L = N if kv_len is None else kv_len[b]
        for h in range(H):
            kh = h // (H // H_kv)
            for i in range(N):
                keys = [j for j in range(N) if j < L and (not causal or j <= i)]
                if not keys:
                    continue
                s = {j: scale * sum(q[b, h, i, c] * k[b, kh, j, c] for c in range(d)) for j in keys}
                mx = max(s.values())
                w = {j: math.exp(s[j] - mx) for j in keys}
                tot = sum(w.values())
                for c in range(d):
                    O[b, h, i, c] = sum(w[j] * v[b, kh, j, c] for j in keys) / tot
                LSE[b, h, i] = mx + math.log(tot)
    return O, LSE


def check_brute_force(attn):
    rng = _rng(6)
    B, H, H_kv, N, d = 2, 4, 2, 6, 3
    q = _f32n(rng, (B, H, N, d))
    k = _f32n(rng, (B, H_kv, N, d))
    v = _f32n(rng, (B, H_kv, N, d))
    for causal in (False, True):
        for lens in (None, [3, 6], [1, 0]):
            O, LSE = attn(q, k, v, 0.7, causal, lens)
            Ob, Lb = brute_force(q, k, v, 0.7, causal, lens)
            np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
            assert np.array_equal(np.isfinite(LSE), np.isfinite(Lb))
            fin = np.isfinite(Lb)
            np.testing.assert_allclose(LSE[fin], Lb[fin], rtol=0, atol=1e-12)


ALL_PINS = [check_golden, check_identical_keys, check_dominant, check_single_key_and_causal_row0,
            check_library, check_gqa_replication, check_brute_force]


def failing_pins(attn):
    """Names of the pins that ``attn`` fails (empty list = all pass)."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(attn)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            bad.append(f"{pin.__name__}: {type(e).__name__}")
    return bad
