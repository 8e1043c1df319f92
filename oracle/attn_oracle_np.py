"""NumPy fp64 restatement of the attention forward: a second, independent oracle for small cases.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``). It is written with whole-matrix NumPy
operations, unlike the C oracle's scalar loops, so that a slip in one restatement shows up as a
disagreement with the other.

Definition followed (the standard_attention listings on "AI训练的最大障碍不是算力,而是'内存墙'"
(zsdodo.com) and "闪电注意力：革命性地提高Transformer效率" (unite.ai); the max-subtracted softmax of
formula 1 in the latter's section "闪电注意力的数学原理"; padded keys ignored as in
"基于AIFI多头注意力机制的高效序列建模实战", "动态序列处理"; grouped heads as in the unite.ai section
"闪电注意力-2"):

    S = scale * Q K^T over the key axis, masked entries set to -inf,
    P = softmax(S) row-wise with the row maximum subtracted,
    O = P V,  LSE = m + ln(sum exp(S - m)).
"""
from __future__ import annotations

import numpy as np


def key_mask(N: int, causal: bool, kv_len: int) -> np.ndarray:
    """Boolean [N, N] matrix: True where query i may attend to key j."""
    j = np.arange(N)[None, :]
    i = np.arange(N)[:, None]
    ok = j < max(0, min(int(kv_len), N))
    if causal:
        ok = ok & (j <= i)
    return np.broadcast_to(ok, (N, N))


def attention_np(q, k, v, scale, causal=False, kv_len=None, return_p=False):
    """q [B,H,N,d], k/v [B,H_kv,N,d] (any float dtype, upcast to fp64). Returns O, LSE (and P)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    assert H % H_kv == 0
    g = H // H_kv
    O = np.zeros((B, H, N, d))
    LSE = np.zeros((B, H, N))
    P_all = np.zeros((B, H, N, N)) if return_p else None
    for b in range(B):
        L = N if kv_len is None else int(kv_len[b])
        mask = key_mask(N, causal, L)
        for h in range(H):
            kh = h // g
            S = float(scale) * (q[b, h] @ k[b, kh].T)
            S = np.where(mask, S, -np.inf)
            m = S.max(axis=1)
            has = np.isfinite(m)
            m_safe = np.where(has, m, 0.0)
            E = np.exp(S - m_safe[:, None])  # exp(-inf) = 0 on masked entries
            l = E.sum(axis=1)
            P = np.where(has[:, None], E / np.where(has, l, 1.0)[:, None], 0.0)
            O[b, h] = P @ v[b, kh]
            with np.errstate(divide="ignore"):
                LSE[b, h] = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
            if return_p:
                P_all[b, h] = P
    if return_p:
        return O, LSE, P_all
    return O, LSE


def merge_np(O_parts, LSE_parts):
    """Combine attention results computed over disjoint key sets (fp64).

    O_parts [P, ..., d] (each part normalised over its own keys), LSE_parts [P, ...] (natural log).
    Softmax merge rule, formula 2 of "闪电注意力的数学原理" on "闪电注意力：革命性地提高Transformer效率"
    (unite.ai), in its corrected form: with m = max_i LSE_i, the union's log-sum-exp is
    m + ln(sum_i exp(LSE_i - m)) and its output is sum_i exp(LSE_i - LSE) O_i. Parts whose LSE is -inf
    (no valid key) get weight 0; if every part is -inf the row is O = 0, LSE = -inf.
    """
    O_parts = np.asarray(O_parts, dtype=np.float64)
    L = np.asarray(LSE_parts, dtype=np.float64)
    m = L.max(axis=0)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    w = np.where(np.isfinite(L), np.exp(L - m_safe[None]), 0.0)
    s = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(has, m_safe + np.log(np.where(has, s, 1.0)), -np.inf)
        wn = np.where(has[None], w / np.where(has, s, 1.0)[None], 0.0)
    O = (wn[..., None] * O_parts).sum(axis=0)
    return O, lse


def attention_bwd_np(q, k, v, dO, scale, causal=False, kv_len=None):
    """Gradients of the attention output with respect to Q, K and V (fp64).

    The pages give the forward only; the backward of the same exact attention is the chain rule
    through it, in the recompute form the pages motivate (the score matrix is not stored; P is
    rebuilt from the row log-sum-exp): with P = softmax(S), S = scale Q K^T (masked), O = P V,
        dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic,   dS = P * (dP - D),
        dQ = scale dS K,   dK = scale dS^T Q.
    Grouped heads: dK and dV of a key/value head sum over the query heads that read it. Rows without
    valid keys contribute nothing. Returns dQ [B,H,N,d], dK [B,H_kv,N,d], dV [B,H_kv,N,d].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    g = H // H_kv
    _, _, P = attention_np(q, k, v, scale, causal=causal, kv_len=kv_len, return_p=True)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            kh = h // g
            Pm = P[b, h]
            O = Pm @ v[b, kh]
            dV[b, kh] += Pm.T @ dO[b, h]
            dP = dO[b, h] @ v[b, kh].T
            D = np.sum(dO[b, h] * O, axis=1)
            dS = Pm * (dP - D[:, None])
            dQ[b, h] = float(scale) * (dS @ k[b, kh])
            dK[b, kh] += float(scale) * (dS.T @ q[b, h])
    return dQ, dK, dV
