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


def _head_stats_np(qh, kh, vh, scale, mask, block=512):
    """O [N, d] and LSE [N] of one head, exact in fp64, computed over blocks of query rows (the same
    definition as attention_np, without holding the N x N matrix at once)."""
    N, d = qh.shape
    O = np.zeros((N, d))
    LSE = np.full(N, -np.inf)
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        S = float(scale) * (qh[r0:r1] @ kh.T)
        S = np.where(mask[r0:r1], S, -np.inf)
        m = S.max(axis=1)
        has = np.isfinite(m)
        m_safe = np.where(has, m, 0.0)
        E = np.exp(S - m_safe[:, None])
        l = E.sum(axis=1)
        O[r0:r1] = np.where(has[:, None], (E @ vh) / np.where(has, l, 1.0)[:, None], 0.0)
        with np.errstate(divide="ignore"):
            LSE[r0:r1] = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    return O, LSE


def attention_bwd_sampled_np(q, k, v, dO, scale, b, h, rows, keys, causal=False, kv_len=None):
    """The gradients of attention_bwd_np at selected positions, exact in fp64, for sequences too long
    for the whole N x N matrices: dQ[b, h, rows] of query head h, and dK[b, kh, keys], dV[b, kh, keys]
    of the key/value head kh = h / (H / H_kv) that head reads (summed over every query head of its
    group, as in attention_bwd_np). Each entry is the same chain rule, evaluated over all N keys or
    all N query rows:
        P_ij = exp(S_ij - LSE_i) (0 where masked),  D_i = sum_c dO_ic O_ic,
        dS_ij = P_ij (dO_i . V_j - D_i),
        dQ_i = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i,  dV_j = sum_i P_ij dO_i,
    with O and LSE of every query row from the exact forward (computed in blocks of rows).
    Returns a dict with dq [len(rows), d], dk and dv [len(keys), d], and O [g, N, d], LSE [g, N] of
    the group's query heads (h's own at index h mod g), P_rows [len(rows), N] and P_keys
    [g, N, len(keys)] (the probabilities used) and dS_rows / dS_keys likewise.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    dO = np.asarray(dO)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    g = H // H_kv
    kh = h // g
    rows = np.asarray(rows, dtype=np.int64)
    keys = np.asarray(keys, dtype=np.int64)
    L = N if kv_len is None else int(kv_len[b])
    mask = key_mask(N, causal, L)
    K = np.asarray(k[b, kh], dtype=np.float64)
    V = np.asarray(v[b, kh], dtype=np.float64)
    out = dict(dk=np.zeros((len(keys), d)), dv=np.zeros((len(keys), d)), O=np.zeros((g, N, d)),
               LSE=np.zeros((g, N)), P_keys=np.zeros((g, N, len(keys))), dS_keys=np.zeros((g, N, len(keys))))
    for t in range(g):
        hq = kh * g + t
        Q = np.asarray(q[b, hq], dtype=np.float64)
        G = np.asarray(dO[b, hq], dtype=np.float64)
        O, LSE = _head_stats_np(Q, K, V, scale, mask)
        D = np.sum(G * O, axis=1)
        has = np.isfinite(LSE)
        lse_safe = np.where(has, LSE, 0.0)
        out["O"][t], out["LSE"][t] = O, LSE
        # columns `keys` of P and dS over every query row
        Sk = float(scale) * (Q @ K[keys].T)
        Pk = np.where(mask[:, keys] & has[:, None], np.exp(np.where(mask[:, keys], Sk, 0.0) - lse_safe[:, None]), 0.0)
        dSk = Pk * (G @ V[keys].T - D[:, None])
        out["dv"] += Pk.T @ G
        out["dk"] += float(scale) * (dSk.T @ Q)
        out["P_keys"][t], out["dS_keys"][t] = Pk, dSk
        if hq == h:
            # rows `rows` of P and dS over every key
            Sr = float(scale) * (Q[rows] @ K.T)
            mr = mask[rows] & has[rows][:, None]
            Pr = np.where(mr, np.exp(np.where(mask[rows], Sr, 0.0) - lse_safe[rows][:, None]), 0.0)
            dSr = Pr * (G[rows] @ V.T - D[rows][:, None])
            out["dq"] = float(scale) * (dSr @ K)
            out["P_rows"], out["dS_rows"] = Pr, dSr
    return out


# ------------------------------------------------------------------------------------------------
# fp8 forward with incoherent processing (section "闪电注意力-3" of "闪电注意力：革命性地提高Transformer
# 效率", unite.ai: FP8 computation, and a processing step that lowers the quantisation error of the
# low-precision format). The pages name the two steps without defining them; the reading taken here:
#   1. rotate Q and K by the same orthogonal matrix, (1/sqrt d) H_d diag(s), H_d the Sylvester
#      Hadamard matrix and s a caller-supplied vector of random signs; Q K^T is unchanged, and an
#      outlier channel is spread over all d channels before rounding;
#   2. round Q, K and V to the 8-bit floating-point format E4M3 with one power-of-two scale per tile
#      of 128 rows;
#   3. exact attention over the rounded values.
# The rotation is applied unnormalised (H_d diag(s)); the factor 1/d of the two rotations moves into
# the softmax scale. Rounding decisions are taken in fp32, the precision in which the rotated values
# exist, with the butterflies in the order of the fast transform below.
# ------------------------------------------------------------------------------------------------
E4M3_MAX = 448.0
FP8_TILE_ROWS = 128


def e4m3_round(x):
    """Nearest value of the E4M3 format (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
    subnormals below 2^-6 with spacing 2^-9; largest finite 448; no infinities), ties to even, values
    beyond the largest finite one clamped to +-448. Returns fp64 values on that grid."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))       # a = f * 2^ex, f in [0.5, 1): binade 2^(ex - 1)
    e = np.clip(ex - 1, -6, 8)                        # normal binades 2^-6 .. 2^8; below: subnormal spacing
    step = np.ldexp(1.0, (e - 3).astype(np.int64))    # 3 mantissa bits
    r = np.round(a / step) * step                     # numpy rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(x < 0, -r, r)


def fwht_f32(x):
    """Unnormalised Walsh-Hadamard transform (Sylvester order) along the last axis, in fp32: spans
    h = 1, 2, 4, ...; for each pair (i, i + h) with bit h of i clear, (x_i, x_i+h) <- (x_i + x_i+h,
    x_i - x_i+h), every output one rounded fp32 addition or subtraction."""
    y = np.array(x, dtype=np.float32, copy=True)
    n = y.shape[-1]
    assert n & (n - 1) == 0
    lead = y.shape[:-1]
    h = 1
    while h < n:
        z = y.reshape(*lead, n // (2 * h), 2, h)
        a = z[..., 0, :].copy()
        b = z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        y = z.reshape(*lead, n)
        h *= 2
    return y


def tile_exponent(x32):
    """Power-of-two scale 2^e of one tile (any shape, fp32): with e8 the biased fp32 exponent field of
    the tile's largest |x| (so that max |x| < 2^(e8 - 126)), e = max(e8 - 134, -100): the tile's values
    times 2^-e stay below 2^8 = 256, inside the E4M3 range. An all-zero tile gets e = 0."""
    m = np.float32(np.max(np.abs(np.asarray(x32, dtype=np.float32)))) if np.size(x32) else np.float32(0)
    if m == 0:
        return 0
    e8 = int((np.array(m, dtype=np.float32).view(np.uint32) >> 23) & 0xFF)
    return max(e8 - 134, -100)


def quantize_e4m3_tiles(x32, rows=FP8_TILE_ROWS):
    """x [..., N, d] fp32 -> (dequantised values fp64, exponents [..., ceil(N / rows)]): each tile of
    `rows` rows is rounded as e4m3_round(x * 2^-e) and stands for that times 2^e."""
    x32 = np.asarray(x32, dtype=np.float32)
    N = x32.shape[-2]
    nt = (N + rows - 1) // rows
    lead = x32.shape[:-2]
    out = np.zeros(x32.shape, np.float64)
    ex = np.zeros(lead + (nt,), np.int64)
    for idx in np.ndindex(*lead):
        for t in range(nt):
            tile = x32[idx][t * rows:(t + 1) * rows]
            e = tile_exponent(tile)
            ex[idx + (t,)] = e
            out[idx][t * rows:(t + 1) * rows] = e4m3_round(tile.astype(np.float64) * 2.0 ** -e) * 2.0 ** e
    return out, ex


def attention_fp8_np(q, k, v, scale, signs=None, causal=False, kv_len=None, return_p=False):
    """Attention over E4M3-rounded inputs after the optional rotation (steps 1-3 above), fp64.

    q [B,H,N,d], k/v [B,H_kv,N,d] (their values read as fp32), signs: None (no rotation) or d values
    +-1. Returns O, LSE (and P), computed by the exact definition of ``attention_np`` on the rounded
    values, plus a dict with the rounded tensors and the tile exponents."""
    q32 = np.asarray(q, dtype=np.float32)
    k32 = np.asarray(k, dtype=np.float32)
    v32 = np.asarray(v, dtype=np.float32)
    d = q32.shape[-1]
    sc = float(scale)
    if signs is not None:
        s = np.asarray(signs, dtype=np.float32).reshape(d)
        assert np.all(np.abs(s) == 1)
        q32 = fwht_f32(q32 * s)
        k32 = fwht_f32(k32 * s)
        sc = sc / d
    qd, eq = quantize_e4m3_tiles(q32)
    kd, ek = quantize_e4m3_tiles(k32)
    vd, ev = quantize_e4m3_tiles(v32)
    res = attention_np(qd, kd, vd, sc, causal=causal, kv_len=kv_len, return_p=return_p)
    parts = dict(q=qd, k=kd, v=vd, eq=eq, ek=ek, ev=ev, scale=sc)
    return (*res, parts)


# ------------------------------------------------------------------------------------------------
# Additive bias and dropout (the xFormers call of the EfficientAttention module on "AI训练的最大障碍
# 不是算力,而是'内存墙'" (zsdodo.com): memory-efficient attention with attn_bias and a dropout
# probability p). Reading taken: the bias is added to the scaled scores, the softmax is taken over
# them (LSE likewise, without dropout), and every probability is kept with probability 1 - p and
# then divided by that keep probability (inverted dropout) before P V.
# The keep decisions come from the counter-based generator Philox4x32-10 of Salmon, Moraes, Dror and
# Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011), so that any tiling reproduces them:
#   counter (j >> 3, i, b * H + h, offset), key (seed mod 2^32, seed >> 32) for query row i and key j;
#   the four 32-bit output words give eight 16-bit values u_0..u_7 (word w: low half u_2w, high half
#   u_2w+1); key j takes u_(j mod 8) and is dropped iff u < t, t = floor(p * 65536). The effective
#   drop probability is t / 65536 and kept values are scaled by 65536 / (65536 - t).
# ------------------------------------------------------------------------------------------------
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57        # round multipliers
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85        # key increments (Weyl sequence)
_U32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds on arrays of counters ([..., 4] uint32) and keys ([..., 2] uint32).
    One round: (hi0, lo0) = M0 * x0, (hi1, lo1) = M1 * x2 (64-bit products split into 32-bit halves),
    x <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0); the key advances by (W0, W1) after every round."""
    x = [np.asarray(ctr[..., i], dtype=np.uint64) & _U32 for i in range(4)]
    k0 = np.asarray(key[..., 0], dtype=np.uint64) & _U32
    k1 = np.asarray(key[..., 1], dtype=np.uint64) & _U32
    for _ in range(10):
        p0 = np.uint64(PHILOX_M0) * x[0]
        p1 = np.uint64(PHILOX_M1) * x[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _U32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _U32
        x = [hi1 ^ x[1] ^ k0, lo1, hi0 ^ x[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(PHILOX_W0)) & _U32
        k1 = (k1 + np.uint64(PHILOX_W1)) & _U32
    return np.stack([a.astype(np.uint32) for a in x], axis=-1)


def dropout_threshold(p):
    """t = floor(p * 65536) for 0 <= p < 1 (p read as the fp32 value the C ABI receives)."""
    p = float(np.float32(p))
    assert 0.0 <= p < 1.0
    return int(np.floor(p * 65536.0))


def dropout_keep_mask(B, H, N, p, seed, offset):
    """Boolean [B, H, N, N]: True where probability (b, h, i, j) is kept (see the section text)."""
    t = dropout_threshold(p)
    G = (N + 7) // 8
    g, i, bh = np.meshgrid(np.arange(G), np.arange(N), np.arange(B * H), indexing="ij")
    ctr = np.stack([g, i, bh, np.full_like(g, int(offset) & 0xFFFFFFFF)], axis=-1).astype(np.uint64)
    key = np.broadcast_to(np.array([int(seed) & 0xFFFFFFFF, (int(seed) >> 32) & 0xFFFFFFFF], np.uint64),
                          ctr.shape[:-1] + (2,))
    w = philox4x32_10(ctr, key).astype(np.uint32)                      # [G, N, BH, 4]
    u = np.stack([w & 0xFFFF, w >> 16], axis=-1).reshape(G, N, B * H, 8)  # u_(2w), u_(2w+1)
    keep = u >= t                                                      # [G, N, BH, 8]
    keep = np.transpose(keep, (2, 1, 0, 3)).reshape(B * H, N, G * 8)[:, :, :N]
    return keep.reshape(B, H, N, N)


def attention_bias_dropout_np(q, k, v, scale, bias=None, p=0.0, seed=0, offset=0, causal=False, kv_len=None,
                              return_p=False):
    """O, LSE of the biased, dropped-out attention (fp64). bias: None or an array broadcastable to
    [B, H, N, N] (natural-log units, added to scale * Q K^T). LSE is that of the biased scores."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    g = H // H_kv
    bias_full = np.zeros((B, H, N, N)) if bias is None else np.broadcast_to(np.asarray(bias, dtype=np.float64),
                                                                              (B, H, N, N))
    t = dropout_threshold(p)
    keep = dropout_keep_mask(B, H, N, p, seed, offset) if t > 0 else np.ones((B, H, N, N), bool)
    inv_keep = 65536.0 / (65536.0 - t)
    O = np.zeros((B, H, N, d))
    LSE = np.zeros((B, H, N))
    P_all = np.zeros((B, H, N, N)) if return_p else None
    for b in range(B):
        L = N if kv_len is None else int(kv_len[b])
        mask = key_mask(N, causal, L)
        for h in range(H):
            S = float(scale) * (q[b, h] @ k[b, h // g].T) + bias_full[b, h]
            S = np.where(mask, S, -np.inf)
            m = S.max(axis=1)
            has = np.isfinite(m)
            m_safe = np.where(has, m, 0.0)
            E = np.exp(S - m_safe[:, None])
            l = E.sum(axis=1)
            P = np.where(has[:, None], E / np.where(has, l, 1.0)[:, None], 0.0)
            O[b, h] = (P * keep[b, h] * inv_keep) @ v[b, h // g]
            with np.errstate(divide="ignore"):
                LSE[b, h] = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
            if return_p:
                P_all[b, h] = P
    if return_p:
        return O, LSE, P_all
    return O, LSE


def attention_bias_dropout_rows_np(q, k, v, scale, b, h, rows, bias_rows=None, p=0.0, seed=0, offset=0,
                                   causal=False, kv_len=None):
    """O [len(rows), d], LSE [len(rows)] of attention_bias_dropout_np for the query rows `rows` of head
    (b, h) alone, each row over all N keys: the same definition restricted to those rows, for sizes whose
    full [B, H, N, N] scores and mask do not fit on the host. bias_rows: None or the rows' biases
    [len(rows), N] (natural-log units). The keep decisions of row i come from the same Philox4x32-10
    counters (j >> 3, i, b * H + h, offset) as dropout_keep_mask."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, N, d = q.shape
    kvh = h // (H // k.shape[1])
    L = N if kv_len is None else int(kv_len[b])
    t = dropout_threshold(p)
    inv_keep = 65536.0 / (65536.0 - t)
    G = (N + 7) // 8
    key = np.array([int(seed) & 0xFFFFFFFF, (int(seed) >> 32) & 0xFFFFFFFF], np.uint64)
    O = np.zeros((len(rows), d))
    LSE = np.zeros(len(rows))
    for n, i in enumerate(rows):
        s = float(scale) * (k[b, kvh] @ q[b, h, i])
        if bias_rows is not None:
            s = s + np.asarray(bias_rows[n], dtype=np.float64)
        jk = np.arange(N)  # row i of key_mask: keys below kv_len (and, causal, not after the query)
        s = np.where((jk < max(0, min(L, N))) & ((jk <= i) if causal else True), s, -np.inf)
        m = s.max()
        if not np.isfinite(m):
            O[n] = 0.0
            LSE[n] = -np.inf
            continue
        e = np.exp(s - m)
        l = e.sum()
        if t > 0:
            ctr = np.stack([np.arange(G), np.full(G, i), np.full(G, b * H + h), np.full(G, int(offset) & 0xFFFFFFFF)],
                           axis=-1).astype(np.uint64)
            w = philox4x32_10(ctr, np.broadcast_to(key, (G, 2))).astype(np.uint32)    # [G, 4]
            u = np.stack([w & 0xFFFF, w >> 16], axis=-1).reshape(G * 8)[:N]          # u_(j mod 8) of group j >> 3
            keep = u >= t
        else:
            keep = np.ones(N, bool)
        O[n] = ((e / l) * keep * inv_keep) @ v[b, kvh]
        LSE[n] = m + np.log(l)
    return O, LSE
