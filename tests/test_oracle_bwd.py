"""The backward oracle against its pins (CPU only): torch autograd in fp64 (a library routine), central
finite differences of the forward oracle (independent of the chain-rule formulas), and the softmax's
invariance to shifting every key by one vector (S changes by a per-row constant, so O and every
gradient but none of them depend on it)."""
import numpy as np
import pytest
import torch

import oracle


def _inputs(seed, B=2, H=4, H_kv=2, N=9, d=5):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H_kv, N, d)) * np.where(rng.random((B, H_kv, N, 1)) < 0.2, 3, 1)
    v = rng.standard_normal((B, H_kv, N, d))
    dO = rng.standard_normal((B, H, N, d))
    return q, k, v, dO


def _torch_grads(q, k, v, dO, scale, causal, kv_len):
    B, H, N, d = q.shape
    g = H // k.shape[1]
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    kr, vr = tk.repeat_interleave(g, dim=1), tv.repeat_interleave(g, dim=1)
    S = scale * tq @ kr.transpose(-1, -2)
    j = torch.arange(N)
    mask = torch.ones(B, 1, N, N, dtype=torch.bool)
    if kv_len is not None:
        mask = mask & (j[None, None, None, :] < torch.tensor(kv_len)[:, None, None, None])
    if causal:
        mask = mask & (j[None, :] <= j[:, None])
    S = S.masked_fill(~mask, float("-inf"))
    P = torch.softmax(S, dim=-1).nan_to_num(0.0)
    O = P @ vr
    O.backward(torch.tensor(dO))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kv_len", [None, [5, 9], [0, 3]])
def test_bwd_equals_torch_autograd(causal, kv_len):
    q, k, v, dO = _inputs(1)
    ours = oracle.attention_bwd_np(q, k, v, dO, 0.45, causal=causal, kv_len=kv_len)
    ref = _torch_grads(q, k, v, dO, 0.45, causal, kv_len)
    for a, b in zip(ours, ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_bwd_equals_finite_differences():
    q, k, v, dO = _inputs(2, B=1, H=2, H_kv=1, N=5, d=3)
    scale, eps = 0.6, 1e-6

    def loss(q_, k_, v_):
        O, _ = oracle.attention_np(q_, k_, v_, scale, causal=True, kv_len=[4])
        return float(np.sum(O * dO))

    grads = oracle.attention_bwd_np(q, k, v, dO, scale, causal=True, kv_len=[4])
    for which, (arr, gr) in enumerate(zip((q, k, v), grads)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus, minus = [a.copy() for a in (q, k, v)], [a.copy() for a in (q, k, v)]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
        np.testing.assert_allclose(gr, num, rtol=0, atol=1e-7)


def test_bwd_invariant_under_shifting_all_keys():
    q, k, v, dO = _inputs(3)
    shift = np.random.default_rng(9).standard_normal(k.shape[-1])
    a = oracle.attention_bwd_np(q, k, v, dO, 0.3, causal=True)
    b = oracle.attention_bwd_np(q, k + shift, v, dO, 0.3, causal=True)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-10)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_key_gradients_sum_to_zero(causal):
    # every row of dS sums to zero over its valid keys (P sums to one), so the key gradients of a
    # head sum to zero over the keys: sum_j dK_j = scale sum_i (sum_j dS_ij) q_i = 0
    q, k, v, dO = _inputs(4)
    _, dK, dV = oracle.attention_bwd_np(q, k, v, dO, 0.5, causal=causal, kv_len=[6, 9])
    np.testing.assert_allclose(dK.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    # and dV of a key is the P-weighted sum of the dO rows that attend to it: sum_j dV_j = sum_i dO_i
    # over rows with at least one valid key (every row here has key 0)
    np.testing.assert_allclose(dV.sum(axis=2), dO.reshape(2, 2, 2, 9, 5).sum(axis=(2, 3)), rtol=0, atol=1e-12)


BWD_MUTANTS = {
    "no_D": ("dS = Pm * (dP - D[:, None])", "dS = Pm * dP"),
    "dK_untransposed": ("dK[b, kh] += float(scale) * (dS.T @ q[b, h])", "dK[b, kh] += float(scale) * (dS @ q[b, h])"),
    "dQ_no_scale": ("dQ[b, h] = float(scale) * (dS @ k[b, kh])", "dQ[b, h] = (dS @ k[b, kh])"),
    "dV_untransposed": ("dV[b, kh] += Pm.T @ dO[b, h]", "dV[b, kh] += Pm @ dO[b, h]"),
    "gqa_overwrite": ("dK[b, kh] += float(scale)", "dK[b, kh] = float(scale)"),
}


@pytest.mark.parametrize("name", list(BWD_MUTANTS))
def test_planted_backward_mistake_is_caught(name):
    import inspect
    from oracle import attn_oracle_np
    old, new = BWD_MUTANTS[name]
    src = inspect.getsource(attn_oracle_np)
    assert old in src
    ns = {}
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    q, k, v, dO = _inputs(1)
    ours = ns["attention_bwd_np"](q, k, v, dO, 0.45, causal=True, kv_len=[5, 9])
    ref = _torch_grads(q, k, v, dO, 0.45, True, [5, 9])
    assert any(not np.allclose(a, b, rtol=0, atol=1e-9) for a, b in zip(ours, ref))


# ---------------------------------------------------------------- the row/key-sampled backward oracle
SAMPLED_CASES = [
    dict(causal=False, kv_len=None, H_kv=4),
    dict(causal=True, kv_len=None, H_kv=2),
    dict(causal=False, kv_len=[37, 0], H_kv=1),
    dict(causal=True, kv_len=[50, 23], H_kv=4),
]


@pytest.mark.parametrize("case", SAMPLED_CASES)
def test_sampled_backward_equals_torch_autograd(case):
    """Every sampled entry equals torch's fp64 autograd of the explicit masked softmax (a library
    routine), over sizes that span several blocks of the forward pass (N = 1100 > its 512-row blocks)."""
    rng = np.random.default_rng(5)
    B, H, N, d = 2, 4, 1100, 8
    q, k, v, dO = _inputs(11, B=B, H=H, H_kv=case["H_kv"], N=N, d=d)
    scale = 0.37
    tq, tk, tv = _torch_grads(q, k, v, dO, scale, case["causal"], case["kv_len"])
    g = H // case["H_kv"]
    for b, h in [(0, 1), (1, H - 1)]:
        rows = np.sort(rng.choice(N, size=17, replace=False))
        keys = np.sort(rng.choice(N, size=13, replace=False))
        r = oracle.attention_bwd_sampled_np(q, k, v, dO, scale, b, h, rows, keys, causal=case["causal"],
                                            kv_len=case["kv_len"])
        np.testing.assert_allclose(r["dq"], tq[b, h, rows], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["dk"], tk[b, h // g, keys], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["dv"], tv[b, h // g, keys], rtol=0, atol=1e-12)


def test_sampled_backward_equals_the_whole_backward():
    q, k, v, dO = _inputs(12, B=1, H=4, H_kv=2, N=300, d=16)
    full = oracle.attention_bwd_np(q, k, v, dO, 0.25, causal=True, kv_len=[290])
    O, L = oracle.attention_np(q, k, v, 0.25, causal=True, kv_len=[290])
    rows, keys = np.arange(0, 300, 7), np.arange(3, 300, 11)
    r = oracle.attention_bwd_sampled_np(q, k, v, dO, 0.25, 0, 3, rows, keys, causal=True, kv_len=[290])
    np.testing.assert_allclose(r["dq"], full[0][0, 3, rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dk"], full[1][0, 1, keys], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dv"], full[2][0, 1, keys], rtol=0, atol=1e-12)
    # the forward statistics it returns are the forward oracle's (query heads 2 and 3 read kv head 1)
    np.testing.assert_allclose(r["O"], O[0, 2:4], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["LSE"][np.isfinite(r["LSE"])], L[0, 2:4][np.isfinite(L[0, 2:4])], rtol=0, atol=1e-12)


@pytest.mark.parametrize("mutant", ["D_dropped", "dK_without_group_sum", "dV_from_dS"])
def test_sampled_backward_planted_mistakes_fail_the_pin(mutant, monkeypatch):
    """Mistakes planted in a copy of the sampled oracle (the D term dropped, a grouped key/value head
    taking one query head only, dV from dS instead of P) each break agreement with torch autograd."""
    import oracle.attn_oracle_np as onp
    src = __import__("inspect").getsource(onp.attention_bwd_sampled_np)
    plant = {
        "D_dropped": ("dSk = Pk * (G @ V[keys].T - D[:, None])", "dSk = Pk * (G @ V[keys].T)"),
        "dK_without_group_sum": ('out["dk"] += float(scale) * (dSk.T @ Q)',
                                 'out["dk"] = float(scale) * (dSk.T @ Q) if t == 0 else out["dk"]'),
        "dV_from_dS": ('out["dv"] += Pk.T @ G', 'out["dv"] += dSk.T @ G'),
    }[mutant]
    assert plant[0] in src
    ns = dict(vars(onp))
    exec(src.replace(plant[0], plant[1]), ns)
    q, k, v, dO = _inputs(13, B=1, H=4, H_kv=2, N=40, d=6)
    tq, tk, tv = _torch_grads(q, k, v, dO, 0.5, False, None)
    keys = np.arange(40)
    r = ns["attention_bwd_sampled_np"](q, k, v, dO, 0.5, 0, 1, np.arange(40), keys)
    ok = (np.allclose(r["dq"], tq[0, 1], atol=1e-9) and np.allclose(r["dk"], tk[0, 0], atol=1e-9)
          and np.allclose(r["dv"], tv[0, 0], atol=1e-9))
    assert not ok
