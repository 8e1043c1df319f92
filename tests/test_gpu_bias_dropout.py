"""GPU attention with an additive bias and dropout (attn_fwd_ex, through the C ABI) against the oracle.

The keep decisions are integer work (Philox4x32-10 draws against a 16-bit threshold), so they must
agree exactly: with them equal, the outputs differ only by the forward's own arithmetic and share its
bar (bf16 inputs: max |dO| <= 2e-3, mean <= 2e-4; |dLSE| <= 1e-3). A single differing keep decision
moves an output by about P_ij |V_j| / (1 - p), far above that bar for the rows where it matters, and
the exact-mask test below checks the decisions directly on a one-key-per-row construction.
"""
import numpy as np
import pytest
import torch

from oracle import attn_oracle_np as o
from exact_tiled_attention_50_b300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


def _bias(shape, N, seed, scale=2.0, pad_to=8):
    """bf16 bias of `shape` (last dim N) stored on the device with its rows padded to a multiple of 8
    elements (the library reads 16-byte aligned rows); returns (device view [.., N], fp64 values)."""
    g = torch.Generator().manual_seed(seed)
    npad = (N + pad_to - 1) // pad_to * pad_to
    full = (torch.randn(tuple(shape[:-1]) + (npad,), generator=g) * scale).to(torch.bfloat16)
    return full.cuda()[..., :N], full[..., :N].double().numpy()


def _run(x, bias=None, bias_np=None, p=0.0, seed=0, offset=0):
    from exact_tiled_attention_50_b300 import attn
    kv = x.kv_len.cuda() if x.kv_len is not None else None
    O, L = attn.attn_fwd_ex(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale, causal=x.causal, kv_len=kv,
                            bias=bias, dropout_p=p, seed=seed, offset=offset)
    rc = attn.check()
    assert rc == attn.ATTN_OK, f"{attn.status_string(rc)} bits {attn.lib.attn_debug_last_error_bits():#x}"
    lens = None if x.kv_len is None else x.kv_len.numpy()
    O_ref, L_ref = o.attention_bias_dropout_np(x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy(),
                                               x.scale, bias=bias_np, p=p, seed=seed, offset=offset,
                                               causal=x.causal, kv_len=lens)
    return O, L, O_ref, L_ref


@pytest.mark.parametrize("d", [64, 128])
def test_full_bias_no_dropout(d):
    x = inputs.custom(2, 4, 2, 300, d, seed=101 + d)
    b, bn = _bias((2, 4, 300, 300), 300, seed=1)
    parity.compare(*_run(x, b, bn), "bf16", what=f"full bias d={d}")


def test_broadcast_bias_causal_gqa_dropout():
    x = inputs.custom(2, 8, 2, 384, 128, causal=True, seed=102)
    b, bn = _bias((384, 384), 384, seed=2)  # one [N, N] bias for every batch and head (zero strides)
    parity.compare(*_run(x, b, bn, p=0.1, seed=1234, offset=3), "bf16", what="broadcast bias, causal, p=0.1")


def test_key_bias_with_masked_keys_and_padding():
    N = 257
    x = inputs.custom(2, 4, 1, N, 64, kv_len=[200, 257], seed=103)
    g = torch.Generator().manual_seed(3)
    full = torch.zeros((2, 1, 1, 264), dtype=torch.bfloat16)  # one bias per key (row stride 0)
    full[..., :N] = (torch.randn((2, 1, 1, N), generator=g) * 2).to(torch.bfloat16)
    full[0, ..., 10:20] = float("-inf")  # masking by bias
    parity.compare(*_run(x, full.cuda()[..., :N], full[..., :N].double().numpy(), p=0.2, seed=77), "bf16",
                   what="key bias, -inf, kv_len")


@pytest.mark.parametrize("N", [1, 129, 1000])
def test_dropout_only_ragged(N):
    x = inputs.custom(1, 4, 4, N, 128, causal=N > 1, seed=104 + N)
    parity.compare(*_run(x, p=0.1, seed=2 ** 40 + 5, offset=N), "bf16", what=f"dropout N={N}")


def test_no_bias_no_dropout_equals_attn_fwd():
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(2, 4, 2, 513, 128, causal=True, seed=105)
    O, L, O_ref, L_ref = _run(x)
    parity.compare(O, L, O_ref, L_ref, "bf16", what="plain")
    O2, L2 = attn.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale, causal=True)
    # the two kernels form the scaled scores with different roundings (the bias variant adds its bias
    # to S * scale*log2e), which can flip the fp16 rounding of a probability, and the row sum takes the
    # rounded values: O and LSE then agree within the forward's bars, not bit for bit
    assert torch.allclose(O, O2, rtol=0, atol=parity.TOL["bf16"]["max_abs"])
    assert torch.allclose(L, L2, rtol=0, atol=parity.LSE_TOL)


def test_split_units_of_the_persistent_schedule():
    x = inputs.custom(1, 24, 24, 1536, 128, seed=106)
    b, bn = _bias((1, 24, 1536, 1536), 1536, seed=4, scale=1.0)
    parity.compare(*_run(x, b, bn, p=0.1, seed=9), "bf16", what="B1 H24 N1536 bias + dropout")


def test_keep_decisions_exactly():
    """Each row attends to one key only (bias -inf elsewhere), with V_j = e_(j mod d) * (j + 1): row i's
    output is then its single key's V scaled by keep / (1 - p), so every keep decision the kernel took
    is read off the output and compared with the oracle's mask."""
    from exact_tiled_attention_50_b300 import attn
    B, H, N, d, p, seed, off = 1, 2, 256, 64, 0.5, 31337, 11
    x = inputs.custom(B, H, H, N, d, seed=107)
    v = torch.zeros((B, H, N, d))
    for j in range(N):
        v[:, :, j, j % d] = float(j + 1)
    rng = np.random.default_rng(5)
    target = rng.integers(0, N, size=(H, N))  # the key each row attends to
    bias = torch.full((B, H, N, N), float("-inf"))
    for h in range(H):
        bias[0, h, np.arange(N), target[h]] = 0.0
    bias = bias.to(torch.bfloat16)
    O, _ = attn.attn_fwd_ex(x.q.cuda(), x.k.cuda(), v.to(torch.bfloat16).cuda(), scale=x.scale,
                            bias=bias.cuda(), dropout_p=p, seed=seed, offset=off)
    assert attn.check() == attn.ATTN_OK
    O = O.cpu().numpy()
    keep = o.dropout_keep_mask(B, H, N, p, seed, off)
    t = o.dropout_threshold(p)
    for h in range(H):
        j = target[h]
        got = O[0, h, np.arange(N), j % d] * (1 - t / 65536.0) / (j + 1)  # 1 if kept, 0 if dropped
        np.testing.assert_allclose(got, keep[0, h, np.arange(N), j].astype(np.float64), rtol=0, atol=1e-3)


@pytest.mark.parametrize("with_bias", [True, False])
def test_full_size_sampled_rows(with_bias):
    """The bench's bias + dropout and dropout-only workloads as bench.py times them: B1 H16 N8192 d128
    (peaky keys), a full [B, H, N, N] bf16 bias drawn on the device with the bench's seed, p = 0.1,
    seed 1, offset 0. Rows sampled in four heads (tile edges and random rows), each checked element by
    element against the row-restricted oracle with the forward's bar; every keep decision of a sampled
    row enters its output."""
    from exact_tiled_attention_50_b300 import attn
    x = inputs.make_inputs(inputs.WORKLOADS[inputs.HEADLINE])
    B, H, N, d = x.q.shape
    bias = None
    if with_bias:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(inputs.SEED_BASE + 4000)
        bias = torch.randn((B, H, N, N), generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    O, L = attn.attn_fwd_ex(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale, bias=bias, dropout_p=0.1, seed=1,
                            offset=0)
    rc = attn.check()
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    q, k, v = x.q.double().numpy(), x.k.double().numpy(), x.v.double().numpy()
    rng = np.random.default_rng(17)
    for h in (0, 5, 10, 15):
        rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 12)]))
        bias_rows = None if bias is None else bias[0, h, torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
        Or, Lr = o.attention_bias_dropout_rows_np(q, k, v, x.scale, 0, h, rows, bias_rows=bias_rows, p=0.1, seed=1,
                                                  offset=0)
        parity.compare(O[0, h, torch.as_tensor(rows, device="cuda")], L[0, h, torch.as_tensor(rows, device="cuda")],
                       Or, Lr, "bf16", what=f"{'bias + ' if with_bias else ''}dropout, head {h}")
