"""The seeded input generator: deterministic, the stated shapes/dtypes, masks and peaky rows."""
import math

import torch

from exact_tiled_attention_50_b300 import inputs


def test_deterministic_and_shapes():
    w = inputs.WORKLOADS["b4h8_n1024_d64"]
    a, b = inputs.make_inputs(w), inputs.make_inputs(w)
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert a.q.shape == (4, 8, 1024, 64) and a.q.dtype == torch.bfloat16
    assert a.kv_len is None and not a.causal
    assert a.scale == float(torch.tensor(1 / 8, dtype=torch.float32))


def test_padding_lengths_in_range():
    w = inputs.WORKLOADS["b8h16_n4096_d128_causal_padded"].with_(N=256, H=2, H_kv=2)
    x = inputs.make_inputs(w)
    assert x.kv_len.dtype == torch.int32 and x.kv_len.shape == (8,)
    assert bool(((x.kv_len >= 128) & (x.kv_len <= 256)).all())


def test_peaky_rows_are_scaled_by_eight():
    w = inputs.WORKLOADS["sweep_b1h16_d128_n512_noncausal_peaky"].with_(H=2, H_kv=2)
    x = inputs.make_inputs(w)
    plain = inputs.make_inputs(w.with_(peaky=False))
    ratio = (x.k.float() / plain.k.float()).nan_to_num(nan=1.0)
    scaled = (ratio == 8).all(dim=-1)
    assert torch.equal(x.q, plain.q) and torch.equal(x.v, plain.v)
    assert int(scaled.sum()) == 2 * math.ceil(0.01 * 512)


def test_headline_workload():
    w = inputs.WORKLOADS[inputs.HEADLINE]
    assert (w.B, w.H, w.N, w.d, w.causal) == (1, 16, 8192, 128, False)
    assert w.nominal_flops() == 4 * 16 * 8192 ** 2 * 128


def test_effective_flops_counts_the_unmasked_pairs():
    """4 d per (query, key) pair the masks leave, against a brute-force count."""
    import numpy as np
    for causal in (False, True):
        for lens in (None, [5, 13, 0]):
            w = inputs.Workload("t", 3, 2, 1, 13, 64, "bf16", causal=causal, padded=lens is not None)
            count = 0
            for b in range(3):
                L = 13 if lens is None else lens[b]
                i, j = np.meshgrid(np.arange(13), np.arange(13), indexing="ij")
                ok = (j < L) & ((j <= i) if causal else True)
                count += int(ok.sum()) * 2  # two heads
            assert inputs.effective_flops(w, lens) == 4.0 * 64 * count
