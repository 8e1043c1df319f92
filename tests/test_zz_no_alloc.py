"""attn_fwd_noalloc: the entry point for callers that cannot allocate device memory where they run
attention (host callbacks, allocator hooks, fixed start-up memory pools, plug-in hosts that forbid
allocation after initialisation). It takes its scratch from one fixed device array inside the library
instead of a caller workspace, so its results must match attn_fwd's, call after call, even though the
array keeps whatever the previous call left in it, and a call must not allocate device memory.

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test.
"""
import pytest
import torch

from exact_tiled_attention_50_b300 import inputs
from tests import parity


def test_oversized_request_is_rejected_without_launch():
    from exact_tiled_attention_50_b300 import attn
    # B=8, H=H_kv=16, N=16384, d=128: the fp16 copy of V alone is 512 MiB, beyond the 64 MiB scratch
    rc = attn.lib.attn_fwd_noalloc(4096, 4096, 4096, 4096, None, 8, 16, 16, 16384, 128, 0.088, 0, None,
                                   attn.ATTN_BF16, attn.ATTN_F32, None)
    assert rc == attn.ATTN_ERR_UNSUPPORTED
    # invalid sizes give attn_fwd's own error
    rc = attn.lib.attn_fwd_noalloc(4096, 4096, 4096, 4096, None, 1, 3, 2, 128, 64, 0.125, 0, None,
                                   attn.ATTN_BF16, attn.ATTN_F32, None)
    assert rc == attn.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("d, n_max", [(64, 438378), (128, 178261)])
def test_size_limit_is_the_workspace_of_attn_fwd(d, n_max):
    """The documented limit: accepted exactly when attn_workspace_bytes fits the 64 MiB array."""
    from exact_tiled_attention_50_b300 import attn
    lim = attn.lib.attn_workspace_bytes
    assert 0 < lim(1, 1, 1, n_max, d, attn.ATTN_BF16) <= 64 << 20 < lim(1, 1, 1, n_max + 1, d, attn.ATTN_BF16)
    rc = attn.lib.attn_fwd_noalloc(4096, 4096, 4096, 4096, None, 1, 1, 1, n_max + 1, d, 0.1, 0, None,
                                   attn.ATTN_BF16, attn.ATTN_F32, None)
    assert rc == attn.ATTN_ERR_UNSUPPORTED


def test_wrapper_rejects_what_it_would_have_to_copy():
    """The Python wrapper creates no tensor, so non-contiguous or mismatched inputs are errors (CPU
    tensors are rejected before any of them reaches the library)."""
    from exact_tiled_attention_50_b300 import attn
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd_noalloc(q, q, q, torch.zeros(1, 2, 8, 64), None)


def _both(x, out_dtype=torch.float32):
    from exact_tiled_attention_50_b300 import attn
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    kv = x.kv_len.cuda() if x.kv_len is not None else None
    B, H, N, d = q.shape
    O_ref, L_ref = attn.attn_fwd(q, k, v, scale=x.scale, causal=x.causal, kv_len=kv, out_dtype=out_dtype)
    O = torch.full((B, H, N, d), float("nan"), dtype=out_dtype, device="cuda")
    L = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    attn.attn_fwd_noalloc(q, k, v, O, L, scale=x.scale, causal=x.causal, kv_len=kv)
    assert attn.check() == attn.ATTN_OK
    return O, L, O_ref, L_ref


def _close(O, L, O_ref, L_ref):
    d = (O.double() - O_ref.double()).abs()
    assert bool(torch.isfinite(O).all())
    assert float(d.max()) <= parity.TOL["bf16"]["max_abs"]
    assert float(d.mean()) <= parity.TOL["bf16"]["mean_abs"]
    fin = torch.isfinite(L_ref)
    assert torch.equal(torch.isfinite(L), fin)
    assert float((L[fin] - L_ref[fin]).abs().max()) <= parity.LSE_TOL


@pytest.mark.gpu
def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row():
    # first call: large enough to fill a good part of the scratch (causal, padded, grouped heads, peaky K)
    x1 = inputs.custom(2, 8, 2, 1000, 128, causal=True, padded=True, peaky=True, seed=41)
    # second call: a different, smaller shape, so the scratch still holds the first call's data beyond
    # what this call writes
    x2 = inputs.custom(1, 4, 4, 300, 64, causal=False, seed=42)
    for x in (x1, x2):
        _close(*_both(x))
    # and the second result is still right against the fp64 oracle
    import oracle
    O, L, _, _ = _both(x2)
    O_o, L_o = oracle.attention(x2.q, x2.k, x2.v, x2.scale, causal=x2.causal, kv_len=x2.kv_len)
    parity.compare(O, L, O_o, L_o, "bf16", what="noalloc second call")


@pytest.mark.gpu
def test_noalloc_call_allocates_nothing():
    """After a first call (which looks up the array's address), further calls with every tensor
    already created leave torch's allocated and reserved device memory unchanged."""
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(1, 4, 2, 700, 128, causal=True, seed=43)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    O = torch.empty((1, 4, 700, 128), dtype=torch.float32, device="cuda")
    L = torch.empty((1, 4, 700), dtype=torch.float32, device="cuda")
    attn.attn_fwd_noalloc(q, k, v, O, L, scale=x.scale, causal=True)
    assert attn.check() == attn.ATTN_OK
    torch.cuda.synchronize()
    alloc, reserved = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(3):
        attn.attn_fwd_noalloc(q, k, v, O, L, scale=x.scale, causal=True)
    assert attn.check() == attn.ATTN_OK
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc
    assert torch.cuda.memory_reserved() == reserved
