"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Small and ragged shapes are compared element by element against the full oracle; the full-size
workloads (the ones the benchmark times) are compared on sampled rows, each evaluated exactly by the
row-sampled oracle over all keys.
"""
import numpy as np
import pytest
import torch

from exact_tiled_attention_50_b300 import inputs
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from exact_tiled_attention_50_b300 import attn  # noqa: F401  (fails loudly without libattn.so)
    assert torch.cuda.is_available()
    yield


# ---------------------------------------------------------------- the five workload families
def test_tiny_fp32_full():
    x = inputs.make_inputs(inputs.WORKLOADS["tiny_b1h1_n256_d64_f32"])
    parity.check_full(x, "f32", what="tiny fp32")


def test_b4h8_n1024_d64_full():
    x = inputs.make_inputs(inputs.WORKLOADS["b4h8_n1024_d64"])
    parity.check_full(x, "bf16", what="b4h8 n1024 d64")


def test_b8h16_n4096_causal_padded_sampled():
    x = inputs.make_inputs(inputs.WORKLOADS["b8h16_n4096_d128_causal_padded"])
    parity.check_sampled(x, "bf16", per_head=24, what="b8h16 n4096 causal padded")


@pytest.mark.parametrize("name", ["gqa_b2h32kv8_n8192_d128_causal", "mqa_b2h32kv1_n8192_d128_causal"])
def test_gqa_mqa_n8192_sampled(name):
    x = inputs.make_inputs(inputs.WORKLOADS[name])
    parity.check_sampled(x, "bf16", per_head=16, what=name)


@pytest.mark.parametrize("n", [512, 1024, 2048, 4096, 8192, 16384])
@pytest.mark.parametrize("causal", [False, True])
def test_peaky_sweep_sampled(n, causal):
    tag = "causal" if causal else "noncausal"
    x = inputs.make_inputs(inputs.WORKLOADS[f"sweep_b1h16_d128_n{n}_{tag}_peaky"])
    parity.check_sampled(x, "bf16", per_head=64 if n >= 8192 else 128, what=f"sweep n{n} {tag}")


def test_peaky_sweep_n2048_full():
    x = inputs.make_inputs(inputs.WORKLOADS["sweep_b1h16_d128_n2048_causal_peaky"])
    parity.check_full(x, "bf16", what="sweep n2048 causal (full)")


# ---------------------------------------------------------------- rows whose scores are all far below 0
@pytest.mark.parametrize("N", [1, 3, 200])
@pytest.mark.parametrize("d", [64, 128])
def test_rows_with_only_negative_scores(N, d):
    """Q shifted by +2 and K by -2 in every channel: every score is about -4 d scale (about -45 for
    d = 128), the softmax is still well defined. The running maximum must be the row's own (a larger
    reference, such as 0, would underflow every fp16 probability: O = 0)."""
    x = inputs.custom(1, 2, 1, N, d, causal=True, seed=90 + N)
    x.q = (x.q.float() + 2.0).to(torch.bfloat16).contiguous()
    x.k = (x.k.float() - 2.0).to(torch.bfloat16).contiguous()
    parity.check_full(x, "bf16", what=f"negative scores N={N} d={d}")


# ---------------------------------------------------------------- edges: ragged sizes, masks, heads
@pytest.mark.parametrize("N", [1, 2, 100, 127, 128, 129, 200, 255, 256, 257, 384, 513])
@pytest.mark.parametrize("d", [64, 128])
def test_ragged_lengths(N, d):
    x = inputs.custom(2, 4, 2, N, d, causal=False, seed=N * 7 + d)
    parity.check_full(x, "bf16", what=f"N={N} d={d}")
    x = inputs.custom(2, 4, 2, N, d, causal=True, seed=N * 7 + d + 1)
    parity.check_full(x, "bf16", what=f"N={N} d={d} causal")


@pytest.mark.parametrize("H,H_kv", [(8, 8), (8, 2), (8, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_head_groups(H, H_kv, causal):
    x = inputs.custom(2, H, H_kv, 300, 128, causal=causal, padded=True, peaky=True, seed=H * 10 + H_kv)
    parity.check_full(x, "bf16", what=f"H={H} H_kv={H_kv} causal={causal}")


@pytest.mark.parametrize("lens", [[1, 1], [299, 300], [300, 300], [0, 171], [129, 128], [256, 1]])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding(lens, causal):
    x = inputs.custom(2, 2, 1, 300, 64, causal=causal, kv_len=lens, seed=sum(lens))
    parity.check_full(x, "bf16", what=f"kv_len={lens} causal={causal}")


def test_kv_len_out_of_range_is_clamped():
    x = inputs.custom(2, 2, 2, 200, 64, kv_len=[-5, 10_000], seed=9)
    O, L = parity.run_gpu(x)
    import oracle
    O_ref, L_ref = oracle.attention(x.q, x.k, x.v, x.scale, kv_len=[0, 200])
    parity.compare(O, L, O_ref, L_ref, "bf16", what="clamped kv_len")


@pytest.mark.parametrize("N", [1, 33, 256, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_path(N, causal):
    for d in (64, 128):
        x = inputs.custom(2, 4, 2, N, d, dtype="f32", causal=causal, padded=True, seed=N + d)
        parity.check_full(x, "f32", what=f"fp32 N={N} d={d}")


def test_bf16_output():
    x = inputs.custom(2, 4, 4, 513, 128, causal=True, peaky=True, seed=5)
    parity.check_full(x, "bf16", out_dtype=torch.bfloat16, what="bf16 out")


def test_large_v_values_use_the_per_head_scale():
    # V beyond the fp16 range (|V| up to ~1e6): the fp16 copy is scaled by a power of two per head
    x = inputs.custom(1, 2, 2, 256, 64, seed=11)
    x.v = (x.v.float() * 2.0 ** 18).to(torch.bfloat16)
    O, L = parity.run_gpu(x)
    import oracle
    O_ref, L_ref = oracle.attention(x.q, x.k, x.v, x.scale)
    rel = (O.double().cpu().numpy() - O_ref) / 2.0 ** 18
    assert np.abs(rel).max() <= 2e-3 and np.abs(rel).mean() <= 2e-4


@pytest.mark.parametrize("causal", [False, True])
def test_v_magnitude_varies_across_key_tiles(causal):
    """Key tiles of very different |V|: the fp16 copy of V takes one power-of-two exponent per 128-key
    tile, the accumulator follows the largest exponent seen (exactly, like the running maximum), and
    work units split between CTAs merge pieces with different exponents. The error of each output is
    bounded relative to the magnitude it is made of, sum_j P_ij |V_j| (fp16 P rounding is relative)."""
    import oracle
    x = inputs.custom(2, 4, 2, 1000, 128, causal=causal, seed=31)
    v = x.v.float()
    v[:, :, 128:256] *= 2.0 ** 10
    v[:, :, 640:768] *= 2.0 ** 20
    v[:, 1, 900:1000] *= 2.0 ** 17
    x.v = v.to(torch.bfloat16)
    O, L = parity.run_gpu(x)
    O_ref, L_ref, P = oracle.attention(x.q, x.k, x.v, x.scale, causal=causal, return_p=True)
    vabs = np.repeat(np.abs(x.v.float().numpy()).astype(np.float64), 2, axis=1)  # kv head of each query head
    mag = np.einsum("bhij,bhjd->bhid", P, vabs)
    err = np.abs(O.double().cpu().numpy() - O_ref)
    assert np.all(err <= 2e-3 * mag + 1e-30), float(np.max(err / (mag + 1e-30)))
    assert float(np.abs(L.cpu().numpy() - L_ref).max()) <= parity.LSE_TOL


# ---------------------------------------------------------------- merge over disjoint key sets
@pytest.mark.parametrize("d", [64, 128])
def test_merge_kernel_against_oracle(d):
    """attn_merge on fp64 oracle parts over keys [0, L) and [L, N) (rounded to fp32) equals the oracle
    over all keys, within the fp32 bar; a part without keys contributes nothing."""
    import oracle
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(2, 4, 2, 300, d, dtype="f32", peaky=True, seed=17)
    q, k, v = (t.numpy() for t in (x.q, x.k, x.v))
    O_full, L_full = oracle.attention(q, k, v, x.scale)
    for L in (0, 128, 171):
        A = oracle.attention(q, k, v, x.scale, kv_len=[L, L])
        Bp = oracle.attention(q, np.roll(k, -L, axis=2), np.roll(v, -L, axis=2), x.scale, kv_len=[300 - L] * 2)
        Op = torch.tensor(np.stack([A[0], Bp[0]]), dtype=torch.float32, device="cuda")
        Lp = torch.tensor(np.stack([A[1], Bp[1]]), dtype=torch.float32, device="cuda")
        O, LSE = attn.merge(Op, Lp)
        assert float(np.abs(O.double().cpu().numpy() - O_full).max()) <= 1e-5
        assert float(np.abs(LSE.double().cpu().numpy() - L_full).max()) <= 1e-5


def test_split_kv_attention_merged_on_gpu():
    """Sequence-parallel use: two attn_fwd calls over disjoint key ranges (the second through rotated
    K/V and kv_len), merged by attn_merge, equal attention over all keys (bf16 bar)."""
    import oracle
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(2, 8, 2, 1000, 128, peaky=True, seed=23)
    L = 389
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    OA, LA = attn.attn_fwd(q, k, v, scale=x.scale, kv_len=torch.full((2,), L, dtype=torch.int32, device="cuda"))
    OB, LB = attn.attn_fwd(q, torch.roll(k, -L, 2).contiguous(), torch.roll(v, -L, 2).contiguous(), scale=x.scale,
                           kv_len=torch.full((2,), 1000 - L, dtype=torch.int32, device="cuda"))
    O, LSE = attn.merge(torch.stack([OA, OB]), torch.stack([LA, LB]))
    assert attn.check() == attn.ATTN_OK
    O_ref, L_ref = oracle.attention(x.q, x.k, x.v, x.scale)
    parity.compare(O, LSE, O_ref, L_ref, "bf16", what="split-KV merged")


# ---------------------------------------------------------------- guard bands, determinism
def test_guard_bands_untouched():
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(2, 4, 2, 300, 128, causal=True, padded=True, seed=21)
    B, H, N, d = x.q.shape
    pad = 4096
    canary = 1234.5
    Obuf = torch.full((pad + B * H * N * d + pad,), canary, dtype=torch.float32, device="cuda")
    Lbuf = torch.full((pad + B * H * N + pad,), canary, dtype=torch.float32, device="cuda")
    O = Obuf[pad:pad + B * H * N * d].view(B, H, N, d)
    L = Lbuf[pad:pad + B * H * N].view(B, H, N)
    attn.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale, causal=True, kv_len=x.kv_len.cuda(),
                  out=O, lse=L)
    assert attn.check() == attn.ATTN_OK
    for buf, n in ((Obuf, B * H * N * d), (Lbuf, B * H * N)):
        assert bool((buf[:pad] == canary).all()) and bool((buf[pad + n:] == canary).all())
    import oracle
    O_ref, L_ref = oracle.attention(x.q, x.k, x.v, x.scale, causal=True, kv_len=x.kv_len)
    parity.compare(O, L, O_ref, L_ref, "bf16", what="guarded")


def test_bitwise_deterministic():
    x = inputs.custom(1, 8, 2, 1000, 128, causal=True, padded=True, peaky=True, seed=3)
    O1, L1 = parity.run_gpu(x)
    O2, L2 = parity.run_gpu(x)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


# ---------------------------------------------------------------- failure path (bounded waits)
def test_bounded_wait_timeout_is_reported_and_context_survives():
    """The producer skips one load (a barrier that nothing completes); the kernel's bounded wait runs
    out, it records ATTN_ERR_TIMEOUT and exits; the next call on the same context works."""
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(1, 1, 1, 256, 64, seed=4)
    attn.lib.attn_debug_set_wait_limit_ns(50_000_000)
    attn.lib.attn_debug_set_skip_kv_load(1)
    try:
        attn.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale)
        assert attn.check() == attn.ATTN_ERR_TIMEOUT
    finally:
        attn.lib.attn_debug_set_skip_kv_load(0)
        attn.lib.attn_debug_set_wait_limit_ns(0)
    assert attn.check() == attn.ATTN_OK  # the error word was cleared
    parity.check_full(x, "bf16", what="after timeout")


# ---------------------------------------------------------------- both work plans
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_both_work_plans_match_the_oracle(mode, causal):
    """Whole units in rounds (mode 1) and stream-K with split units merged (mode 2) give the same
    attention, whichever the cost model would pick for the shape."""
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(2, 8, 2, 1000, 128, causal=causal, padded=True, peaky=True, seed=300 + mode)
    attn.lib.attn_debug_set_plan_mode(mode)
    try:
        parity.check_full(x, "bf16", what=f"plan mode {mode} causal={causal}")
    finally:
        attn.lib.attn_debug_set_plan_mode(0)


# ---------------------------------------------------------------- host buffers, pipelined over head groups
@pytest.mark.parametrize("B,H,H_kv,N,d,dtype,causal,padded,n_groups", [
    (2, 8, 2, 600, 128, "bf16", True, True, 0),     # 2 batches x 2 kv heads: 4 groups
    (1, 16, 16, 384, 64, "bf16", False, False, 3),  # tapered groups (3, 5, 5, 3 kv heads)
    (2, 4, 1, 300, 128, "bf16", True, False, 64),   # MQA: one group per batch
    (1, 2, 2, 256, 64, "f32", False, False, 0),
])
def test_host_pipeline_matches_the_oracle(B, H, H_kv, N, d, dtype, causal, padded, n_groups):
    """attn_fwd_host: host inputs copied in, attention, host outputs copied back, pipelined over
    groups of heads; its host results match the oracle (and attn_fwd's) on every head."""
    import oracle
    from exact_tiled_attention_50_b300 import attn
    x = inputs.custom(B, H, H_kv, N, d, dtype, causal=causal, padded=padded, peaky=dtype == "bf16",
                      seed=400 + n_groups)
    qh, kh, vh = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
    oh = torch.full((B, H, N, d), float("nan"), dtype=torch.float32).pin_memory()
    lh = torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()
    kvh = x.kv_len.pin_memory() if x.kv_len is not None else None
    qd, kd, vd = torch.empty_like(x.q, device="cuda"), torch.empty_like(x.k, device="cuda"), torch.empty_like(x.v, device="cuda")
    od = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    ld = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    kvd = torch.empty((B,), dtype=torch.int32, device="cuda") if kvh is not None else None
    attn.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, scale=x.scale, causal=causal, kv_len_h=kvh,
                       kv_len_d=kvd, n_groups=n_groups)
    torch.cuda.synchronize()
    assert attn.check() == attn.ATTN_OK
    O_ref, L_ref = oracle.attention(x.q, x.k, x.v, x.scale, causal=causal, kv_len=x.kv_len)
    parity.compare(oh, lh, O_ref, L_ref, dtype, what=f"host pipeline {B}x{H}/{H_kv} N={N} groups={n_groups}")
    assert torch.equal(od.cpu(), oh)  # the device buffers hold the same result


def test_host_pipeline_full_size_sampled_rows():
    """attn_fwd_host on the bench workload (B1 H16 N8192 d128, the end-to-end leg's call with its default
    tapered head groups): sampled rows of every head against the oracle, and the whole host result within
    twice the forward's bar of attn_fwd's on the device inputs. The two need not agree bit for bit: a
    group of one or two heads gets its own schedule, in which the persistent kernel splits the units
    into pieces merged in fp32 (shorter tensor-core accumulations, slightly different rounding)."""
    import oracle
    from exact_tiled_attention_50_b300 import attn
    x = inputs.make_inputs(inputs.WORKLOADS[inputs.HEADLINE])
    B, H, N, d = x.q.shape
    qh, kh, vh = x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory()
    oh = torch.full((B, H, N, d), float("nan"), dtype=torch.float32).pin_memory()
    lh = torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()
    qd, kd, vd = torch.empty_like(x.q, device="cuda"), torch.empty_like(x.k, device="cuda"), torch.empty_like(x.v, device="cuda")
    od = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    ld = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    attn.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, scale=x.scale)
    torch.cuda.synchronize()
    assert attn.check() == attn.ATTN_OK
    rows = parity.sample_rows(B, H, N, None, per_head=24, seed=5)
    O_ref, L_ref = oracle.attention_rows(x.q, x.k, x.v, x.scale, rows)
    parity.compare(oh.reshape(-1, d)[torch.as_tensor(rows)], lh.reshape(-1)[torch.as_tensor(rows)], O_ref, L_ref,
                   "bf16", what="host pipeline, bench workload")
    O2, L2 = attn.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale)
    assert float((O2.cpu() - oh).abs().max()) <= 2 * parity.TOL["bf16"]["max_abs"]
    assert float((L2.cpu() - lh).abs().max()) <= 2 * parity.LSE_TOL


def test_bf16_output_full_size_sampled_rows():
    """bf16 output on the bench workload (B1 H16 N8192 d128): its epilogue rounds O to bf16 straight from
    the registers; sampled rows against the oracle with the bar widened by half an output ulp."""
    x = inputs.make_inputs(inputs.WORKLOADS[inputs.HEADLINE])
    parity.check_sampled(x, "bf16", per_head=24, out_dtype=torch.bfloat16, what="bf16 out, bench workload", seed=9)


@pytest.mark.parametrize("name,heads", [("sweep_b1h16_d128_n8192_noncausal_peaky", (0, 9)),
                                        ("sweep_b1h16_d128_n16384_causal_peaky", (3, 12))])
def test_whole_heads_at_the_longest_sizes(name, heads):
    """Every element of two whole heads at N = 8192 and 16384 (peaky keys) against the oracle: the
    largest errors sit in single rows dominated by one key (fp16 P rounding plus the tensor core's long
    accumulation), which row sampling may miss."""
    import oracle
    from exact_tiled_attention_50_b300 import attn
    w = inputs.WORKLOADS[name]
    x = inputs.make_inputs(w)
    B, H, N, d = x.q.shape
    O, L = attn.attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), scale=x.scale, causal=w.causal)
    rc = attn.check()
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    for h in heads:
        rows = np.arange(h * N, (h + 1) * N, dtype=np.int64)
        O_ref, L_ref = oracle.attention_rows(x.q, x.k, x.v, x.scale, rows, causal=w.causal)
        parity.compare(O[0, h], L[0, h], O_ref, L_ref, "bf16", what=f"{name} head {h}, every row")
