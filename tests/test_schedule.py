"""The persistent tensor-core kernel's work schedule, checked on the host (no GPU): every key step of
every work unit is computed exactly once, the pieces of a split unit sit where the merge expects them,
and the work is balanced across CTAs. The unit costs are checked against a direct count of the key
tiles each 128-row query tile needs (keys below kv_len, and below the row for causal attention)."""
import math

import numpy as np
import pytest

COMPLETE, OWNER, WRITER = 0, 1, 2


@pytest.fixture(scope="module")
def attn():
    from exact_tiled_attention_50_b300 import build
    build.build()
    from exact_tiled_attention_50_b300 import attn
    return attn


def unit_cost(N, causal, kv, pair):
    """Key steps of the two 128-row query tiles of `pair` (at least 1)."""
    best = 0
    for t in range(2):
        q0 = 256 * pair + 128 * t
        if q0 >= N:
            continue
        tiles = 0
        for j in range(math.ceil(N / 128)):  # key tile j holds keys [128 j, 128 j + 128)
            first_key = 128 * j
            if first_key < kv and (not causal or first_key <= q0 + 127):
                tiles += 1
        best = max(best, tiles)
    return max(best, 1)


CASES = [
    (1, 16, 8192, False, None, 148),
    (1, 16, 8192, True, None, 148),
    (2, 32, 8192, True, None, 148),
    (8, 16, 4096, True, [2048, 4096, 3000, 2049, 4095, 1, 0, 3333], 148),
    (4, 8, 1024, False, None, 148),
    (1, 16, 512, False, None, 148),
    (1, 16, 512, True, None, 148),
    (2, 4, 300, True, [299, 0], 148),
    (1, 1, 1, False, None, 148),
    (3, 5, 1000, False, [1000, 999, 500], 148),
    (1, 16, 16384, False, None, 148),
    (2, 3, 777, False, None, 7),
    (5, 7, 2000, True, None, 13),
    (64, 4, 256, False, None, 148),
]


@pytest.mark.parametrize("B,H,N,causal,kv_len,sms", CASES)
def test_schedule_covers_every_key_step_once(attn, B, H, N, causal, kv_len, sms):
    segs = attn.schedule(B, H, N, causal, kv_len, sms)
    n_pairs = math.ceil(N / 256)
    G = max(s[0] for s in segs) + 1
    assert G <= min(sms, 160)
    covered = {}
    for cta, b, h, pair, k0, k1, cost, kind in segs:
        kv = N if kv_len is None else min(max(kv_len[b], 0), N)
        assert cost == unit_cost(N, causal, kv, pair), (b, pair)
        assert 0 <= k0 < k1 <= cost
        covered.setdefault((b, h, pair), []).append((k0, k1, cta, kind))
    assert len(covered) == B * H * n_pairs  # every unit appears
    for key, pieces in covered.items():
        pieces.sort()
        cost = unit_cost(N, causal, N if kv_len is None else min(max(kv_len[key[0]], 0), N), key[2])
        assert pieces[0][0] == 0 and pieces[-1][1] == cost
        for (a0, a1, *_), (b0, b1, *_) in zip(pieces, pieces[1:]):
            assert a1 == b0  # disjoint and contiguous
        head = pieces[0]
        if len(pieces) == 1:
            assert head[3] == COMPLETE
        else:
            assert head[3] == OWNER
            # the later pieces are writers on the CTAs right after the owner, in key order
            ctas = [p[2] for p in pieces]
            assert ctas == list(range(head[2], head[2] + len(pieces)))
            assert all(p[3] == WRITER for p in pieces[1:])


SPLIT_PENALTY = 10  # key steps a stream-K plan costs beyond its even share (the plan's cost model)
UNIT_OVERHEAD = 2   # line positions of a unit before its key steps (a segment's fixed time)


def plan_kind(segs):
    """'stream' when some unit is computed in pieces (or the plan could split), 'whole' otherwise."""
    return "stream" if any(s[7] != COMPLETE for s in segs) else "whole"


@pytest.mark.parametrize("B,H,N,causal,kv_len,sms", CASES)
def test_schedule_roles_and_balance(attn, B, H, N, causal, kv_len, sms):
    segs = attn.schedule(B, H, N, causal, kv_len, sms)
    G = max(s[0] for s in segs) + 1
    per_cta = {c: [s for s in segs if s[0] == c] for c in range(G)}
    load = []
    for c, lst in per_cta.items():
        kinds = [s[7] for s in lst]
        # at most one partial result per CTA (its slot), written by the first piece of its stream-K
        # chunk; only whole units (the data-parallel rounds) run before it
        assert kinds.count(WRITER) <= 1
        if WRITER in kinds:
            assert all(k == COMPLETE for k in kinds[:kinds.index(WRITER)])
        assert kinds.count(OWNER) <= 1 and (OWNER not in kinds or kinds[-1] == OWNER)
        # key steps plus the overhead of every unit the CTA starts (a writer piece starts none)
        load.append(sum(s[5] - s[4] + (UNIT_OVERHEAD if s[4] == 0 else 0) for s in lst))
    assert min(load) >= 1  # no CTA is launched without work
    n_pairs = math.ceil(N / 256)
    units = B * H * n_pairs
    if plan_kind(segs) == "stream":
        # every CTA gets an equal chunk of the line up to rounding; a chunk boundary inside (or at the
        # end of) a unit's overhead moves that overhead to the CTA that starts the unit: at most
        # UNIT_OVERHEAD more on one CTA and as much less on the one before it
        assert max(load) - min(load) <= 1 + 2 * UNIT_OVERHEAD, (min(load), max(load), sum(load) / G)
    else:
        # whole units in rounds: unit r * G + c on CTA c, no CTA idle in the first round
        assert G == math.ceil(units / math.ceil(units / G))
        for c, lst in per_cta.items():
            us = [(s[1] * H + s[2]) * n_pairs + s[3] for s in lst]
            assert us == list(range(c, units, G))


def model_makespans(B, H, N, causal, padded, sms):
    """Busiest CTA's key steps plus unit overheads under each plan (kv_len counted as N), as the
    plan's cost model states."""
    nb = math.ceil(N / 128)
    n_pairs = math.ceil(N / 256)
    costs = [unit_cost(N, causal, N, p) for p in range(n_pairs)]
    w = B * H * (sum(costs) + UNIT_OVERHEAD * n_pairs)
    g_cap = min(sms, 160)
    g = max(1, min(g_cap, math.ceil(w / 2)))
    t_stream = math.ceil(w / g) + SPLIT_PENALTY
    units = B * H * n_pairs
    rounds = math.ceil(units / g_cap)
    uniform = not causal and not padded
    t_whole = rounds * (nb + UNIT_OVERHEAD) if uniform else (max(costs) + UNIT_OVERHEAD if rounds == 1 else None)
    return t_whole, t_stream


@pytest.mark.parametrize("B,H,N,causal,kv_len,sms", CASES)
def test_schedule_takes_the_cheaper_plan(attn, B, H, N, causal, kv_len, sms):
    segs = attn.schedule(B, H, N, causal, kv_len, sms)
    t_whole, t_stream = model_makespans(B, H, N, causal, kv_len is not None, sms)
    want = "whole" if t_whole is not None and t_whole < t_stream else "stream"
    got = plan_kind(segs)
    # a stream-K plan whose chunk boundaries all fall on unit boundaries splits nothing: it looks whole
    assert got == want or (want == "stream" and got == "whole")


@pytest.mark.parametrize("B,H,N,causal,kv_len,expect_G,expect", [
    (4, 8, 1024, False, None, 128, "whole"),       # 128 units of 8 steps: one round, no merges
    (1, 16, 512, False, None, 32, "whole"),        # 32 units of 4 steps
    (1, 16, 512, True, None, 32, "whole"),
    (1, 16, 1024, True, None, 64, "whole"),        # causal: the costliest unit (8 steps) beats 3 + merges
    (1, 16, 2048, False, None, 128, "whole"),
    (1, 16, 8192, False, None, 148, "stream"),     # 512 units of 64 steps: 3.46 rounds -> stream-K
    (1, 16, 16384, False, None, 148, "stream"),
    (2, 32, 8192, True, None, 148, "stream"),
])
def test_schedule_choice_on_the_workloads(attn, B, H, N, causal, kv_len, expect_G, expect):
    segs = attn.schedule(B, H, N, causal, kv_len, 148)
    assert max(s[0] for s in segs) + 1 == expect_G
    assert plan_kind(segs) == expect


def test_schedule_rejects_bad_arguments(attn):
    assert attn.lib.attn_debug_schedule(0, 1, 128, 0, None, 148, None, 0) == -1
    assert attn.lib.attn_debug_schedule(1, 1, 128, 0, None, 0, None, 0) == -1
