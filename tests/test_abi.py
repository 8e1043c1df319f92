"""The C-ABI library: it loads without a GPU, exports every function include/attn.h declares, and
rejects invalid arguments on the host before launching anything (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_50_b300 import build
    build.build()
    from exact_tiled_attention_50_b300 import attn
    return attn


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(attn_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_check", "attn_status_string", "attn_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, missing
    assert set(lib.EXPORTED) <= set(declared_functions())


def test_status_strings(lib):
    assert lib.status_string(0) == "ATTN_OK"
    assert lib.status_string(4) == "ATTN_ERR_TIMEOUT"
    assert lib.status_string(99) == "ATTN_UNKNOWN_STATUS"


def test_workspace_bytes(lib):
    import torch
    assert lib.workspace_bytes(1, 1, 1, 256, 64, torch.float32) == 0
    w = lib.workspace_bytes(2, 32, 8, 8192, 128, torch.bfloat16)
    assert w >= 2 * 8 * 8192 * 128 * 2 and w % 256 == 0
    assert lib.workspace_bytes(1, 3, 2, 128, 64, torch.bfloat16) == 0  # H % H_kv != 0
    assert lib.workspace_bytes(1, 1, 1, 128, 96, torch.bfloat16) == 0  # unsupported d


def _call(lib, **kw):
    a = dict(Q=4096, K=4096, V=4096, O=4096, LSE=None, B=1, H=2, H_kv=1, N=128, d=64, scale=0.125, causal=0,
             kv_len=None, ind=1, outd=0, ws=4096, ws_bytes=1 << 30)
    a.update(kw)
    return lib.lib.attn_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["H_kv"], a["N"], a["d"],
                            a["scale"], a["causal"], a["kv_len"], a["ind"], a["outd"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("bad", [
    dict(Q=None), dict(K=None), dict(V=None), dict(O=None),
    dict(B=0), dict(H=0), dict(H_kv=0), dict(N=0), dict(N=-5),
    dict(H=3, H_kv=2), dict(d=96), dict(d=256), dict(d=0),
    dict(scale=0.0), dict(scale=-1.0), dict(scale=float("inf")), dict(scale=float("nan")),
    dict(causal=2), dict(Q=4100), dict(O=4104), dict(ind=7), dict(outd=9),
    dict(ws=None), dict(ws=4096 + 16), dict(ws_bytes=100),
])
def test_invalid_arguments_rejected_without_launch(lib, bad):
    assert _call(lib, **bad) == lib.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(O_parts=None), dict(n=0), dict(rows=0), dict(d=96), dict(O=4100)])
def test_merge_invalid_arguments(lib, bad):
    a = dict(O_parts=4096, L_parts=4096, n=2, rows=128, d=128, O=8192, L=8192)
    a.update(bad)
    assert lib.lib.attn_merge(a["O_parts"], a["L_parts"], a["n"], a["rows"], a["d"], a["O"], a["L"], None) == \
        lib.ATTN_ERR_INVALID_ARG


def test_unsupported_combination(lib):
    assert _call(lib, ind=0, outd=1) == lib.ATTN_ERR_UNSUPPORTED


def test_fp8_workspace_bytes(lib):
    w = lib.lib.attn_fwd_fp8_workspace_bytes(2, 8, 2, 1000, 128)
    # E4M3 copies of Q (B H N d), K (B H_kv N d), V^T (B H_kv d N padded to 128) at least
    assert w >= 2 * 8 * 1000 * 128 + 2 * 2 * 1000 * 128 + 2 * 2 * 128 * 1024 and w % 256 == 0
    assert lib.lib.attn_fwd_fp8_workspace_bytes(2, 8, 2, 1000, 64) == 0  # d = 128 only
    assert lib.lib.attn_fwd_fp8_workspace_bytes(2, 8, 3, 1000, 128) == 0


def _call_fp8(lib, **kw):
    a = dict(Q=4096, K=4096, V=4096, O=4096, LSE=None, B=1, H=2, H_kv=1, N=128, d=128, scale=0.125, causal=0,
             kv_len=None, signs=None, ws=4096, ws_bytes=1 << 30)
    a.update(kw)
    return lib.lib.attn_fwd_fp8(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["H_kv"], a["N"],
                                a["d"], a["scale"], a["causal"], a["kv_len"], a["signs"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("bad", [
    dict(Q=None), dict(O=None), dict(B=0), dict(N=0), dict(H=3, H_kv=2), dict(scale=0.0),
    dict(scale=float("nan")), dict(causal=3), dict(K=4100), dict(ws=None), dict(ws=4096 + 64), dict(ws_bytes=1000),
])
def test_fp8_invalid_arguments_rejected_without_launch(lib, bad):
    assert _call_fp8(lib, **bad) == lib.ATTN_ERR_INVALID_ARG


def test_fp8_head_dim_other_than_128_unsupported(lib):
    assert _call_fp8(lib, d=64) == lib.ATTN_ERR_UNSUPPORTED


def _call_ex(lib, **kw):
    a = dict(Q=4096, K=4096, V=4096, O=4096, LSE=None, B=1, H=2, H_kv=1, N=128, d=64, scale=0.125, causal=0,
             kv_len=None, bias=None, sb=0, sh=0, sr=128, p=0.1, seed=1, off=0, ws=4096, ws_bytes=1 << 30)
    a.update(kw)
    return lib.lib.attn_fwd_ex(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["H_kv"], a["N"], a["d"],
                               a["scale"], a["causal"], a["kv_len"], a["bias"], a["sb"], a["sh"], a["sr"], a["p"],
                               a["seed"], a["off"], a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("bad", [
    dict(Q=None), dict(O=None), dict(N=0), dict(d=96), dict(H=3, H_kv=2), dict(scale=-1.0), dict(causal=5),
    dict(p=1.0), dict(p=-0.1), dict(p=float("nan")), dict(bias=4100), dict(bias=4096, sr=100),
    dict(bias=4096, sb=-8), dict(bias=4096, sh=12), dict(ws=None), dict(ws_bytes=64),
])
def test_ex_invalid_arguments_rejected_without_launch(lib, bad):
    assert _call_ex(lib, **bad) == lib.ATTN_ERR_INVALID_ARG


def _groups_per_batch(B, H_kv, n_groups):
    """The host pipeline's groups per batch, restated: about n_groups in all (8 by default, at most
    64), one more per batch when there are at least two (half-size groups at both ends), at most one
    per key/value head, and at most 64 over every batch (0: unsupported)."""
    per = -(-min(n_groups if n_groups > 0 else 8, 64) // B)
    if per >= 2:
        per += 1
    per = min(per, H_kv)
    if per * B > 64:
        per = 64 // B
    return per


@pytest.mark.parametrize("B,H_kv,n_groups", [
    (1, 16, 0), (1, 16, 3), (2, 2, 0), (2, 1, 64), (8, 16, 64), (64, 1, 0), (65, 1, 0), (3, 5, 7), (1, 1, 0),
    (4, 32, 16), (33, 4, 64),
])
def test_host_pipeline_group_count(lib, B, H_kv, n_groups):
    per = _groups_per_batch(B, H_kv, n_groups)
    assert lib.lib.attn_fwd_host_groups(B, H_kv, n_groups) == (B * per if per > 0 else -1)


def test_host_pipeline_invalid_sizes(lib):
    assert lib.lib.attn_fwd_host_groups(0, 4, 0) == -1
    assert lib.lib.attn_fwd_host_groups(2, 0, 0) == -1
