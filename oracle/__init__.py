"""CPU oracle for the attention forward (fp64): test infrastructure, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline and reference legs)
may import this package. The CUDA library never links, loads or calls it, and it shares no code with
the CUDA path; the two meet only in the seeded inputs of ``exact_tiled_attention_50_b300.inputs``.

``attn_oracle.c`` is the plain definition (full N x N score matrix per head, fp64) plus a row-sampled
evaluator of the same definition and a tiled restatement of the online-softmax recurrence;
``attn_oracle_np.py`` is an independent NumPy restatement for small cases, the merge of results over
disjoint key sets (split-KV), and the backward pass (dQ, dK, dV) of the same attention, whole or at
selected rows and keys (for sequences too long for the whole matrices).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, OpenMP, no fast-math) into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ci, cd = ctypes.c_int, ctypes.c_double
        lib.oracle_attn_f64.argtypes = [f32p, f32p, f32p, f64p, f64p, f64p, ci, ci, ci, ci, ci, cd, ci, i32p]
        lib.oracle_attn_rows_f64.argtypes = [f32p, f32p, f32p, i64p, ci, f64p, f64p, ci, ci, ci, ci, ci, cd, ci, i32p]
        lib.oracle_attn_tiled_f64.argtypes = [f32p, f32p, f32p, f64p, f64p, ci, ci, ci, ci, ci, cd, ci, i32p, ci, ci]
        for fn in (lib.oracle_attn_f64, lib.oracle_attn_rows_f64, lib.oracle_attn_tiled_f64):
            fn.restype = ci
        lib.oracle_num_threads.restype = ci
        lib.oracle_set_num_threads.argtypes = [ci]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    """Exact fp32 copy of the input values (bf16 and fp32 values are representable in fp32)."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach().to("cpu", torch.float32).numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _lens(kv_len, B):
    if kv_len is None:
        return None
    if hasattr(kv_len, "detach"):
        kv_len = kv_len.detach().cpu().numpy()
    a = np.ascontiguousarray(np.asarray(kv_len).reshape(B), dtype=np.int32)
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the following C-oracle calls (all host cores by default)."""
    _load().oracle_set_num_threads(int(n))


def attention(q, k, v, scale, causal=False, kv_len=None, return_p=False):
    """Full oracle. q [B,H,N,d], k/v [B,H_kv,N,d]. Returns fp64 O [B,H,N,d], LSE [B,H,N] (and P)."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    O = np.empty((B, H, N, d), np.float64)
    LSE = np.empty((B, H, N), np.float64)
    P = np.empty((B, H, N, N), np.float64) if return_p else None
    lens = _lens(kv_len, B)
    rc = lib.oracle_attn_f64(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                             _ptr(O, ctypes.c_double), _ptr(LSE, ctypes.c_double),
                             _ptr(P, ctypes.c_double) if return_p else None,
                             B, H, H_kv, N, d, float(scale), int(bool(causal)),
                             _ptr(lens, ctypes.c_int32) if lens is not None else None)
    if rc != 0:
        raise ValueError(f"oracle_attn_f64 failed with code {rc}")
    return (O, LSE, P) if return_p else (O, LSE)


def attention_rows(q, k, v, scale, rows, causal=False, kv_len=None):
    """Row-sampled oracle: rows are flat indices (b*H + h)*N + i. Returns O [R,d], LSE [R]."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = rows.shape[0]
    O = np.empty((R, d), np.float64)
    LSE = np.empty((R,), np.float64)
    lens = _lens(kv_len, B)
    rc = lib.oracle_attn_rows_f64(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                                  _ptr(rows, ctypes.c_int64), R, _ptr(O, ctypes.c_double),
                                  _ptr(LSE, ctypes.c_double), B, H, H_kv, N, d, float(scale),
                                  int(bool(causal)), _ptr(lens, ctypes.c_int32) if lens is not None else None)
    if rc != 0:
        raise ValueError(f"oracle_attn_rows_f64 failed with code {rc}")
    return O, LSE


def attention_tiled(q, k, v, scale, causal=False, kv_len=None, Br=16, Bc=16):
    """Tiled online-softmax restatement (fp64); used only to show it equals the full oracle."""
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    O = np.empty((B, H, N, d), np.float64)
    LSE = np.empty((B, H, N), np.float64)
    lens = _lens(kv_len, B)
    rc = lib.oracle_attn_tiled_f64(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float), _ptr(v, ctypes.c_float),
                                   _ptr(O, ctypes.c_double), _ptr(LSE, ctypes.c_double), B, H, H_kv, N, d,
                                   float(scale), int(bool(causal)),
                                   _ptr(lens, ctypes.c_int32) if lens is not None else None, int(Br), int(Bc))
    if rc != 0:
        raise ValueError(f"oracle_attn_tiled_f64 failed with code {rc}")
    return O, LSE


from .attn_oracle_np import (attention_bias_dropout_np, attention_bwd_np, attention_bwd_sampled_np,  # noqa: E402
                             attention_fp8_np,
                             attention_np, dropout_keep_mask, dropout_threshold, e4m3_round, fwht_f32, merge_np,
                             philox4x32_10, quantize_e4m3_tiles, tile_exponent)
