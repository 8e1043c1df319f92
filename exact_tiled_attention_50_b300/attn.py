"""Python binding of libattn.so (argument marshalling only; every step runs in the CUDA kernels).

Importing this module loads the in-tree ``libattn.so`` and raises if it is missing: there is no
fallback implementation. Tensors are torch CUDA tensors (torch provides device memory and streams).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
ATTN_F32, ATTN_BF16 = 0, 1

EXPORTED = ("attn_fwd", "attn_check", "attn_status_string", "attn_workspace_bytes", "attn_launches_per_call",
            "attn_debug_set_wait_limit_ns", "attn_debug_set_skip_kv_load", "attn_set_kernel_events",
            "attn_event_elapsed_ms", "attn_fwd_noalloc", "attn_debug_schedule",
            "attn_debug_last_error_bits", "attn_merge", "attn_bwd", "attn_bwd_workspace_bytes", "attn_fwd_fp8",
            "attn_fwd_fp8_workspace_bytes", "attn_fwd_ex", "attn_debug_set_plan_mode", "attn_fwd_host",
            "attn_fwd_host_groups")


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m exact_tiled_attention_50_b300.build` "
                          "(there is no CPU or PyTorch fallback)")
    lib = ctypes.CDLL(path)
    vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci, ci, vp, sz, vp]
    lib.attn_fwd.restype = ci
    lib.attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci, ci, vp]
    lib.attn_fwd_noalloc.restype = ci
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, ci, ci,
                                  vp, vp, vp, vp, vp, vp, vp, sz, ci, vp]
    lib.attn_fwd_host.restype = ci
    lib.attn_fwd_host_groups.argtypes = [ci, ci, ci]
    lib.attn_fwd_host_groups.restype = ci
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, vp, sz, vp]
    lib.attn_bwd.restype = ci
    ll = ctypes.c_longlong
    lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, vp, ll, ll, ll, cf,
                                ctypes.c_uint64, ctypes.c_uint32, vp, sz, vp]
    lib.attn_fwd_ex.restype = ci
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, vp, vp, vp, sz, vp]
    lib.attn_fwd_fp8.restype = ci
    lib.attn_fwd_fp8_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
    lib.attn_fwd_fp8_workspace_bytes.restype = sz
    lib.attn_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_merge.argtypes = [vp, vp, ci, ctypes.c_longlong, ci, vp, vp, vp]
    lib.attn_merge.restype = ci
    lib.attn_check.argtypes = [vp]
    lib.attn_check.restype = ci
    lib.attn_status_string.argtypes = [ci]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
    lib.attn_workspace_bytes.restype = sz
    lib.attn_launches_per_call.argtypes = [ci]
    lib.attn_launches_per_call.restype = ci
    lib.attn_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.attn_debug_set_wait_limit_ns.restype = None
    lib.attn_debug_set_skip_kv_load.argtypes = [ci]
    lib.attn_debug_set_skip_kv_load.restype = None
    lib.attn_debug_set_plan_mode.argtypes = [ci]
    lib.attn_debug_set_plan_mode.restype = None
    lib.attn_set_kernel_events.argtypes = [vp, vp]
    lib.attn_set_kernel_events.restype = None
    lib.attn_debug_last_error_bits.argtypes = []
    lib.attn_debug_last_error_bits.restype = ctypes.c_uint32
    lib.attn_debug_schedule.argtypes = [ci, ci, ci, ci, vp, ci, vp, ci]
    lib.attn_debug_schedule.restype = ci
    lib.attn_event_elapsed_ms.argtypes = [vp, vp]
    lib.attn_event_elapsed_ms.restype = ctypes.c_float
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.attn_status_string(int(code)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return ATTN_F32
    if t == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t}")


def workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int, in_dtype: torch.dtype) -> int:
    return int(lib.attn_workspace_bytes(B, H, H_kv, N, d, _dtype_code(in_dtype)))


_ws_cache: dict = {}


def _workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """A cached device workspace per (device, stream); torch allocations are 256-byte aligned."""
    key = (device, torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: Optional[float] = None,
             causal: bool = False, kv_len: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.float32,
             workspace: Optional[torch.Tensor] = None, want_lse: bool = True):
    """O, LSE = softmax(scale q k^T) v on the current CUDA stream.

    q [B,H,N,d], k/v [B,H_kv,N,d] (bf16 or fp32, contiguous, on one CUDA device); kv_len int32 [B]
    on the device or None. Returns (O [B,H,N,d] in out_dtype, LSE [B,H,N] fp32 or None).
    """
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if k.shape != (B, H_kv, N, d) or v.shape != (B, H_kv, N, d):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    ws_bytes = workspace_bytes(B, H, H_kv, N, d, q.dtype)
    if workspace is None and ws_bytes > 0:
        workspace = _workspace(ws_bytes, q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                      lse.data_ptr() if lse is not None else None, B, H, H_kv, N, d, float(scale), int(bool(causal)),
                      kv_len.data_ptr() if kv_len is not None else None, _dtype_code(q.dtype), _dtype_code(out.dtype),
                      workspace.data_ptr() if workspace is not None else None,
                      workspace.numel() * workspace.element_size() if workspace is not None else 0, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_fwd_ex(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: Optional[float] = None,
                causal: bool = False, kv_len: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                dropout_p: float = 0.0, seed: int = 0, offset: int = 0, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """O, LSE of the attention with an additive bias and dropout (bf16 q, k, v; fp32 O, LSE).

    bias: bf16 CUDA tensor broadcastable to [B, H, N, N] whose last dimension is contiguous; broadcast
    dimensions are passed as zero strides (no copy). The library needs 16-byte aligned rows: strides
    that are multiples of 8 elements (pad the last dimension when N is not). dropout_p, seed, offset:
    the dropout probability and the generator's key and counter word (see attn_fwd_ex in attn.h)."""
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise TypeError("attn_fwd_ex takes bf16 q, k, v")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    strides = (0, 0, 0)
    if bias is not None:
        if bias.dtype != torch.bfloat16 or not bias.is_cuda:
            raise TypeError("bias must be a bf16 CUDA tensor")
        bias = bias.expand(B, H, N, N)
        if bias.stride(3) != 1:
            raise ValueError("the bias's last dimension must be contiguous")
        strides = (bias.stride(0), bias.stride(1), bias.stride(2))
    nbytes = workspace_bytes(B, H, H_kv, N, d, q.dtype)
    if workspace is None:
        workspace = _workspace(max(nbytes, 256), q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, H_kv, N, d,
                         float(scale), int(bool(causal)), kv_len.data_ptr() if kv_len is not None else None,
                         bias.data_ptr() if bias is not None else None, *strides, float(dropout_p),
                         int(seed) & 0xFFFFFFFFFFFFFFFF, int(offset) & 0xFFFFFFFF, workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_ex")
    return out, lse


def attn_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: Optional[float] = None,
                 causal: bool = False, kv_len: Optional[torch.Tensor] = None, signs: Optional[torch.Tensor] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None):
    """O, LSE of the fp8 path (E4M3 tensor cores; Q, K rotated by the random signs `signs` (int8 [d],
    +-1, on the device) or not rotated when None). q, k, v bf16 CUDA tensors, d = 128; O, LSE fp32."""
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise TypeError("attn_fwd_fp8 takes bf16 q, k, v")
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    if signs is not None:
        signs = signs.to(device=q.device, dtype=torch.int8).contiguous()
    nbytes = int(lib.attn_fwd_fp8_workspace_bytes(B, H, H_kv, N, d))
    if workspace is None:
        workspace = _workspace(max(nbytes, 256), q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, H_kv, N, d,
                          float(scale), int(bool(causal)), kv_len.data_ptr() if kv_len is not None else None,
                          signs.data_ptr() if signs is not None else None, workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_fp8")
    return out, lse


def attn_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor],
                     *, scale: Optional[float] = None, causal: bool = False,
                     kv_len: Optional[torch.Tensor] = None) -> None:
    """attn_fwd through the entry point that allocates nothing: the library's fixed device scratch
    replaces the workspace. q, k, v, out, lse (and kv_len) must already be contiguous CUDA tensors of
    the shapes attn_fwd takes; this wrapper creates no tensor either, so it rejects (ValueError or
    TypeError) what attn_fwd would have copied or converted instead of calling the library."""
    tensors = {"q": q, "k": k, "v": v, "out": out, "lse": lse, "kv_len": kv_len}
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda or t.device != q.device:
            raise ValueError(f"{name} must be a CUDA tensor on {q.device}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (this entry point makes no copies)")
    if q.dim() != 4:
        raise ValueError(f"q must be [B, H, N, d], got {tuple(q.shape)}")
    B, H, N, d = q.shape
    H_kv = k.shape[1] if k.dim() == 4 else -1
    if k.shape != (B, H_kv, N, d) or v.shape != (B, H_kv, N, d):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    _dtype_code(q.dtype)
    if out.shape != (B, H, N, d):
        raise ValueError(f"out must be [B, H, N, d] = {(B, H, N, d)}, got {tuple(out.shape)}")
    _dtype_code(out.dtype)
    if lse is not None and (lse.shape != (B, H, N) or lse.dtype != torch.float32):
        raise ValueError(f"lse must be fp32 [B, H, N] = {(B, H, N)}")
    if kv_len is not None and (kv_len.dtype != torch.int32 or kv_len.numel() != B):
        raise ValueError("kv_len must be an int32 tensor of B elements")
    if scale is None:
        scale = d ** -0.5
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr() if lse is not None else None, B, H, H_kv, N, d, float(scale),
                              int(bool(causal)), kv_len.data_ptr() if kv_len is not None else None,
                              _dtype_code(q.dtype), _dtype_code(out.dtype), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_noalloc")


def attn_fwd_host(q_h: torch.Tensor, k_h: torch.Tensor, v_h: torch.Tensor, o_h: torch.Tensor,
                  lse_h: Optional[torch.Tensor], q_d: torch.Tensor, k_d: torch.Tensor, v_d: torch.Tensor,
                  o_d: torch.Tensor, lse_d: Optional[torch.Tensor], *, scale: Optional[float] = None,
                  causal: bool = False, kv_len_h: Optional[torch.Tensor] = None,
                  kv_len_d: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  n_groups: int = 0) -> None:
    """attn_fwd with host inputs and outputs, copies and compute pipelined over groups of heads.

    q_h, k_h, v_h, o_h, lse_h (and kv_len_h): contiguous CPU tensors (pinned for overlap) of the shapes
    and dtypes attn_fwd takes and returns; q_d .. lse_d (and kv_len_d): contiguous CUDA tensors of the
    same shapes. On return the work is enqueued on the current stream; o_h and lse_h hold the result
    once that stream reaches this point."""
    for name, t in (("q_h", q_h), ("k_h", k_h), ("v_h", v_h), ("o_h", o_h)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    for name, t in (("q_d", q_d), ("k_d", k_d), ("v_d", v_d), ("o_d", o_d)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    B, H, N, d = q_h.shape
    H_kv = k_h.shape[1]
    if q_d.shape != q_h.shape or k_d.shape != k_h.shape or v_d.shape != v_h.shape or o_d.shape != o_h.shape:
        raise ValueError("host and device tensors differ in shape")
    if (lse_h is None) != (lse_d is None) or (kv_len_h is None) != (kv_len_d is None):
        raise ValueError("give lse (and kv_len) on both sides or on neither")
    if scale is None:
        scale = d ** -0.5
    ws_bytes = workspace_bytes(B, H, H_kv, N, d, q_h.dtype)
    if workspace is None and ws_bytes > 0:
        workspace = _workspace(ws_bytes, q_d.device)
    stream = torch.cuda.current_stream(q_d.device).cuda_stream
    ptr = (lambda t: t.data_ptr() if t is not None else None)
    rc = lib.attn_fwd_host(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(), ptr(lse_h), B, H, H_kv, N,
                           d, float(scale), int(bool(causal)), ptr(kv_len_h), _dtype_code(q_h.dtype),
                           _dtype_code(o_h.dtype), q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(), o_d.data_ptr(),
                           ptr(lse_d), ptr(kv_len_d), ptr(workspace),
                           workspace.numel() * workspace.element_size() if workspace is not None else 0,
                           int(n_groups), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, do: torch.Tensor,
             lse: torch.Tensor, *, scale: Optional[float] = None, causal: bool = False,
             kv_len: Optional[torch.Tensor] = None):
    """Gradients (dQ, dK, dV, fp32) of attn_fwd's output for upstream gradient do; q, k, v, do bf16,
    o and lse the fp32 outputs of attn_fwd on the same inputs."""
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if not (q.dtype == k.dtype == v.dtype == do.dtype == torch.bfloat16):
        raise TypeError("attn_bwd takes bf16 q, k, v, do")
    if o.dtype != torch.float32 or lse.dtype != torch.float32:
        raise TypeError("attn_bwd takes the fp32 O and LSE of attn_fwd")
    q, k, v, o, do, lse = (t.contiguous() for t in (q, k, v, o, do, lse))
    if scale is None:
        scale = d ** -0.5
    if kv_len is not None:
        kv_len = kv_len.to(device=q.device, dtype=torch.int32).contiguous()
    dq = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    dk = torch.empty((B, H_kv, N, d), dtype=torch.float32, device=q.device)
    dv = torch.empty((B, H_kv, N, d), dtype=torch.float32, device=q.device)
    nbytes = int(lib.attn_bwd_workspace_bytes(B, H, N, d))
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H_kv, N, d, float(scale), int(bool(causal)),
                      kv_len.data_ptr() if kv_len is not None else None, ws.data_ptr(), nbytes, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def merge(o_parts: torch.Tensor, lse_parts: torch.Tensor):
    """Merge attention results over disjoint key sets: o_parts [P, ..., d] fp32, lse_parts [P, ...] fp32
    (CUDA, contiguous) -> (O [..., d], LSE [...])."""
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise TypeError("merge takes fp32 parts")
    o_parts, lse_parts = o_parts.contiguous(), lse_parts.contiguous()
    P, d = o_parts.shape[0], o_parts.shape[-1]
    rows = lse_parts[0].numel()
    if o_parts[0].numel() != rows * d or lse_parts.shape[0] != P:
        raise ValueError("shape mismatch between o_parts and lse_parts")
    out = torch.empty(o_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    stream = torch.cuda.current_stream(o_parts.device).cuda_stream
    rc = lib.attn_merge(o_parts.data_ptr(), lse_parts.data_ptr(), P, rows, d, out.data_ptr(), lse.data_ptr(), stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_merge")
    return out, lse


def schedule(B: int, H: int, N: int, causal: bool, kv_len=None, sms: int = 148):
    """The persistent kernel's work schedule for these sizes (host computation, no GPU): a list of
    (cta, b, h, pair, k0, k1, cost, kind) tuples in each CTA's run order."""
    import numpy as np
    kv = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, dtype=np.int32).reshape(B))
    kv_ptr = kv.ctypes.data if kv is not None else None
    n = lib.attn_debug_schedule(B, H, N, int(bool(causal)), kv_ptr, sms, None, 0)
    if n < 0:
        raise ValueError("invalid schedule arguments")
    out = np.zeros((max(n, 1), 8), dtype=np.int32)
    lib.attn_debug_schedule(B, H, N, int(bool(causal)), kv_ptr, sms, out.ctypes.data, n)
    return [tuple(int(v) for v in row) for row in out[:n]]


def check(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return (and clear) the device error status (ATTN_OK on success)."""
    s = (stream or torch.cuda.current_stream()).cuda_stream
    return int(lib.attn_check(s))


def launches_per_call(in_dtype: torch.dtype) -> int:
    return int(lib.attn_launches_per_call(_dtype_code(in_dtype)))


def set_kernel_events(start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]) -> None:
    """Record ``start``/``stop`` around the main attention kernel of every following call (None: off)."""
    if start is None or stop is None:
        lib.attn_set_kernel_events(None, None)
    else:
        lib.attn_set_kernel_events(start.cuda_event, stop.cuda_event)


def event_elapsed_ms(start: torch.cuda.Event, stop: torch.cuda.Event) -> float:
    """Elapsed time between two events recorded by the library's timing hook."""
    ms = float(lib.attn_event_elapsed_ms(start.cuda_event, stop.cuda_event))
    if ms < 0:
        raise RuntimeError("cudaEventElapsedTime failed")
    return ms
