"""Thin ctypes binding over libattn.so (argument marshalling only).

Every step of the computation runs in the CUDA library; this module checks
tensor shapes, allocates outputs and workspaces with PyTorch (device memory
and streams are all PyTorch is used for) and passes raw device pointers and
the current CUDA stream to the C entry points of ``include/libattn.h``.

There is no fallback: if the library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libattn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "libattn.h")

F16, BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
          3: "workspace missing or too small", 4: "CUDA error", 5: "device wait timed out",
          6: "device-side data check failed"}

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "attn_version": ([], ctypes.c_char_p),
    "attn_status_str": ([_i], ctypes.c_char_p),
    "attn_fwd": ([_vp] * 5 + [_i] * 7 + [_f, _i, _i, _i, _f, _vp], _i),
    "attn_fwd_strided": ([_vp] * 5 + [ctypes.c_int64] * 3 + [_i] * 7 +
                         [_f, _i, _i, _i, _f, _i, _vp], _i),
    "attn_bwd_workspace_size": ([_i] * 7, _sz),
    "attn_bwd_strided": ([_vp] * 9 + [ctypes.c_int64] * 6 + [_i] * 7 +
                         [_f, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "attn_bwd": ([_vp] * 9 + [_i] * 7 + [_f, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "attn_fwd_varlen": ([_vp] * 7 + [_i] * 9 + [_f, _i, _i, _i, _f, _vp], _i),
    "attn_bwd_varlen_workspace_size": ([_i] * 9, _sz),
    "attn_bwd_varlen": ([_vp] * 11 + [_i] * 9 + [_f, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "attn_kvcache_num_splits": ([_i] * 7, _i),
    "attn_kvcache_workspace_size": ([_i] * 7, _sz),
    "attn_fwd_kvcache": ([_vp] * 7 + [_i] * 3 + [_vp, _vp] + [_i] * 7 +
                         [_f, _i, _i, _i, _f, _i, _vp, _sz, _vp], _i),
    "attn_fwd_kvcache_noalloc": ([_vp] * 7 + [_i] * 3 + [_vp, _vp] + [_i] * 7 +
                                 [_f, _i, _i, _i, _f, _i, _vp], _i),
    "attn_fwd_fp8_workspace_size": ([_i] * 4, _sz),
    "attn_fwd_fp8": ([_vp] * 5 + [_f] * 3 + [_i] * 6 + [_f, _i, _i, _i, _f, _vp, _sz, _vp], _i),
    "attn_fwd_probs": ([_vp] * 4 + [_i] * 7 + [_f, _i, _i, _i, _f, _vp], _i),
    "attn_kvcache_advance": ([_vp, _i, _i, _vp], _i),
    "attn_get_device_error": ([_vp, ctypes.POINTER(_i)], _i),
    "attn_launch_count": ([], ctypes.c_ulonglong),
    "attn_set_wait_limit_ns": ([ctypes.c_ulonglong], ctypes.c_ulonglong),
    "attn_set_test_stall": ([_i], _i),
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} (status {status})")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions include/libattn.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^(?:[a-z_0-9]+\s+)+\*?\s*(attn_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def lib() -> ctypes.CDLL:
    """Loads libattn.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libattn.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(l, name)
            fn.argtypes = args
            fn.restype = res
        _lib = l
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise AttnError(status, what)


def _torch():
    import torch

    return torch


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"dtype {t.dtype} is not fp16/bf16")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(*ts):
    for t in ts:
        if t is not None:
            _need(t.is_cuda, "tensors must be on a CUDA device")
            _need(t.is_contiguous(), "tensors must be contiguous (Inference Cookbook FAQ Q13)")


def _win(window):
    wl, wr = window
    return int(wl), int(wr)


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def _row_stride(t):
    """Token stride (elements) of a (b, s, h, d) tensor whose heads are dense
    within a token: 0 when fully contiguous, the stride when it is a view of a
    packed layout (e.g. qkv[:, :, 0] of a (b, s, 3, h, d) tensor)."""
    if t is None or t.is_contiguous():
        return 0
    b, s, h, d = t.shape
    _need(t.is_cuda, "tensors must be on a CUDA device")
    _need(t.stride(3) == 1 and t.stride(2) == d and (b == 1 or t.stride(0) == s * t.stride(1)),
          "a non-contiguous q/k/v must be a token-strided view with dense heads "
          "(e.g. of a packed (b, s, 3, h, d) tensor)")
    return t.stride(1)


def fwd(q, k, v, *, scale=None, causal=False, window=(-1, -1), softcap=0.0, out=None, lse=None,
        pack_gqa=None):
    """Dense forward.  q (b,sq,hq,d), k/v (b,sk,hkv,d) -> out (b,sq,hq,d), lse (b,hq,sq) fp32.
    q/k/v may be token-strided views of packed qkv / kv tensors (no copies).
    pack_gqa: None = automatic, False/True = off/on (Inference Cookbook FAQ Q15)."""
    torch = _torch()
    b, sq, hq, d = q.shape
    _, sk, hkv, _ = k.shape
    _need(k.shape == v.shape and k.shape[0] == b and k.shape[3] == d, "k/v shape mismatch")
    _need(q.dtype == k.dtype == v.dtype, "q, k, v must share a dtype")
    out = torch.empty_like(q, memory_format=torch.contiguous_format) if out is None else out
    lse = torch.empty((b, hq, sq), device=q.device, dtype=torch.float32) if lse is None else lse
    rs = [_row_stride(t) for t in (q, k, v)]
    _cuda_contig(out, lse)
    wl, wr = _win(window)
    args = (_dt(q), b, sq, sk, hq, hkv, d, _scale(scale, d), int(bool(causal)), wl, wr,
            float(softcap), _stream())
    if any(rs) or pack_gqa is not None:
        pk = -1 if pack_gqa is None else int(bool(pack_gqa))
        st = lib().attn_fwd_strided(_p(q), _p(k), _p(v), _p(out), _p(lse), *rs, *args[:-1], pk,
                                    args[-1])
    else:
        _cuda_contig(q, k, v)
        st = lib().attn_fwd(_p(q), _p(k), _p(v), _p(out), _p(lse), *args)
    _check(st, "attn_fwd")
    return out, lse


def fwd_qkvpacked(qkv, **kw):
    """Forward on a packed (b, s, 3, h, d) tensor ("flash_attn FlashAttention
    完整说明" §六.1's qkvpacked call), read in place."""
    return fwd(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], **kw)


def fwd_kvpacked(q, kv, **kw):
    """Forward with a packed (b, sk, 2, hkv, d) key/value tensor (Inference
    Cookbook FAQ Q7's kvpacked call), read in place."""
    return fwd(q, kv[:, :, 0], kv[:, :, 1], **kw)


def bwd_workspace(q, k, deterministic=False):
    torch = _torch()
    b, sq, hq, d = q.shape
    n = lib().attn_bwd_workspace_size(b, sq, k.shape[1], hq, k.shape[2], d, int(bool(deterministic)))
    return torch.empty(max(n, 1), device=q.device, dtype=torch.uint8)


def bwd(q, k, v, out, lse, dout, *, scale=None, causal=False, window=(-1, -1), softcap=0.0,
        deterministic=False, workspace=None, dq=None, dk=None, dv=None):
    """Dense backward -> dq, dk, dv (same shapes and dtype as q, k, v)."""
    torch = _torch()
    b, sq, hq, d = q.shape
    _, sk, hkv, _ = k.shape
    cf = torch.contiguous_format
    dq = torch.empty_like(q, memory_format=cf) if dq is None else dq
    dk = torch.empty_like(k, memory_format=cf) if dk is None else dk
    dv = torch.empty_like(v, memory_format=cf) if dv is None else dv
    ws = bwd_workspace(q, k, deterministic) if workspace is None else workspace
    rs = [_row_stride(t) for t in (q, k, v, dq, dk, dv)]
    _cuda_contig(out, lse, dout, ws)
    wl, wr = _win(window)
    ptrs = (_p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv))
    args = (_dt(q), b, sq, sk, hq, hkv, d, _scale(scale, d), int(bool(causal)), wl, wr,
            float(softcap), int(bool(deterministic)), _p(ws), ws.numel(), _stream())
    if any(rs):
        st = lib().attn_bwd_strided(*ptrs, *rs, *args)
    else:
        _cuda_contig(q, k, v, dq, dk, dv)
        st = lib().attn_bwd(*ptrs, *args)
    _check(st, "attn_bwd")
    return dq, dk, dv


def bwd_qkvpacked(qkv, out, lse, dout, *, dqkv=None, **kw):
    """Backward of fwd_qkvpacked: the gradients land in a packed (b, s, 3, h, d)
    tensor ``dqkv`` (allocated if not given) with no copies."""
    torch = _torch()
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    bwd(qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2], out, lse, dout,
        dq=dqkv[:, :, 0], dk=dqkv[:, :, 1], dv=dqkv[:, :, 2], **kw)
    return dqkv


def fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *, scale=None,
               causal=False, window=(-1, -1), softcap=0.0, out=None, lse=None):
    """Packed forward.  q (Tq,hq,d), k/v (Tk,hkv,d) -> out (Tq,hq,d), lse (hq,Tq)."""
    torch = _torch()
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    _need(cu_seqlens_q.dtype == torch.int32 and cu_seqlens_k.dtype == torch.int32,
          "cu_seqlens must be int32")
    _need(cu_seqlens_k.numel() == batch + 1, "cu_seqlens_q/k length mismatch")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((hq, tq), device=q.device, dtype=torch.float32) if lse is None else lse
    _cuda_contig(q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k)
    wl, wr = _win(window)
    st = lib().attn_fwd_varlen(_p(q), _p(k), _p(v), _p(out), _p(lse), _p(cu_seqlens_q),
                               _p(cu_seqlens_k), batch, int(max_seqlen_q), int(max_seqlen_k), tq,
                               tk, _dt(q), hq, hkv, d, _scale(scale, d), int(bool(causal)), wl,
                               wr, float(softcap), _stream())
    _check(st, "attn_fwd_varlen")
    return out, lse


def bwd_varlen(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
               *, scale=None, causal=False, window=(-1, -1), softcap=0.0, deterministic=False,
               workspace=None):
    torch = _torch()
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        n = lib().attn_bwd_varlen_workspace_size(batch, int(max_seqlen_q), int(max_seqlen_k), tq,
                                                 tk, hq, hkv, d, int(bool(deterministic)))
        workspace = torch.empty(max(n, 1), device=q.device, dtype=torch.uint8)
    _cuda_contig(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_k, workspace)
    wl, wr = _win(window)
    st = lib().attn_bwd_varlen(_p(q), _p(k), _p(v), _p(out), _p(lse), _p(dout), _p(dq), _p(dk),
                               _p(dv), _p(cu_seqlens_q), _p(cu_seqlens_k), batch,
                               int(max_seqlen_q), int(max_seqlen_k), tq, tk, _dt(q), hq, hkv, d,
                               _scale(scale, d), int(bool(causal)), wl, wr, float(softcap),
                               int(bool(deterministic)), _p(workspace), workspace.numel(),
                               _stream())
    _check(st, "attn_bwd_varlen")
    return dq, dk, dv


def kvcache_workspace(q, k_cache, page_size, max_pages_per_seq, num_splits=0):
    torch = _torch()
    b, sq, hq, d = q.shape
    hkv = k_cache.shape[2]
    n = lib().attn_kvcache_workspace_size(b, sq, hq, hkv, d, page_size * max_pages_per_seq,
                                          int(num_splits))
    return torch.empty(max(n, 1), device=q.device, dtype=torch.uint8)


def fwd_kvcache(q, k_cache, v_cache, cache_seqlens, *, k_new=None, v_new=None, block_table=None,
                scale=None, causal=False, window=(-1, -1), softcap=0.0, num_splits=0,
                workspace=None, out=None, lse=None):
    """Decode against a (paged) KV cache, appending k_new/v_new (Inference
    Cookbook FAQ Q17/Q18).  Does not modify cache_seqlens."""
    torch = _torch()
    b, sq, hq, d = q.shape
    if block_table is not None:
        num_pages, page_size, hkv, _ = k_cache.shape
        max_pages = block_table.shape[1]
        _need(block_table.dtype == torch.int32, "block_table must be int32")
    else:
        num_pages, page_size, hkv, _ = k_cache.shape
        max_pages = 1
    s_new = 0 if k_new is None else k_new.shape[1]
    _need(cache_seqlens.dtype == torch.int32, "cache_seqlens must be int32")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((b, hq, sq), device=q.device, dtype=torch.float32) if lse is None else lse
    ws = kvcache_workspace(q, k_cache, page_size, max_pages, num_splits) if workspace is None \
        else workspace
    _cuda_contig(q, k_cache, v_cache, k_new, v_new, cache_seqlens, block_table, out, lse, ws)
    wl, wr = _win(window)
    st = lib().attn_fwd_kvcache(_p(q), _p(k_cache), _p(v_cache), _p(k_new), _p(v_new),
                                _p(cache_seqlens), _p(block_table), num_pages, page_size,
                                max_pages, _p(out), _p(lse), _dt(q), b, sq, s_new, hq, hkv, d,
                                _scale(scale, d), int(bool(causal)), wl, wr, float(softcap),
                                int(num_splits), _p(ws), ws.numel(), _stream())
    _check(st, "attn_fwd_kvcache")
    return out, lse


def num_splits(b, sq, hq, hkv, d, max_seqlen_k, requested=0) -> int:
    return lib().attn_kvcache_num_splits(b, sq, hq, hkv, d, max_seqlen_k, requested)


def launch_count() -> int:
    """Kernels the library has enqueued since it was loaded."""
    return int(lib().attn_launch_count())


def set_wait_limit_ns(ns: int) -> int:
    """Wall-clock limit of each device-side wait for the calls that follow
    (0 = the default 2 s); returns the previous limit.  For error-path tests."""
    return int(lib().attn_set_wait_limit_ns(int(ns)))


def set_test_stall(on: bool) -> bool:
    """Test hook: while on, the tensor-core kernels' first wait can only run
    out (see attn_set_test_stall); returns the previous setting."""
    return bool(lib().attn_set_test_stall(int(bool(on))))


def device_error() -> tuple[int, int]:
    """(status, raw error word) of the sticky device error word; clears it."""
    detail = ctypes.c_int(0)
    st = lib().attn_get_device_error(_stream(), ctypes.byref(detail))
    return st, detail.value


def fwd_probs(q, k, lse, *, scale=None, causal=False, window=(-1, -1), softcap=0.0, out=None):
    """Debug only (Inference Cookbook FAQ Q9): the (b,hq,sq,sk) fp32 attention
    probabilities of the forward that produced ``lse`` -- O(N^2) memory."""
    torch = _torch()
    b, sq, hq, d = q.shape
    _, sk, hkv, _ = k.shape
    _need(k.shape[0] == b and k.shape[3] == d, "k shape mismatch")
    _need(q.dtype == k.dtype, "q, k must share a dtype")
    _need(tuple(lse.shape) == (b, hq, sq) and lse.dtype == torch.float32, "lse must be (b,hq,sq) fp32")
    out = torch.empty((b, hq, sq, sk), device=q.device, dtype=torch.float32) if out is None else out
    _cuda_contig(q, k, lse, out)
    wl, wr = _win(window)
    st = lib().attn_fwd_probs(_p(q), _p(k), _p(lse), _p(out), _dt(q), b, sq, sk, hq, hkv, d,
                              _scale(scale, d), int(bool(causal)), wl, wr, float(softcap),
                              _stream())
    _check(st, "attn_fwd_probs")
    return out


def kvcache_advance(cache_seqlens, s_new: int):
    """cache_seqlens += s_new on the current stream (Inference Cookbook FAQ
    Q17), as a kernel so a decode step can be captured in a CUDA graph (FAQ Q19)."""
    torch = _torch()
    _need(cache_seqlens.dtype == torch.int32, "cache_seqlens must be int32")
    _cuda_contig(cache_seqlens)
    st = lib().attn_kvcache_advance(_p(cache_seqlens), cache_seqlens.numel(), int(s_new), _stream())
    _check(st, "attn_kvcache_advance")


def fwd_fp8(q, k, v, descale_q=1.0, descale_k=1.0, descale_v=1.0, *, scale=None, causal=False,
            window=(-1, -1), softcap=0.0, out=None, lse=None, workspace=None):
    """FP8 forward (Inference Cookbook FAQ Q20): q, k, v are float8_e4m3fn (or
    uint8 E4M3 bytes) standing for q*descale_q etc.; returns bf16 out and fp32 lse."""
    torch = _torch()
    b, sq, hq, d = q.shape
    _, sk, hkv, _ = k.shape
    _need(k.shape == v.shape and k.shape[0] == b and k.shape[3] == d, "k/v shape mismatch")
    for t in (q, k, v):
        _need(t.element_size() == 1, "q, k, v must be 1-byte E4M3 tensors")
    out = torch.empty((b, sq, hq, d), device=q.device, dtype=torch.bfloat16) if out is None else out
    lse = torch.empty((b, hq, sq), device=q.device, dtype=torch.float32) if lse is None else lse
    if workspace is None:
        n = lib().attn_fwd_fp8_workspace_size(b, sk, hkv, d)
        workspace = torch.empty(max(n, 1), device=q.device, dtype=torch.uint8)
    _cuda_contig(q, k, v, out, lse, workspace)
    wl, wr = _win(window)
    st = lib().attn_fwd_fp8(_p(q), _p(k), _p(v), _p(out), _p(lse), float(descale_q),
                            float(descale_k), float(descale_v), b, sq, sk, hq, hkv, d,
                            _scale(scale, d), int(bool(causal)), wl, wr, float(softcap),
                            _p(workspace), workspace.numel(), _stream())
    _check(st, "attn_fwd_fp8")
    return out, lse
