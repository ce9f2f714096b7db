"""PyTorch-facing wrappers of the C ABI (argument marshalling only).

Every function checks dtypes, devices, shapes and contiguity, allocates the
outputs with torch (PyTorch is the device-memory and stream provider here),
and calls the matching ``fa_*`` entry point on the current CUDA stream.  All
arithmetic happens in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import functools
import math
from typing import Optional, Tuple

import torch

from . import _lib

_lib_handle = None


def lib():
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _lib.load()
    return _lib_handle


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _on_tensor_device(fn):
    """Runs a wrapper with the CUDA device of its tensors current (the library
    launches on the current device); tensors on two devices are refused."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        tensors = [a for a in list(args) + list(kwargs.values()) if isinstance(a, torch.Tensor) and a.is_cuda]
        if not tensors:
            return fn(*args, **kwargs)
        dev = tensors[0].device
        if any(t.device != dev for t in tensors):
            raise ValueError("all CUDA tensors of a call must be on one device")
        with torch.cuda.device(dev):
            return fn(*args, **kwargs)
    return wrapper


def _check_bf16(name, t, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def set_option(opt: int, value: float) -> None:
    _lib.check(lib().fa_set_option(opt, float(value)), "fa_set_option")


def device_error() -> int:
    """Synchronises and returns the recorded device error code (0 = none)."""
    code = ctypes.c_uint(0)
    lib().fa_device_error(ctypes.byref(code))
    return int(code.value)


@_on_tensor_device
def fwd(q, k, v, causal: bool = False, scale: Optional[float] = None, out=None, lse=None,
        stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Dense forward.  q, k, v [B, N, H, d] bf16 -> (o [B, N, H, d], lse [B, H, N] fp32)."""
    _check_bf16("q", q)
    B, N, H, d = q.shape
    _check_bf16("k", k, q.shape)
    _check_bf16("v", v, q.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_bf16("out", o, q.shape)
    st = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, H, N, d, int(bool(causal)), scale,
                      _stream(stream))
    _lib.check(st, "fa_fwd")
    return o, l


@_on_tensor_device
def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None, workspace=None,
        stream=None, out=None):
    """Dense backward -> (dq, dk, dv), each [B, N, H, d] bf16 (written into
    ``out`` = (dq, dk, dv) when given)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_bf16(name, t, q.shape)
    B, N, H, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, N]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is not None:
        dq, dk, dv = out
        for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            _check_bf16(name, t, q.shape)
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = lib().fa_bwd_workspace_bytes(B, H, N, d)
    ws = workspace if workspace is not None else torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError("workspace too small")
    st = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                      _ptr(ws), B, H, N, d, int(bool(causal)), scale, _stream(stream))
    _lib.check(st, "fa_bwd")
    return dq, dk, dv


def _check_cu(cu_seqlens, q):
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor")
    if cu_seqlens.device != q.device:
        raise ValueError("cu_seqlens must be on the device of q")


@_on_tensor_device
def fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale: Optional[float] = None,
               stream=None):
    """Packed forward.  q, k, v [total, H, d]; cu_seqlens int32 [S+1] on the device.
    Returns (o [total, H, d], lse [H, total])."""
    _check_bf16("q", q)
    total, H, d = q.shape
    _check_bf16("k", k, q.shape)
    _check_bf16("v", v, q.shape)
    _check_cu(cu_seqlens, q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    l = torch.empty((H, total), dtype=torch.float32, device=q.device)
    st = lib().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                             int(max_seqlen), total, H, d, int(bool(causal)), scale, _stream(stream))
    _lib.check(st, "fa_fwd_varlen")
    return o, l


@_on_tensor_device
def bwd_varlen(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int, causal: bool = False,
               scale: Optional[float] = None, stream=None):
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_bf16(name, t, q.shape)
    total, H, d = q.shape
    _check_cu(cu_seqlens, q)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, total) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [H, total]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = lib().fa_bwd_varlen_workspace_bytes(total, H, d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(ws), _ptr(cu_seqlens), cu_seqlens.numel() - 1, int(max_seqlen), total,
                             H, d, int(bool(causal)), scale, _stream(stream))
    _lib.check(st, "fa_bwd_varlen")
    return dq, dk, dv


@_on_tensor_device
def decode(q, k_cache, v_cache, num_splits: int = 0, scale: Optional[float] = None, stream=None,
           workspace=None):
    """Single-token decode.  q [B, 1, H, d]; caches [B, L, H, d].
    Returns (o [B, 1, H, d], lse [B, H])."""
    _check_bf16("q", q)
    B, one, H, d = q.shape
    if one != 1:
        raise ValueError("q must be [B, 1, H, d]")
    _check_bf16("k_cache", k_cache)
    L = k_cache.shape[1]
    if tuple(k_cache.shape) != (B, L, H, d):
        raise ValueError("k_cache must be [B, L, H, d]")
    _check_bf16("v_cache", v_cache, k_cache.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    splits = num_splits if num_splits > 0 else lib().fa_decode_num_splits(B, H, L, d)
    nbytes = lib().fa_decode_workspace_bytes(B, H, d, max(splits, 1))
    ws = workspace if workspace is not None else torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    l = torch.empty((B, H), dtype=torch.float32, device=q.device)
    st = lib().fa_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(l), B, H, L, d, splits,
                                 _ptr(ws), scale, _stream(stream))
    _lib.check(st, "fa_decode_splitkv")
    return o, l


@_on_tensor_device
def decode_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len: int, num_splits: int = 0,
                 scale: Optional[float] = None, stream=None, workspace=None):
    """Single-token decode over a paged cache.  q [B, 1, H, d]; pages
    [num_pages, page_size, H, d]; block_table int32 [B, max_blocks] and
    seq_lens int32 [B] on the device.  Returns (o [B, 1, H, d], lse [B, H])."""
    _check_bf16("q", q)
    B, one, H, d = q.shape
    if one != 1:
        raise ValueError("q must be [B, 1, H, d]")
    _check_bf16("k_pages", k_pages)
    num_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    if tuple(k_pages.shape) != (num_pages, page_size, H, d):
        raise ValueError("k_pages must be [num_pages, page_size, H, d]")
    _check_bf16("v_pages", v_pages, k_pages.shape)
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_blocks] and seq_lens [B]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    splits = num_splits if num_splits > 0 else lib().fa_decode_num_splits(B, H, int(max_seq_len), d)
    nbytes = lib().fa_decode_workspace_bytes(B, H, d, max(splits, 1))
    ws = workspace if workspace is not None else torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    l = torch.empty((B, H), dtype=torch.float32, device=q.device)
    st = lib().fa_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), _ptr(o),
                               _ptr(l), B, H, d, page_size, num_pages, block_table.shape[1], int(max_seq_len), splits,
                               _ptr(ws), scale, _stream(stream))
    _lib.check(st, "fa_decode_paged")
    return o, l


# ---------------------------------------------------------------- grouped-query attention

@_on_tensor_device
def fwd_gqa(q, k, v, causal: bool = False, scale: Optional[float] = None, stream=None):
    """q [B, N, Hq, d]; k, v [B, N, Hkv, d] with Hkv dividing Hq.
    Returns (o [B, N, Hq, d], lse [B, Hq, N])."""
    _check_bf16("q", q)
    B, N, Hq, d = q.shape
    _check_bf16("k", k)
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, N, Hkv, d):
        raise ValueError("k must be [B, N, Hkv, d]")
    _check_bf16("v", v, k.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    l = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    st = lib().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, Hq, Hkv, N, d, int(bool(causal)), scale,
                          _stream(stream))
    _lib.check(st, "fa_fwd_gqa")
    return o, l


@_on_tensor_device
def bwd_gqa(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None, stream=None):
    """Gradients of fwd_gqa: (dq [B, N, Hq, d], dk, dv [B, N, Hkv, d])."""
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _check_bf16(name, t, q.shape)
    B, N, Hq, d = q.shape
    _check_bf16("k", k)
    Hkv = k.shape[2]
    _check_bf16("v", v, k.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = lib().fa_bwd_workspace_bytes(B, Hq, N, d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                          _ptr(ws), B, Hq, Hkv, N, d, int(bool(causal)), scale, _stream(stream))
    _lib.check(st, "fa_bwd_gqa")
    return dq, dk, dv


@_on_tensor_device
def decode_gqa(q, k_cache, v_cache, num_splits: int = 0, scale: Optional[float] = None, stream=None):
    """q [B, 1, Hq, d]; caches [B, L, Hkv, d].  Returns (o [B, 1, Hq, d], lse [B, Hq])."""
    _check_bf16("q", q)
    B, one, Hq, d = q.shape
    _check_bf16("k_cache", k_cache)
    L, Hkv = k_cache.shape[1], k_cache.shape[2]
    if one != 1 or tuple(k_cache.shape) != (B, L, Hkv, d):
        raise ValueError("q must be [B, 1, Hq, d] and the caches [B, L, Hkv, d]")
    _check_bf16("v_cache", v_cache, k_cache.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    splits = num_splits if num_splits > 0 else lib().fa_decode_num_splits(B, Hkv, L, d)
    nbytes = lib().fa_decode_workspace_bytes(B, Hq, d, max(splits, 1))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    l = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib().fa_decode_gqa(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(l), B, Hq, Hkv, L, d, splits,
                             _ptr(ws), scale, _stream(stream))
    _lib.check(st, "fa_decode_gqa")
    return o, l


# ---------------------------------------------------------------- masks: causal / sliding window, Nq != Nk

def _window(causal: bool, window: Optional[Tuple[int, int]]):
    """(window_left, window_right) of the C ABI; ``causal`` alone is (-1, 0)."""
    if window is None:
        return (-1, 0) if causal else (-1, -1)
    wl, wr = int(window[0]), int(window[1])
    if causal:
        wr = 0 if wr < 0 else min(wr, 0)
    return wl, wr


@_on_tensor_device
def fwd_masked(q, k, v, causal: bool = False, window: Optional[Tuple[int, int]] = None,
               scale: Optional[float] = None, stream=None):
    """q [B, Nq, Hq, d]; k, v [B, Nk, Hkv, d].  Bottom-right aligned mask:
    query i sees keys i + Nk - Nq - window[0] .. i + Nk - Nq + window[1]
    (-1 = open side; ``causal`` caps window[1] at 0).
    Returns (o [B, Nq, Hq, d], lse [B, Hq, Nq])."""
    _check_bf16("q", q)
    B, Nq, Hq, d = q.shape
    _check_bf16("k", k)
    Nk, Hkv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Nk, Hkv, d):
        raise ValueError("k must be [B, Nk, Hkv, d]")
    _check_bf16("v", v, k.shape)
    wl, wr = _window(causal, window)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    l = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    st = lib().fa_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), B, Hq, Hkv, Nq, Nk, d, wl, wr, scale,
                             _stream(stream))
    _lib.check(st, "fa_fwd_masked")
    return o, l


@_on_tensor_device
def bwd_masked(q, k, v, o, lse, dout, causal: bool = False, window: Optional[Tuple[int, int]] = None,
               scale: Optional[float] = None, stream=None):
    """Gradients of fwd_masked: (dq [B, Nq, Hq, d], dk, dv [B, Nk, Hkv, d])."""
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _check_bf16(name, t, q.shape)
    B, Nq, Hq, d = q.shape
    _check_bf16("k", k)
    Nk, Hkv = k.shape[1], k.shape[2]
    _check_bf16("v", v, k.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, Hq, Nq]")
    wl, wr = _window(causal, window)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = lib().fa_bwd_workspace_bytes(B, Hq, Nq, d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(ws), B, Hq, Hkv, Nq, Nk, d, wl, wr, scale, _stream(stream))
    _lib.check(st, "fa_bwd_masked")
    return dq, dk, dv


@_on_tensor_device
def fwd_masked_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                      causal: bool = False, window: Optional[Tuple[int, int]] = None,
                      scale: Optional[float] = None, stream=None):
    """Packed fwd_masked: q [total_q, Hq, d]; k, v [total_k, Hkv, d]; int32
    offsets on the device.  Returns (o [total_q, Hq, d], lse [Hq, total_q])."""
    _check_bf16("q", q)
    total_q, Hq, d = q.shape
    _check_bf16("k", k)
    total_k, Hkv = k.shape[0], k.shape[1]
    if tuple(k.shape) != (total_k, Hkv, d):
        raise ValueError("k must be [total_k, Hkv, d]")
    _check_bf16("v", v, k.shape)
    _check_cu(cu_seqlens_q, q)
    _check_cu(cu_seqlens_k, q)
    if cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    wl, wr = _window(causal, window)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    l = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    st = lib().fa_fwd_masked_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(l), _ptr(cu_seqlens_q),
                                    _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, int(max_seqlen_q),
                                    int(max_seqlen_k), total_q, total_k, Hq, Hkv, d, wl, wr, scale, _stream(stream))
    _lib.check(st, "fa_fwd_masked_varlen")
    return o, l


@_on_tensor_device
def bwd_masked_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                      causal: bool = False, window: Optional[Tuple[int, int]] = None,
                      scale: Optional[float] = None, stream=None):
    """Gradients of fwd_masked_varlen: (dq [total_q, Hq, d], dk, dv [total_k, Hkv, d])."""
    for name, t in (("q", q), ("o", o), ("dout", dout)):
        _check_bf16(name, t, q.shape)
    total_q, Hq, d = q.shape
    _check_bf16("k", k)
    total_k, Hkv = k.shape[0], k.shape[1]
    _check_bf16("v", v, k.shape)
    _check_cu(cu_seqlens_q, q)
    _check_cu(cu_seqlens_k, q)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (Hq, total_q) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [Hq, total_q]")
    wl, wr = _window(causal, window)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = lib().fa_bwd_varlen_workspace_bytes(total_q, Hq, d)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = lib().fa_bwd_masked_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                    _ptr(dv), _ptr(ws), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                    cu_seqlens_q.numel() - 1, int(max_seqlen_q), int(max_seqlen_k), total_q, total_k,
                                    Hq, Hkv, d, wl, wr, scale, _stream(stream))
    _lib.check(st, "fa_bwd_masked_varlen")
    return dq, dk, dv


# ---------------------------------------------------------------- FP8 forward

@_on_tensor_device
def fp8_quantize(x, signs=None, transpose: bool = False, stream=None):
    """e4m3 block quantisation of x [B, N, H, d] (bf16).  With ``signs`` (int8
    [d] of +-1 on the device) the rows are first rotated by the Hadamard matrix
    and the signs.  Returns (codes uint8 [B, N, H, d], or [B, H, d, n_pad] when
    transposed; scales fp32 [B, H, ceil(N / 128)])."""
    _check_bf16("x", x)
    B, N, H, d = x.shape
    nblk = (N + 127) // 128
    if signs is not None:
        if signs.dtype != torch.int8 or tuple(signs.shape) != (d,) or signs.device != x.device:
            raise ValueError("signs must be int8 [d] on the device of x")
    if transpose:
        codes = torch.empty((B, H, d, nblk * 128), dtype=torch.uint8, device=x.device)
    else:
        codes = torch.empty((B, N, H, d), dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    st = lib().fa_fp8_quantize(_ptr(x), _ptr(signs), _ptr(codes), _ptr(scales), B, N, H, d,
                               int(signs is not None), int(bool(transpose)), _stream(stream))
    _lib.check(st, "fa_fp8_quantize")
    return codes, scales


@_on_tensor_device
def fwd_fp8_codes(q_codes, k_codes, vt_codes, q_scale, k_scale, v_scale, causal: bool = False,
                  window: Optional[Tuple[int, int]] = None, rotated: bool = True, scale: Optional[float] = None,
                  stream=None):
    """Attention on e4m3 operands from fp8_quantize (V transposed).
    Returns (o [B, Nq, Hq, d] bf16, lse [B, Hq, Nq])."""
    B, Nq, Hq, d = q_codes.shape
    Nk, Hkv = k_codes.shape[1], k_codes.shape[2]
    for name, t in (("q_codes", q_codes), ("k_codes", k_codes), ("vt_codes", vt_codes)):
        if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous uint8 CUDA tensor")
    if tuple(vt_codes.shape) != (B, Hkv, d, (Nk + 127) // 128 * 128):
        raise ValueError("vt_codes must be [B, Hkv, d, ceil(Nk / 128) * 128]")
    wl, wr = _window(causal, window)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((B, Nq, Hq, d), dtype=torch.bfloat16, device=q_codes.device)
    l = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q_codes.device)
    st = lib().fa_fwd_fp8(_ptr(q_codes), _ptr(k_codes), _ptr(vt_codes), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                          _ptr(o), _ptr(l), B, Hq, Hkv, Nq, Nk, d, wl, wr, int(bool(rotated)), scale,
                          _stream(stream))
    _lib.check(st, "fa_fwd_fp8")
    return o, l


@_on_tensor_device
def fwd_fp8(q, k, v, signs=None, causal: bool = False, window: Optional[Tuple[int, int]] = None,
            scale: Optional[float] = None, stream=None):
    """The FP8 forward from bf16 inputs: quantise Q and K (rotated when signs
    are given) and V (transposed), then attend.  Returns (o, lse)."""
    qc, qs = fp8_quantize(q, signs, stream=stream)
    kc, ks = fp8_quantize(k, signs, stream=stream)
    vc, vs = fp8_quantize(v, None, transpose=True, stream=stream)
    return fwd_fp8_codes(qc, kc, vc, qs, ks, vs, causal=causal, window=window, rotated=signs is not None,
                         scale=scale, stream=stream)


# ---------------------------------------------------------------- paged cache: write side

class PagePool:
    """Host page allocator of the C library (block tables, free list,
    reference counts); see fa_pool_* in fa.h.  Pages themselves are device
    tensors [num_pages, page_size, Hkv, d] that the caller owns."""

    def __init__(self, num_pages: int, page_size: int, max_seqs: int, max_blocks: int):
        self._lib = lib()
        self.handle = self._lib.fa_pool_create(num_pages, page_size, max_seqs, max_blocks)
        if not self.handle:
            raise _lib.FaError(_lib.FA_ERR_INVALID_ARG, "fa_pool_create")
        self.num_pages, self.page_size, self.max_seqs, self.max_blocks = num_pages, page_size, max_seqs, max_blocks

    def close(self):
        if self.handle:
            self._lib.fa_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()

    def free_pages(self) -> int:
        return self._lib.fa_pool_free_pages(self.handle)

    def refcount(self, page: int) -> int:
        return self._lib.fa_pool_refcount(self.handle, page)

    def add_seq(self) -> int:
        s = ctypes.c_int(-1)
        _lib.check(self._lib.fa_pool_add_seq(self.handle, ctypes.byref(s)), "fa_pool_add_seq")
        return s.value

    def fork(self, parent: int) -> int:
        s = ctypes.c_int(-1)
        _lib.check(self._lib.fa_pool_fork(self.handle, parent, ctypes.byref(s)), "fa_pool_fork")
        return s.value

    def release(self, seq: int) -> None:
        _lib.check(self._lib.fa_pool_release(self.handle, seq), "fa_pool_release")

    def reserve_append(self, seqs):
        """Next token of each sequence: int32 host tensors (page, slot, copy_src)."""
        seqs_t = torch.as_tensor(list(seqs), dtype=torch.int32)
        n = seqs_t.numel()
        page, slot, src = (torch.empty(n, dtype=torch.int32) for _ in range(3))
        _lib.check(self._lib.fa_pool_reserve_append(self.handle, _ptr(seqs_t), n, _ptr(page), _ptr(slot), _ptr(src)),
                   "fa_pool_reserve_append")
        return page, slot, src

    def export(self):
        """(block_table int32 [max_seqs, max_blocks], seq_lens int32 [max_seqs]), host."""
        table = torch.empty((self.max_seqs, self.max_blocks), dtype=torch.int32)
        lens = torch.empty(self.max_seqs, dtype=torch.int32)
        _lib.check(self._lib.fa_pool_export(self.handle, _ptr(table), _ptr(lens)), "fa_pool_export")
        return table, lens


@_on_tensor_device
def paged_append(k_new, v_new, k_pages, v_pages, page, slot, copy_src, stream=None):
    """Copies shared pages where copy_src >= 0, then writes each token's K, V
    rows ([n, Hkv, d] bf16) into (page, slot); index tensors int32 on the device."""
    _check_bf16("k_new", k_new)
    n, Hkv, d = k_new.shape
    _check_bf16("v_new", v_new, k_new.shape)
    _check_bf16("k_pages", k_pages)
    num_pages, P = k_pages.shape[0], k_pages.shape[1]
    if tuple(k_pages.shape) != (num_pages, P, Hkv, d):
        raise ValueError("k_pages must be [num_pages, page_size, Hkv, d]")
    _check_bf16("v_pages", v_pages, k_pages.shape)
    for name, t in (("page", page), ("slot", slot), ("copy_src", copy_src)):
        if t.dtype != torch.int32 or not t.is_cuda or t.numel() != n or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor of {n} entries")
    st = lib().fa_paged_append(_ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages), _ptr(page), _ptr(slot),
                               _ptr(copy_src), n, Hkv, d, P, num_pages, _stream(stream))
    _lib.check(st, "fa_paged_append")


# ---------------------------------------------------------------- decode with a sliding window

def _window_span(L: int, window_left: int) -> int:
    return L if window_left < 0 or window_left >= L else window_left + 1


@_on_tensor_device
def decode_window(q, k_cache, v_cache, window_left: int, num_splits: int = 0, scale: Optional[float] = None,
                  stream=None):
    """Decode that sees only the last window_left + 1 keys of each cache.
    q [B, 1, Hq, d]; caches [B, L, Hkv, d].  Returns (o [B, 1, Hq, d], lse [B, Hq])."""
    _check_bf16("q", q)
    B, one, Hq, d = q.shape
    _check_bf16("k_cache", k_cache)
    L, Hkv = k_cache.shape[1], k_cache.shape[2]
    if one != 1 or tuple(k_cache.shape) != (B, L, Hkv, d):
        raise ValueError("q must be [B, 1, Hq, d] and the caches [B, L, Hkv, d]")
    _check_bf16("v_cache", v_cache, k_cache.shape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    span = _window_span(L, int(window_left))
    splits = num_splits if num_splits > 0 else lib().fa_decode_num_splits(B, Hkv, span, d)
    nbytes = lib().fa_decode_workspace_bytes(B, Hq, d, max(splits, 1))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    l = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib().fa_decode_window(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(l), B, Hq, Hkv, L, d,
                                int(window_left), splits, _ptr(ws), scale, _stream(stream))
    _lib.check(st, "fa_decode_window")
    return o, l


@_on_tensor_device
def decode_paged_window(q, k_pages, v_pages, block_table, seq_lens, max_seq_len: int, window_left: int = -1,
                        num_splits: int = 0, scale: Optional[float] = None, stream=None):
    """Paged decode with grouped K/V heads and a sliding window.  q [B, 1, Hq, d];
    pages [num_pages, page_size, Hkv, d]; block_table int32 [B, max_blocks] and
    seq_lens int32 [B] on the device.  Returns (o [B, 1, Hq, d], lse [B, Hq])."""
    _check_bf16("q", q)
    B, one, Hq, d = q.shape
    if one != 1:
        raise ValueError("q must be [B, 1, Hq, d]")
    _check_bf16("k_pages", k_pages)
    num_pages, page_size, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if tuple(k_pages.shape) != (num_pages, page_size, Hkv, d):
        raise ValueError("k_pages must be [num_pages, page_size, Hkv, d]")
    _check_bf16("v_pages", v_pages, k_pages.shape)
    for name, t in (("block_table", block_table), ("seq_lens", seq_lens)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_blocks] and seq_lens [B]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    span = _window_span(int(max_seq_len), int(window_left))
    splits = num_splits if num_splits > 0 else lib().fa_decode_num_splits(B, Hkv, span, d)
    nbytes = lib().fa_decode_workspace_bytes(B, Hq, d, max(splits, 1))
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    l = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    st = lib().fa_decode_paged_window(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                      _ptr(o), _ptr(l), B, Hq, Hkv, d, page_size, num_pages, block_table.shape[1],
                                      int(max_seq_len), int(window_left), splits, _ptr(ws), scale, _stream(stream))
    _lib.check(st, "fa_decode_paged_window")
    return o, l
