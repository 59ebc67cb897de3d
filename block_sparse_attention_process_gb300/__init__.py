"""GB300-native block-sparse ("splash") attention: Python binding of libbsa.so.

The functions here have the names of the C entry points in ``include/bsa.h``
(without the ``bsa_`` prefix) and do argument marshalling only: torch
supplies device memory and the current stream, and every step of the path
runs in the library's CUDA kernels.  When the library is missing every call
raises; nothing falls back to another implementation.

    info = mask_compile("causal", S, S)                     # MaskInfo (fwd orientation)
    o, lse = fwd(q, k, v, info)                              # bf16 O, fp32 logsumexp
    dkv = mask_compile("causal", S, S, orientation="dkv")
    dq, dk, dv = bwd(q, k, v, o, lse, do, info, dkv)
"""
from __future__ import annotations

import ctypes as C
import math
from dataclasses import dataclass
from typing import Optional

import torch

from . import _abi
from ._abi import BsaError, check

__all__ = ["mask_compile", "MaskInfo", "fwd", "fwd_partial", "fwd_merge", "bwd", "bwd_noalloc", "bwd_rowsum",
           "bwd_dkv", "bwd_dq",
           "get_device_error", "set_wait_limit_ns", "debug_wait_timeout", "debug_selfcheck", "version", "BsaError",
           "library_path"]

_KINDS = {"dense": _abi.MASK_DENSE, "causal": _abi.MASK_CAUSAL, "local": _abi.MASK_LOCAL,
          "chunked": _abi.MASK_CHUNKED_CAUSAL, "full": _abi.MASK_FULL}
_ORIENT = {"fwd": _abi.ORIENT_FWD, "dkv": _abi.ORIENT_DKV}
_IDX_DTYPES = {1: torch.int8, 2: torch.int16, 4: torch.int32}


def library_path() -> str:
    return _abi.LIB_PATH


def version() -> str:
    return _abi.lib().bsa_version().decode()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


class _DevArray:
    """A borrowed device array (no copy) usable with torch.as_tensor."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def _view(ptr: int, shape, dtype: torch.dtype) -> torch.Tensor:
    n = 1
    for s in shape:
        n *= s
    if n == 0 or not ptr:
        return torch.empty(shape, dtype=dtype, device="cuda")
    typestr = {torch.int8: "|i1", torch.uint8: "|u1", torch.int16: "<i2", torch.int32: "<i4"}[dtype]
    return torch.as_tensor(_DevArray(ptr, shape, typestr), device="cuda")


class MaskInfo:
    """A compiled mask owned by the library (freed when this object dies)."""

    def __init__(self, handle: int):
        self._h = C.c_void_p(handle)

    @property
    def handle(self) -> C.c_void_p:
        if not self._h:
            raise RuntimeError("MaskInfo was destroyed")
        return self._h

    def desc(self) -> _abi.MaskInfoDesc:
        d = _abi.MaskInfoDesc()
        check(_abi.lib().bsa_mask_info_view(self.handle, C.byref(d)), "bsa_mask_info_view")
        return d

    def arrays(self) -> dict:
        """Borrowed device views of the MaskInfo arrays (valid while self lives)."""
        d = self.desc()
        shp = (d.heads, d.rows, d.width)
        out = {
            "block_mask": _view(d.block_mask, shp, torch.int8),
            "data_next": _view(d.data_next, shp, _IDX_DTYPES[d.data_next_bytes]),
            "mask_next": None if not d.mask_next else _view(d.mask_next, shp, _IDX_DTYPES[d.mask_next_bytes]),
            "partial_mask_blocks": None if not d.partial_mask_blocks else
            _view(d.partial_mask_blocks, (d.num_partial, 128, 128), torch.uint8),
            "q_sequence": _view(d.q_sequence, (d.q_len,), torch.int32),
            "row_len": _view(d.row_len, (d.heads * d.rows,), torch.int32),
            "row_order": _view(d.row_order, (d.heads * d.rows,), torch.int32),
        }
        return out

    def to_host(self) -> dict:
        """Copies of every array plus the counts, as numpy (for inspection and tests)."""
        torch.cuda.synchronize()
        d = self.desc()
        out = {k: (None if v is None else v.cpu().numpy()) for k, v in self.arrays().items()}
        out.update(width=d.width, cols=d.cols, num_partial=d.num_partial, n_empty=d.n_empty,
                   n_partial=d.n_partial, n_full=d.n_full, heads=d.heads, rows=d.rows)
        return out

    def destroy(self) -> None:
        if self._h:
            _abi.lib().bsa_mask_info_destroy(self._h)
            self._h = C.c_void_p(None)

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def mask_compile(kind: str, q_len: int, kv_len: int, *, mask_heads: int = 1, local_left: Optional[int] = None,
                 local_right: Optional[int] = None, chunk: int = 0, dense: Optional[torch.Tensor] = None,
                 shrink: bool = True, orientation: str = "fwd", stream=None) -> MaskInfo:
    """bsa_mask_compile.  ``dense`` is a CUDA uint8 tensor [mask_heads, q_len, kv_len] (or 2-D)."""
    spec = _abi.MaskSpec()
    spec.kind = _KINDS[kind]
    spec.q_len, spec.kv_len = q_len, kv_len
    spec.mask_heads = mask_heads
    spec.local_left = -1 if local_left is None else local_left
    spec.local_right = -1 if local_right is None else local_right
    spec.chunk = chunk
    if dense is not None:
        if dense.dtype != torch.uint8 or not dense.is_cuda or not dense.is_contiguous():
            raise ValueError("dense mask must be a contiguous CUDA uint8 tensor")
        spec.mask_heads = 1 if dense.dim() == 2 else dense.shape[0]
        spec.dense = dense.data_ptr()
    opts = _abi.MaskOpts(128, 128, 1 if shrink else 0, _ORIENT[orientation])
    out = C.c_void_p()
    check(_abi.lib().bsa_mask_compile(C.byref(spec), C.byref(opts), _stream(stream), C.byref(out)),
          "bsa_mask_compile")
    return MaskInfo(out.value)


def _check_bf16(name: str, t: torch.Tensor) -> None:
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")


def _sink_fields(sinks: Optional[torch.Tensor], Hkv: int):
    """(pointer, count, per-kv-head flag) of an fp32 CUDA sinks tensor [Hkv, n] or [n]."""
    if sinks is None:
        return None, 0, 0
    if sinks.dtype != torch.float32 or not sinks.is_cuda or not sinks.is_contiguous():
        raise ValueError("sinks must be a contiguous CUDA float32 tensor")
    if sinks.dim() == 2:
        if sinks.shape[0] != Hkv:
            raise ValueError("a 2-D sinks tensor must be [Hkv, num_sinks]")
        return _ptr(sinks), sinks.shape[1], 1
    if sinks.dim() != 1:
        raise ValueError("sinks must be [Hkv, num_sinks] or [num_sinks]")
    return _ptr(sinks), sinks.shape[0], 0


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, info: MaskInfo, *, o: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
        logits_soft_cap: Optional[float] = None, sinks: Optional[torch.Tensor] = None, stream=None):
    """bsa_fwd.  q [B,Hq,S,D], k/v [B,Hkv,Skv,D] bf16 -> (o bf16 [B,Hq,S,D], lse fp32 [B,Hq,S]).
    Optional soft cap c (scores -> c*tanh(s/c)) and sinks (fp32 [Hkv, n] or [n])."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(n, t)
    B, Hq, S, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    sp, sn, skv = _sink_fields(sinks, Hkv)
    a = _abi.FwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, D, S, Skv,
                     math.nan if softmax_scale is None else softmax_scale, logits_soft_cap or 0.0, sp, sn, skv)
    check(_abi.lib().bsa_fwd(C.byref(a), info.handle, _stream(stream)), "bsa_fwd")
    return o, lse


def fwd_partial(q: torch.Tensor, k_shard: torch.Tensor, v_shard: torch.Tensor, info: MaskInfo, kv_offset: int, *,
                softmax_scale: Optional[float] = None, logits_soft_cap: Optional[float] = None, stream=None):
    """bsa_fwd_partial: attention of q over one key shard (k_shard / v_shard hold keys
    kv_offset .. kv_offset + Skv_shard - 1 of the MaskInfo's key axis).
    -> (o_acc fp32 [B,Hq,S,D], m fp32 [B,Hq,S], l fp32 [B,Hq,S])."""
    for n, t in (("q", q), ("k", k_shard), ("v", v_shard)):
        _check_bf16(n, t)
    B, Hq, S, D = q.shape
    Hkv, Skv = k_shard.shape[1], k_shard.shape[2]
    o_acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=q.device)
    m = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    l = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    a = _abi.FwdPartialArgs(_ptr(q), _ptr(k_shard), _ptr(v_shard), _ptr(o_acc), _ptr(m), _ptr(l), B, Hq, Hkv, D, S,
                            Skv, kv_offset, math.nan if softmax_scale is None else softmax_scale,
                            logits_soft_cap or 0.0)
    check(_abi.lib().bsa_fwd_partial(C.byref(a), info.handle, _stream(stream)), "bsa_fwd_partial")
    return o_acc, m, l


def fwd_merge(o_acc: torch.Tensor, m: torch.Tensor, l: torch.Tensor, stream=None):
    """bsa_fwd_merge over stacked shards: o_acc [n, B,Hq,S,D], m / l [n, B,Hq,S] fp32
    -> (o bf16 [B,Hq,S,D], lse fp32 [B,Hq,S])."""
    for n_, t in (("o_acc", o_acc), ("m", m), ("l", l)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n_} must be a contiguous CUDA float32 tensor")
    n = o_acc.shape[0]
    D = o_acc.shape[-1]
    rows = o_acc[0].numel() // D
    o = torch.empty(o_acc.shape[1:], dtype=torch.bfloat16, device=o_acc.device)
    lse = torch.empty(m.shape[1:], dtype=torch.float32, device=o_acc.device)
    a = _abi.MergeArgs(n, _ptr(o_acc), _ptr(m), _ptr(l), _ptr(o), _ptr(lse), rows, D)
    check(_abi.lib().bsa_fwd_merge(C.byref(a), _stream(stream)), "bsa_fwd_merge")
    return o, lse


@dataclass
class _BwdBufs:
    args: _abi.BwdArgs
    dq: torch.Tensor
    dk: torch.Tensor
    dv: torch.Tensor
    dsum: torch.Tensor
    dsinks: Optional[torch.Tensor] = None


def _bwd_args(q, k, v, o, lse, do, dq, dk, dv, dsum, softmax_scale, grad_fp32, logits_soft_cap=None,
              sinks=None) -> _BwdBufs:
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_bf16(n, t)
    B, Hq, S, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    gdt = torch.float32 if grad_fp32 else torch.bfloat16
    dq = torch.empty(q.shape, dtype=gdt, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=gdt, device=q.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=gdt, device=q.device) if dv is None else dv
    dsum = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if dsum is None else dsum
    sp, sn, skv = _sink_fields(sinks, Hkv)
    dsinks = None if sinks is None else torch.empty_like(sinks)
    a = _abi.BwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                     _ptr(dsum), B, Hq, Hkv, D, S, Skv, math.nan if softmax_scale is None else softmax_scale,
                     1 if grad_fp32 else 0, logits_soft_cap or 0.0, sp, _ptr(dsinks), sn, skv)
    return _BwdBufs(a, dq, dk, dv, dsum, dsinks)


def bwd(q, k, v, o, lse, do, fwd_info: MaskInfo, dkv_info: MaskInfo, *, dq=None, dk=None, dv=None, dsum=None,
        softmax_scale=None, grad_fp32: bool = False, logits_soft_cap=None, sinks=None, stream=None):
    """bsa_bwd: rowsum, then dK/dV, then dQ.  Returns (dq, dk, dv), plus dsinks when sinks are given."""
    b = _bwd_args(q, k, v, o, lse, do, dq, dk, dv, dsum, softmax_scale, grad_fp32, logits_soft_cap, sinks)
    check(_abi.lib().bsa_bwd(C.byref(b.args), fwd_info.handle, dkv_info.handle, _stream(stream)), "bsa_bwd")
    return (b.dq, b.dk, b.dv) if sinks is None else (b.dq, b.dk, b.dv, b.dsinks)


def bwd_noalloc(q, k, v, o, lse, do, fwd_info: MaskInfo, dkv_info: MaskInfo, *, dq, dk, dv, softmax_scale=None,
                grad_fp32: bool = False, logits_soft_cap=None, sinks=None, dsinks=None, stream=None):
    """bsa_bwd_noalloc: the backward pass with no device allocation inside the
    library (its rowsum scratch is a fixed 4 MiB device array); the caller
    supplies the gradient buffers (and ``dsinks``, the sinks' shape, when the
    sinks' gradient is wanted)."""
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_bf16(n, t)
    B, Hq, S, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    sp, sn, skv = _sink_fields(sinks, Hkv)
    a = _abi.BwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                     None, B, Hq, Hkv, D, S, Skv, math.nan if softmax_scale is None else softmax_scale,
                     1 if grad_fp32 else 0, logits_soft_cap or 0.0, sp, _ptr(dsinks), sn, skv)
    check(_abi.lib().bsa_bwd_noalloc(C.byref(a), fwd_info.handle, dkv_info.handle, _stream(stream)),
          "bsa_bwd_noalloc")
    return (dq, dk, dv) if dsinks is None else (dq, dk, dv, dsinks)


def bwd_rowsum(o, do, *, dsum=None, stream=None) -> torch.Tensor:
    """bsa_bwd_rowsum: dsum[b,h,s] = sum_d dO*O (fp32)."""
    _check_bf16("o", o)
    _check_bf16("do", do)
    B, H, S, D = o.shape
    dsum = torch.empty((B, H, S), dtype=torch.float32, device=o.device) if dsum is None else dsum
    a = _abi.BwdArgs(_ptr(o), _ptr(o), _ptr(o), _ptr(o), _ptr(dsum), _ptr(do), _ptr(o), _ptr(o), _ptr(o),
                     _ptr(dsum), B, H, H, D, S, S, math.nan, 0)
    check(_abi.lib().bsa_bwd_rowsum(C.byref(a), _stream(stream)), "bsa_bwd_rowsum")
    return dsum


def bwd_dkv(q, k, v, o, lse, do, dsum, dkv_info: MaskInfo, *, dk=None, dv=None, softmax_scale=None,
            grad_fp32=False, stream=None):
    b = _bwd_args(q, k, v, o, lse, do, None, dk, dv, dsum, softmax_scale, grad_fp32)
    check(_abi.lib().bsa_bwd_dkv(C.byref(b.args), dkv_info.handle, _stream(stream)), "bsa_bwd_dkv")
    return b.dk, b.dv


def bwd_dq(q, k, v, o, lse, do, dsum, fwd_info: MaskInfo, *, dq=None, softmax_scale=None, grad_fp32=False,
           stream=None):
    b = _bwd_args(q, k, v, o, lse, do, dq, None, None, dsum, softmax_scale, grad_fp32)
    check(_abi.lib().bsa_bwd_dq(C.byref(b.args), fwd_info.handle, _stream(stream)), "bsa_bwd_dq")
    return b.dq


def get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word; raises if non-zero."""
    w = C.c_uint32(0)
    st = _abi.lib().bsa_get_device_error(_stream(stream), C.byref(w))
    if st != _abi.OK:
        raise BsaError(st, f"device error word {w.value:#x}")
    return w.value


def set_wait_limit_ns(ns: int) -> None:
    check(_abi.lib().bsa_set_wait_limit_ns(ns), "bsa_set_wait_limit_ns")


def debug_wait_timeout(stream=None) -> None:
    check(_abi.lib().bsa_debug_wait_timeout(_stream(stream)), "bsa_debug_wait_timeout")


def debug_selfcheck(stream=None) -> None:
    """bsa_debug_selfcheck: out-of-range indices through the range checks
    (recorded only by the range-checked build)."""
    check(_abi.lib().bsa_debug_selfcheck(_stream(stream)), "bsa_debug_selfcheck")
