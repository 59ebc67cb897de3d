"""The C ABI library builds, loads and exports every symbol include/bsa.h declares.

Also host-side argument checking: calls with bad arguments must return the
documented status before anything touches the GPU (these run without one).
"""
import ctypes as C
import math
import os
import re

import pytest

from helpers import ROOT, ensure_built


def declared_symbols():
    with open(os.path.join(ROOT, "include", "bsa.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"BSA_API\s+[\w\s\*]+?\b(bsa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("bsa_mask_compile", "bsa_mask_info_view", "bsa_mask_info_destroy", "bsa_fwd", "bsa_bwd",
              "bsa_bwd_rowsum", "bsa_bwd_dkv", "bsa_bwd_dq", "bsa_get_device_error", "bsa_status_string",
              "bsa_last_error"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    for n in declared_symbols():
        assert hasattr(L, n), n
        assert n in _abi.SIGNATURES, f"{n} has no ctypes signature"
    assert L.bsa_version().decode().count(".") == 2


def test_status_strings():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    assert L.bsa_status_string(_abi.OK) == b"ok"
    assert L.bsa_status_string(_abi.INVALID_ARG) == b"invalid argument"
    assert L.bsa_status_string(99) == b"unknown status"


def _fwd_args(**kw):
    from block_sparse_attention_process_gb300 import _abi
    a = _abi.FwdArgs(16, 32, 48, 64, 80, 1, 2, 2, 128, 256, 256, math.nan)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,status", [
    ({"S_q": 200}, "INVALID_ARG"),
    ({"Hq": 3}, "INVALID_ARG"),
    ({"B": 0}, "INVALID_ARG"),
    ({"D": 96}, "UNSUPPORTED"),
    ({"q": None}, "INVALID_ARG"),
    ({"o": 8}, "INVALID_ARG"),  # misaligned
])
def test_fwd_rejects_bad_arguments_on_host(kw, status):
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _fwd_args(**kw)
    st = L.bsa_fwd(C.byref(a), C.c_void_p(1), None)
    assert st == getattr(_abi, status), L.bsa_last_error()
    assert len(L.bsa_last_error()) > 0


def test_fwd_rejects_null_maskinfo():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _fwd_args()
    assert L.bsa_fwd(C.byref(a), None, None) == _abi.INVALID_ARG


@pytest.mark.parametrize("field,value,status", [
    ("q_len", 100, "INVALID_ARG"),
    ("kind", 9, "INVALID_ARG"),
    ("mask_heads", 0, "INVALID_ARG"),
    ("chunk", 0, "INVALID_ARG"),
    ("kv_len", 512, "UNSUPPORTED"),   # computable mask with q_len != kv_len
])
def test_mask_compile_rejects_bad_specs_on_host(field, value, status):
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    spec = _abi.MaskSpec(kind=_abi.MASK_CHUNKED_CAUSAL, mask_heads=1, q_len=256, kv_len=256, local_left=-1,
                         local_right=-1, chunk=128, dense=None)
    setattr(spec, field, value)
    opts = _abi.MaskOpts(128, 128, 1, 0)
    out = C.c_void_p()
    st = L.bsa_mask_compile(C.byref(spec), C.byref(opts), None, C.byref(out))
    assert st == getattr(_abi, status)
    assert out.value is None


@pytest.mark.parametrize("opts,status", [((64, 128, 1, 0), "UNSUPPORTED"), ((128, 128, 2, 0), "INVALID_ARG"),
                                          ((128, 128, 1, 5), "INVALID_ARG")])
def test_mask_compile_rejects_bad_options(opts, status):
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    spec = _abi.MaskSpec(kind=_abi.MASK_CAUSAL, mask_heads=1, q_len=256, kv_len=256, local_left=-1,
                         local_right=-1, chunk=0, dense=None)
    o = _abi.MaskOpts(*opts)
    out = C.c_void_p()
    assert L.bsa_mask_compile(C.byref(spec), C.byref(o), None, C.byref(out)) == getattr(_abi, status)


def test_dense_mask_needs_a_pointer():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    spec = _abi.MaskSpec(kind=_abi.MASK_DENSE, mask_heads=1, q_len=256, kv_len=384, local_left=-1,
                         local_right=-1, chunk=0, dense=None)
    o = _abi.MaskOpts(128, 128, 1, 0)
    out = C.c_void_p()
    assert L.bsa_mask_compile(C.byref(spec), C.byref(o), None, C.byref(out)) == _abi.INVALID_ARG


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from block_sparse_attention_process_gb300 import _abi
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _abi.lib()


def _partial_args(**kw):
    from block_sparse_attention_process_gb300 import _abi
    a = _abi.FwdPartialArgs(16, 32, 48, 64, 80, 96, 1, 2, 2, 128, 256, 128, 128, math.nan)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,status", [
    ({"S_kv_shard": 100}, "INVALID_ARG"),
    ({"kv_offset": 64}, "INVALID_ARG"),
    ({"kv_offset": -128}, "INVALID_ARG"),
    ({"D": 96}, "UNSUPPORTED"),
    ({"o_acc": None}, "INVALID_ARG"),
    ({"m": 8}, "INVALID_ARG"),  # misaligned
])
def test_fwd_partial_rejects_bad_arguments_on_host(kw, status):
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _partial_args(**kw)
    st = L.bsa_fwd_partial(C.byref(a), C.c_void_p(1), None)
    assert st == getattr(_abi, status), L.bsa_last_error()


def test_fwd_partial_rejects_null_maskinfo():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    assert L.bsa_fwd_partial(C.byref(_partial_args()), None, None) == _abi.INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    ({"n_shards": 0}, "INVALID_ARG"),
    ({"rows": 0}, "INVALID_ARG"),
    ({"D": 96}, "UNSUPPORTED"),
    ({"lse": None}, "INVALID_ARG"),
    ({"o_acc": 8}, "INVALID_ARG"),  # misaligned
])
def test_fwd_merge_rejects_bad_arguments_on_host(kw, status):
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _abi.MergeArgs(2, 16, 32, 48, 64, 80, 256, 128)
    for k, v in kw.items():
        setattr(a, k, v)
    assert L.bsa_fwd_merge(C.byref(a), None) == getattr(_abi, status), L.bsa_last_error()


def _bwd_args(**kw):
    from block_sparse_attention_process_gb300 import _abi
    a = _abi.BwdArgs(16, 32, 48, 64, 80, 96, 112, 128, 144, 160, 1, 2, 2, 128, 256, 256, math.nan, 1,
                     0.0, 176, 192, 2, 0)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("entry", ["bsa_bwd", "bsa_bwd_noalloc"])
@pytest.mark.parametrize("kw,status", [
    ({"sinks": 178}, "INVALID_ARG"),     # sinks not 4-byte aligned
    ({"dsinks": 194}, "INVALID_ARG"),    # dsinks not 4-byte aligned
    ({"sinks": None}, "INVALID_ARG"),    # num_sinks > 0 without sinks
    ({"num_sinks": 65}, "UNSUPPORTED"),
    ({"logits_soft_cap": -1.0}, "INVALID_ARG"),
    ({"dk": 8}, "INVALID_ARG"),          # misaligned tensor
    ({"D": 96}, "UNSUPPORTED"),
    ({"Hq": 3}, "INVALID_ARG"),
])
def test_backward_entry_points_reject_bad_arguments_on_host(entry, kw, status):
    """Both backward entry points make the same host-side checks, before any
    launch (so they run without a GPU)."""
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _bwd_args(**kw)
    fn = getattr(L, entry)
    st = fn(C.byref(a), C.c_void_p(1), C.c_void_p(1), None)
    assert st == getattr(_abi, status), (entry, kw, L.bsa_last_error())


def test_noalloc_ignores_the_dsum_pointer_but_bwd_needs_it():
    ensure_built()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _bwd_args(dsum=None, num_sinks=0, sinks=None, dsinks=None)
    assert L.bsa_bwd(C.byref(a), C.c_void_p(1), C.c_void_p(1), None) == _abi.INVALID_ARG
    # the allocation-free entry point gets past the argument checks to the
    # MaskInfo checks (null MaskInfo -> invalid argument, with that message)
    assert L.bsa_bwd_noalloc(C.byref(a), None, None, None) == _abi.INVALID_ARG
    assert b"MaskInfo" in L.bsa_last_error()


def test_range_checked_library_exports_the_same_symbols():
    """The range-checked variant (built by build(), loaded when
    BSA_LIBRARY_VARIANT=debug) exports every symbol the header declares."""
    import ctypes
    from block_sparse_attention_process_gb300 import build as b
    if not os.path.exists(b.LIB_DEBUG):
        pytest.skip("range-checked library not built")
    L = ctypes.CDLL(b.LIB_DEBUG)
    for n in declared_symbols():
        assert hasattr(L, n), n
