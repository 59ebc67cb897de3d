"""bsa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (their memory is fixed up front by a pool or budget, or they must not
hit the device-wide synchronisation an allocation can cause).

Each case calls it through the C ABI twice in a row; both calls must give
the fp64 oracle's gradients (fp32 outputs, max-abs 2e-2) and the same
gradients as bsa_bwd within that tolerance, the second call reusing the
static rowsum scratch the first one filled, and the device error word must
read 0 after each call.  The cases reach the round-robin tile decoding of
this entry point with a shared mask, per-head dense masks (one MaskInfo row
per query head), D = 64, the soft cap and sinks with their gradient.  A
MaskInfo entry made out of range on purpose must show up in the device
error word (the kernels check every index they read and skip a bad one).

The file is named to be collected last, and works alone in a fresh process
as well as after the other tests.
"""
import ctypes as C
import math

import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, compare, need_gpu
from oracle import attention as oatt
from workloads import bernoulli_mask, qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _args(abi, q, k, v, o, lse, do, dq, dk, dv, dsum, cap=0.0, sinks=None, dsinks=None, per_kv=0):
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    n_sinks = 0 if sinks is None else sinks.shape[-1]
    return abi.BwdArgs(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None if dsum is None else dsum.data_ptr(),
                       B, Hq, Hkv, D, S, S, math.nan, 1, cap,
                       None if sinks is None else sinks.data_ptr(), None if dsinks is None else dsinks.data_ptr(),
                       n_sinks, per_kv)


def _error_word(L, stream):
    w = C.c_uint32(0)
    st = L.bsa_get_device_error(C.c_void_p(stream), C.byref(w))
    return st, w.value


CASES = [
    # id, B, Hq, Hkv, S, D, mask kind, mask kwargs, cap, sink shape
    ("causal-gqa", 2, 4, 2, 1024, 128, "causal", {}, 0.0, None),
    ("local-mha", 2, 2, 2, 768, 128, "local", {"local_left": 200, "local_right": 0}, 0.0, None),
    ("perhead-dense-gqa", 1, 4, 2, 512, 128, "dense-perhead", {}, 0.0, None),
    ("causal-d64-cap-sinks", 1, 4, 2, 512, 64, "causal", {}, 1.5, (2, 3)),
]


def _dense_per_head(Hq, S):
    m = np.stack([bernoulli_mask(S, p, seed=s) for p, s in zip((0.05, 0.5, 0.9, 0.3), range(1, Hq + 1))])
    m[1, :, 256:] = 0
    return m


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_noalloc_backward_matches_oracle_and_bwd_twice(case):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    _, B, Hq, Hkv, S, D, kind, kw, cap, sink_shape = case
    q, k, v, do = (t.cuda() for t in qkvdo(B, Hq, Hkv, S, D, seed=31))
    om = {"kind": kind, "kv_len": S}
    if kind == "dense-perhead":
        dense = _dense_per_head(Hq, S)
        dd = torch.from_numpy(dense).cuda()
        info = bsa.mask_compile("dense", S, S, dense=dd)
        dkv = bsa.mask_compile("dense", S, S, dense=dd, orientation="dkv")
        om = {"kind": "dense", "kv_len": S, "dense": dense}
    else:
        info = bsa.mask_compile(kind, S, S, **kw)
        dkv = bsa.mask_compile(kind, S, S, orientation="dkv", **kw)
        if kind == "local":
            om.update(left=kw["local_left"], right=kw["local_right"])
    sinks = None
    if sink_shape is not None:
        sinks = torch.from_numpy(np.random.default_rng(5).standard_normal(sink_shape).astype(np.float32) * 2).cuda()
    o, lse = bsa.fwd(q, k, v, info, logits_soft_cap=cap or None, sinks=sinks)
    stream = torch.cuda.current_stream().cuda_stream
    per_kv = 1 if sinks is not None and sinks.dim() == 2 else 0

    # the ordinary backward, for comparison
    ref = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in (q, k, v)]
    dsum = torch.empty(lse.shape, dtype=torch.float32, device="cuda")
    ref_ds = None if sinks is None else torch.empty_like(sinks)
    a = _args(_abi, q, k, v, o, lse, do, *ref, dsum, cap, sinks, ref_ds, per_kv)
    assert L.bsa_bwd(C.byref(a), info.handle, dkv.handle, C.c_void_p(stream)) == _abi.OK, L.bsa_last_error()
    assert _error_word(L, stream) == (_abi.OK, 0)

    zs = None if sinks is None else sinks.double().cpu().numpy()
    want = oatt.backward(f64(q), f64(k), f64(v), f64(do), om, cap=cap or None, sinks=zs)

    for call in range(2):
        got = [torch.full(t.shape, float("nan"), dtype=torch.float32, device="cuda") for t in (q, k, v)]
        ds = None if sinks is None else torch.full_like(sinks, float("nan"))
        b = _args(_abi, q, k, v, o, lse, do, *got, None, cap, sinks, ds, per_kv)
        st = L.bsa_bwd_noalloc(C.byref(b), info.handle, dkv.handle, C.c_void_p(stream))
        assert st == _abi.OK, L.bsa_last_error()
        assert _error_word(L, stream) == (_abi.OK, 0), call
        for name, g, r, w in zip(("dQ", "dK", "dV"), got, ref, want):
            gh = g.cpu().numpy()
            compare(f"{name} vs oracle (call {call})", gh, w, TOL_GRAD)
            compare(f"{name} vs bsa_bwd (call {call})", gh, r.cpu().numpy(), TOL_GRAD)
        if sinks is not None:
            g, w = ds.cpu().numpy().astype(np.float64), want[3]
            assert np.abs(g - w).max() <= 1e-2 * np.abs(w).max() + 1e-4, (call, g, w)


def test_noalloc_reports_a_bad_maskinfo_index_through_the_error_word():
    """A label out of range in the dK/dV MaskInfo: the kernel's own index
    check turns it into an empty block and sets the bounds bit, which
    bsa_get_device_error must return (and then clear)."""
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    B, H, S, D = 1, 2, 512, 128
    q, k, v, do = (t.cuda() for t in qkvdo(B, H, H, S, D, seed=32))
    info = bsa.mask_compile("causal", S, S)
    dkv = bsa.mask_compile("causal", S, S, orientation="dkv")
    o, lse = bsa.fwd(q, k, v, info)
    stream = torch.cuda.current_stream().cuda_stream
    assert _error_word(L, stream) == (_abi.OK, 0)
    dkv.arrays()["block_mask"][0, 1, 0] = 7   # a label no MaskInfo holds
    got = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in (q, k, v)]
    b = _args(_abi, q, k, v, o, lse, do, *got, None)
    assert L.bsa_bwd_noalloc(C.byref(b), info.handle, dkv.handle, C.c_void_p(stream)) == _abi.OK
    st, word = _error_word(L, stream)
    assert st == _abi.DEVICE and word & 2, (st, word)
    assert _error_word(L, stream) == (_abi.OK, 0)   # read once, then cleared


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need_gpu()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _abi.BwdArgs(16, 16, 16, 16, 16, 16, 16, 16, 16, None, 8, 128, 8, 128, 2048, 2048, math.nan, 1)
    st = L.bsa_bwd_noalloc(C.byref(a), C.c_void_p(1), C.c_void_p(1), None)
    assert st == _abi.UNSUPPORTED
    assert b"exceeds its fixed scratch" in L.bsa_last_error()
