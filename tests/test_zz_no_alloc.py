"""bsa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (their memory is fixed up front by a pool or budget, or they must not
hit the device-wide synchronisation an allocation can cause).

It is called through the C ABI twice in a row and must give the same
gradients as bsa_bwd (within the backward tolerance) both times; the second
call reuses the static rowsum scratch the first one filled.  The file is
named to be collected last, and works alone in a fresh process as well as
after the other tests.
"""
import ctypes as C
import math

import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, need_gpu
from workloads import qkvdo

pytestmark = pytest.mark.gpu


def _args(abi, q, k, v, o, lse, do, dq, dk, dv, dsum):
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    return abi.BwdArgs(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), None if dsum is None else dsum.data_ptr(),
                       B, Hq, Hkv, D, S, S, math.nan, 1)


@pytest.mark.parametrize("kind,Hq,Hkv,S", [("causal", 4, 2, 1024), ("local", 2, 2, 768)])
def test_noalloc_backward_matches_bwd_twice(kind, Hq, Hkv, S):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    kw = {"local_left": 200, "local_right": 0} if kind == "local" else {}
    q, k, v, do = (t.cuda() for t in qkvdo(2, Hq, Hkv, S, 128, seed=31))
    info = bsa.mask_compile(kind, S, S, **kw)
    dkv = bsa.mask_compile(kind, S, S, orientation="dkv", **kw)
    o, lse = bsa.fwd(q, k, v, info)
    stream = torch.cuda.current_stream().cuda_stream

    ref = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in (q, k, v)]
    dsum = torch.empty(lse.shape, dtype=torch.float32, device="cuda")
    a = _args(_abi, q, k, v, o, lse, do, *ref, dsum)
    assert L.bsa_bwd(C.byref(a), info.handle, dkv.handle, C.c_void_p(stream)) == _abi.OK, L.bsa_last_error()

    for call in range(2):
        got = [torch.full(t.shape, float("nan"), dtype=torch.float32, device="cuda") for t in (q, k, v)]
        b = _args(_abi, q, k, v, o, lse, do, *got, None)
        st = L.bsa_bwd_noalloc(C.byref(b), info.handle, dkv.handle, C.c_void_p(stream))
        assert st == _abi.OK, L.bsa_last_error()
        torch.cuda.synchronize()
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            err = (g - r).abs().max().item()
            assert np.isfinite(err) and err <= TOL_GRAD, (call, name, err)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    need_gpu()
    from block_sparse_attention_process_gb300 import _abi
    L = _abi.lib()
    a = _abi.BwdArgs(16, 16, 16, 16, 16, 16, 16, 16, 16, None, 8, 128, 8, 128, 2048, 2048, math.nan, 1)
    st = L.bsa_bwd_noalloc(C.byref(a), C.c_void_p(1), C.c_void_p(1), None)
    assert st == _abi.UNSUPPORTED
    assert b"exceeds its fixed scratch" in L.bsa_last_error()
