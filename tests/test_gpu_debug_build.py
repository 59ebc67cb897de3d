"""The range-checked build (libbsa_debug.so, compiled with -DBSA_DEBUG=1):
tensor-memory addresses, the global rows the kernels compute from the
schedule and MaskInfo, and the phase of every mbarrier after each completed
wait are checked on the device, a violation recorded in the error word.

A child process loads it (BSA_LIBRARY_VARIANT=debug) and runs the forward
and backward over every mask kind, GQA/MQA head maps, D = 64 and 128, the
soft cap and sinks, key shards with their merge and the allocation-free
backward: results within the usual tolerances of the oracle, and the device
error word 0 after each (no check fired); and out-of-range indices planted
by bsa_debug_selfcheck set the debug bit with a source line.  The release
build compiles the checks out: the same call leaves the word 0.
"""
import os
import subprocess
import sys

import pytest

from helpers import ROOT, need_gpu

pytestmark = pytest.mark.gpu

SCRIPT = r'''
import math, sys
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import numpy as np, torch
import block_sparse_attention_process_gb300 as bsa
from block_sparse_attention_process_gb300 import _abi
assert _abi.LIB_PATH.endswith("libbsa_debug.so"), _abi.LIB_PATH
from helpers import TOL_GRAD, TOL_LSE, TOL_O, compare
from oracle import attention as oatt
from workloads import bernoulli_mask, qkvdo
f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
cases = [
    # B, Hq, Hkv, S, D, kind, library kwargs, oracle kwargs, cap, sinks
    (1, 2, 2, 512, 64, "causal", {}, {}, None, None),
    (2, 8, 2, 1024, 128, "causal", {}, {}, None, None),
    (1, 4, 4, 1024, 128, "local", {"local_left": 300, "local_right": 40}, {"left": 300, "right": 40}, None, None),
    (1, 4, 1, 768, 128, "chunked", {"chunk": 256}, {"chunk": 256}, None, None),
    (1, 4, 2, 512, 128, "dense", {}, {}, None, None),
    (1, 4, 2, 512, 64, "causal", {}, {}, 2.0, (2, 3)),
]
for B, Hq, Hkv, S, D, kind, lkw, okw, cap, sink_shape in cases:
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=50)
    dense = bernoulli_mask(S, 0.3, 3) if kind == "dense" else None
    dd = None if dense is None else torch.from_numpy(dense).cuda()
    info = bsa.mask_compile(kind, S, S, dense=dd, **lkw)
    dkv = bsa.mask_compile(kind, S, S, dense=dd, orientation="dkv", **lkw)
    sinks = None if sink_shape is None else torch.from_numpy(
        np.random.default_rng(1).standard_normal(sink_shape).astype(np.float32)).cuda()
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info, logits_soft_cap=cap, sinks=sinks)
    grads = bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=True, logits_soft_cap=cap, sinks=sinks)
    assert bsa.get_device_error() == 0, (kind, S)
    mask = {"kind": kind, "kv_len": S, **okw}
    if dense is not None:
        mask["dense"] = dense
    zs = None if sinks is None else sinks.double().cpu().numpy()
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), mask, cap=cap, sinks=zs)
    compare("O", o.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), mask, cap=cap, sinks=zs)
    for name, g, r in zip(("dQ", "dK", "dV"), grads[:3], ref[:3]):
        compare(name, g.cpu().numpy(), r, TOL_GRAD)
    if sinks is None and kind == "causal" and D == 128:
        # the allocation-free backward and two key shards merged
        got = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in (qd, kd, vd)]
        bsa.bwd_noalloc(qd, kd, vd, o, lse, dod, info, dkv, dq=got[0], dk=got[1], dv=got[2], grad_fp32=True)
        assert bsa.get_device_error() == 0
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref[:3]):
            compare(name + " noalloc", g.cpu().numpy(), r, TOL_GRAD)
        half = S // 2
        parts = [bsa.fwd_partial(qd, kd[:, :, a:a + half].contiguous(), vd[:, :, a:a + half].contiguous(), info, a)
                 for a in (0, half)]
        om, lm = bsa.fwd_merge(*(torch.stack(list(x)) for x in zip(*parts)))
        assert bsa.get_device_error() == 0
        compare("O shards", om.float().cpu().numpy(), ro, TOL_O)
        compare("LSE shards", lm.cpu().numpy(), rl, TOL_LSE)
# the range checks report what they find: out-of-range indices planted by
# bsa_debug_selfcheck (nothing is accessed with them) set the debug bit
# and a source line
w = __import__("ctypes").c_uint32(0)
bsa.debug_selfcheck()
st = _abi.lib().bsa_get_device_error(None, __import__("ctypes").byref(w))
assert st == _abi.DEVICE and (w.value & 8) and (w.value >> 16) > 0, (st, hex(w.value))
assert bsa.get_device_error() == 0
print("ok")
'''


def test_range_checked_build_runs_clean():
    need_gpu()
    from block_sparse_attention_process_gb300 import build as b
    if not os.path.exists(b.LIB_DEBUG):
        b.build(debug=True)
    env = dict(os.environ, BSA_LIBRARY_VARIANT="debug")
    r = subprocess.run([sys.executable, "-c", SCRIPT.replace("ROOT", repr(ROOT))], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_release_build_compiles_the_checks_out():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    from block_sparse_attention_process_gb300 import _abi
    if _abi.LIB_PATH.endswith("libbsa_debug.so"):
        pytest.skip("this process runs the range-checked build")
    bsa.debug_selfcheck()
    assert bsa.get_device_error() == 0
