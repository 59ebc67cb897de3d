"""Degenerate shapes and masks through the whole path against the oracle:
one 128 x 128 block (a single partial block on the diagonal), an odd GQA
group (3 query heads per KV head) with B = 3, and a mask with no visible
key at all (MaskInfo of width 0: O = 0, LSE = -inf and zero gradients, the
reading the pages leave open for rows that see nothing).
"""
import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, TOL_LSE, TOL_O, compare, need_gpu
from oracle import attention as oatt
from workloads import qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("D", [64, 128])
def test_single_block_odd_group(D):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    B, Hq, Hkv, S = 3, 3, 1, 128
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=23)
    info = bsa.mask_compile("causal", S, S)
    dkv = bsa.mask_compile("causal", S, S, orientation="dkv")
    assert info.to_host()["width"] == 1
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info)
    dq, dk, dv = bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=True)
    assert bsa.get_device_error() == 0
    mask = {"kind": "causal", "kv_len": S}
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), mask)
    compare("O", o.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)
    for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), oatt.backward(f64(q), f64(k), f64(v), f64(do), mask)):
        compare(name, got.cpu().numpy(), want, TOL_GRAD)
    info.destroy()
    dkv.destroy()


def test_mask_with_no_visible_key():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    B, Hq, Hkv, S, D = 1, 4, 2, 384, 128
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=29)
    dd = torch.zeros((S, S), dtype=torch.uint8, device="cuda")
    info = bsa.mask_compile("dense", S, S, dense=dd)
    dkv = bsa.mask_compile("dense", S, S, dense=dd, orientation="dkv")
    assert info.to_host()["width"] == 0 and dkv.to_host()["width"] == 0
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info)
    for fp32 in (True, False):
        dq, dk, dv = bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=fp32)
        assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)
    assert bsa.get_device_error() == 0
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), {"kind": "dense", "kv_len": S, "dense": np.zeros((S, S), np.uint8)})
    assert np.all(ro == 0) and np.all(np.isneginf(rl))
    info.destroy()
    dkv.destroy()
