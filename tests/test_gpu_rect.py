"""Dense masks with different query and key lengths (S_q != S_kv): MaskInfo
rows are query blocks and its columns key blocks in the forward orientation,
the other way round in the dK/dV one, so a rectangular mask exercises both
extents separately (a square workload cannot tell them apart).  Forward O
and LSE and the fp32 and bf16 gradients against the fp64 oracle, GQA with a
shared mask and MQA with one mask per query head, with an all-masked query
block and an all-masked key block planted.
"""
import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, TOL_LSE, TOL_O, bf16_half_ulp, compare, need_gpu
from oracle import attention as oatt
from workloads import qkvdo

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, S_q, S_kv, D, per-head mask, p
    (1, 4, 2, 384, 896, 128, False, 0.3),
    (2, 2, 1, 1024, 256, 64, True, 0.5),
]


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rect_mask(Hm, Sq, Skv, p, seed):
    rng = np.random.default_rng(seed)
    m = (rng.random((Hm, Sq, Skv)) < p).astype(np.uint8)
    m[:, 128:256, :] = 0        # a query block that sees nothing
    m[:, :, Skv - 128:] = 0     # a key block nobody sees
    m[:, :, :128] |= np.eye(Sq, 128, dtype=np.uint8)[None]  # some rows see their first keys
    return m


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}_Hq{c[1]}_Hkv{c[2]}_Sq{c[3]}_Skv{c[4]}_D{c[5]}" for c in CASES])
def test_rectangular_dense_mask_forward_and_backward(case):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    B, Hq, Hkv, Sq, Skv, D, per_head, p = case
    Hm = Hq if per_head else 1
    q, k, v, do = qkvdo(B, Hq, Hkv, Sq, D, seed=11, Skv=Skv)
    m = rect_mask(Hm, Sq, Skv, p, seed=5)
    dd = torch.from_numpy(m if per_head else m[0]).cuda()
    info = bsa.mask_compile("dense", Sq, Skv, dense=dd)
    dkv = bsa.mask_compile("dense", Sq, Skv, dense=dd, orientation="dkv")
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info)
    grads = {g: bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=g) for g in (True, False)}
    assert bsa.get_device_error() == 0

    mask = {"kind": "dense", "kv_len": Skv, "dense": m if per_head else m[0]}
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), mask)
    compare("O", o.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)  # (-inf where a row sees nothing)
    assert np.all(np.isneginf(rl[:, :, 128:256]))   # the planted query block sees nothing
    assert torch.all(o[:, :, 128:256] == 0)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), mask)
    for fp32, gr in grads.items():
        for name, got, want in zip(("dQ", "dK", "dV"), gr, ref):
            compare(f"{name} ({'fp32' if fp32 else 'bf16'})", got.float().cpu().numpy(), want, TOL_GRAD,
                    None if fp32 else bf16_half_ulp(want))
        # the key block nobody sees gets zero gradients
        assert torch.all(gr[1][:, :, Skv - 128:] == 0) and torch.all(gr[2][:, :, Skv - 128:] == 0)
    info.destroy()
    dkv.destroy()
