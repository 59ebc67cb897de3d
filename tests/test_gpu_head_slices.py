"""Calls on head slices of the step's tensors (B = 1, a contiguous range of
KV heads with their query heads), so that every pointer starts inside its
tensor.  The end-to-end benchmark runs the forward in two such halves and
dQ in four parts, each part behind its inputs' copy or ahead of its
output's.  Heads are independent and each launch computes a query head's
tile the same way whatever else it runs, so the parts must equal the
single calls over all heads bit for bit; one sliced head is also checked
against the oracle (O, LSE and dQ within the usual tolerances).
"""
import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, TOL_LSE, TOL_O, bf16_half_ulp, compare, need_gpu
from oracle import attention as oatt
from workloads import qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def parts(n, Hq, Hkv):
    G, kv = Hq // Hkv, Hkv // n
    return [(slice(c * kv * G, (c + 1) * kv * G), slice(c * kv, (c + 1) * kv)) for c in range(n)]


def test_head_slice_calls_equal_the_call_over_all_heads():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    B, Hq, Hkv, S, D = 1, 8, 4, 1280, 128
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=31)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    info = bsa.mask_compile("causal", S, S)

    o, lse = bsa.fwd(qd, kd, vd, info)
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    for hs, gs in parts(2, Hq, Hkv):
        bsa.fwd(qd[:, hs], kd[:, gs], vd[:, gs], info, o=o2[:, hs], lse=lse2[:, hs])
    dsum = bsa.bwd_rowsum(o, dod)
    dq = bsa.bwd_dq(qd, kd, vd, o, lse, dod, dsum, info)
    dq2 = torch.empty_like(dq)
    for hs, gs in parts(4, Hq, Hkv):
        bsa.bwd_dq(qd[:, hs], kd[:, gs], vd[:, gs], o[:, hs], lse[:, hs], dod[:, hs], dsum[:, hs], info,
                   dq=dq2[:, hs])
    torch.cuda.synchronize()
    assert bsa.get_device_error() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(dq, dq2)

    # a head of the last forward half and of the third dQ part, against the oracle
    hq, g = 5, 5 // (Hq // Hkv)
    mask = oatt.mask_rows_for({"kind": "causal", "kv_len": S}, 0)
    scale = 1 / np.sqrt(D)
    rdq, _, _, _, ro, rl, _ = oatt.head_backward(f64(q[0, hq]), f64(k[0, g]), f64(v[0, g]), f64(do[0, hq]),
                                                 mask, scale)
    compare(f"O[0,{hq}] (half call) vs oracle", o2[0, hq].float().cpu().numpy(), ro, TOL_O)
    compare(f"LSE[0,{hq}] (half call) vs oracle", lse2[0, hq].cpu().numpy(), rl, TOL_LSE)
    compare(f"dQ[0,{hq}] (part call) vs oracle", dq2[0, hq].float().cpu().numpy(), rdq, TOL_GRAD,
            bf16_half_ulp(rdq))
    info.destroy()
