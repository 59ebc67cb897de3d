"""A long sequence: GQA 8/2, local window (1024, 0) at 65,536 tokens (512
block rows, 32,768 forward tiles, row indices into Q/O up to 2^19) through
the forward and both gradient launches, against the oracle on samples it
can compute one by one: O and LSE on sampled rows, dQ on whole row chunks
(a row's dQ needs only that row and all keys), and dK/dV of sampled key
blocks from every query that sees them (the window bounds those queries).
"""
import math

import numpy as np
import pytest

from helpers import TOL_GRAD, TOL_LSE, TOL_O, compare, need_gpu
from oracle import attention as oatt
from workloads import qkvdo

pytestmark = pytest.mark.gpu

B, HQ, HKV, S, D, LEFT = 1, 8, 2, 65536, 128, 1024


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def test_local_window_at_65536_tokens():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    q, k, v, do = qkvdo(B, HQ, HKV, S, D, seed=41)
    info = bsa.mask_compile("local", S, S, local_left=LEFT, local_right=0)
    dkv = bsa.mask_compile("local", S, S, local_left=LEFT, local_right=0, orientation="dkv")
    assert info.to_host()["width"] == 9
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info)
    dq, dk, dv = bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=True)
    assert bsa.get_device_error() == 0
    o, lse, dq, dk, dv = (t.float().cpu().numpy() for t in (o, lse, dq, dk, dv))
    info.destroy()
    dkv.destroy()

    mask = oatt.mask_rows_for({"kind": "local", "kv_len": S, "left": LEFT, "right": 0}, 0)
    scale = 1 / math.sqrt(D)
    G = HQ // HKV
    rng = np.random.default_rng(3)
    for h in (0, HQ - 1):
        g = h // G
        rows = np.array(sorted(set(rng.choice(S, size=96, replace=False).tolist()) | {0, 127, 1024, S - 1}))
        ro, rl = oatt.head_forward(f64(q[0, h]), f64(k[0, g]), f64(v[0, g]), mask, scale, rows=rows)
        compare(f"O[0,{h}] rows", o[0, h, rows], ro, TOL_O)
        compare(f"LSE[0,{h}] rows", lse[0, h, rows], rl, TOL_LSE)
        for r0 in (0, S // 2 + 128, S - 256):
            r1 = r0 + 256
            rows_fn = lambda r, r0=r0: mask(np.asarray(r) + r0)  # noqa: E731
            rdq = oatt.head_backward(f64(q[0, h, r0:r1]), f64(k[0, g]), f64(v[0, g]), f64(do[0, h, r0:r1]),
                                     rows_fn, scale)[0]
            compare(f"dQ[0,{h}] rows {r0}..{r1}", dq[0, h, r0:r1], rdq, TOL_GRAD)
    # key block j is seen by the queries [128 j, 128 j + 127 + LEFT]
    for g, j in ((0, 0), (HKV - 1, S // 256), (HKV - 1, S // 128 - 1)):
        r0, r1 = 128 * j, min(S, 128 * j + 128 + LEFT)
        rows_fn = lambda r, r0=r0: mask(np.asarray(r) + r0)  # noqa: E731
        rdk = np.zeros((S, D))
        rdv = np.zeros((S, D))
        for h in range(g * G, (g + 1) * G):
            _, dkh, dvh, _, _, _, _ = oatt.head_backward(f64(q[0, h, r0:r1]), f64(k[0, g]), f64(v[0, g]),
                                                         f64(do[0, h, r0:r1]), rows_fn, scale)
            rdk += dkh
            rdv += dvh
        sl = slice(128 * j, 128 * j + 128)
        compare(f"dK[0,{g}] block {j}", dk[0, g, sl], rdk[sl], TOL_GRAD)
        compare(f"dV[0,{g}] block {j}", dv[0, g, sl], rdv[sl], TOL_GRAD)
