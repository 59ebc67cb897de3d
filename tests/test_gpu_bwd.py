"""GPU backward (rowsum, dK/dV launch, dQ launch) vs the fp64 oracle.

dQ/dK/dV: fp32 outputs within max-abs 2e-2 of the oracle; bf16 outputs within
2e-2 plus half a bf16 ulp of the reference value (the rounding of the
output itself, which exceeds 2e-2 once |x| >= 8).  GQA/MQA sum dK/dV over
each query-head group inside the dK/dV launch; dense masks load their
partial blocks in both launches.  Small cases compare every element; the
full-size workloads compare whole sampled heads.
"""
import math

import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, bf16_half_ulp, compare, lib_mask_args, need_gpu, oracle_mask_args
from oracle import attention as oatt
from workloads import WORKLOADS, MaskSpec, bernoulli_mask, planted_block_mask, qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def gpu_fwd_bwd(q, k, v, do, spec, dense=None, grad_fp32=True, shrink=True, scale=None):
    import block_sparse_attention_process_gb300 as bsa
    S, Skv = q.shape[2], k.shape[2]
    dd = None if dense is None else torch.from_numpy(np.ascontiguousarray(dense)).cuda()
    info = bsa.mask_compile(spec.kind, S, Skv, dense=dd, shrink=shrink, **lib_mask_args(spec))
    dkv = bsa.mask_compile(spec.kind, S, Skv, dense=dd, shrink=shrink, orientation="dkv", **lib_mask_args(spec))
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info, softmax_scale=scale)
    dq, dk, dv = bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=grad_fp32, softmax_scale=scale)
    assert bsa.get_device_error() == 0
    return [t.float().cpu().numpy() for t in (dq, dk, dv, o)] + [lse.cpu().numpy()]


def omask(spec, S, dense=None):
    m = {"kind": spec.kind, "kv_len": S}
    m.update(oracle_mask_args(spec, S))
    if dense is not None:
        m["dense"] = dense
    return m


def check_grads(got, ref, fp32):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        compare(name, g, r, TOL_GRAD, None if fp32 else bf16_half_ulp(r))


SMALL = [
    (1, 2, 2, 512, 64, MaskSpec("causal")),
    (2, 2, 2, 384, 128, MaskSpec("causal")),
    (1, 4, 1, 512, 128, MaskSpec("local", left=200, right=70)),
    (1, 4, 2, 640, 64, MaskSpec("chunked", chunk=192)),
    (1, 4, 4, 512, 128, MaskSpec("dense", p=0.3, seed=2)),
    (1, 2, 2, 256, 128, MaskSpec("full")),
    (1, 8, 2, 768, 128, MaskSpec("local", left=300, right=None)),
]


@pytest.mark.parametrize("fp32", [True, False], ids=["fp32", "bf16"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}H{c[1]}/{c[2]}S{c[3]}D{c[4]}-{c[5].kind}")
def test_small_cases_elementwise(case, fp32):
    need_gpu()
    B, Hq, Hkv, S, D, spec = case
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=21)
    dense = bernoulli_mask(S, spec.p, spec.seed) if spec.kind == "dense" else None
    dq, dk, dv, _, _ = gpu_fwd_bwd(q, k, v, do, spec, dense=dense, grad_fp32=fp32)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), omask(spec, S, dense))
    check_grads((dq, dk, dv), ref, fp32)


def test_rowsum_matches_definition():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    _, _, o, do = qkvdo(2, 3, 3, 512, 128, seed=4)
    ds = bsa.bwd_rowsum(o.cuda(), do.cuda()).cpu().numpy()
    ref = oatt.rowsum_do_o(f64(do), f64(o))
    # fp32 sum of 128 exact products: error far below 1e-4 relative to the row's sum of |terms|
    scale = (np.abs(f64(do) * f64(o))).sum(-1)
    assert np.all(np.abs(ds - ref) <= 1e-5 * scale + 1e-6)


def test_planted_dense_with_empty_rows_and_columns():
    need_gpu()
    S = 640
    m = planted_block_mask(1, 5, 5, seed=12)[0]
    m[128:256, :] = 0
    m[300, :] = 0
    m[:, 512:] = 0
    q, k, v, do = qkvdo(1, 2, 1, S, 128, seed=5)
    dq, dk, dv, _, _ = gpu_fwd_bwd(q, k, v, do, MaskSpec("dense"), dense=m)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), {"kind": "dense", "kv_len": S, "dense": m})
    check_grads((dq, dk, dv), ref, True)
    assert np.all(dq[0, :, 128:256] == 0) and np.all(dk[0, :, 512:] == 0) and np.all(dv[0, :, 512:] == 0)


def test_per_head_dense_masks_gqa():
    need_gpu()
    S, Hq = 512, 4
    m = np.stack([bernoulli_mask(S, p, seed=s) for p, s in ((0.05, 1), (0.5, 2), (0.9, 3), (0.3, 4))])
    m[1, :, 256:] = 0
    q, k, v, do = qkvdo(1, Hq, 2, S, 128, seed=6)
    import block_sparse_attention_process_gb300 as bsa
    dd = torch.from_numpy(m).cuda()
    info = bsa.mask_compile("dense", S, S, dense=dd)
    dkv = bsa.mask_compile("dense", S, S, dense=dd, orientation="dkv")
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.fwd(qd, kd, vd, info)
    dq, dk, dv = bsa.bwd(qd, kd, vd, o, lse, dod, info, dkv, grad_fp32=True)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), {"kind": "dense", "kv_len": S, "dense": m})
    check_grads([t.cpu().numpy() for t in (dq, dk, dv)], ref, True)


def test_unshrunk_maskinfo_same_gradients():
    need_gpu()
    q, k, v, do = qkvdo(1, 2, 2, 768, 128, seed=7)
    spec = MaskSpec("local", left=256, right=0)
    a = gpu_fwd_bwd(q, k, v, do, spec, shrink=True)
    b = gpu_fwd_bwd(q, k, v, do, spec, shrink=False)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_explicit_scale():
    need_gpu()
    q, k, v, do = qkvdo(1, 2, 2, 384, 128, seed=8)
    spec = MaskSpec("causal")
    dq, dk, dv, _, _ = gpu_fwd_bwd(q, k, v, do, spec, scale=0.05)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), omask(spec, 384), scale=0.05)
    check_grads((dq, dk, dv), ref, True)


def test_backward_is_deterministic():
    need_gpu()
    q, k, v, do = qkvdo(1, 4, 2, 1024, 128, seed=9)
    a = gpu_fwd_bwd(q, k, v, do, MaskSpec("causal"))
    b = gpu_fwd_bwd(q, k, v, do, MaskSpec("causal"))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ---------------------------------------------------------------- full size

@pytest.mark.parametrize("name,heads", [
    ("mha_causal_s4096_fwdbwd", [(0, 0), (1, 15)]),
    ("mqa_bernoulli_s2048", None),        # one kv head: all 16 q heads contribute to dK/dV
    ("mha_local1024_s8192", [(0, 7)]),
    ("gqa_causal_s8192", [(0, 2)]),       # kv group 0 of 4 q heads
])
def test_full_size_sampled_heads(name, heads):
    need_gpu()
    w = WORKLOADS[name]
    q, k, v, do = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed)
    dense = bernoulli_mask(w.S, w.mask.p, w.mask.seed) if w.mask.kind == "dense" else None
    dq, dk, dv, o, lse = gpu_fwd_bwd(q, k, v, do, w.mask, dense=dense, grad_fp32=True)
    group = w.Hq // w.Hkv
    mask = omask(w.mask, w.S, dense)
    if heads is None:
        kv_heads = [(b, g) for b in range(w.B) for g in range(w.Hkv)]
    else:
        kv_heads = sorted({(b, h // group) for b, h in heads})
    scale = 1 / math.sqrt(w.D)
    for b, g in kv_heads:
        rdk = np.zeros(k.shape[2:])
        rdv = np.zeros(v.shape[2:])
        for h in range(g * group, (g + 1) * group):
            rdq, dkh, dvh, _, _, _, _ = oatt.head_backward(f64(q[b, h]), f64(k[b, g]), f64(v[b, g]), f64(do[b, h]),
                                                        oatt.mask_rows_for(mask, 0), scale)
            rdk += dkh
            rdv += dvh
            compare(f"dQ[{b},{h}]", dq[b, h], rdq, TOL_GRAD)
        compare(f"dK[{b},{g}]", dk[b, g], rdk, TOL_GRAD)
        compare(f"dV[{b},{g}]", dv[b, g], rdv, TOL_GRAD)


# ------------------------------------------------- the benchmarked configuration

def test_small_gqa_bf16_unsplit_tensor_store_epilogue():
    """bf16 gradients of a GQA case with enough key/value tiles (B * Hkv *
    S/128 = 4 * 8 * 10 = 320, two per SM) that the dK/dV launch keeps each
    q-head group in one CTA and writes bf16 dK/dV through its tensor-store
    epilogue (the path the GQA benchmark times), compared in full."""
    need_gpu()
    B, Hq, Hkv, S, D = 4, 16, 8, 1280, 128
    assert B * Hkv * (S // 128) >= 2 * torch.cuda.get_device_properties(0).multi_processor_count
    spec = MaskSpec("causal")
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=22)
    dq, dk, dv, _, _ = gpu_fwd_bwd(q, k, v, do, spec, grad_fp32=False)
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), omask(spec, S))
    check_grads((dq, dk, dv), ref, False)


def _group_reference(q, k, v, do, mask, b, g, group, D):
    """Oracle dQ of the group's q heads and the group's summed dK/dV."""
    scale = 1 / math.sqrt(D)
    rdk = np.zeros(k.shape[2:])
    rdv = np.zeros(v.shape[2:])
    rdq = {}
    for h in range(g * group, (g + 1) * group):
        dqh, dkh, dvh, _, _, _, _ = oatt.head_backward(f64(q[b, h]), f64(k[b, g]), f64(v[b, g]), f64(do[b, h]),
                                                       oatt.mask_rows_for(mask, h), scale)
        rdq[h] = dqh
        rdk += dkh
        rdv += dvh
    return rdq, rdk, rdv


def test_benchmarked_backward_bf16_gqa_causal_s8192():
    """The backward exactly as the benchmark runs it (GQA 32/8, causal, 8192
    tokens, D = 128, bf16 dQ/dK/dV, unsplit dK/dV with the tensor-store
    epilogue): dK/dV of kv group 0 and dQ of its four q heads, every element,
    against the oracle at 2e-2 plus half a bf16 ulp."""
    need_gpu()
    w = WORKLOADS["gqa_causal_s8192"]
    q, k, v, do = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed)
    dq, dk, dv, _, _ = gpu_fwd_bwd(q, k, v, do, w.mask, grad_fp32=False)
    group = w.Hq // w.Hkv
    rdq, rdk, rdv = _group_reference(q, k, v, do, omask(w.mask, w.S), 0, 0, group, w.D)
    for h, r in rdq.items():
        compare(f"dQ[0,{h}]", dq[0, h], r, TOL_GRAD, bf16_half_ulp(r))
    compare("dK[0,0]", dk[0, 0], rdk, TOL_GRAD, bf16_half_ulp(rdk))
    compare("dV[0,0]", dv[0, 0], rdv, TOL_GRAD, bf16_half_ulp(rdv))


def test_bf16_gradients_over_plain_tolerance_are_rounding_only(record_property):
    """The forward + backward workload (B 2, H 16, causal 4096): bf16 dQ/dK/dV
    of two sampled heads against the oracle.  Counts the elements whose error
    exceeds the plain 2e-2 and checks that each of them sits where the bf16
    rounding of the output is a large part of it (|x| >= 2, where half a bf16
    ulp is 1/128 or more), and that the fp32 outputs of the same heads are within the
    plain 2e-2 everywhere."""
    need_gpu()
    w = WORKLOADS["mha_causal_s4096_fwdbwd"]
    q, k, v, do = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed)
    bf = gpu_fwd_bwd(q, k, v, do, w.mask, grad_fp32=False)
    fp = gpu_fwd_bwd(q, k, v, do, w.mask, grad_fp32=True)
    mask = omask(w.mask, w.S)
    total, over, worst, worst_fp32 = 0, 0, 0.0, 0.0
    for b, h in ((0, 0), (1, 15)):
        rdq, rdk, rdv = _group_reference(q, k, v, do, mask, b, h, 1, w.D)
        for name, i, r in (("dQ", 0, rdq[h]), ("dK", 1, rdk), ("dV", 2, rdv)):
            got = bf[i][b, h].astype(np.float64)
            err = np.abs(got - r)
            hi = err > TOL_GRAD
            total += err.size
            over += int(hi.sum())
            worst = max(worst, float(err.max()))
            assert np.all(np.abs(r[hi]) >= 2.0), f"{name}[{b},{h}]: an element over 2e-2 at |x| < 2"
            compare(f"{name}[{b},{h}] bf16", got, r, TOL_GRAD, bf16_half_ulp(r))
            worst_fp32 = max(worst_fp32, compare(f"{name}[{b},{h}] fp32", fp[i][b, h], r, TOL_GRAD))
    record_property("bf16_over_2e-2", over)
    record_property("bf16_elements", total)
    print(f"\nbf16 gradient elements over 2e-2: {over} of {total} ({over / total:.2e}); "
          f"max-abs bf16 {worst:.3e}, fp32 {worst_fp32:.3e}")
