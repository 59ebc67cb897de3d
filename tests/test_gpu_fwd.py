"""GPU forward vs the fp64 oracle.

O (bf16) within max-abs 2e-2 and LSE (fp32) within 1e-5 of the oracle,
element by element, on small cases that span several tiles, ragged block
counts, GQA/MQA head maps, D = 64 and 128, every mask kind, per-head masks,
unshrunk MaskInfo and fully masked rows; and on the full-size workloads
(in the bench's launch configuration) on sampled heads and rows.
"""
import math

import numpy as np
import pytest
import torch

from helpers import TOL_LSE, TOL_O, compare, lib_mask_args, need_gpu, oracle_mask_args
from oracle import attention as oatt
from workloads import WORKLOADS, MaskSpec, bernoulli_mask, planted_block_mask, qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(q, k, v, spec: MaskSpec, dense=None, shrink=True, scale=None):
    import block_sparse_attention_process_gb300 as bsa
    S, Skv = q.shape[2], k.shape[2]
    dev_dense = None if dense is None else torch.from_numpy(np.ascontiguousarray(dense)).cuda()
    info = bsa.mask_compile(spec.kind, S, Skv, dense=dev_dense, shrink=shrink, **lib_mask_args(spec))
    o, lse = bsa.fwd(q.cuda(), k.cuda(), v.cuda(), info, softmax_scale=scale)
    assert bsa.get_device_error() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def oracle_mask(spec: MaskSpec, S, dense=None):
    m = {"kind": spec.kind, "kv_len": S}
    m.update(oracle_mask_args(spec, S))
    if dense is not None:
        m["dense"] = dense
    return m


SMALL = [
    # B, Hq, Hkv, S, D, mask
    (1, 2, 2, 512, 64, MaskSpec("causal")),
    (2, 4, 2, 384, 128, MaskSpec("causal")),
    (1, 4, 1, 512, 128, MaskSpec("local", left=200, right=70)),
    (1, 2, 2, 640, 64, MaskSpec("chunked", chunk=192)),
    (1, 4, 4, 512, 128, MaskSpec("dense", p=0.3, seed=2)),
    (1, 2, 2, 256, 128, MaskSpec("full")),
    (1, 8, 2, 1024, 128, MaskSpec("local", left=300, right=None)),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}H{c[1]}/{c[2]}S{c[3]}D{c[4]}-{c[5].kind}")
def test_small_cases_elementwise(case):
    need_gpu()
    B, Hq, Hkv, S, D, spec = case
    q, k, v, _ = qkvdo(B, Hq, Hkv, S, D, seed=3, with_do=False)
    dense = bernoulli_mask(S, spec.p, spec.seed) if spec.kind == "dense" else None
    o, lse = run_gpu(q, k, v, spec, dense=dense)
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), oracle_mask(spec, S, dense))
    compare("O", o, ro, TOL_O)
    compare("LSE", lse, rl, TOL_LSE)


def test_unshrunk_maskinfo_gives_same_result():
    need_gpu()
    q, k, v, _ = qkvdo(1, 2, 2, 1024, 128, seed=4, with_do=False)
    spec = MaskSpec("local", left=256, right=0)
    o1, l1 = run_gpu(q, k, v, spec, shrink=True)
    o2, l2 = run_gpu(q, k, v, spec, shrink=False)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), oracle_mask(spec, 1024))
    compare("O", o2, ro, TOL_O)
    compare("LSE", l2, rl, TOL_LSE)


def test_planted_dense_with_empty_rows_and_columns():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    S = 640
    m = planted_block_mask(1, 5, 5, seed=11)[0]
    m[128:256, :] = 0          # a whole block row with no visible key
    m[300, :] = 0              # one row inside a partial block
    m[:, 512:] = 0             # an empty block column
    q, k, v, _ = qkvdo(1, 2, 1, S, 128, seed=5, with_do=False)
    o, lse = run_gpu(q, k, v, MaskSpec("dense"), dense=m)
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), {"kind": "dense", "kv_len": S, "dense": m})
    assert np.all(o[0, :, 128:256] == 0) and np.all(np.isneginf(lse[0, :, 128:256]))
    assert np.all(o[0, :, 300] == 0) and np.all(np.isneginf(lse[0, :, 300]))
    compare("O", o, ro, TOL_O)
    compare("LSE", lse, rl, TOL_LSE)


def test_per_head_dense_masks():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    S, Hq = 512, 3
    m = np.stack([bernoulli_mask(S, p, seed=s) for p, s in ((0.05, 1), (0.5, 2), (0.9, 3))])
    m[1, :, 256:] = 0
    q, k, v, _ = qkvdo(2, Hq, 1, S, 128, seed=6, with_do=False)
    info = bsa.mask_compile("dense", S, S, dense=torch.from_numpy(m).cuda())
    o, lse = bsa.fwd(q.cuda(), k.cuda(), v.cuda(), info)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), {"kind": "dense", "kv_len": S, "dense": m})
    compare("O", o, ro, TOL_O)
    compare("LSE", lse, rl, TOL_LSE)


def test_explicit_softmax_scale():
    need_gpu()
    q, k, v, _ = qkvdo(1, 2, 2, 384, 128, seed=7, with_do=False)
    spec = MaskSpec("causal")
    o, lse = run_gpu(q, k, v, spec, scale=0.05)
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), oracle_mask(spec, 384), scale=0.05)
    compare("O", o, ro, TOL_O)
    compare("LSE", lse, rl, TOL_LSE)


def test_repeat_run_is_deterministic():
    need_gpu()
    q, k, v, _ = qkvdo(1, 4, 2, 1024, 128, seed=8, with_do=False)
    a = run_gpu(q, k, v, MaskSpec("causal"))
    b = run_gpu(q, k, v, MaskSpec("causal"))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_maskinfo_shared_by_two_streams():
    """A MaskInfo's launch-time tile schedule is uploaded in stream order on
    the first launch's stream; a launch on another stream waits for that
    upload and gives the same result."""
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    q, k, v, _ = qkvdo(1, 4, 2, 1024, 128, seed=9, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    info = bsa.mask_compile("causal", 1024, 1024)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        o1, l1 = bsa.fwd(q, k, v, info)
    with torch.cuda.stream(s2):
        o2, l2 = bsa.fwd(q, k, v, info)
    torch.cuda.synchronize()
    assert bsa.get_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), {"kind": "causal", "kv_len": 1024})
    compare("O", o2.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", l2.cpu().numpy(), rl, TOL_LSE)


# ---------------------------------------------------------------- full size

def sampled_rows(S, n, rng):
    rows = set(rng.choice(S, size=n, replace=False).tolist())
    rows.update([0, 1, 127, 128, S - 129, S - 128, S - 1])
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", [n for n in WORKLOADS])
def test_full_size_workloads_sampled(name):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    w = WORKLOADS[name]
    q, k, v, _ = qkvdo(w.B, w.Hq, w.Hkv, w.S, w.D, seed=w.seed, with_do=False)
    dense = bernoulli_mask(w.S, w.mask.p, w.mask.seed) if w.mask.kind == "dense" else None
    dev_dense = None if dense is None else torch.from_numpy(dense).cuda()
    info = bsa.mask_compile(w.mask.kind, w.S, w.S, dense=dev_dense, **lib_mask_args(w.mask))
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = bsa.fwd(qd, kd, vd, info)
    assert bsa.get_device_error() == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all()
    rng = np.random.default_rng(0)
    group = w.Hq // w.Hkv
    heads = sorted({(0, 0), (w.B - 1, w.Hq - 1), (int(rng.integers(w.B)), int(rng.integers(w.Hq)))})
    mask = oracle_mask(w.mask, w.S, dense)
    for b, h in heads:
        rows = sampled_rows(w.S, 200, rng)
        g = h // group
        ro, rl = oatt.head_forward(f64(q[b, h]), f64(k[b, g]), f64(v[b, g]), oatt.mask_rows_for(mask, 0),
                                   1 / math.sqrt(w.D), rows=rows)
        compare(f"O[{b},{h}]", o[b, h, rows], ro, TOL_O)
        compare(f"LSE[{b},{h}]", lse[b, h, rows], rl, TOL_LSE)


def test_wait_timeout_reports_error_instead_of_hanging():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    bsa.get_device_error()
    bsa.set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        bsa.debug_wait_timeout()
        with pytest.raises(bsa.BsaError, match="timed out"):
            bsa.get_device_error()
    finally:
        bsa.set_wait_limit_ns(0)
    assert bsa.get_device_error() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_row_with_one_visible_key_returns_its_value_row_exactly(D):
    """Closed form: a query row that sees a single key has P = 1 on it, so
    O is that key's value row (bf16, exactly) and LSE its scaled score.
    Causal row 0 sees key 0 only; the scores are made negative for half of
    the heads (Q negated) so that the row maximum is below zero there too.
    The running maximum must be the row's true maximum for P = 1 to come
    out exactly (a maximum taken over anything else leaves P < 1, rounded
    to bf16, and O off by up to an ulp)."""
    need_gpu()
    B, Hq, Hkv, S = 2, 8, 4, 384
    q, k, v, _ = qkvdo(B, Hq, Hkv, S, D, seed=41, with_do=False)
    # s00 = q0 . k0 / sqrt(D): flip the sign of Q's row 0 where it is positive
    s00 = (q[:, :, 0].float() * k[:, :, 0].float().repeat_interleave(Hq // Hkv, dim=1)).sum(-1)
    flip = torch.ones((B, Hq), dtype=torch.bfloat16)
    flip[:, ::2] = torch.where(s00[:, ::2] > 0, -1.0, 1.0).to(torch.bfloat16)
    q[:, :, 0] = q[:, :, 0] * flip[..., None]
    o, lse = run_gpu(q, k, v, MaskSpec("causal"))
    v0 = v[:, :, 0].float().repeat_interleave(Hq // Hkv, dim=1).numpy()
    assert np.array_equal(o[:, :, 0], v0), np.abs(o[:, :, 0] - v0).max()
    want = (q[:, :, 0].double() * k[:, :, 0].double().repeat_interleave(Hq // Hkv, dim=1)).sum(-1) / math.sqrt(D)
    assert (want[:, ::2] < 0).all()
    assert np.abs(lse[:, :, 0] - want.numpy()).max() <= TOL_LSE
