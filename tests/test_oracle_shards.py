"""Pins of the key-sharded partial attention and its merge (oracle/shards.py),
following "Splash Attention: When the Mask Stops Being Arithmetic and
Becomes the Loop", section "What does ring attention add on top of the
splash kernel?": per-shard maximum, normaliser and unnormalised
accumulator, merged with the flash rescaling and one final divide; a shard
with no active key contributes zeros.

Checked against what does not depend on the shard code: the unsharded
forward (a different code path: one softmax over all keys), a pure-Python
loop on tiny inputs, and closed forms with Q = 0.
"""
import math

import numpy as np
import pytest

from oracle import attention as oatt
from oracle import shards as osh
from workloads import bernoulli_mask, qkvdo


def f64(t):
    return t.float().numpy().astype(np.float64)


CASES = [
    ("causal", {}, 1, 2, 2, 512, 64),
    ("local", {"left": 100, "right": 30}, 1, 2, 1, 384, 64),
    ("chunked", {"chunk": 128}, 2, 2, 2, 256, 32),
]


@pytest.mark.parametrize("kind,params,B,Hq,Hkv,S,D", CASES)
@pytest.mark.parametrize("cuts", [[0, 512], [0, 128, 512], [0, 256, 384, 512]])
def test_merge_of_shards_equals_unsharded_forward(kind, params, B, Hq, Hkv, S, D, cuts):
    cuts = [min(c, S) for c in cuts]
    cuts[-1] = S
    q, k, v, _ = qkvdo(B, Hq, Hkv, S, D, seed=5, with_do=False)
    q, k, v = f64(q), f64(k), f64(v)
    mask = {"kind": kind, "kv_len": S, **params}
    o_ref, lse_ref = oatt.forward(q, k, v, mask)
    parts = [osh.forward_partial(q, k, v, mask, a, b) for a, b in zip(cuts, cuts[1:]) if b > a]
    o, lse = osh.merge_partials(*zip(*parts))
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
    assert np.allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)


def test_dense_mask_shards_and_order_independence():
    S = 256
    q, k, v, _ = qkvdo(1, 2, 2, S, 32, seed=6, with_do=False)
    q, k, v = f64(q), f64(k), f64(v)
    mask = {"kind": "dense", "kv_len": S, "dense": bernoulli_mask(S, 0.2, 3)}
    parts = [osh.forward_partial(q, k, v, mask, a, a + 128) for a in (0, 128)]
    o1, l1 = osh.merge_partials(*zip(*parts))
    o2, l2 = osh.merge_partials(*zip(*parts[::-1]))
    o_ref, lse_ref = oatt.forward(q, k, v, mask)
    assert np.allclose(o1, o_ref, atol=1e-12) and np.allclose(l1, lse_ref, atol=1e-12)
    assert np.allclose(o1, o2, atol=1e-14) and np.allclose(l1, l2, atol=1e-14)


def test_empty_shard_contributes_zeros():
    # causal: query rows < 256 see no key of the shard [256, 384)
    S = 384
    q, k, v, _ = qkvdo(1, 1, 1, S, 16, seed=7, with_do=False)
    q, k, v = f64(q), f64(k), f64(v)
    mask = {"kind": "causal", "kv_len": S}
    acc, m, l = osh.forward_partial(q, k, v, mask, 256, 384)
    assert np.all(acc[0, 0, :256] == 0) and np.all(l[0, 0, :256] == 0) and np.all(np.isneginf(m[0, 0, :256]))
    assert np.all(l[0, 0, 256:] >= 1.0)  # the row's own key is visible; its weight is exp(0) at the max
    # merging the empty shard changes nothing
    a0, m0, l0 = osh.forward_partial(q, k, v, mask, 0, 256)
    o_a, lse_a = osh.merge_partials([a0], [m0], [l0])
    o_b, lse_b = osh.merge_partials([a0, acc], [m0, m], [l0, l])
    assert np.array_equal(o_a[0, 0, :256], o_b[0, 0, :256]) and np.array_equal(lse_a[0, 0, :256], lse_b[0, 0, :256])


def test_all_empty_row_gives_zero_and_minus_inf():
    z = np.zeros((3, 4))
    ninf = np.full(3, -np.inf)
    o, lse = osh.merge_partials([z, z], [ninf, ninf], [np.zeros(3), np.zeros(3)])
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_zero_queries_closed_form():
    # Q = 0: every visible score is 0, so m = 0, l = number of visible keys,
    # acc = sum of their value rows
    S, D = 256, 8
    rng = np.random.default_rng(0)
    q = np.zeros((1, 1, S, D))
    k = rng.standard_normal((1, 1, S, D))
    v = rng.standard_normal((1, 1, S, D))
    acc, m, l = osh.forward_partial(q, k, v, {"kind": "causal", "kv_len": S}, 128, 256)
    for i in (0, 127, 128, 200, 255):
        vis = [j for j in range(128, 256) if j <= i]
        if not vis:
            assert l[0, 0, i] == 0 and np.isneginf(m[0, 0, i])
        else:
            assert m[0, 0, i] == 0 and l[0, 0, i] == len(vis)
            assert np.allclose(acc[0, 0, i], v[0, 0, vis].sum(axis=0), atol=1e-12)


def test_brute_force_loop_tiny():
    S, D = 128, 4
    rng = np.random.default_rng(1)
    q, k, v = (rng.standard_normal((1, 1, S, D)) for _ in range(3))
    mask = {"kind": "local", "kv_len": S, "left": 20, "right": 5}
    scale = 0.37
    acc, m, l = osh.forward_partial(q, k, v, mask, 40, 100, scale=scale)
    for i in (0, 10, 45, 99, 127):
        vis = [j for j in range(40, 100) if i - 20 <= j <= i + 5]
        if not vis:
            assert l[0, 0, i] == 0
            continue
        s = [scale * sum(q[0, 0, i, d] * k[0, 0, j, d] for d in range(D)) for j in vis]
        mm = max(s)
        w = [math.exp(x - mm) for x in s]
        assert abs(m[0, 0, i] - mm) < 1e-12 and abs(l[0, 0, i] - sum(w)) < 1e-12
        for d in range(D):
            assert abs(acc[0, 0, i, d] - sum(wj * v[0, 0, j, d] for wj, j in zip(w, vis))) < 1e-12
