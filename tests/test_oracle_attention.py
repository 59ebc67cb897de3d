"""Pins for the attention oracle (CPU only).

Each check ties the fp64 oracle to something outside it:
* closed forms with Q = 0 (uniform weights over the visible keys);
* invariants: rows of P sum to one, constant V gives constant O;
* special cases that are library routines: torch's scaled_dot_product_attention
  in fp64 (no mask, is_causal, boolean attn_mask) for O, and torch
  autograd through it for dQ, dK, dV (GQA by repeating K/V heads, which makes
  autograd sum the group);
* central finite differences of the oracle's own forward for its backward.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as att
from oracle import masks
from workloads import bernoulli_mask, qkvdo


def f64(t):
    return t.to(torch.float64).numpy()


def mask_dict(kind, S, **kw):
    d = {"kind": kind, "kv_len": S}
    d.update(kw)
    return d


@pytest.mark.parametrize("kind,kw", [("causal", {}), ("local", {"left": 100, "right": 0}),
                                     ("chunked", {"chunk": 96}), ("full", {})])
def test_zero_query_closed_form(kind, kw):
    # With Q = 0 every visible score is 0, so P is uniform over the visible
    # keys: O_i = mean of V over them and LSE_i = ln(count).
    S, D = 256, 32
    rng = np.random.default_rng(3)
    q = np.zeros((1, 1, S, D))
    k = rng.standard_normal((1, 1, S, D))
    v = rng.standard_normal((1, 1, S, D))
    o, lse = att.forward(q, k, v, mask_dict(kind, S, **kw))
    full = masks.materialise(kind, S, S, **kw)
    for i in range(S):
        vis = np.nonzero(full[i])[0]
        assert np.allclose(o[0, 0, i], v[0, 0, vis].mean(axis=0), atol=1e-12)
        assert abs(lse[0, 0, i] - math.log(vis.size)) < 1e-12
    if kind == "causal":
        assert np.allclose(lse[0, 0], np.log(np.arange(1, S + 1)), atol=1e-12)


def test_probs_rows_sum_to_one_and_respect_mask():
    S, D = 384, 64
    q, k, v, _ = qkvdo(1, 1, 1, S, D, seed=5, with_do=False)
    dense = bernoulli_mask(S, 0.2, seed=4)
    mrows = att.mask_rows_for(mask_dict("dense", S, dense=dense), 0)
    p = att.head_probs(f64(q)[0, 0], f64(k)[0, 0], mrows, 1 / math.sqrt(D))
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(p[dense == 0] == 0)


def test_constant_v_gives_constant_o():
    S, D = 256, 64
    q, k, _, _ = qkvdo(1, 2, 2, S, D, seed=2, with_do=False)
    v = np.full((1, 2, S, D), 0.375)
    o, _ = att.forward(f64(q), f64(k), v, mask_dict("causal", S))
    assert np.allclose(o, 0.375, atol=1e-12)


def _sdpa(q, k, v, attn_mask=None, is_causal=False, scale=None):
    return F.scaled_dot_product_attention(q, k, v, attn_mask=attn_mask, is_causal=is_causal,
                                          scale=scale)


@pytest.mark.parametrize("case", ["full", "causal", "dense"])
def test_forward_matches_sdpa_fp64(case):
    B, H, S, D = 2, 3, 256, 64
    q, k, v, _ = qkvdo(B, H, H, S, D, seed=11, with_do=False)
    qd, kd, vd = (t.to(torch.float64) for t in (q, k, v))
    if case == "full":
        ref = _sdpa(qd, kd, vd)
        m = mask_dict("full", S)
    elif case == "causal":
        ref = _sdpa(qd, kd, vd, is_causal=True)
        m = mask_dict("causal", S)
    else:
        dense = bernoulli_mask(S, 0.1, seed=1)
        ref = _sdpa(qd, kd, vd, attn_mask=torch.from_numpy(dense != 0))
        m = mask_dict("dense", S, dense=dense)
    o, _ = att.forward(f64(q), f64(k), f64(v), m)
    assert np.abs(o - ref.numpy()).max() < 1e-12


def test_lse_matches_logsumexp_of_sdpa_weights():
    # exp(s - lse) must be the softmax torch computes; check via its weights.
    S, D = 256, 32
    q, k, v, _ = qkvdo(1, 1, 1, S, D, seed=9, with_do=False)
    s = (q.double()[0, 0] @ k.double()[0, 0].T) / math.sqrt(D)
    s = s.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=1).numpy()
    _, lse = att.forward(f64(q), f64(k), f64(v), mask_dict("causal", S))
    assert np.abs(lse[0, 0] - ref_lse).max() < 1e-12


@pytest.mark.parametrize("Hq,Hkv,case", [(2, 2, "causal"), (4, 2, "local"), (4, 1, "dense")])
def test_backward_matches_autograd_fp64(Hq, Hkv, case):
    B, S, D = 1, 256, 32
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=13)
    if case == "causal":
        m = mask_dict("causal", S)
        bool_mask = torch.ones(S, S, dtype=torch.bool).tril()
    elif case == "local":
        m = mask_dict("local", S, left=50, right=10)
        bool_mask = torch.from_numpy(masks.materialise("local", S, S, left=50, right=10))
    else:
        dense = bernoulli_mask(S, 0.15, seed=3)
        m = mask_dict("dense", S, dense=dense)
        bool_mask = torch.from_numpy(dense != 0)
    qd = q.double().requires_grad_(True)
    kd = k.double().requires_grad_(True)
    vd = v.double().requires_grad_(True)
    rep = Hq // Hkv
    out = _sdpa(qd, kd.repeat_interleave(rep, dim=1), vd.repeat_interleave(rep, dim=1),
                attn_mask=bool_mask)
    out.backward(do.double())
    dq, dk, dv = att.backward(f64(q), f64(k), f64(v), f64(do), m)
    assert np.abs(dq - qd.grad.numpy()).max() < 1e-10
    assert np.abs(dk - kd.grad.numpy()).max() < 1e-10
    assert np.abs(dv - vd.grad.numpy()).max() < 1e-10


def test_backward_finite_differences():
    # loss = sum(O * dO); central differences of the oracle's forward.
    rng = np.random.default_rng(0)
    S, D = 128, 16
    q = rng.standard_normal((1, 1, S, D))
    k = rng.standard_normal((1, 1, S, D))
    v = rng.standard_normal((1, 1, S, D))
    do = rng.standard_normal((1, 1, S, D))
    m = mask_dict("local", S, left=40, right=3)
    dq, dk, dv = att.backward(q, k, v, do, m)

    def loss(q_, k_, v_):
        o, _ = att.forward(q_, k_, v_, m)
        return float((o * do).sum())

    eps = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = (0, 0, int(rng.integers(S)), int(rng.integers(D)))
            ap = arr.copy(); ap[idx] += eps
            am = arr.copy(); am[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = ap
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = am
            fd = (loss(**{f"{x}_": args_p[x] for x in "qkv"})
                  - loss(**{f"{x}_": args_m[x] for x in "qkv"})) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_fully_masked_row_gives_zero_output_and_minus_inf_lse():
    S, D = 256, 32
    q, k, v, do = qkvdo(1, 1, 1, S, D, seed=1)
    dense = np.ones((S, S), np.uint8)
    dense[5] = 0
    m = mask_dict("dense", S, dense=dense)
    o, lse = att.forward(f64(q), f64(k), f64(v), m)
    assert np.all(o[0, 0, 5] == 0) and lse[0, 0, 5] == -np.inf
    dq, dk, dv = att.backward(f64(q), f64(k), f64(v), f64(do), m)
    assert np.all(dq[0, 0, 5] == 0)
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def test_rowsum_matches_definition_on_integers():
    do = np.arange(24, dtype=np.float64).reshape(1, 1, 3, 8)
    o = np.ones((1, 1, 3, 8))
    assert att.rowsum_do_o(do, o)[0, 0].tolist() == [28.0, 92.0, 156.0]
