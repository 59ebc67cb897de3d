"""Pins of the soft cap and attention sinks in the oracle (oracle/attention.py),
the arguments ``logits_soft_cap`` and ``softmax_aux`` of the EasyDeL
``blocksparse_attention`` operator.  The page names them without formulas;
the readings checked here: the cap maps each visible scaled score s to
c*tanh(s/c); sinks are extra logits of each row in the normaliser, with no
value.

Checked against an independent formulation (torch autograd in fp64 through
tanh, a sink column concatenated to the scores and a softmax), closed forms
with Q = 0, limits (c -> inf, z -> -inf), an identity linking the sink and
sink-free results, and finite differences of the sink gradient.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import masks as omasks
from workloads import qkvdo


def f64(t):
    return t.to(torch.float64).numpy()


def torch_reference(q, k, v, do, allowed, scale, cap, sinks):
    """Plain torch fp64 with autograd: O, LSE and dq, dk, dv, dsinks (one kv group)."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    z = None if sinks is None else torch.tensor(sinks, dtype=torch.float64, requires_grad=True)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    kk = k.repeat_interleave(g, dim=1)
    vv = v.repeat_interleave(g, dim=1)
    s = scale * q @ kk.transpose(-1, -2)
    if cap:
        s = cap * torch.tanh(s / cap)
    s = s.masked_fill(~torch.tensor(allowed), -math.inf)
    if z is not None:
        zz = z.repeat_interleave(g, dim=0) if z.dim() == 2 else z.expand(Hq, -1)
        zcol = zz[None, :, None, :].expand(B, Hq, S, zz.shape[-1])
        full = torch.cat([s, zcol], dim=-1)
    else:
        full = s
    lse = torch.logsumexp(full, dim=-1)
    p = torch.exp(s - lse[..., None])
    o = p @ vv
    (o * torch.tensor(do)).sum().backward()
    out = [o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()]
    out.append(None if z is None else z.grad.numpy())
    return out


@pytest.mark.parametrize("cap,sink_shape", [(None, (2, 3)), (5.0, None), (2.0, (3,)), (8.0, (2, 1))])
def test_matches_torch_autograd(cap, sink_shape):
    B, Hq, Hkv, S, D = 1, 4, 2, 256, 16
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=21)
    q, k, v, do = f64(q) * 2.0, f64(k), f64(v), f64(do)   # larger scores so the cap matters
    rng = np.random.default_rng(4)
    sinks = None if sink_shape is None else rng.standard_normal(sink_shape) * 2.0
    mask = {"kind": "local", "kv_len": S, "left": 40, "right": 10}
    allowed = omasks.rows("local", np.arange(S), S, left=40, right=10)
    scale = 1 / math.sqrt(D)
    o, lse = oatt.forward(q, k, v, mask, cap=cap, sinks=sinks)
    grads = oatt.backward(q, k, v, do, mask, cap=cap, sinks=sinks)
    ref = torch_reference(q, k, v, do, np.broadcast_to(allowed, (B, Hq, S, S)), scale, cap, sinks)
    assert np.allclose(o, ref[0], atol=1e-12) and np.allclose(lse, ref[1], atol=1e-12)
    for got, want in zip(grads[:3], ref[2:5]):
        assert np.allclose(got, want, atol=1e-11)
    if sinks is not None:
        assert np.allclose(grads[3], ref[5], atol=1e-11)


def test_zero_queries_with_one_sink_closed_form():
    # Q = 0: every visible score is 0 (and tanh(0) = 0), so the row's
    # normaliser is n_visible + e^z and O is the mean of the visible values
    # shrunk by n / (n + e^z)
    S, D, z = 128, 8, 0.7
    rng = np.random.default_rng(2)
    q = np.zeros((1, 1, S, D))
    k = rng.standard_normal((1, 1, S, D))
    v = rng.standard_normal((1, 1, S, D))
    o, lse = oatt.forward(q, k, v, {"kind": "causal", "kv_len": S}, cap=3.0, sinks=np.array([z]))
    for i in (0, 5, 127):
        n = i + 1
        assert abs(lse[0, 0, i] - math.log(n + math.exp(z))) < 1e-12
        assert np.allclose(o[0, 0, i], v[0, 0, :n].sum(axis=0) / (n + math.exp(z)), atol=1e-12)


def test_limits():
    S, D = 256, 16
    q, k, v, _ = qkvdo(1, 2, 2, S, D, seed=22, with_do=False)
    q, k, v = f64(q), f64(k), f64(v)
    mask = {"kind": "causal", "kv_len": S}
    o0, l0 = oatt.forward(q, k, v, mask)
    o1, l1 = oatt.forward(q, k, v, mask, cap=1e9)
    o2, l2 = oatt.forward(q, k, v, mask, sinks=np.array([-1e4, -1e4]))
    assert np.allclose(o0, o1, atol=1e-12) and np.allclose(l0, l1, atol=1e-12)
    assert np.allclose(o0, o2, atol=1e-12) and np.allclose(l0, l2, atol=1e-12)


def test_sink_identity_against_sink_free_forward():
    # lse_z = logaddexp(lse, logsumexp(z)) and O_z = O * exp(lse - lse_z)
    S, D = 256, 16
    q, k, v, _ = qkvdo(1, 2, 1, S, D, seed=23, with_do=False)
    q, k, v = f64(q), f64(k), f64(v)
    mask = {"kind": "chunked", "kv_len": S, "chunk": 96}
    z = np.array([[0.3, -1.2, 2.0]])
    o0, l0 = oatt.forward(q, k, v, mask)
    oz, lz = oatt.forward(q, k, v, mask, sinks=z)
    lsz = np.log(np.exp(z[0]).sum())
    assert np.allclose(lz, np.logaddexp(l0, lsz), atol=1e-12)
    assert np.allclose(oz, o0 * np.exp(l0 - lz)[..., None], atol=1e-12)


def test_sink_gradient_finite_differences():
    S, D = 128, 8
    q, k, v, do = qkvdo(1, 2, 1, S, D, seed=24)
    q, k, v, do = f64(q), f64(k), f64(v), f64(do)
    mask = {"kind": "local", "kv_len": S, "left": 20, "right": 0}
    z = np.array([[0.5, -0.4]])
    _, _, _, dz = oatt.backward(q, k, v, do, mask, cap=4.0, sinks=z)
    eps = 1e-6
    for j in range(2):
        zp, zm = z.copy(), z.copy()
        zp[0, j] += eps
        zm[0, j] -= eps
        fp = (oatt.forward(q, k, v, mask, cap=4.0, sinks=zp)[0] * do).sum()
        fm = (oatt.forward(q, k, v, mask, cap=4.0, sinks=zm)[0] * do).sum()
        assert abs((fp - fm) / (2 * eps) - dz[0, j]) < 1e-6
