"""GPU forward and backward with the logit soft cap and attention sinks vs
the fp64 oracle (oracle/attention.py, the ``logits_soft_cap`` and
``softmax_aux`` readings): O and the gradients within 2e-2, LSE within
1e-5, the sinks' gradient within 1% of its largest entry (it sums Dsum,
which the GPU computes from bf16 O, over every row of a head)."""
import numpy as np
import pytest
import torch

from helpers import TOL_GRAD, TOL_LSE, TOL_O, compare, lib_mask_args, need_gpu, oracle_mask_args
from oracle import attention as oatt
from workloads import MaskSpec, bernoulli_mask, qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


CASES = [
    # B, Hq, Hkv, S, D, mask, cap, sink shape
    (1, 2, 2, 512, 128, MaskSpec("causal"), 2.0, None),
    (1, 4, 2, 384, 128, MaskSpec("local", left=150, right=20), None, (2, 3)),
    (2, 4, 1, 256, 64, MaskSpec("causal"), 1.0, (2,)),
    (1, 2, 2, 512, 128, MaskSpec("dense", p=0.3, seed=2), 1.5, (2, 1)),
    (1, 4, 4, 384, 64, MaskSpec("chunked", chunk=128), 3.0, (4, 2)),
]


def setup(case, seed):
    B, Hq, Hkv, S, D, spec, cap, sink_shape = case
    q, k, v, do = qkvdo(B, Hq, Hkv, S, D, seed=seed)
    dense = bernoulli_mask(S, spec.p, spec.seed) if spec.kind == "dense" else None
    om = {"kind": spec.kind, "kv_len": S}
    om.update(oracle_mask_args(spec, S))
    if dense is not None:
        om["dense"] = dense
    sinks = None
    if sink_shape is not None:
        sinks = torch.from_numpy(np.random.default_rng(seed).standard_normal(sink_shape).astype(np.float32) * 2)
    return q, k, v, do, dense, om, sinks


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[5].kind}-cap{c[6]}-sinks{c[7]}-D{c[4]}")
def test_forward_and_backward(case):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    B, Hq, Hkv, S, D, spec, cap, _ = case
    q, k, v, do, dense, om, sinks = setup(case, 31)
    dd = None if dense is None else torch.from_numpy(np.ascontiguousarray(dense)).cuda()
    info = bsa.mask_compile(spec.kind, S, S, dense=dd, **lib_mask_args(spec))
    dkv = bsa.mask_compile(spec.kind, S, S, dense=dd, orientation="dkv", **lib_mask_args(spec))
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    sg = None if sinks is None else sinks.cuda()
    o, lse = bsa.fwd(qg, kg, vg, info, logits_soft_cap=cap, sinks=sg)
    zs = None if sinks is None else sinks.double().numpy()
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), om, cap=cap, sinks=zs)
    compare("O", o.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)
    out = bsa.bwd(qg, kg, vg, o, lse, dog, info, dkv, logits_soft_cap=cap, sinks=sg, grad_fp32=True)
    assert bsa.get_device_error() == 0
    ref = oatt.backward(f64(q), f64(k), f64(v), f64(do), om, cap=cap, sinks=zs)
    for name, g, r in zip(("dQ", "dK", "dV"), out[:3], ref[:3]):
        compare(name, g.cpu().numpy(), r, TOL_GRAD)
    if sinks is not None:
        got, want = out[3].cpu().numpy().astype(np.float64), ref[3]
        assert np.abs(got - want).max() <= 1e-2 * np.abs(want).max() + 1e-4, (got, want)


def test_rows_with_no_visible_key_take_the_sinks_logsumexp():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    # local window right-only (keys k >= q+1 .. q+64): the last query block sees
    # nothing in its last rows; a planted dense mask with empty block rows too
    S, D = 256, 64
    q, k, v, _ = qkvdo(1, 2, 1, S, D, seed=33, with_do=False)
    dense = np.zeros((S, S), np.uint8)
    dense[:128, :64] = 1  # query block 1 is empty
    info = bsa.mask_compile("dense", S, S, dense=torch.from_numpy(dense).cuda())
    z = torch.tensor([0.25, -1.0], dtype=torch.float32)
    o, lse = bsa.fwd(q.cuda(), k.cuda(), v.cuda(), info, sinks=z.cuda())
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), {"kind": "dense", "kv_len": S, "dense": dense},
                          sinks=z.double().numpy())
    want = float(np.log(np.exp(z.double().numpy()).sum()))
    assert np.allclose(lse.cpu().numpy()[:, :, 128:], want, atol=1e-6)
    assert torch.all(o[:, :, 128:] == 0)
    compare("O", o.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)


def test_soft_cap_in_a_key_shard():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    from oracle import shards as osh
    S, D = 512, 128
    q, k, v, _ = qkvdo(1, 2, 2, S, D, seed=34, with_do=False)
    info = bsa.mask_compile("causal", S, S)
    parts = [bsa.fwd_partial(q.cuda(), k[:, :, a:a + 256].contiguous().cuda(), v[:, :, a:a + 256].contiguous().cuda(),
                             info, a, logits_soft_cap=3.0) for a in (0, 256)]
    o, lse = bsa.fwd_merge(*(torch.stack(list(x)) for x in zip(*parts)))
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), {"kind": "causal", "kv_len": S}, cap=3.0)
    compare("O", o.float().cpu().numpy(), ro, TOL_O)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)
