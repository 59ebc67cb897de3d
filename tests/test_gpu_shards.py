"""GPU key-shard forward (bsa_fwd_partial) and merge (bsa_fwd_merge) vs the
fp64 oracle (oracle/shards.py).

Per shard, what is unique is compared: the row's m + log(l) (its
logsumexp over the shard, 1e-5) and o_acc / l (2e-2, like O); the kernel's m
is a lazy reference that may lag the true maximum, so m alone is not.  Rows
with no visible key in a shard must come back exactly as o_acc = 0, l = 0,
m = -inf.  The merge of the GPU shards must equal the unsharded forward of
the oracle (O 2e-2, LSE 1e-5), and the merge kernel alone, fed the oracle's
shards, must equal the oracle's merge.  At the benchmark's size (GQA 32/8
causal, 8192, two shards) the merge is compared with the unsharded GPU
forward in full and with the oracle on sampled rows.
"""
import numpy as np
import pytest
import torch

from helpers import TOL_LSE, TOL_O, compare, lib_mask_args, need_gpu, oracle_mask_args
from oracle import attention as oatt
from oracle import shards as osh
from workloads import MaskSpec, bernoulli_mask, qkvdo

pytestmark = pytest.mark.gpu


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


CASES = [
    # B, Hq, Hkv, S, D, mask, shard cuts (keys)
    (1, 2, 2, 512, 64, MaskSpec("causal"), [0, 256, 512]),
    (2, 4, 2, 384, 128, MaskSpec("causal"), [0, 128, 384]),
    (1, 4, 1, 640, 128, MaskSpec("local", left=200, right=70), [0, 256, 384, 640]),
    (1, 2, 2, 512, 128, MaskSpec("dense", p=0.3, seed=2), [0, 384, 512]),
    (1, 2, 2, 512, 64, MaskSpec("chunked", chunk=192), [0, 128, 256, 384, 512]),
]


def oracle_mask(spec, S, dense):
    m = {"kind": spec.kind, "kv_len": S}
    m.update(oracle_mask_args(spec, S))
    if dense is not None:
        m["dense"] = dense
    return m


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}/{c[2]}S{c[3]}D{c[4]}-{c[5].kind}-{len(c[6])-1}")
def test_shards_and_merge_match_oracle(case):
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    B, Hq, Hkv, S, D, spec, cuts = case
    q, k, v, _ = qkvdo(B, Hq, Hkv, S, D, seed=11, with_do=False)
    dense = bernoulli_mask(S, spec.p, spec.seed) if spec.kind == "dense" else None
    dd = None if dense is None else torch.from_numpy(np.ascontiguousarray(dense)).cuda()
    info = bsa.mask_compile(spec.kind, S, S, dense=dd, **lib_mask_args(spec))
    om = oracle_mask(spec, S, dense)
    qg = q.cuda()
    accs, ms, ls = [], [], []
    for a, b in zip(cuts, cuts[1:]):
        acc, m, l = bsa.fwd_partial(qg, k[:, :, a:b].contiguous().cuda(), v[:, :, a:b].contiguous().cuda(), info, a)
        assert bsa.get_device_error() == 0
        r_acc, r_m, r_l = osh.forward_partial(f64(q), f64(k), f64(v), om, a, b)
        acc, m, l = acc.cpu().numpy().astype(np.float64), m.cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64)
        empty = r_l == 0
        assert np.array_equal(l == 0, empty), "empty rows differ"
        assert np.all(np.isneginf(m[empty])) and np.all(acc[empty] == 0)
        live = ~empty
        with np.errstate(divide="ignore"):
            compare("shard lse", (m + np.log(l))[live], (r_m + np.log(r_l))[live], TOL_LSE)
        compare("shard o_acc/l", (acc / np.where(live, l, 1)[..., None])[live],
                (r_acc / np.where(live, r_l, 1)[..., None])[live], TOL_O)
        accs.append(acc); ms.append(m); ls.append(l)
    # merge on the GPU of the GPU shards vs the unsharded oracle forward
    st = lambda xs: torch.from_numpy(np.stack(xs).astype(np.float32)).cuda().contiguous()
    o, lse = bsa.fwd_merge(st(accs), st(ms), st(ls))
    ro, rl = oatt.forward(f64(q), f64(k), f64(v), om)
    compare("merged O", o.float().cpu().numpy(), ro, TOL_O)
    compare("merged LSE", lse.cpu().numpy(), rl, TOL_LSE)


def test_merge_kernel_alone_matches_oracle_merge():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    S, D = 512, 128
    q, k, v, _ = qkvdo(1, 2, 2, S, D, seed=12, with_do=False)
    om = {"kind": "local", "kv_len": S, "left": 150, "right": 0}
    parts = [osh.forward_partial(f64(q), f64(k), f64(v), om, a, a + 128) for a in range(0, S, 128)]
    accs, ms, ls = zip(*parts)
    st = lambda xs: torch.from_numpy(np.stack(xs).astype(np.float32)).cuda().contiguous()
    o, lse = bsa.fwd_merge(st(accs), st(ms), st(ls))
    ro, rl = osh.merge_partials(accs, ms, ls)
    # inputs rounded to fp32, output to bf16: O within a bf16 half-ulp plus fp32 rounding
    compare("O", o.float().cpu().numpy(), ro, 1e-2)
    compare("LSE", lse.cpu().numpy(), rl, TOL_LSE)


def test_two_shards_match_unsharded_forward_at_full_size():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    # the GQA causal 8192 shape, split in the middle of the key axis
    B, Hq, Hkv, S, D = 1, 32, 8, 8192, 128
    q, k, v, _ = qkvdo(B, Hq, Hkv, S, D, seed=13, with_do=False)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    info = bsa.mask_compile("causal", S, S)
    o_ref, lse_ref = bsa.fwd(q, k, v, info)
    h = S // 2
    p1 = bsa.fwd_partial(q, k[:, :, :h].contiguous(), v[:, :, :h].contiguous(), info, 0)
    p2 = bsa.fwd_partial(q, k[:, :, h:].contiguous(), v[:, :, h:].contiguous(), info, h)
    assert bsa.get_device_error() == 0
    o, lse = bsa.fwd_merge(*(torch.stack([a, b]) for a, b in zip(p1, p2)))
    # the second shard is empty for the first half of the queries
    assert torch.all(p2[2][:, :, :h] == 0) and torch.all(torch.isneginf(p2[1][:, :, :h]))
    assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O
    assert (lse - lse_ref).abs().max().item() <= 1e-4
    # and the merged result against the oracle on sampled rows of three
    # heads (both shards' sides of the cut, the ends of the axis)
    rng = np.random.default_rng(7)
    mask = {"kind": "causal", "kv_len": S}
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    for hq in (0, 13, Hq - 1):
        rows = np.array(sorted(set(rng.choice(S, size=120, replace=False).tolist())
                               | {0, 127, h - 1, h, h + 1, S - 1}))
        g = hq // (Hq // Hkv)
        ro, rl = oatt.head_forward(f64(q[0, hq]), f64(k[0, g]), f64(v[0, g]), oatt.mask_rows_for(mask, 0),
                                   1 / np.sqrt(D), rows=rows)
        compare(f"merged O[0,{hq}] vs oracle", on[0, hq, rows], ro, TOL_O)
        compare(f"merged LSE[0,{hq}] vs oracle", ln[0, hq, rows], rl, TOL_LSE)
