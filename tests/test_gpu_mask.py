"""GPU mask compiler vs the oracle: every MaskInfo array bit-exact, same dtypes.

Covers the workloads' masks in both orientations, planted dense masks with
empty, full and duplicated blocks (several heads, shrink on and off), the
integer-downcast boundaries, an all-empty mask and determinism.
"""
import numpy as np
import pytest
import torch

from helpers import lib_mask_args, need_gpu, oracle_mask_args
from oracle import mask_info as omi
from workloads import WORKLOADS, bernoulli_mask, planted_block_mask

pytestmark = pytest.mark.gpu


def compile_both(kind, q_len, kv_len, *, dense=None, orientation="fwd", shrink=True, okw=None, lkw=None):
    import block_sparse_attention_process_gb300 as bsa
    okw = okw or {}
    lkw = lkw or {}
    ref = omi.compile_mask_info(kind, q_len, kv_len, dense=dense, orientation=orientation, shrink_grid=shrink,
                                **okw)
    dev_dense = None
    if dense is not None:
        dev_dense = torch.from_numpy(np.ascontiguousarray(dense)).cuda()
    info = bsa.mask_compile(kind, q_len, kv_len, dense=dev_dense, orientation=orientation, shrink=shrink, **lkw)
    got = info.to_host()
    info.destroy()
    return ref, got


def assert_same(ref, got):
    assert got["width"] == ref.width
    assert (got["n_empty"], got["n_partial"], got["n_full"]) == (ref.n_empty, ref.n_partial, ref.n_full)
    for name in ("block_mask", "data_next"):
        r, g = getattr(ref, name), got[name]
        assert g.dtype == r.dtype, (name, g.dtype, r.dtype)
        assert np.array_equal(g, r), name
    if ref.mask_next is None:
        assert got["mask_next"] is None and got["partial_mask_blocks"] is None
    else:
        assert got["mask_next"].dtype == ref.mask_next.dtype
        assert np.array_equal(got["mask_next"], ref.mask_next)
        assert got["num_partial"] == ref.num_partial_blocks
        assert np.array_equal(got["partial_mask_blocks"], ref.partial_mask_blocks)
    assert np.array_equal(got["q_sequence"], ref.q_sequence)


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("orientation", ["fwd", "dkv"])
def test_workload_masks_bit_exact(name, orientation):
    need_gpu()
    w = WORKLOADS[name]
    dense = None
    if w.mask.kind == "dense":
        dense = bernoulli_mask(w.S, w.mask.p, w.mask.seed)
    ref, got = compile_both(w.mask.kind, w.S, w.S, dense=dense, orientation=orientation,
                            okw=oracle_mask_args(w.mask, w.S), lkw=lib_mask_args(w.mask))
    assert_same(ref, got)


def test_page_counts_on_gpu():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    c = bsa.mask_compile("causal", 8192, 8192).to_host()
    assert c["n_empty"] == 2016 and c["width"] == 64
    loc = bsa.mask_compile("local", 8192, 8192, local_left=1024, local_right=0).to_host()
    assert loc["width"] == 9
    dense = torch.from_numpy(bernoulli_mask(2048, 0.1, 1)).cuda()
    d = bsa.mask_compile("dense", 2048, 2048, dense=dense).to_host()
    assert d["n_partial"] == 256 and d["partial_mask_blocks"].nbytes == 4 * 1024 * 1024


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("orientation", ["fwd", "dkv"])
@pytest.mark.parametrize("shrink", [True, False])
def test_planted_dense_bit_exact(seed, orientation, shrink):
    need_gpu()
    heads, nq, nk = 3, 4, 6
    m = planted_block_mask(heads, nq, nk, seed=seed)
    ref, got = compile_both("dense", nq * 128, nk * 128, dense=m, orientation=orientation, shrink=shrink)
    assert_same(ref, got)


@pytest.mark.parametrize("kind,okw,lkw", [
    ("local", {"left": 200, "right": 70}, {"local_left": 200, "local_right": 70}),
    ("local", {"left": None, "right": 5}, {"local_left": None, "local_right": 5}),
    ("local", {"left": 0, "right": 0}, {"local_left": 0, "local_right": 0}),
    ("chunked", {"chunk": 192}, {"chunk": 192}),
    ("causal", {}, {}),
    ("full", {}, {}),
])
@pytest.mark.parametrize("orientation", ["fwd", "dkv"])
@pytest.mark.parametrize("shrink", [True, False])
def test_computable_masks_bit_exact(kind, okw, lkw, orientation, shrink):
    need_gpu()
    ref, got = compile_both(kind, 1152, 1152, orientation=orientation, shrink=shrink, okw=okw, lkw=lkw)
    assert_same(ref, got)


@pytest.mark.parametrize("cols", [128, 129])
def test_downcast_boundary(cols):
    need_gpu()
    dense = np.ones((128, cols * 128), np.uint8)
    ref, got = compile_both("dense", 128, cols * 128, dense=dense)
    assert_same(ref, got)


def test_mask_next_int16_when_256_partial_blocks():
    need_gpu()
    dense = bernoulli_mask(2048, 0.1, 1)
    ref, got = compile_both("dense", 2048, 2048, dense=dense)
    assert got["mask_next"].dtype == np.int16
    assert_same(ref, got)


def test_all_empty_mask():
    need_gpu()
    dense = np.zeros((256, 384), np.uint8)
    ref, got = compile_both("dense", 256, 384, dense=dense)
    assert got["width"] == 0
    assert_same(ref, got)


def test_nonbinary_dense_bytes_are_normalised():
    need_gpu()
    rng = np.random.default_rng(5)
    m = (rng.random((256, 256)) < 0.5).astype(np.uint8) * rng.integers(1, 255, (256, 256)).astype(np.uint8)
    ref, got = compile_both("dense", 256, 256, dense=m)
    assert_same(ref, got)


def test_compile_is_deterministic():
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    dense = torch.from_numpy(planted_block_mask(2, 5, 5, seed=9)).cuda()
    a = bsa.mask_compile("dense", 640, 640, dense=dense).to_host()
    b = bsa.mask_compile("dense", 640, 640, dense=dense).to_host()
    for k in ("block_mask", "data_next", "mask_next", "partial_mask_blocks"):
        assert np.array_equal(a[k], b[k])


def per_head_dense_mask(H, S, seed=0):
    """[H, S, S] uint8 with four kinds of heads: scattered Bernoulli(0.1)
    (every block partial and distinct), a causal pattern (all diagonal
    blocks partial and equal, shared across heads), planted blocks (zeros,
    ones, three repeated patterns, fresh random ones) and a band
    |q - k| <= 700 (repeating partial edge blocks)."""
    m = np.zeros((H, S, S), np.uint8)
    idx = np.arange(S)
    for h in range(H):
        kind = h % 4
        if kind == 0:
            m[h] = bernoulli_mask(S, 0.1, seed + h)
        elif kind == 1:
            m[h] = idx[:, None] >= idx[None, :]
        elif kind == 2:
            m[h] = planted_block_mask(1, S // 128, S // 128, seed=seed + h)[0]
        else:
            m[h] = np.abs(idx[:, None] - idx[None, :]) <= 700
    return m


@pytest.mark.parametrize("orientation", ["fwd", "dkv"])
def test_per_head_dense_mask_s8192_bit_exact(orientation):
    """Sixteen mask heads of 8192 x 8192 (1 GiB of mask bytes, 65536 blocks,
    tens of thousands partial): every MaskInfo array against the oracle."""
    need_gpu()
    H, S = 16, 8192
    m = per_head_dense_mask(H, S)
    ref, got = compile_both("dense", S, S, dense=m, orientation=orientation)
    assert got["heads"] == H
    assert_same(ref, got)


@pytest.mark.parametrize("bits", [0, 3])
def test_dedup_settles_shared_hashes_by_bytes(bits, tmp_path):
    """With the block hashes cut to `bits` bits (BSA_DEDUP_HASH_BITS, read
    when the library is loaded, hence a child process) different partial
    blocks share hashes; the first-occurrence search must still pick the
    first block with equal bytes."""
    need_gpu()
    import os
    import subprocess
    import sys
    from helpers import ROOT
    script = r'''
import sys, numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
from test_gpu_mask import compile_both, assert_same
from workloads import planted_block_mask, bernoulli_mask
for seed in (0, 1):
    m = planted_block_mask(3, 5, 7, seed=seed)
    for o in ("fwd", "dkv"):
        assert_same(*compile_both("dense", 5 * 128, 7 * 128, dense=m, orientation=o))
m = np.stack([bernoulli_mask(1024, 0.2, 9)] * 2)
assert_same(*compile_both("dense", 1024, 1024, dense=m))
print("ok")
'''.replace("ROOT", repr(ROOT))
    env = dict(os.environ, BSA_DEDUP_HASH_BITS=str(bits))
    r = subprocess.run([sys.executable, "-c", script], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_many_partial_blocks_with_duplicates_across_chunks():
    """More than a thousand partial blocks (the list, the slot numbering and
    the row order each span several 1024-entry chunks), many of them
    repeated across rows and heads."""
    need_gpu()
    H, nq, nk = 4, 24, 24
    rng = np.random.default_rng(5)
    pats = [(rng.random((128, 128)) < 0.5).astype(np.uint8) for _ in range(40)]
    m = np.zeros((H, nq * 128, nk * 128), np.uint8)
    for h in range(H):
        for i in range(nq):
            for j in range(nk):
                r = rng.random()
                blk = pats[int(rng.integers(0, 40))] if r < 0.7 else (
                    np.ones((128, 128), np.uint8) if r < 0.8 else np.zeros((128, 128), np.uint8))
                m[h, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] = blk
    for o in ("fwd", "dkv"):
        ref, got = compile_both("dense", nq * 128, nk * 128, dense=m, orientation=o)
        assert ref.n_partial > 1024 and got["num_partial"] == 40
        assert_same(ref, got)


@pytest.mark.parametrize("orientation", ["fwd", "dkv"])
@pytest.mark.parametrize("heads", [1, 3])
def test_rectangular_dense_bit_exact(orientation, heads):
    """S_q != S_kv (384 x 896): rows and columns have different extents in
    each orientation; a query block with no visible key and a key block no
    query sees are planted."""
    need_gpu()
    rng = np.random.default_rng(17 + heads)
    m = (rng.random((heads, 384, 896)) < 0.3).astype(np.uint8)
    m[:, 128:256, :] = 0
    m[:, :, 768:] = 0
    m[:, 256:, 128:256] = 1  # full blocks
    dense = m if heads > 1 else m[0]
    for shrink in (True, False):
        ref, got = compile_both("dense", 384, 896, dense=dense, orientation=orientation, shrink=shrink)
        assert_same(ref, got)


@pytest.mark.parametrize("orientation", ["fwd", "dkv"])
@pytest.mark.parametrize("case", ["causal_8192", "local_8192", "per_head_64x2048", "per_head_72x2048"])
def test_row_lengths_and_order(case, orientation):
    """The library's own row arrays, from which the launches build their tile
    schedules: row_len is each mask row's number of non-empty blocks (the
    oracle's count), row_order the rows by decreasing length, ties in
    increasing row order.  Up to 1024 rows one CTA sorts them (64 per-head
    masks of 16 block rows: exactly 1024); above that a counting sort over
    1024-row chunks does (72 x 16 = 1152 rows)."""
    need_gpu()
    import block_sparse_attention_process_gb300 as bsa
    kind, dense, S, kw, okw = "dense", None, 2048, {}, {}
    if case == "causal_8192":
        kind, S = "causal", 8192
    elif case == "local_8192":
        kind, S, kw, okw = "local", 8192, dict(local_left=1024, local_right=0), dict(left=1024, right=0)
    else:
        dense = per_head_dense_mask(int(case.split("_")[2].split("x")[0]), S)
    ref = omi.compile_mask_info(kind, S, S, dense=dense, orientation=orientation, **okw)
    dd = None if dense is None else torch.from_numpy(dense).cuda()
    info = bsa.mask_compile(kind, S, S, dense=dd, orientation=orientation, **kw)
    host = {k: v.cpu().numpy() for k, v in info.arrays().items() if k in ("row_len", "row_order")}
    info.destroy()
    want_len = (ref.labels_unshrunk != 0).sum(axis=-1).reshape(-1)
    assert np.array_equal(host["row_len"], want_len)
    assert np.array_equal(host["row_order"], np.argsort(-want_len, kind="stable"))
