"""Pins for the MaskInfo oracle (CPU only).

The oracle is held to things other than itself:
* the block counts and grid widths the splash-attention explainer prints
  (tests/golden/page_counts.json);
* closed forms for causal, local-window and chunked-causal block counts,
  derived by hand in the comments below;
* hand-built masks whose labels, stack slots, next-block pointers and
  shrunk arrays are known by construction;
* a round trip: decoding MaskInfo back into an element mask must give the
  mask it was compiled from.
"""
import json
import os

import numpy as np
import pytest

from oracle import mask_info as mi
from workloads import bernoulli_mask, planted_block_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_counts.json")
B = 128


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Numbers printed on the page
# --------------------------------------------------------------------------

def test_page_causal_8192_skips_2016_of_4096():
    g = golden()["causal_8192_empty"]
    info = mi.compile_mask_info("causal", g["q_len"], g["kv_len"])
    total = info.n_empty + info.n_partial + info.n_full
    assert total == g["total_blocks"]
    assert info.n_empty == g["empty_blocks"]


def test_page_causal_8192_does_not_shrink():
    g = golden()["causal_8192_no_shrink"]
    info = mi.compile_mask_info("causal", g["q_len"], g["kv_len"])
    assert g["kv_len"] // B == g["grid_width_before"]
    assert info.width == g["grid_width_after"]


def test_page_local_1024_shrinks_64_to_9():
    g = golden()["local_1024_8192_shrink"]
    m = g["mask"]
    info = mi.compile_mask_info("local", g["q_len"], g["kv_len"], left=m["left"], right=m["right"])
    assert g["kv_len"] // B == g["grid_width_before"]
    assert info.width == g["grid_width_after"]
    assert info.block_mask.shape == (1, 64, 9)


def test_page_bernoulli_2048_all_partial_4mib():
    g = golden()["bernoulli_2048_partial"]
    dense = bernoulli_mask(g["q_len"], g["mask"]["p"], g["mask"]["seed"])
    info = mi.compile_mask_info("dense", g["q_len"], g["kv_len"], dense=dense)
    assert info.n_partial == g["partial_blocks"]
    assert info.n_empty == g["skipped_blocks"]
    assert info.n_partial + info.n_full == g["visited_blocks"]
    assert info.partial_mask_blocks.nbytes == g["partial_mask_bytes"]
    assert info.width == g["grid_width_after"]
    # mask_next's largest slot is 255: it no longer fits int8
    assert info.mask_next.dtype == np.int16
    assert info.data_next.dtype == np.int8


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("S", [512, 4096])
def test_causal_closed_form(S):
    # n block rows: the strictly upper triangle is empty (n(n-1)/2 blocks),
    # the diagonal is mixed (n), the strictly lower triangle full (n(n-1)/2).
    n = S // B
    info = mi.compile_mask_info("causal", S, S)
    assert (info.n_empty, info.n_partial, info.n_full) == (n * (n - 1) // 2, n, n * (n - 1) // 2)
    assert info.width == n
    # row i visits columns 0..i; the label is 2 below the diagonal, 1 on it
    for i in range(n):
        assert list(info.data_next[0, i, :i + 1]) == list(range(i + 1))
        assert list(info.block_mask[0, i, :i + 1]) == [2] * i + [1]
        assert all(info.block_mask[0, i, i + 1:] == 0)
        assert all(info.data_next[0, i, i + 1:] == i)


def test_local_closed_form_8192():
    # Window q-1024 <= k <= q at 128-blocks (1024 = 8 blocks).  Block row i
    # touches key blocks i-8 .. i.  Block j is full iff 128j >= 128i+127-1024
    # and 128j+127 <= 128i, i.e. i-7 <= j <= i-1 (7 blocks); j = i-8 and
    # j = i are mixed.  Rows i < 8 lose the columns below 0: i full and 1
    # mixed.  Full = 56*7 + (0+...+7) = 420; mixed = 56*2 + 8 = 120.
    info = mi.compile_mask_info("local", 8192, 8192, left=1024, right=0)
    assert (info.n_full, info.n_partial) == (420, 120)
    assert info.n_empty == 4096 - 540
    assert info.width == 9
    i = 20
    assert list(info.data_next[0, i]) == list(range(i - 8, i + 1))
    assert list(info.block_mask[0, i]) == [1] + [2] * 7 + [1]


def test_local_exclusive_bound_gives_same_counts():
    # Reading the window as q-1023 <= k <= q changes no block count.
    a = mi.compile_mask_info("local", 8192, 8192, left=1024, right=0)
    b = mi.compile_mask_info("local", 8192, 8192, left=1023, right=0)
    assert (a.n_empty, a.n_partial, a.n_full, a.width) == (b.n_empty, b.n_partial, b.n_full, b.width)


def test_chunked_closed_form_16384():
    # Chunk 2048 = 16 blocks: each of the 8 chunks is a causal 16x16 block
    # square on the diagonal (16 mixed, 120 full), everything else empty.
    info = mi.compile_mask_info("chunked", 16384, 16384, chunk=2048)
    assert (info.n_partial, info.n_full) == (8 * 16, 8 * 120)
    assert info.n_empty == 128 * 128 - 8 * 136
    assert info.width == 16
    # max data_next is 127 (the last block column): still int8
    assert info.data_next.dtype == np.int8
    assert info.data_next.max() == 127


@pytest.mark.parametrize("cols,dtype", [(128, np.int8), (129, np.int16)])
def test_downcast_boundary(cols, dtype):
    # One query block against `cols` key blocks, all visible: data_next holds
    # 0..cols-1, so 127 still fits int8 and 128 needs int16.
    info = mi.compile_mask_info("full", 128, cols * 128)
    assert info.data_next.max() == cols - 1
    assert info.data_next.dtype == dtype
    assert info.block_mask.dtype == np.int8


# --------------------------------------------------------------------------
# Hand-built mask with known answers
# --------------------------------------------------------------------------

def _hand_mask():
    rng = np.random.default_rng(7)
    Z = np.zeros((B, B), np.uint8)
    O = np.ones((B, B), np.uint8)
    A = (rng.random((B, B)) < 0.5).astype(np.uint8)
    Bp = (rng.random((B, B)) < 0.5).astype(np.uint8)
    C = (rng.random((B, B)) < 0.5).astype(np.uint8)
    grid = [[Z, A, O, A],
            [Z, Z, Z, Z],
            [Bp, Z, A.copy(), Z],
            [O, Z, Z, C]]
    m = np.block(grid)
    return m, (A, Bp, C)


def test_hand_mask_fwd():
    m, (A, Bp, C) = _hand_mask()
    info = mi.compile_mask_info("dense", 512, 512, dense=m)
    assert info.labels_unshrunk[0].tolist() == [[0, 1, 2, 1], [0, 0, 0, 0], [1, 0, 1, 0], [2, 0, 0, 1]]
    assert info.num_partial_blocks == 3
    assert np.array_equal(info.partial_mask_blocks[0], A)
    assert np.array_equal(info.partial_mask_blocks[1], Bp)
    assert np.array_equal(info.partial_mask_blocks[2], C)
    assert info.width == 3
    assert info.block_mask[0].tolist() == [[1, 2, 1], [0, 0, 0], [1, 1, 0], [2, 1, 0]]
    assert info.data_next[0].tolist() == [[1, 2, 3], [0, 0, 0], [0, 2, 2], [0, 3, 3]]
    assert info.mask_next[0].tolist() == [[0, 0, 0], [0, 0, 0], [1, 0, 0], [0, 2, 0]]
    assert (info.n_empty, info.n_partial, info.n_full) == (9, 5, 2)


def test_hand_mask_unshrunk_data_next():
    m, _ = _hand_mask()
    info = mi.compile_mask_info("dense", 512, 512, dense=m, shrink_grid=False)
    assert info.width == 4
    # row 0: cell 0 empty -> next non-empty is column 1
    # row 1: whole row empty -> 0
    # row 2: cell 1 -> 2; cell 3 has nothing to its right -> last one to its left (2)
    # row 3: cells 1, 2 -> 3
    assert info.data_next[0].tolist() == [[1, 1, 2, 3], [0, 0, 0, 0], [0, 2, 2, 2], [0, 3, 3, 3]]
    assert info.mask_next[0].tolist() == [[0, 0, 0, 0], [0, 0, 0, 0], [1, 0, 0, 0], [0, 0, 0, 2]]


def test_hand_mask_dkv_is_transpose():
    m, (A, Bp, C) = _hand_mask()
    info = mi.compile_mask_info("dense", 512, 512, dense=m, orientation="dkv")
    fwd = mi.compile_mask_info("dense", 512, 512, dense=m)
    assert np.array_equal(info.labels_unshrunk[0], fwd.labels_unshrunk[0].T)
    # transposed rows in order: row0 [Z, Z, B^T, O]; row1 [A^T, Z, Z, Z];
    # row2 [O, Z, A^T, Z]; row3 [A^T, Z, Z, C^T]  ->  stack B^T, A^T, C^T
    assert info.num_partial_blocks == 3
    assert np.array_equal(info.partial_mask_blocks[0], Bp.T)
    assert np.array_equal(info.partial_mask_blocks[1], A.T)
    assert np.array_equal(info.partial_mask_blocks[2], C.T)
    # rows hold 2, 1, 2, 2 non-empty blocks, so the shrunk width is 2
    assert info.width == 2
    assert info.mask_next[0].tolist() == [[0, 0], [1, 0], [0, 1], [1, 2]]


# --------------------------------------------------------------------------
# Round trip: decode MaskInfo and get the mask back
# --------------------------------------------------------------------------

def decode(info: mi.MaskInfo, n_rows: int, n_cols: int) -> np.ndarray:
    heads = info.block_mask.shape[0]
    out = np.full((heads, n_rows * B, n_cols * B), 7, np.uint8)
    seen = np.zeros((heads, n_rows, n_cols), bool)
    for h in range(heads):
        for r in range(n_rows):
            for t in range(info.width):
                lab = int(info.block_mask[h, r, t])
                if lab == 0:
                    continue
                c = int(info.data_next[h, r, t])
                assert not seen[h, r, c], "column listed twice"
                seen[h, r, c] = True
                if lab == 2:
                    blk = np.ones((B, B), np.uint8)
                else:
                    blk = info.partial_mask_blocks[int(info.mask_next[h, r, t])]
                out[h, r * B:(r + 1) * B, c * B:(c + 1) * B] = blk
    out[out == 7] = 0
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_round_trip_planted(seed):
    heads, nq, nk = 2, 3, 5
    m = planted_block_mask(heads, nq, nk, seed=seed)
    info = mi.compile_mask_info("dense", nq * B, nk * B, dense=m)
    assert np.array_equal(decode(info, nq, nk), m)
    # stack blocks are pairwise distinct and all mixed
    P = info.num_partial_blocks
    flat = info.partial_mask_blocks.reshape(P, -1)
    assert len({r.tobytes() for r in flat}) == P
    assert all(0 < r.sum() < B * B for r in flat)
    # dkv orientation decodes to the transpose
    dkv = mi.compile_mask_info("dense", nq * B, nk * B, dense=m, orientation="dkv")
    assert np.array_equal(decode(dkv, nk, nq), np.transpose(m, (0, 2, 1)))


@pytest.mark.parametrize("kind,kw", [("causal", {}), ("local", {"left": 200, "right": 70}),
                                     ("chunked", {"chunk": 192}), ("local", {"left": None, "right": 5})])
def test_round_trip_computable_labels(kind, kw):
    # For computable masks the labels alone must agree with the element mask:
    # label 2 blocks are all ones, label 0 blocks all zeros, label 1 mixed.
    from oracle import masks
    S = 640
    full = masks.materialise(kind, S, S, **kw)
    info = mi.compile_mask_info(kind, S, S, **kw)
    assert info.mask_next is None and info.partial_mask_blocks is None
    n = S // B
    lab = info.labels_unshrunk[0]
    for i in range(n):
        for j in range(n):
            blk = full[i * B:(i + 1) * B, j * B:(j + 1) * B]
            want = 2 if blk.all() else (1 if blk.any() else 0)
            assert lab[i, j] == want
    assert np.array_equal(info.q_sequence, np.arange(S, dtype=np.int32))


def test_empty_mask_has_width_zero():
    m = np.zeros((256, 384), np.uint8)
    info = mi.compile_mask_info("dense", 256, 384, dense=m)
    assert info.width == 0
    assert info.block_mask.shape == (1, 2, 0)
    assert info.num_partial_blocks == 0
    assert info.n_empty == 6
