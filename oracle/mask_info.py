"""MaskInfo, the compiled form of a mask, computed the slow and obvious way.

Source: "Splash Attention: When the Mask Stops Being Arithmetic and Becomes
the Loop".  Each step below follows one section of that page:

1. ``classify_blocks``: cut the mask into grid-step blocks and label each
   one 0 (all zeros), 1 (mixed) or 2 (all ones) by asking ``any()`` and
   ``all()`` of the block ("What is splash attention and how is it different
   from flash attention?", "Does splash attention make every sparse mask
   faster?").
2. ``dedup_partial_blocks``: the mixed blocks of a dense mask go into a
   deduplicated stack ``partial_mask_blocks``; ``mask_next`` points into it
   ("What is MaskInfo in splash attention?").  Computable masks (causal,
   local, chunked causal) have neither: both are None (same section).
3. ``data_next_unshrunk``: for each grid position, the next non-empty
   key/value block (same section).
4. ``shrink``: per block row, keep only the non-empty columns, padded to
   the widest row ("What does grid shrinking do in splash attention?").
5. ``downcast``: integer arrays take the smallest type their largest value
   fits in (int8 / int16 / int32) ("What is MaskInfo in splash attention?").

Readings where the page is silent (this library's own contract):

* Equality of partial blocks is byte equality of the 0/1 block; stack slots
  are handed out in order of first occurrence, walking (head, row, column)
  in row-major order.
* ``data_next`` at an empty cell: the smallest non-empty column to its
  right in the same row; if none, the largest non-empty column to its
  left; if the row is empty, 0.
* ``mask_next`` at label-0 and label-2 cells is 0.
* Shrink padding slots carry label 0, ``data_next`` = the row's last real
  column (0 for an empty row), ``mask_next`` = 0.  The grid width W is the
  largest row count (0 when the whole mask is empty).
* Downcast is to signed types: max <= 127 -> int8, <= 32767 -> int16,
  else int32.  ``block_mask`` is int8 and the stack uint8 0/1.
* ``q_sequence`` is always present: int32 arange(q_len).
* The dkv orientation (for the key/value-gradient grid, whose rows are key
  blocks) is every step above applied to the transposed mask.
* Counts (empty / partial / full) are taken over the unshrunk grid, summed
  over mask heads.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Optional

import numpy as np

from . import masks

BLOCK = 128


@dataclass
class MaskInfo:
    block_mask: np.ndarray                 # int8 [Hm, n_rows, W]
    data_next: np.ndarray                  # int8/16/32 [Hm, n_rows, W]
    mask_next: Optional[np.ndarray]        # int8/16/32 [Hm, n_rows, W]; None if computable
    partial_mask_blocks: Optional[np.ndarray]  # uint8 [P, block, block]; None if computable
    q_sequence: np.ndarray                 # int32 [q_len]
    n_empty: int
    n_partial: int
    n_full: int
    width: int                             # W
    num_partial_blocks: int                # P (0 if computable)
    labels_unshrunk: np.ndarray            # int8 [Hm, n_rows, n_cols] (for tests)


StripFn = Callable[[int, int], np.ndarray]


def classify_blocks(strip: StripFn, heads: int, n_rows: int, n_cols: int,
                    block: int = BLOCK) -> np.ndarray:
    """Label every block: 2 if all entries are 1, 1 if any is 1, else 0.

    ``strip(h, r)`` returns the boolean rows of block-row ``r`` of head ``h``
    ([block, n_cols*block]).
    """
    lab = np.zeros((heads, n_rows, n_cols), dtype=np.int8)
    for h in range(heads):
        for r in range(n_rows):
            s = strip(h, r)
            for c in range(n_cols):
                blk = s[:, c * block:(c + 1) * block]
                if blk.all():
                    lab[h, r, c] = 2
                elif blk.any():
                    lab[h, r, c] = 1
    return lab


def dedup_partial_blocks(strip: StripFn, labels: np.ndarray, block: int = BLOCK):
    """Stack of distinct mixed blocks, and for each cell its slot in the stack.

    Returns (stack uint8 [P, block, block], mask_next int64 [Hm, n_rows, n_cols]).
    Walks label-1 cells in (head, row, column) order; a block whose bytes equal
    an earlier stacked block's reuses that slot, otherwise it takes slot P
    and P grows by one.
    """
    heads, n_rows, n_cols = labels.shape
    seen: dict[bytes, int] = {}
    stack: list[np.ndarray] = []
    nxt = np.zeros(labels.shape, dtype=np.int64)
    for h in range(heads):
        for r in range(n_rows):
            if not (labels[h, r] == 1).any():
                continue
            s = strip(h, r)
            for c in range(n_cols):
                if labels[h, r, c] != 1:
                    continue
                blk = s[:, c * block:(c + 1) * block].astype(np.uint8)
                key = blk.tobytes()
                slot = seen.get(key)
                if slot is None:
                    slot = len(stack)
                    seen[key] = slot
                    stack.append(blk)
                nxt[h, r, c] = slot
    if stack:
        arr = np.stack(stack).astype(np.uint8)
    else:
        arr = np.zeros((0, block, block), dtype=np.uint8)
    return arr, nxt


def data_next_unshrunk(labels: np.ndarray) -> np.ndarray:
    """For each cell, the key/value block the pipeline should hold there."""
    heads, n_rows, n_cols = labels.shape
    out = np.zeros(labels.shape, dtype=np.int64)
    for h in range(heads):
        for r in range(n_rows):
            nonempty = [c for c in range(n_cols) if labels[h, r, c] != 0]
            for c in range(n_cols):
                if labels[h, r, c] != 0:
                    out[h, r, c] = c
                    continue
                later = [x for x in nonempty if x > c]
                earlier = [x for x in nonempty if x < c]
                if later:
                    out[h, r, c] = later[0]
                elif earlier:
                    out[h, r, c] = earlier[-1]
                else:
                    out[h, r, c] = 0
    return out


def shrink(labels: np.ndarray, mask_next: Optional[np.ndarray]):
    """Row compaction of the non-empty columns, padded to the widest row.

    Returns (block_mask, data_next, mask_next or None, W, row_len).
    """
    heads, n_rows, n_cols = labels.shape
    cols = [[[c for c in range(n_cols) if labels[h, r, c] != 0] for r in range(n_rows)]
            for h in range(heads)]
    row_len = np.array([[len(cols[h][r]) for r in range(n_rows)] for h in range(heads)],
                       dtype=np.int64).reshape(heads, n_rows)
    W = int(row_len.max()) if row_len.size else 0
    bm = np.zeros((heads, n_rows, W), dtype=np.int8)
    dn = np.zeros((heads, n_rows, W), dtype=np.int64)
    mn = None if mask_next is None else np.zeros((heads, n_rows, W), dtype=np.int64)
    for h in range(heads):
        for r in range(n_rows):
            cs = cols[h][r]
            for t in range(W):
                if t < len(cs):
                    c = cs[t]
                    bm[h, r, t] = labels[h, r, c]
                    dn[h, r, t] = c
                    if mn is not None:
                        mn[h, r, t] = mask_next[h, r, c]
                else:
                    bm[h, r, t] = 0
                    dn[h, r, t] = cs[-1] if cs else 0
                    if mn is not None:
                        mn[h, r, t] = 0
    return bm, dn, mn, W, row_len


def downcast(a: np.ndarray) -> np.ndarray:
    """The array in the smallest signed integer type that holds its largest value."""
    mx = int(a.max()) if a.size else 0
    if mx <= np.iinfo(np.int8).max:
        return a.astype(np.int8)
    if mx <= np.iinfo(np.int16).max:
        return a.astype(np.int16)
    return a.astype(np.int32)


def _strip_fn(kind: str, q_len: int, kv_len: int, orientation: str, block: int, dense,
              params) -> StripFn:
    def strip(h: int, r: int) -> np.ndarray:
        lo, hi = r * block, (r + 1) * block
        d = None if dense is None else dense[h]
        if orientation == "fwd":
            q = np.arange(lo, hi)[:, None]
            k = np.arange(kv_len)[None, :]
            return masks.allowed(kind, q, k, dense=d, **params)
        # dkv: rows are key positions, columns are query positions (mask transposed)
        k = np.arange(lo, hi)[:, None]
        q = np.arange(q_len)[None, :]
        return masks.allowed(kind, q, k, dense=d, **params)
    return strip


def compile_mask_info(kind: str, q_len: int, kv_len: int, *, heads: int = 1,
                      dense: Optional[np.ndarray] = None, left: Optional[int] = None,
                      right: Optional[int] = None, chunk: Optional[int] = None,
                      orientation: str = "fwd", shrink_grid: bool = True,
                      block: int = BLOCK) -> MaskInfo:
    """Compile a mask into MaskInfo (steps 1-5 of the module docstring).

    ``dense`` is [heads, q_len, kv_len] (or [q_len, kv_len] for one head).
    """
    if q_len % block or kv_len % block:
        raise ValueError("sequence lengths must be multiples of the block size")
    if orientation not in ("fwd", "dkv"):
        raise ValueError("orientation is 'fwd' or 'dkv'")
    if kind == "dense":
        dense = np.asarray(dense)
        if dense.ndim == 2:
            dense = dense[None]
        heads = dense.shape[0]
    params = {}
    if kind == "local":
        params = dict(left=left, right=right)
    elif kind == "chunked":
        params = dict(chunk=chunk)
    strip = _strip_fn(kind, q_len, kv_len, orientation, block, dense, params)
    n_q, n_k = q_len // block, kv_len // block
    n_rows, n_cols = (n_q, n_k) if orientation == "fwd" else (n_k, n_q)

    labels = classify_blocks(strip, heads, n_rows, n_cols, block)
    computable = kind != "dense"
    if computable:
        stack, mnext_full = None, None
    else:
        stack, mnext_full = dedup_partial_blocks(strip, labels, block)
    dnext_full = data_next_unshrunk(labels)

    if shrink_grid:
        bm, dn, mn, W, _ = shrink(labels, mnext_full)
    else:
        bm, dn, mn, W = labels.copy(), dnext_full, mnext_full, n_cols

    return MaskInfo(
        block_mask=bm.astype(np.int8),
        data_next=downcast(dn),
        mask_next=None if mn is None else downcast(mn),
        partial_mask_blocks=stack,
        q_sequence=np.arange(q_len, dtype=np.int32),
        n_empty=int((labels == 0).sum()),
        n_partial=int((labels == 1).sum()),
        n_full=int((labels == 2).sum()),
        width=int(W),
        num_partial_blocks=0 if stack is None else int(stack.shape[0]),
        labels_unshrunk=labels,
    )
