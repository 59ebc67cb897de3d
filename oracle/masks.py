"""Element-wise attention masks, written out as boolean arrays.

Source: "Splash Attention: When the Mask Stops Being Arithmetic and Becomes
the Loop", section "What is MaskInfo in splash attention?", which names
CausalMask, LocalMask and ChunkedCausalMask as computable masks and a dense
NumPy array as the general case.  The page gives names, not formulas; the
plain readings used here are:

* causal:           key k is visible from query q iff k <= q
* local(left,right):           q - left <= k <= q + right, both ends
                               inclusive; None means that side is unbounded
* chunked causal(c):           q // c == k // c and k <= q
* dense:                       the given 0/1 array (nonzero = visible)
* full:                        every key visible
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def allowed(kind: str, q: np.ndarray, k: np.ndarray, *, left: Optional[int] = None,
            right: Optional[int] = None, chunk: Optional[int] = None,
            dense: Optional[np.ndarray] = None) -> np.ndarray:
    """Whether key index ``k`` is visible from query index ``q`` (broadcasting).

    ``dense`` (kind == "dense") is a 2-D [q_len, kv_len] array indexed by
    (q, k).
    """
    q = np.asarray(q, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    if kind == "causal":
        return k <= q
    if kind == "local":
        ok = np.ones(np.broadcast_shapes(q.shape, k.shape), dtype=bool)
        if left is not None:
            ok &= k >= q - left
        if right is not None:
            ok &= k <= q + right
        return ok
    if kind == "chunked":
        if chunk is None or chunk <= 0:
            raise ValueError("chunked mask needs a positive chunk")
        return (q // chunk == k // chunk) & (k <= q)
    if kind == "dense":
        if dense is None:
            raise ValueError("dense mask needs an array")
        return np.asarray(dense)[q, k] != 0
    if kind == "full":
        return np.ones(np.broadcast_shapes(q.shape, k.shape), dtype=bool)
    raise ValueError(f"unknown mask kind {kind!r}")


def rows(kind: str, q_idx, kv_len: int, **kw) -> np.ndarray:
    """Boolean mask rows [len(q_idx), kv_len] for the given query indices."""
    q = np.asarray(q_idx, dtype=np.int64)[:, None]
    k = np.arange(kv_len, dtype=np.int64)[None, :]
    return allowed(kind, q, k, **kw)


def materialise(kind: str, q_len: int, kv_len: int, **kw) -> np.ndarray:
    """The whole [q_len, kv_len] boolean mask."""
    return rows(kind, np.arange(q_len), kv_len, **kw)
