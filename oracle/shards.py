"""Key-sharded attention: per-shard partial results and their merge, fp64.

Source: "Splash Attention: When the Mask Stops Being Arithmetic and Becomes
the Loop", section "What does ring attention add on top of the splash
kernel?".  The keys and values are split into shards along the key axis and
the same masked attention runs on each shard, with the MaskInfo cut to the
shard's key range.  Each shard yields its own running maximum and
normaliser together with its unnormalised accumulator; the shards are
combined with the flash-attention rescaling and the accumulator is divided
by the final normaliser once, at the end.  A shard with no active key for a
row contributes zeros (never uninitialised values).

Definitions, for one (batch, q head) row and a shard K of keys:

    s_k  = scale * q . k_k  for visible k in K
    m    = max_k s_k                       (-inf when no key of K is visible)
    l    = sum_k exp(s_k - m)              (0 then)
    acc  = sum_k exp(s_k - m) v_k          (0 then)

and the merge of shards 1..n:

    M    = max_i m_i over shards with l_i > 0
    L    = sum_i exp(m_i - M) l_i
    O    = sum_i exp(m_i - M) acc_i / L,   LSE = M + log L
           (O = 0 and LSE = -inf when every shard is empty for the row)

Test infrastructure only (see ``oracle/__init__.py``).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .attention import ROW_CHUNK, MaskRows, _mask_head, _scores, default_scale, mask_rows_for


def head_partial(qm: np.ndarray, km: np.ndarray, vm: np.ndarray, mask_rows: MaskRows, scale: float,
                 k0: int, k1: int):
    """(acc [S, Dv], m [S], l [S]) of one (batch, q head) over keys [k0, k1).

    ``km`` and ``vm`` hold the whole key axis; the mask is evaluated on the
    global key indices and cut to the shard."""
    S = qm.shape[0]
    acc = np.zeros((S, vm.shape[1]))
    m = np.full(S, -np.inf)
    l = np.zeros(S)
    ks, vs = km[k0:k1], vm[k0:k1]
    for c0 in range(0, S, ROW_CHUNK):
        r = np.arange(c0, min(S, c0 + ROW_CHUNK))
        allowed = mask_rows(r)[:, k0:k1]
        s = _scores(qm[r], ks, allowed, scale)
        mr = s.max(axis=1) if s.shape[1] else np.full(r.size, -np.inf)
        live = np.isfinite(mr)
        w = np.where(live[:, None], np.exp(s - np.where(live, mr, 0.0)[:, None]), 0.0)
        acc[r] = w @ vs
        l[r] = w.sum(axis=1)
        m[r] = mr
    return acc, m, l


def forward_partial(q, k, v, mask: dict, k0: int, k1: int, scale: Optional[float] = None):
    """Batch version of :func:`head_partial`: acc [B,Hq,S,Dv], m and l [B,Hq,S]."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    scale = default_scale(D) if scale is None else scale
    group = Hq // Hkv
    acc = np.zeros((B, Hq, S, v.shape[3]))
    m = np.zeros((B, Hq, S))
    l = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            g = h // group
            acc[b, h], m[b, h], l[b, h] = head_partial(q[b, h], k[b, g], v[b, g],
                                                       mask_rows_for(mask, _mask_head(mask, h)), scale, k0, k1)
    return acc, m, l


def merge_partials(accs: Sequence[np.ndarray], ms: Sequence[np.ndarray], ls: Sequence[np.ndarray]):
    """Merge shard results (any leading shape, last axis of acc = Dv) into (O, LSE)."""
    accs = [np.asarray(a, np.float64) for a in accs]
    ms = [np.asarray(x, np.float64) for x in ms]
    ls = [np.asarray(x, np.float64) for x in ls]
    live = [(l > 0) & np.isfinite(m) for m, l in zip(ms, ls)]
    M = np.full(ms[0].shape, -np.inf)
    for m, lv in zip(ms, live):
        M = np.where(lv, np.maximum(M, m), M)
    anyl = np.isfinite(M)
    Ms = np.where(anyl, M, 0.0)
    L = np.zeros(M.shape)
    O = np.zeros(accs[0].shape)
    for a, m, l, lv in zip(accs, ms, ls, live):
        w = np.where(lv, np.exp(np.where(lv, m, 0.0) - Ms), 0.0)
        L += w * l
        O += w[..., None] * a
    with np.errstate(divide="ignore", invalid="ignore"):
        O = np.where(anyl[..., None], O / np.where(anyl, L, 1.0)[..., None], 0.0)
        lse = np.where(anyl, Ms + np.log(np.where(anyl, L, 1.0)), -np.inf)
    return O, lse
