"""Dense masked softmax attention and its gradients in fp64.

Sources:
* Forward: "Splash Attention: When the Mask Stops Being Arithmetic and
  Becomes the Loop", section "What is splash attention and how is it
  different from flash attention?" -- attention whose masked-out scores do
  not contribute; the online softmax of the kernel reaches the same
  result as the plain row softmax written here.
* Saved residuals and backward: "Flash Attention on a TPU, Line by Line",
  sections "What does the TPU flash attention kernel save for the backward
  pass?" (the scores are rebuilt from Q and K and the saved row statistics;
  rowsum(dO*O) is computed once outside the gradient kernels) and "Why does
  the TPU flash attention backward pass run two kernels instead of one?"
  (key/value gradients sum over query blocks, query gradients over key
  blocks).  The row statistics are kept as one logsumexp per row.

Definitions, per batch b and query head h, with kv head g = h // (Hq/Hkv):

    s    = scale * q k^T,  s = -inf where the mask is 0
    lse  = log(sum_k exp(s))          (-inf for a row with no visible key)
    P    = exp(s - lse)               (0 in a row with no visible key)
    O    = P v
    Dsum = rowsum(dO * O)
    dV   = P^T dO                     (summed over the q heads of group g)
    dP   = dO v^T
    dS   = P * (dP - Dsum)
    dQ   = scale * dS k
    dK   = scale * dS^T q             (summed over the q heads of group g)

Optional score transforms, from the operator signature on the EasyDeL
``blocksparse_attention`` module page (``logits_soft_cap``, ``softmax_aux``);
the page gives the arguments but not the formulas, so these are the plain
readings:

    soft cap c > 0:  s = c * tanh(s / c) on the visible scaled scores
    sinks z_1..z_n:  extra logits of the row that enter the normaliser (and
                     carry no value):  lse = log(sum_k exp(s_k) + sum_j exp(z_j)),
                     P = exp(s - lse),  O = P v;  per q head h the sinks are
                     z[h // (Hq/Hkv), :] for a [Hkv, n] array, z[:] for [n]
    their gradients: dS = P * (dP - Dsum) * (1 - (s / c)^2)  with the cap,
                     dz_j = -sum over the rows of exp(z_j - lse) * Dsum

Rows are processed in chunks of 1024 to bound memory; nothing is fused.
"""
from __future__ import annotations

import math
from typing import Callable, Optional

import numpy as np

ROW_CHUNK = 1024

MaskRows = Callable[[np.ndarray], np.ndarray]   # query indices -> bool [n, kv_len]


def _scores(qc: np.ndarray, km: np.ndarray, allowed: np.ndarray, scale: float) -> np.ndarray:
    s = scale * (qc @ km.T)
    return np.where(allowed, s, -np.inf)


def _capped(s: np.ndarray, cap: Optional[float]) -> np.ndarray:
    if not cap:
        return s
    with np.errstate(invalid="ignore"):
        return np.where(np.isfinite(s), cap * np.tanh(s / cap), s)


def _logsumexp_rows(s: np.ndarray, sinks: Optional[np.ndarray] = None) -> np.ndarray:
    if sinks is not None and len(sinks):
        s = np.concatenate([s, np.broadcast_to(np.asarray(sinks, np.float64), (s.shape[0], len(sinks)))], axis=1)
    m = s.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    tot = np.exp(s - m_safe[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        return np.where(finite, m_safe + np.log(tot), -np.inf)


def _probs(s: np.ndarray, lse: np.ndarray) -> np.ndarray:
    finite = np.isfinite(lse)
    p = np.exp(s - np.where(finite, lse, 0.0)[:, None])
    return np.where(finite[:, None], p, 0.0)


def head_forward(qm: np.ndarray, km: np.ndarray, vm: np.ndarray, mask_rows: MaskRows,
                 scale: float, rows: Optional[np.ndarray] = None, cap: Optional[float] = None,
                 sinks: Optional[np.ndarray] = None):
    """O [n, Dv] and LSE [n] for one (batch, q head), for query rows ``rows``."""
    S = qm.shape[0]
    rows = np.arange(S) if rows is None else np.asarray(rows)
    o = np.zeros((rows.size, vm.shape[1]))
    lse = np.zeros(rows.size)
    for c0 in range(0, rows.size, ROW_CHUNK):
        r = rows[c0:c0 + ROW_CHUNK]
        s = _capped(_scores(qm[r], km, mask_rows(r), scale), cap)
        l = _logsumexp_rows(s, sinks)
        p = _probs(s, l)
        o[c0:c0 + r.size] = p @ vm
        lse[c0:c0 + r.size] = l
    return o, lse


def head_probs(qm, km, mask_rows: MaskRows, scale: float, rows=None) -> np.ndarray:
    """The attention weights P [n, kv_len] for query rows ``rows``."""
    rows = np.arange(qm.shape[0]) if rows is None else np.asarray(rows)
    s = _scores(qm[rows], km, mask_rows(rows), scale)
    return _probs(s, _logsumexp_rows(s))


def head_backward(qm, km, vm, dom, mask_rows: MaskRows, scale: float, cap: Optional[float] = None,
                  sinks: Optional[np.ndarray] = None):
    """(dQ, dK contribution, dV contribution, Dsum, O, LSE, dsinks) for one (batch, q head)."""
    S = qm.shape[0]
    dq = np.zeros_like(qm)
    dk = np.zeros_like(km)
    dv = np.zeros_like(vm)
    dsum = np.zeros(S)
    o_all = np.zeros((S, vm.shape[1]))
    lse_all = np.zeros(S)
    z = np.zeros(0) if sinks is None else np.asarray(sinks, np.float64)
    dz = np.zeros(z.shape)
    for c0 in range(0, S, ROW_CHUNK):
        r = np.arange(c0, min(S, c0 + ROW_CHUNK))
        s = _capped(_scores(qm[r], km, mask_rows(r), scale), cap)
        lse = _logsumexp_rows(s, z)
        p = _probs(s, lse)
        o = p @ vm
        ds_row = (dom[r] * o).sum(axis=1)
        dp = dom[r] @ vm.T
        dS = p * (dp - ds_row[:, None])
        if cap:
            dS = dS * np.where(np.isfinite(s), 1.0 - (np.where(np.isfinite(s), s, 0.0) / cap) ** 2, 0.0)
        dq[r] = scale * (dS @ km)
        dk += scale * (dS.T @ qm[r])
        dv += p.T @ dom[r]
        if z.size:
            fin = np.isfinite(lse)
            pz = np.where(fin[:, None], np.exp(z[None, :] - np.where(fin, lse, 0.0)[:, None]), 0.0)
            dz -= (pz * ds_row[:, None]).sum(axis=0)
        dsum[r] = ds_row
        o_all[r] = o
        lse_all[r] = lse
    return dq, dk, dv, dsum, o_all, lse_all, dz


def mask_rows_for(mask: dict, head: int) -> MaskRows:
    """Row-producing mask function for mask head ``head`` (0 when the mask is shared)."""
    from . import masks
    kind = mask["kind"]
    dense = mask.get("dense")
    params = {k: mask[k] for k in ("left", "right", "chunk") if k in mask}

    def fn(r: np.ndarray) -> np.ndarray:
        d = None
        if dense is not None:
            d = dense[head] if dense.ndim == 3 else dense
        kv_len = mask["kv_len"]
        return masks.rows(kind, r, kv_len, dense=d, **params)
    return fn


def _mask_head(mask: dict, hq: int) -> int:
    dense = mask.get("dense")
    if dense is not None and dense.ndim == 3 and dense.shape[0] > 1:
        return hq
    return 0


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def head_sinks(sinks: Optional[np.ndarray], h: int, group: int) -> Optional[np.ndarray]:
    """The sink logits of q head h: row h // group of a [Hkv, n] array, or a shared [n] array."""
    if sinks is None:
        return None
    z = np.asarray(sinks, np.float64)
    return z[h // group] if z.ndim == 2 else z


def forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: dict,
            scale: Optional[float] = None, cap: Optional[float] = None, sinks: Optional[np.ndarray] = None):
    """O [B,Hq,S,Dv] and LSE [B,Hq,S] for the whole batch (small cases)."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    scale = default_scale(D) if scale is None else scale
    group = Hq // Hkv
    o = np.zeros((B, Hq, S, v.shape[3]))
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            g = h // group
            o[b, h], lse[b, h] = head_forward(q[b, h], k[b, g], v[b, g],
                                              mask_rows_for(mask, _mask_head(mask, h)), scale,
                                              cap=cap, sinks=head_sinks(sinks, h, group))
    return o, lse


def backward(q, k, v, do, mask: dict, scale: Optional[float] = None, cap: Optional[float] = None,
             sinks: Optional[np.ndarray] = None):
    """dQ, dK, dV (fp64) for the whole batch; dK/dV summed over each kv group.
    With sinks, also their gradient (same shape as ``sinks``)."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    scale = default_scale(D) if scale is None else scale
    group = Hq // Hkv
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    dz = None if sinks is None else np.zeros(np.shape(sinks))
    for b in range(B):
        for h in range(Hq):
            g = h // group
            dqh, dkh, dvh, _, _, _, dzh = head_backward(q[b, h], k[b, g], v[b, g], do[b, h],
                                                        mask_rows_for(mask, _mask_head(mask, h)),
                                                        scale, cap=cap, sinks=head_sinks(sinks, h, group))
            dq[b, h] = dqh
            dk[b, g] += dkh
            dv[b, g] += dvh
            if dz is not None:
                if dz.ndim == 2:
                    dz[g] += dzh
                else:
                    dz += dzh
    return (dq, dk, dv) if dz is None else (dq, dk, dv, dz)


def rowsum_do_o(do: np.ndarray, o: np.ndarray) -> np.ndarray:
    """Dsum = sum over the head dimension of dO * O, in fp64."""
    return (np.asarray(do, np.float64) * np.asarray(o, np.float64)).sum(axis=-1)
