"""Seeded synthetic inputs shared by the tests, the benchmark and smoke().

This module only draws random numbers and describes shapes.  It holds none
of the attention or mask-compilation arithmetic: the oracle (``oracle/``)
and the CUDA library (``block_sparse_attention_process_gb300``) each
implement that on their own, and both consume the arrays made here.

Recipe (the same for every workload):

* Q, K, V, dO: ``torch.Generator('cpu').manual_seed(seed)``, ``randn`` in
  fp32 drawn in the order Q, K, V, dO, then rounded to bf16 (round to
  nearest even, torch's ``.to(torch.bfloat16)``).  Layout BHSD.
* Dense random mask: ``numpy.random.default_rng(seed).random((S, S)) < p``
  with the diagonal forced to 1, stored as uint8 0/1.
* Computable masks are described by parameters only (kind, windows, chunk).

The workloads are the five shapes the splash-attention pages discuss
(causal at 8192 tokens, a 1024-token left window, chunked causal, a
90%-zero scattered mask at 2048 tokens) plus a small case and a
forward+backward case; all data is synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class MaskSpec:
    """Parameters of one mask.  ``kind`` is causal | local | chunked | dense | full."""

    kind: str
    left: Optional[int] = None     # local: keys allowed back to q-left (None = unbounded)
    right: Optional[int] = None    # local: keys allowed up to q+right (None = unbounded)
    chunk: Optional[int] = None    # chunked causal: chunk length in tokens
    p: Optional[float] = None      # dense: probability of a 1
    seed: Optional[int] = None     # dense: numpy seed


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    mask: MaskSpec
    backward: bool = False
    seed: int = 0
    notes: str = field(default="", compare=False)


WORKLOADS = {
    "causal_s512_d64": Workload(
        "causal_s512_d64", B=1, Hq=2, Hkv=2, S=512, D=64, mask=MaskSpec("causal"),
        notes="small causal forward; 6 of 16 blocks empty"),
    "gqa_causal_s8192": Workload(
        "gqa_causal_s8192", B=1, Hq=32, Hkv=8, S=8192, D=128, mask=MaskSpec("causal"),
        notes="GQA 32/8 causal forward; 2016 of 4096 blocks empty, no shrink"),
    "mha_local1024_s8192": Workload(
        "mha_local1024_s8192", B=1, Hq=16, Hkv=16, S=8192, D=128,
        mask=MaskSpec("local", left=1024, right=0),
        notes="MHA local window (1024, 0) forward; shrunk grid width 9"),
    "mqa_chunked2048_s16384": Workload(
        "mqa_chunked2048_s16384", B=1, Hq=16, Hkv=1, S=16384, D=128,
        mask=MaskSpec("chunked", chunk=2048),
        notes="MQA 16/1 chunked-causal forward"),
    "mqa_bernoulli_s2048": Workload(
        "mqa_bernoulli_s2048", B=1, Hq=16, Hkv=1, S=2048, D=128,
        mask=MaskSpec("dense", p=0.1, seed=1),
        notes="MQA 16/1 dense Bernoulli(0.1) mask, diagonal forced; 256 of 256 blocks partial"),
    "mha_causal_s4096_fwdbwd": Workload(
        "mha_causal_s4096_fwdbwd", B=2, Hq=16, Hkv=16, S=4096, D=128, mask=MaskSpec("causal"),
        backward=True, notes="MHA causal forward + backward"),
}


def qkvdo(B: int, Hq: int, Hkv: int, S: int, D: int, seed: int = 0, with_do: bool = True,
          Skv: Optional[int] = None):
    """Q [B,Hq,S,D], K/V [B,Hkv,Skv,D], dO [B,Hq,S,D] as CPU bf16 tensors."""
    Skv = S if Skv is None else Skv
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((B, Hq, S, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Skv, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Skv, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    do = None
    if with_do:
        do = torch.randn((B, Hq, S, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, do


def bernoulli_mask(S: int, p: float, seed: int, Skv: Optional[int] = None,
                   force_diagonal: bool = True) -> np.ndarray:
    """uint8 [S, Skv] with entries 1 w.p. p; the main diagonal forced to 1."""
    Skv = S if Skv is None else Skv
    m = np.random.default_rng(seed).random((S, Skv)) < p
    if force_diagonal:
        d = min(S, Skv)
        m[np.arange(d), np.arange(d)] = True
    return m.astype(np.uint8)


def planted_block_mask(heads: int, nq: int, nk: int, seed: int, block: int = 128,
                       p_cell: float = 0.3) -> np.ndarray:
    """A small dense uint8 mask [heads, nq*block, nk*block] with planted block structure.

    Each block is drawn independently as one of: all zeros, all ones, a copy of
    one of three fixed random patterns (so duplicates occur), or fresh random
    bytes.  Used to exercise the classifier, the dedup of partial blocks, the
    next-block pointers and the shrink pass on small inputs.
    """
    rng = np.random.default_rng(seed)
    patterns = [(rng.random((block, block)) < 0.5).astype(np.uint8) for _ in range(3)]
    out = np.zeros((heads, nq * block, nk * block), dtype=np.uint8)
    for h in range(heads):
        for i in range(nq):
            for j in range(nk):
                r = rng.random()
                if r < p_cell:
                    blk = np.zeros((block, block), np.uint8)
                elif r < p_cell + 0.2:
                    blk = np.ones((block, block), np.uint8)
                elif r < p_cell + 0.5:
                    blk = patterns[int(rng.integers(0, 3))]
                else:
                    blk = (rng.random((block, block)) < 0.5).astype(np.uint8)
                out[h, i * block:(i + 1) * block, j * block:(j + 1) * block] = blk
    return out
