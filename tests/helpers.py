"""Helpers shared by the tests: building the library, oracle comparisons."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances (floating point), stated per output:
#   O (bf16 output): max-abs 2e-2 against the fp64 oracle
#   LSE (fp32 output): max-abs 1e-5 against the fp64 oracle
#   dQ/dK/dV: max-abs 2e-2 on the fp32 outputs; bf16 outputs: 2e-2 plus half
#   a bf16 ulp of the reference value (the rounding of the output itself)
TOL_O = 2e-2
TOL_LSE = 1e-5
TOL_GRAD = 2e-2


def ensure_built():
    from block_sparse_attention_process_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    return b.LIB


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()


def mask_dict(kind: str, S: int, **kw) -> dict:
    d = {"kind": kind, "kv_len": S}
    d.update({k: v for k, v in kw.items() if v is not None})
    return d


def oracle_mask_args(spec, S):
    """Translate a workloads.MaskSpec into oracle / library keyword arguments."""
    if spec.kind == "local":
        return {"left": spec.left, "right": spec.right}
    if spec.kind == "chunked":
        return {"chunk": spec.chunk}
    return {}


def lib_mask_args(spec):
    if spec.kind == "local":
        return {"local_left": spec.left, "local_right": spec.right}
    if spec.kind == "chunked":
        return {"chunk": spec.chunk}
    return {}


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (bf16 keeps 8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def compare(name: str, got: np.ndarray, want: np.ndarray, tol: float, extra: np.ndarray | None = None):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    inf_w = ~np.isfinite(want)
    assert np.array_equal(~np.isfinite(got), inf_w), f"{name}: non-finite pattern differs"
    if inf_w.any():
        assert np.array_equal(got[inf_w], want[inf_w]), f"{name}: infinities differ"
    fin = ~inf_w
    err = np.abs(got[fin] - want[fin])
    bound = tol + (0 if extra is None else extra[fin])
    worst = float((err - bound).max()) if err.size else -1.0
    assert worst <= 0, f"{name}: max-abs err {err.max():.3e} exceeds tolerance (worst excess {worst:.3e})"
    return float(err.max()) if err.size else 0.0
