"""ctypes mirror of include/bsa.h and the loader of libbsa.so.

Argument marshalling only: every step of the attention path runs in the
CUDA library.  If the library is missing this module raises; there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# BSA_LIBRARY_VARIANT=debug loads the range-checked build (see build.py)
LIB_PATH = os.path.join(HERE, "_lib", "libbsa_debug.so" if os.environ.get("BSA_LIBRARY_VARIANT") == "debug"
                        else "libbsa.so")

# status codes
OK, INVALID_ARG, UNSUPPORTED, CUDA, OOM, TIMEOUT, DEVICE = range(7)
# mask kinds
MASK_DENSE, MASK_CAUSAL, MASK_LOCAL, MASK_CHUNKED_CAUSAL, MASK_FULL = range(5)
ORIENT_FWD, ORIENT_DKV = 0, 1


class MaskSpec(C.Structure):
    _fields_ = [("kind", C.c_int32), ("mask_heads", C.c_int32), ("q_len", C.c_int64), ("kv_len", C.c_int64),
                ("local_left", C.c_int64), ("local_right", C.c_int64), ("chunk", C.c_int64),
                ("dense", C.c_void_p)]


class MaskOpts(C.Structure):
    _fields_ = [("block_q", C.c_int32), ("block_kv", C.c_int32), ("shrink", C.c_int32),
                ("orientation", C.c_int32)]


class MaskInfoDesc(C.Structure):
    _fields_ = [("block_mask", C.c_void_p), ("data_next", C.c_void_p), ("data_next_bytes", C.c_int32),
                ("mask_next", C.c_void_p), ("mask_next_bytes", C.c_int32),
                ("partial_mask_blocks", C.c_void_p), ("q_sequence", C.c_void_p),
                ("heads", C.c_int32), ("rows", C.c_int32), ("width", C.c_int32), ("cols", C.c_int32),
                ("num_partial", C.c_int64), ("n_empty", C.c_int64), ("n_partial", C.c_int64),
                ("n_full", C.c_int64), ("kind", C.c_int32), ("orientation", C.c_int32),
                ("shrink", C.c_int32), ("q_len", C.c_int64), ("kv_len", C.c_int64),
                ("row_len", C.c_void_p), ("row_order", C.c_void_p)]


class FwdArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("o", C.c_void_p),
                ("lse", C.c_void_p), ("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32),
                ("D", C.c_int32), ("S_q", C.c_int64), ("S_kv", C.c_int64), ("softmax_scale", C.c_float),
                ("logits_soft_cap", C.c_float), ("sinks", C.c_void_p), ("num_sinks", C.c_int32),
                ("sinks_per_kv_head", C.c_int32)]


class FwdPartialArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("o_acc", C.c_void_p),
                ("m", C.c_void_p), ("l", C.c_void_p), ("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32),
                ("D", C.c_int32), ("S_q", C.c_int64), ("S_kv_shard", C.c_int64), ("kv_offset", C.c_int64),
                ("softmax_scale", C.c_float), ("logits_soft_cap", C.c_float)]


class MergeArgs(C.Structure):
    _fields_ = [("n_shards", C.c_int32), ("o_acc", C.c_void_p), ("m", C.c_void_p), ("l", C.c_void_p),
                ("o", C.c_void_p), ("lse", C.c_void_p), ("rows", C.c_int64), ("D", C.c_int32)]


class BwdArgs(C.Structure):
    _fields_ = [("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("o", C.c_void_p),
                ("lse", C.c_void_p), ("do_", C.c_void_p), ("dq", C.c_void_p), ("dk", C.c_void_p),
                ("dv", C.c_void_p), ("dsum", C.c_void_p), ("B", C.c_int32), ("Hq", C.c_int32),
                ("Hkv", C.c_int32), ("D", C.c_int32), ("S_q", C.c_int64), ("S_kv", C.c_int64),
                ("softmax_scale", C.c_float), ("grad_fp32", C.c_int32), ("logits_soft_cap", C.c_float),
                ("sinks", C.c_void_p), ("dsinks", C.c_void_p), ("num_sinks", C.c_int32),
                ("sinks_per_kv_head", C.c_int32)]


# name -> (restype, argtypes); every symbol include/bsa.h declares
SIGNATURES = {
    "bsa_mask_compile": (C.c_int, [C.POINTER(MaskSpec), C.POINTER(MaskOpts), C.c_void_p, C.POINTER(C.c_void_p)]),
    "bsa_mask_info_view": (C.c_int, [C.c_void_p, C.POINTER(MaskInfoDesc)]),
    "bsa_mask_info_destroy": (C.c_int, [C.c_void_p]),
    "bsa_fwd": (C.c_int, [C.POINTER(FwdArgs), C.c_void_p, C.c_void_p]),
    "bsa_fwd_partial": (C.c_int, [C.POINTER(FwdPartialArgs), C.c_void_p, C.c_void_p]),
    "bsa_fwd_merge": (C.c_int, [C.POINTER(MergeArgs), C.c_void_p]),
    "bsa_bwd": (C.c_int, [C.POINTER(BwdArgs), C.c_void_p, C.c_void_p, C.c_void_p]),
    "bsa_bwd_rowsum": (C.c_int, [C.POINTER(BwdArgs), C.c_void_p]),
    "bsa_bwd_noalloc": (C.c_int, [C.POINTER(BwdArgs), C.c_void_p, C.c_void_p, C.c_void_p]),
    "bsa_bwd_dkv": (C.c_int, [C.POINTER(BwdArgs), C.c_void_p, C.c_void_p]),
    "bsa_bwd_dq": (C.c_int, [C.POINTER(BwdArgs), C.c_void_p, C.c_void_p]),
    "bsa_get_device_error": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint32)]),
    "bsa_set_wait_limit_ns": (C.c_int, [C.c_uint64]),
    "bsa_debug_wait_timeout": (C.c_int, [C.c_void_p]),
    "bsa_debug_selfcheck": (C.c_int, [C.c_void_p]),
    "bsa_debug_tile_schedule": (C.c_int, [C.POINTER(C.c_int32), C.POINTER(C.c_int32), C.c_int32, C.c_int32,
                                          C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                          C.POINTER(C.c_int32), C.c_int32, C.POINTER(C.c_int32)]),
    "bsa_status_string": (C.c_char_p, [C.c_int]),
    "bsa_last_error": (C.c_char_p, []),
    "bsa_version": (C.c_char_p, []),
}

_lib = None


def lib() -> C.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbsa.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                               "or python -m block_sparse_attention_process_gb300.build")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class BsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        L = lib()
        msg = L.bsa_last_error().decode(errors="replace")
        super().__init__(f"{where}: {L.bsa_status_string(status).decode()} ({status}): {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != OK:
        raise BsaError(status, where)
