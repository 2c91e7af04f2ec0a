"""ctypes loader of libcsa_b300.so (built in-tree by build.py).

Raises at first use when the library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(HERE, "libcsa_b300.so")

P = ctypes.c_void_p
I32 = ctypes.c_int
I64 = ctypes.c_int64
F32 = ctypes.c_float
F64 = ctypes.c_double
SZ = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/csa_b300.h
SIGNATURES = {
    "csa_last_error": (ctypes.c_char_p, []),
    "csa_version": (ctypes.c_char_p, []),
    "csa_rope_table": (I32, [I64, I32, F64, P, P]),
    "csa_selftest_wait_timeout": (I32, [P, ctypes.c_uint32, P]),
    "csa_workspace_size": (I64, [I32, I32, I64, I64, I32, I32, I32, I64, I64]),
    "csa_status_reset": (I32, [P, P]),
    "csa_status_read": (I32, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
    "kvcache_pack_fp8_bf16": (I32, [P, I64, P, P]),
    "csa_compress_kv": (I32, [P, I32, P, P, P, P, I64, I64, I32, I64, I32, I32, I32, I32, P, P, P]),
    "csa_compress_kv_channel_logits": (I32, [P, I32, P, P, P, P, I64, I64, I32, I64, I32, I32, I32, I32, P, P,
                                             P]),
    "csa_indexer_topk": (I32, [P, I32, P, P, P, I32, P, I32, I64, I32, I32, I64, I32, I32, P, P,
                               P, SZ, P]),
    "csa_sparse_mqa": (I32, [P, I32, P, I32, I64, I32, I32, I32, I32, P, I64, I32, P, I32, P, P,
                             I64, I32, F32, P, P, I64, P, P, P, SZ, P]),
    "csa_indexer_topk_noalloc": (I32, [P, I32, P, P, P, I32, P, I32, I64, I32, I32, I64, I32, I32, P,
                                       P, P]),
    "hca_dense_attn": (I32, [P, I32, P, I32, I64, I32, I32, I32, I32, P, I64, I32, P, P, I64, I32,
                             F32, P, P, I64, P, P, P, SZ, P]),
    "csa_decode_append": (I32, [P, P, P, P, P, P, P, P, I64, P, I32, I32, I32, I32, I32, P, P, P, P, P, I64, P,
                                P, P, I64, I32, P, P]),
}

_lib = None


class CsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"csa error {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(SO_PATH):
            raise RuntimeError(f"{SO_PATH} is not built: run `python -m long_context_sparse_29_b300.build`"
                               " (the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(SO_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(code: int) -> None:
    if code != 0:
        raise CsaError(code, lib().csa_last_error().decode())
