"""CPU oracle for DeepSeek-V4's hybrid compressed attention (CSA / HCA).

TEST INFRASTRUCTURE ONLY: the test-suite, the package smoke check and the
benchmark's CPU-baseline leg may import it; the CUDA library and its Python
binding never do.

The arithmetic lives in ``csa_oracle.c`` (plain C, fp64 attention, fp32
operation sequences written out where floating point decides a stored code).
This module only builds that file with gcc and marshals numpy arrays into it.
Each wrapper names the step of the method it computes; the sources are cited
in the C file.

Parity pins (tests/test_oracle_*.py) tie every function to something other
than itself: closed forms, exhaustive code tables of the number formats,
brute force on tiny inputs and special cases that reduce to a library routine
(causal attention).  Functions without such a pin are listed here:
parity unpinned -- the choice of the project exponential's polynomial (pinned
only to within 2 ulp of exp, not to a published bit pattern), the RoPE pair
convention, and the softmax scale; these are readings of the pages, not
results the pages fix.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_SO = os.path.join(_HERE, "_build", "libcsa_oracle.so")

FMT_F32 = 0
FMT_MIXED592 = 1


def build(force: bool = False) -> str:
    """Compile csa_oracle.c with gcc (no contraction of a*b+c into fma)."""
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int
F64 = ctypes.c_double


def _declare(L):
    sig = {
        "orc_set_threads": (None, [I32]),
        "orc_get_threads": (I32, []),
        "orc_rope_table": (None, [I64, I32, F64, P, P]),
        "orc_sexp": (ctypes.c_float, [ctypes.c_float]),
        "orc_sexp_vec": (None, [P, I64, P]),
        "orc_e4m3_encode_vec": (None, [P, I64, P]),
        "orc_e2m1_encode_vec": (None, [P, I64, P]),
        "orc_e4m3_decode": (F64, [ctypes.c_uint8]),
        "orc_e2m1_decode": (F64, [ctypes.c_uint8]),
        "orc_compress": (None, [P, P, P, I64, I64, I32, I32, I32, I64, P, P, I64, P]),
        "orc_compress_channel_logits": (None, [P, P, P, I64, I64, I32, I32, I32, I64, P, P, I64, P]),
        "orc_pack_mixed": (None, [P, I64, P]),
        "orc_unpack_mixed": (None, [P, I64, P]),
        "orc_mxfp4_quant": (None, [P, I64, I32, P, P]),
        "orc_mxfp4_dot": (ctypes.c_float, [P, P, P, P, I32]),
        "orc_indexer_topk_fp4": (None, [P, P, P, P, P, I64, I64, I32, I32, I64, I32, I32, P, P]),
        "orc_indexer_topk_f32": (None, [P, P, P, P, I64, I64, I32, I32, I64, I32, I32, P, P]),
        "orc_fp8b32_quant": (None, [P, I64, I32, P, P]),
        "orc_fp4q_fp8k_dot": (ctypes.c_float, [P, P, P, P, I32]),
        "orc_indexer_topk_fp4q_fp8k": (None, [P, P, P, P, P, I64, I64, I32, I32, I64, I32, I32, P, P]),
        "orc_attention": (None, [P, P, I64, I64, I32, I32, I32, I32, P, I64, I32, P, I32,
                                 P, P, I64, I32, F64, P, P, I64, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# --------------------------------------------------------------------------
# number formats and the project exponential
# --------------------------------------------------------------------------
def rope_table(P_rows: int, R: int, base: float = 10000.0):
    """cos/sin fp32 tables [P_rows, R/2] (fp64 evaluation, nearest fp32)."""
    c = np.empty((P_rows, R // 2), np.float32)
    s = np.empty((P_rows, R // 2), np.float32)
    lib().orc_rope_table(P_rows, R, float(base), _p(c), _p(s))
    return c, s


def sexp(x) -> np.ndarray:
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib().orc_sexp_vec(_p(x), x.size, _p(y))
    return y


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty(x.shape, np.uint8)
    lib().orc_e4m3_encode_vec(_p(x), x.size, _p(y))
    return y


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    table = np.array([L.orc_e4m3_decode(c) for c in range(256)], np.float64)
    return table[np.asarray(codes, np.uint8)]


def e2m1_encode(x) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty(x.shape, np.uint8)
    lib().orc_e2m1_encode_vec(_p(x), x.size, _p(y))
    return y


def e2m1_decode(codes) -> np.ndarray:
    L = lib()
    table = np.array([L.orc_e2m1_decode(c) for c in range(16)], np.float64)
    return table[np.asarray(codes, np.uint8) & 15]


# --------------------------------------------------------------------------
# compression and cache formats
# --------------------------------------------------------------------------
def compress(x, z, s, m: int, R: int, pos0: int = 0, rope=None) -> np.ndarray:
    """Block compression + RoPE of the last R channels: x fp32 [B, T, C] -> [B, T//m, C].

    z [B, T]: one logit per token; z [B, T, C]: one logit per token and channel.
    """
    x = _c(x, np.float32)
    B, T, C = x.shape
    per_channel = np.ndim(z) == 3
    z = _c(z, np.float32).reshape((B, T, C) if per_channel else (B, T))
    s = None if s is None else _c(s, np.float32)
    N = T // m
    out = np.empty((B, N, C), np.float32)
    if R > 0:
        rc, rs = (_c(rope[0], np.float32), _c(rope[1], np.float32))
        rows = rc.shape[0]
    else:
        rc = rs = None
        rows = 0
    fn = lib().orc_compress_channel_logits if per_channel else lib().orc_compress
    fn(_p(x), _p(z), _p(s), B, T, C, m, R, int(pos0), _p(rc), _p(rs), rows, _p(out))
    return out


def pack_mixed(v) -> np.ndarray:
    """fp32 [..., 512] post-RoPE rows -> mixed FP8/BF16 rows [..., 592] uint8."""
    v = _c(v, np.float32)
    lead = v.shape[:-1]
    assert v.shape[-1] == 512
    out = np.empty(lead + (592,), np.uint8)
    lib().orc_pack_mixed(_p(v), int(np.prod(lead, dtype=np.int64)), _p(out))
    return out


def unpack_mixed(rows) -> np.ndarray:
    rows = _c(rows, np.uint8)
    lead = rows.shape[:-1]
    out = np.empty(lead + (512,), np.float64)
    lib().orc_unpack_mixed(_p(rows), int(np.prod(lead, dtype=np.int64)), _p(out))
    return out


def mxfp4_quant(v):
    """fp32 [..., d] -> (codes [..., d/2] uint8, scales [..., d/32] uint8)."""
    v = _c(v, np.float32)
    lead, d = v.shape[:-1], v.shape[-1]
    n = int(np.prod(lead, dtype=np.int64))
    codes = np.empty(lead + (d // 2,), np.uint8)
    scales = np.empty(lead + (d // 32,), np.uint8)
    lib().orc_mxfp4_quant(_p(v), n, d, _p(codes), _p(scales))
    return codes, scales


def mxfp4_dequant(codes, scales) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    lo = e2m1_decode(codes & 15)
    hi = e2m1_decode(codes >> 4)
    v = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return v * np.repeat(sc, 32, axis=-1)


def compress_kv(x, z, s, m: int, fmt: str, R: int, pos0: int = 0, rope=None):
    """Oracle of the compress-and-store call.

    fmt 'f32' -> fp32 entries; 'mixed592' -> 592-byte rows; 'mxfp4' ->
    (codes, scales).  x fp32 [B, T, C] (bf16 inputs already widened).
    """
    e = compress(x, z, s, m, R, pos0, rope)
    if fmt == "f32":
        return e
    if fmt == "mixed592":
        return pack_mixed(e)
    if fmt == "mxfp4":
        return mxfp4_quant(e)
    if fmt == "fp8b32":
        return fp8b32_quant(e)
    raise ValueError(fmt)


def fp8b32_quant(v):
    """FP8 indexer keys: E4M3 codes with a power-of-two scale per 32 channels
    (the smallest 2^e with max|v| / 2^e <= 448; byte e + 127).
    v fp32 [..., d] -> (codes uint8 [..., d], scales uint8 [..., d/32])."""
    v = _c(v, np.float32)
    d = v.shape[-1]
    n = v.size // d
    codes = np.empty(v.shape, np.uint8)
    scales = np.empty(v.shape[:-1] + (d // 32,), np.uint8)
    lib().orc_fp8b32_quant(_p(v), n, d, _p(codes), _p(scales))
    return codes, scales


def fp8b32_dequant(codes, scales) -> np.ndarray:
    """fp64 values of FP8 keys (exact)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    d = codes.shape[-1]
    vals = e4m3_decode(codes.ravel()).reshape(codes.shape)
    sc = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return vals * np.repeat(sc, 32, axis=-1)[..., :d]


# --------------------------------------------------------------------------
# indexer + top-k
# --------------------------------------------------------------------------
def indexer_topk_fp8k(qI, w, keys, q_pos, N: int, m: int, k: int):
    """Top-k with MXFP4 queries and FP8 keys (codes [B, N, dI], scales
    [B, N, dI/32]); same order and padding as indexer_topk."""
    qI = _c(qI, np.float32)
    B, Tq, HI, dI = qI.shape
    w = _c(w, np.float32)
    q_pos = _c(q_pos, np.int64)
    kc, ks = _c(keys[0], np.uint8), _c(keys[1], np.uint8)
    idx = np.empty((B, Tq, k), np.int32)
    sc = np.empty((B, Tq, k), np.float32)
    lib().orc_indexer_topk_fp4q_fp8k(_p(qI), _p(w), _p(kc), _p(ks), _p(q_pos), B, Tq, HI, dI, N, m, k,
                                     _p(idx), _p(sc))
    return idx, sc


def indexer_topk(qI, w, keys, q_pos, N: int, m: int, k: int):
    """Top-k entry indices per query (score desc, index asc), -1 padded.

    qI fp32 [B, Tq, HI, dI]; w fp32 [B, Tq, HI]; keys either fp32 [B, N, dI]
    or (codes [B, N, dI/2], scales [B, N, dI/32]); q_pos int64 [B, Tq].
    Returns (idx int32 [B, Tq, k], scores fp32 [B, Tq, k]).
    """
    qI = _c(qI, np.float32)
    B, Tq, HI, dI = qI.shape
    w = _c(w, np.float32)
    q_pos = _c(q_pos, np.int64)
    idx = np.empty((B, Tq, k), np.int32)
    sc = np.empty((B, Tq, k), np.float32)
    if isinstance(keys, tuple):
        kc, ks = _c(keys[0], np.uint8), _c(keys[1], np.uint8)
        lib().orc_indexer_topk_fp4(_p(qI), _p(w), _p(kc), _p(ks), _p(q_pos), B, Tq, HI, dI, N,
                                   m, k, _p(idx), _p(sc))
    else:
        kf = _c(keys, np.float32)
        lib().orc_indexer_topk_f32(_p(qI), _p(w), _p(kf), _p(q_pos), B, Tq, HI, dI, N, m, k,
                                   _p(idx), _p(sc))
    return idx, sc


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def attention(q, q_pos, cache, N: int, m: int, idx, swa, swa_pos0, W: int, scale: float,
              rope, R: int = 64, fmt: int = FMT_MIXED592):
    """Sparse (idx given) or dense (idx None) MQA over entries + window.

    q fp32 [B, Tq, H, D]; cache rows [B, N, 592] uint8 or fp32 [B, N, D];
    swa rows [B, Ts, ...] in the same format; returns (out fp64 [B,Tq,H,D],
    lse fp64 [B,Tq,H], n_invalid).
    """
    q = _c(q, np.float32)
    B, Tq, H, D = q.shape
    q_pos = _c(q_pos, np.int64)
    dt = np.float32 if fmt == FMT_F32 else np.uint8
    cache = _c(cache, dt)
    swa = _c(swa, dt)
    Ts = swa.shape[1]
    swa_pos0 = _c(swa_pos0, np.int64)
    k = 0
    if idx is not None:
        idx = _c(idx, np.int32)
        k = idx.shape[-1]
    rc, rs = _c(rope[0], np.float32), _c(rope[1], np.float32)
    out = np.empty((B, Tq, H, D), np.float64)
    lse = np.empty((B, Tq, H), np.float64)
    bad = ctypes.c_int64(0)
    lib().orc_attention(_p(q), _p(q_pos), B, Tq, H, D, R, fmt, _p(cache), N, m, _p(idx), k,
                        _p(swa), _p(swa_pos0), Ts, W, float(scale), _p(rc), _p(rs), rc.shape[0],
                        _p(out), _p(lse), ctypes.byref(bad))
    return out, lse, int(bad.value)
