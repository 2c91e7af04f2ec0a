"""B300 (sm_103a) compressed attention: DeepSeek-V4's CSA and HCA.

Thin Python binding over the C ABI of libcsa_b300.so (include/csa_b300.h):
argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; torch provides device memory and streams.

Calls (same names as the C ABI):
  compress_kv            block compression + RoPE + packing of KV / indexer keys
  kvcache_pack_fp8_bf16  standalone mixed FP8/BF16 row packing
  indexer_topk           lightning-indexer scores and top-k entry selection
  sparse_mqa             CSA: MQA over selected entries + sliding window
  hca_dense_attn         HCA: MQA over all visible entries + sliding window
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from ._lib import CsaError, check, lib

__all__ = ["CsaError", "Workspace", "ChunkedPrefill", "rope_table", "compress_kv", "kvcache_pack_fp8_bf16",
           "indexer_topk", "sparse_mqa", "hca_dense_attn", "workspace_size", "LayerCache", "decode_append",
           "DTYPE_F32", "DTYPE_BF16", "FMT_F32", "FMT_MIXED592", "FMT_MXFP4", "FMT_FP8B32"]

DTYPE_F32, DTYPE_BF16 = 0, 1
FMT_F32, FMT_MIXED592, FMT_MXFP4, FMT_FP8B32 = 0, 1, 2, 3
OP_INDEXER_TOPK, OP_SPARSE_MQA, OP_HCA_DENSE = 1, 2, 3
FLAG_DEVICE_CHECK, FLAG_TIMEOUT = 1, 2
MIXED_ROW = 592


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _dt(t):
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def workspace_size(op: int, B: int, Tq: int, N: int, k: int, H: int, D: int, max_keys: int,
                   Ts: int = 0) -> int:
    return int(lib().csa_workspace_size(op, B, Tq, N, k, H, D, max_keys, Ts))


class Workspace:
    """Device scratch for the library calls (first 16 bytes: status flags).

    Grows on demand; `flags()` reads the sticky device-check / timeout flags.
    """

    def __init__(self, device=None, nbytes: int = 1 << 20):
        self.device = torch.device(device or "cuda")
        self.buf = None
        self._alloc(nbytes)

    def _alloc(self, nbytes):
        self.buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=self.device)
        check(lib().csa_status_reset(_ptr(self.buf), _stream(self.device)))

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self._alloc(nbytes + (nbytes >> 3))
        return self.buf

    def reset(self):
        check(lib().csa_status_reset(_ptr(self.buf), _stream(self.device)))

    def flags(self) -> int:
        f = ctypes.c_uint32(0)
        code = lib().csa_status_read(_ptr(self.buf), _stream(self.device), ctypes.byref(f))
        if code not in (0, -4, -5):
            check(code)
        return int(f.value)


_default_ws: dict = {}


def _ws(ws, device):
    if ws is not None:
        return ws
    key = torch.device(device).index if torch.device(device).index is not None else torch.cuda.current_device()
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device("cuda", key))
    return _default_ws[key]


def selftest_wait_timeout(ws: Workspace, polls: int = 1000) -> None:
    """Make one bounded device wait expire on purpose; ws's timeout flag is
    then set (see csa_selftest_wait_timeout)."""
    check(lib().csa_selftest_wait_timeout(_ptr(ws.buf), int(polls), _stream(ws.device)))


def rope_table(P: int, R: int = 64, base: float = 10000.0, device="cuda"):
    """cos/sin tables fp32 [P, R/2] on `device` (built on the host by the library)."""
    c = np.empty((P, R // 2), np.float32)
    s = np.empty((P, R // 2), np.float32)
    check(lib().csa_rope_table(P, R, float(base), c.ctypes.data_as(ctypes.c_void_p),
                               s.ctypes.data_as(ctypes.c_void_p)))
    return torch.from_numpy(c).to(device), torch.from_numpy(s).to(device)


def compress_kv(x, z, s, m: int, out_fmt: int, R: int = 0, rope=None, pos0: int = 0, out=None,
                out_scales=None):
    """Compress x [B, T, C] (bf16 or fp32) in blocks of m; see csa_compress_kv.

    z fp32 [B, T] (one logit per token), or [B, T, C] (one per token and
    channel: csa_compress_kv_channel_logits).  Returns fp32 [B, N, C]
    (FMT_F32), uint8 [B, N, 592] (FMT_MIXED592), (codes uint8 [B, N, C/2],
    scales uint8 [B, N, C/32]) (FMT_MXFP4) or (codes uint8 [B, N, C], scales
    uint8 [B, N, C/32]) (FMT_FP8B32).
    """
    _need(x, "x")
    B, T, C = x.shape
    _need(z, "z", torch.float32)
    per_channel = z.dim() == 3
    if tuple(z.shape) != ((B, T, C) if per_channel else (B, T)):
        raise CsaError(f"z has shape {tuple(z.shape)}; [B, T] or [B, T, C] expected")
    if s is not None:
        _need(s, "s", torch.float32)
    N = T // m
    dev = x.device
    if out is None:
        if out_fmt == FMT_F32:
            out = torch.empty((B, N, C), dtype=torch.float32, device=dev)
        elif out_fmt == FMT_MIXED592:
            out = torch.empty((B, N, MIXED_ROW), dtype=torch.uint8, device=dev)
        else:
            out = torch.empty((B, N, C if out_fmt == FMT_FP8B32 else C // 2), dtype=torch.uint8, device=dev)
            out_scales = torch.empty((B, N, C // 32), dtype=torch.uint8, device=dev)
    rc, rs = (rope if rope is not None else (None, None))
    rows = rc.shape[0] if rc is not None else 0
    fn = lib().csa_compress_kv_channel_logits if per_channel else lib().csa_compress_kv
    check(fn(_ptr(x), _dt(x), _ptr(z), _ptr(s), _ptr(rc), _ptr(rs), rows, pos0,
             B, T, C, R, m, out_fmt, _ptr(out), _ptr(out_scales), _stream(dev)))
    return (out, out_scales) if out_fmt in (FMT_MXFP4, FMT_FP8B32) else out


class LayerCache:
    """Device state of one attention layer's decode caches (csa_decode_append):
    compressed entries [B, nmax, 592], indexer keys (CSA layers: CI > 0), the
    window cache [B, Ts, 592] with its first position per sequence, and the
    rings of the last m raw tokens."""

    def __init__(self, B: int, nmax: int, m: int, W: int, Ts: int | None = None, CI: int = 0, C: int = 512,
                 pos0: int = 0, device="cuda"):
        dev = torch.device(device)
        self.B, self.nmax, self.m, self.W, self.CI, self.C = B, nmax, m, W, CI, C
        self.Ts = Ts if Ts is not None else 2 * W
        self.cache = torch.zeros((B, nmax, MIXED_ROW), dtype=torch.uint8, device=dev)
        self.kI_codes = torch.zeros((B, nmax, CI // 2), dtype=torch.uint8, device=dev) if CI else None
        self.kI_scales = torch.zeros((B, nmax, CI // 32), dtype=torch.uint8, device=dev) if CI else None
        self.swa = torch.zeros((B, self.Ts, MIXED_ROW), dtype=torch.uint8, device=dev)
        self.swa_pos0 = torch.full((B,), pos0, dtype=torch.int64, device=dev)
        self.kv_tail = torch.zeros((B, m, C), dtype=torch.bfloat16, device=dev)
        self.z_tail = torch.zeros((B, m), dtype=torch.float32, device=dev)
        self.kI_tail = torch.zeros((B, m, CI), dtype=torch.bfloat16, device=dev) if CI else None
        self.zI_tail = torch.zeros((B, m), dtype=torch.float32, device=dev) if CI else None


def decode_append(lc: LayerCache, kv, z, t_pos, rope, kI=None, zI=None, s=None, sI=None, R: int = 64):
    """Append one token per sequence to lc (see csa_decode_append): kv [B, C]
    bf16, z [B] fp32, t_pos [B] int64 (device), kI [B, CI] bf16 / zI [B] for
    CSA layers."""
    _need(kv, "kv", torch.bfloat16)
    _need(z, "z", torch.float32)
    _need(t_pos, "t_pos", torch.int64)
    B, C = kv.shape
    rc, rs = rope
    check(lib().csa_decode_append(_ptr(kv), _ptr(z), _ptr(kI), _ptr(zI), _ptr(s), _ptr(sI), _ptr(rc), _ptr(rs),
                                  rc.shape[0], _ptr(t_pos), B, C, R, lc.CI, lc.m, _ptr(lc.kv_tail), _ptr(lc.z_tail),
                                  _ptr(lc.kI_tail), _ptr(lc.zI_tail), _ptr(lc.cache), lc.nmax, _ptr(lc.kI_codes),
                                  _ptr(lc.kI_scales), _ptr(lc.swa), lc.Ts, lc.W, _ptr(lc.swa_pos0),
                                  _stream(kv.device)))


class ChunkedPrefill:
    """Prefill of one sequence in query chunks against resident caches that
    grow chunk by chunk (entries [1, N, 592], window rows [1, T, 592], MXFP4
    indexer keys).  run(t0, t1, ...) stores the chunk's tokens at their
    positions (csa_compress_kv: entries, window rows with m = 1, keys), then
    the chunk's queries select among and attend over everything visible so
    far (csa_indexer_topk, csa_sparse_mqa on views of the caches that end at
    the chunk's last visible entry / start at its first window token).  Each
    step is one library call; nothing is computed here."""

    def __init__(self, T: int, m: int, k: int, W: int, rope, C: int = 512, CI: int = 64, R: int = 64,
                 device="cuda"):
        dev = torch.device(device)
        self.T, self.m, self.k, self.W, self.C, self.CI, self.R, self.rope = T, m, k, W, C, CI, R, rope
        N = T // m
        self.cache = torch.zeros((1, N, MIXED_ROW), dtype=torch.uint8, device=dev)
        self.swa = torch.zeros((1, T, MIXED_ROW), dtype=torch.uint8, device=dev)
        self.kc = torch.zeros((1, N, CI // 2), dtype=torch.uint8, device=dev)
        self.ks = torch.zeros((1, N, CI // 32), dtype=torch.uint8, device=dev)
        self.q_pos = torch.arange(T, dtype=torch.int64, device=dev)[None]
        self.ws_ix, self.ws_attn = Workspace(dev), Workspace(dev)
        self._pos0 = {}
        self._idx = None

    def _window_start(self, t0: int):
        lo = max(0, t0 - self.W + 1)   # the first window token of query t0
        if lo not in self._pos0:
            self._pos0[lo] = torch.full((1,), lo, dtype=torch.int64, device=self.cache.device)
        return lo, self._pos0[lo]

    def run(self, t0: int, t1: int, kv, z, kI, zI, s, sI, q, qI, w, scale: float, out=None):
        """Tokens and queries [t0, t1) (t0 a multiple of m; chunk tensors [1, t1 - t0, ...])."""
        m = self.m
        if t0 % m or t1 <= t0 or t1 > self.T:
            raise CsaError(f"chunk [{t0}, {t1}) must start at a multiple of m = {m} and lie in [0, {self.T}]")
        e0, e1 = t0 // m, t1 // m
        compress_kv(kv, z, s, m, FMT_MIXED592, self.R, self.rope, pos0=t0, out=self.cache[:, e0:e1])
        compress_kv(kv, z, None, 1, FMT_MIXED592, self.R, self.rope, pos0=t0, out=self.swa[:, t0:t1])
        compress_kv(kI, zI, sI, m, FMT_MXFP4, 0, out=self.kc[:, e0:e1], out_scales=self.ks[:, e0:e1])
        n = t1 - t0
        if self._idx is None or self._idx.shape[1] < n:
            self._idx = torch.empty((1, n, self.k), dtype=torch.int32, device=self.cache.device)
        idx = self._idx[:, :n]
        qp = self.q_pos[:, t0:t1]
        indexer_topk(qI, w, self.kc[:, :e1], self.ks[:, :e1], qp, e1, m, self.k, scores=False, idx_out=idx,
                     ws=self.ws_ix)
        lo, pos0 = self._window_start(t0)
        return sparse_mqa(q, qp, self.cache[:, :e1], m, idx, self.swa[:, lo:t1], pos0, self.W, scale, self.rope,
                          self.R, out=out, ws=self.ws_attn)


def kvcache_pack_fp8_bf16(v, out=None):
    """Pack post-RoPE rows v fp32 [..., 512] into uint8 [..., 592]."""
    _need(v, "v", torch.float32)
    lead = v.shape[:-1]
    n = int(np.prod(lead)) if len(lead) else 1
    if out is None:
        out = torch.empty(tuple(lead) + (MIXED_ROW,), dtype=torch.uint8, device=v.device)
    check(lib().kvcache_pack_fp8_bf16(_ptr(v), n, _ptr(out), _stream(v.device)))
    return out


def indexer_topk(qI, w, kI, kI_scales, q_pos, N: int, m: int, k: int, scores: bool = True,
                 idx_out=None, score_out=None, ws: Workspace | None = None):
    """Top-k entries per query.  qI [B, Tq, HI, dI] bf16 with MXFP4 keys (codes
    [B, N, dI/2]) or FP8 keys (codes [B, N, dI]), both with kI_scales
    [B, N, dI/32]; or qI fp32 with fp32 keys (kI_scales None)."""
    _need(qI, "qI")
    _need(w, "w", torch.float32)
    _need(q_pos, "q_pos", torch.int64)
    _need(kI, "kI")
    B, Tq, HI, dI = qI.shape
    fmt = FMT_F32 if kI_scales is None else (FMT_FP8B32 if kI.shape[-1] == dI else FMT_MXFP4)
    dev = qI.device
    if idx_out is None:
        idx_out = torch.empty((B, Tq, k), dtype=torch.int32, device=dev)
    if scores and score_out is None:
        score_out = torch.empty((B, Tq, k), dtype=torch.float32, device=dev)
    ws = _ws(ws, dev)
    need = workspace_size(OP_INDEXER_TOPK, B, Tq, N, k, HI, dI, 0, 0)
    buf = ws.get(need)
    check(lib().csa_indexer_topk(_ptr(qI), _dt(qI), _ptr(w), _ptr(kI), _ptr(kI_scales), fmt,
                                 _ptr(q_pos), B, Tq, HI, dI, N, m, k, _ptr(idx_out),
                                 _ptr(score_out if scores else None), _ptr(buf), buf.numel(),
                                 _stream(dev)))
    return (idx_out, score_out) if scores else idx_out


def _attn(q, q_pos, cache, N, m, idx, swa, swa_pos0, W, scale, rope, R, want_lse, out, ws):
    _need(q, "q")
    _need(q_pos, "q_pos", torch.int64)
    B, Tq, H, D = q.shape
    fmt = FMT_MIXED592 if q.dtype == torch.bfloat16 else FMT_F32
    dev = q.device
    if swa is not None:
        _need(swa, "swa")
        _need(swa_pos0, "swa_pos0", torch.int64)
    Ts = swa.shape[1] if swa is not None else 0
    if out is None:
        out = torch.empty_like(q)
    lse = torch.empty((B, Tq, H), dtype=torch.float32, device=dev) if want_lse else None
    rc, rs = rope
    ws = _ws(ws, dev)
    k = idx.shape[-1] if idx is not None else 0
    max_keys = (k if idx is not None else N) + W
    op = OP_SPARSE_MQA if idx is not None else OP_HCA_DENSE
    buf = ws.get(workspace_size(op, B, Tq, N, k, H, D, max_keys, Ts))
    st = _stream(dev)
    if idx is not None:
        _need(idx, "idx", torch.int32)
        check(lib().csa_sparse_mqa(_ptr(q), _dt(q), _ptr(q_pos), B, Tq, H, D, R, fmt, _ptr(cache), N,
                                   m, _ptr(idx), k, _ptr(swa), _ptr(swa_pos0), Ts, W, float(scale),
                                   _ptr(rc), _ptr(rs), rc.shape[0], _ptr(out), _ptr(lse), _ptr(buf),
                                   buf.numel(), st))
    else:
        check(lib().hca_dense_attn(_ptr(q), _dt(q), _ptr(q_pos), B, Tq, H, D, R, fmt, _ptr(cache), N,
                                   m, _ptr(swa), _ptr(swa_pos0), Ts, W, float(scale), _ptr(rc),
                                   _ptr(rs), rc.shape[0], _ptr(out), _ptr(lse), _ptr(buf),
                                   buf.numel(), st))
    return (out, lse) if want_lse else out


def sparse_mqa(q, q_pos, cache, m: int, idx, swa, swa_pos0, W: int, scale: float, rope,
               R: int = 64, lse: bool = False, out=None, ws: Workspace | None = None):
    """CSA: attention of q [B, Tq, H, D] over the idx-selected entries of cache
    [B, N, row] (block size m) and the window rows of swa; see csa_sparse_mqa."""
    return _attn(q, q_pos, cache, cache.shape[1], m, idx, swa, swa_pos0, W, scale, rope, R, lse,
                 out, ws)


def hca_dense_attn(q, q_pos, cache, m: int, swa, swa_pos0, W: int, scale: float, rope,
                   R: int = 64, lse: bool = False, out=None, ws: Workspace | None = None):
    """HCA: attention of q over every visible entry of cache [B, N, row] (block size m)
    and the window rows of swa; see hca_dense_attn."""
    return _attn(q, q_pos, cache, cache.shape[1], m, None, swa, swa_pos0, W, scale, rope, R, lse,
                 out, ws)
