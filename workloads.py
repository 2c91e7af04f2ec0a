"""Seeded synthetic inputs for the compressed-attention workloads.

This module only draws random arrays and names workload shapes. It holds none
of the method's arithmetic (no compression, quantisation, scoring, selection or
attention), so both the CUDA path and the CPU oracle can be fed from it without
sharing any code of the method.

Shapes and distributions follow the five workloads of the compressed sparse /
heavily compressed attention study (DeepSeek-V4: CSA with m=4, top-k and a
128-token window; HCA with m'=128):

* activations (q, kv, indexer q / k) ~ N(0, 1), rounded to bf16 except in the
  fp32 tiny case;
* compression logits ~ N(0, 1) (tiny case) or N(0, 0.5^2);
* per-channel compression scales ~ U(0.5, 1.5); indexer head weights ~ U(0, 1);
* in the hybrid 1M-context case the indexer queries are Student-t with
  3 degrees of freedom (heavy tails).

Every array comes from numpy's Philox counter-based generator keyed by
(seed, config name, tensor name, sequence), so any sequence of a batch can be
regenerated on its own.

bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
of the fp32 draw); fp32 tensors as ``float32``.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
import zlib

import numpy as np

__all__ = ["Config", "CONFIGS", "rng_for", "f32_to_bf16_bits", "bf16_bits_to_f32",
           "gen_tokens", "gen_queries", "gen_channel_scales"]


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    kind: str          # csa_prefill | csa_decode | hca_prefill | hca_decode
    B: int             # sequences
    T: int             # context tokens per sequence
    Tq: int            # query tokens per sequence (T for prefill, 1 for decode)
    m: int             # compression ratio
    k: int             # top-k (0 for dense HCA)
    W: int             # sliding window
    H: int             # query heads (one shared KV: MQA)
    D: int             # KV / head dim
    R: int             # RoPE dims (the last R of D)
    HI: int            # indexer heads
    dI: int            # indexer head dim
    fp32: bool         # fp32 throughout (no FP8/FP4/bf16)
    z_std: float       # std of the compression logits
    rope_base: float = 10000.0
    qI_dist: str = "normal"   # "normal" or "t3"

    @property
    def N(self) -> int:
        """Complete compressed entries per sequence."""
        return self.T // self.m

    @property
    def is_decode(self) -> bool:
        return self.kind.endswith("decode")


def _c(**kw) -> Config:
    return Config(**kw)


CONFIGS: dict[str, Config] = {
    # Tiny CSA causal prefill, fp32 throughout.
    "c1_tiny_csa_prefill": _c(name="c1_tiny_csa_prefill", kind="csa_prefill", B=1, T=512, Tq=512,
                              m=4, k=16, W=32, H=8, D=128, R=64, HI=4, dI=32, fp32=True,
                              z_std=1.0),
    # CSA prefill, 1 x 8192 tokens.
    "c2_csa_prefill_8k": _c(name="c2_csa_prefill_8k", kind="csa_prefill", B=1, T=8192, Tq=8192,
                            m=4, k=512, W=128, H=64, D=512, R=64, HI=16, dI=64, fp32=False,
                            z_std=0.5),
    # CSA prefill of 1 x 131072 tokens, run in query chunks against the growing cache.
    "c2_csa_prefill_128k": _c(name="c2_csa_prefill_128k", kind="csa_prefill", B=1, T=131072, Tq=131072,
                              m=4, k=512, W=128, H=64, D=512, R=64, HI=16, dI=64, fp32=False,
                              z_std=0.5),
    # CSA decode, batch 32 at 128K context.
    "c3_csa_decode_128k": _c(name="c3_csa_decode_128k", kind="csa_decode", B=32, T=131072, Tq=1,
                             m=4, k=1024, W=128, H=64, D=512, R=64, HI=16, dI=64, fp32=False,
                             z_std=0.5),
    # HCA prefill of 1 x 65536 tokens (512 entries at m'=128).
    "c4_hca_prefill_64k": _c(name="c4_hca_prefill_64k", kind="hca_prefill", B=1, T=65536, Tq=65536,
                             m=128, k=0, W=128, H=64, D=512, R=64, HI=0, dI=0, fp32=False,
                             z_std=0.5),
    # HCA decode, batch 16 at 1M context (8192 entries each).
    "c4_hca_decode_1m": _c(name="c4_hca_decode_1m", kind="hca_decode", B=16, T=1 << 20, Tq=1,
                           m=128, k=0, W=128, H=64, D=512, R=64, HI=0, dI=0, fp32=False,
                           z_std=0.5),
    # Hybrid pair at 1M context, decode batch 4: the CSA layer ...
    "c5_hybrid_csa_decode_1m": _c(name="c5_hybrid_csa_decode_1m", kind="csa_decode", B=4,
                                  T=1 << 20, Tq=1, m=4, k=1024, W=128, H=64, D=512, R=64,
                                  HI=16, dI=64, fp32=False, z_std=0.5, qI_dist="t3"),
    # ... followed by the HCA layer (its own activations).
    "c5_hybrid_hca_decode_1m": _c(name="c5_hybrid_hca_decode_1m", kind="hca_decode", B=4,
                                  T=1 << 20, Tq=1, m=128, k=0, W=128, H=64, D=512, R=64,
                                  HI=0, dI=0, fp32=False, z_std=0.5),
}


def rng_for(seed: int, *key) -> np.random.Generator:
    """Philox generator keyed by (seed, *key); key items are str or int."""
    words = [int(seed)]
    for item in key:
        words.append(zlib.crc32(item.encode()) if isinstance(item, str) else int(item))
    return np.random.Generator(np.random.Philox(np.random.SeedSequence(words)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Inputs are finite draws, so NaN handling is not needed here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _act(cfg: Config, rng: np.random.Generator, shape, dist: str = "normal") -> np.ndarray:
    if dist == "t3":
        x = rng.standard_t(3, size=shape).astype(np.float32)
    else:
        x = rng.standard_normal(size=shape, dtype=np.float32)
    return x if cfg.fp32 else f32_to_bf16_bits(x)


def gen_channel_scales(cfg: Config, seed: int = 0) -> dict:
    """Per-channel compression scales of the KV compressor and the indexer-key compressor."""
    out = {"s": rng_for(seed, cfg.name, "s").uniform(0.5, 1.5, size=cfg.D).astype(np.float32)}
    if cfg.dI:
        out["sI"] = rng_for(seed, cfg.name, "sI").uniform(0.5, 1.5, size=cfg.dI).astype(np.float32)
    return out


def gen_tokens(cfg: Config, b: int, t0: int = 0, t1: int | None = None, seed: int = 0,
               parts=("kv", "z", "kI", "zI")) -> dict:
    """Per-token activations of sequence b, tokens [t0, t1) of the context.

    kv [n, D] and z [n]; with an indexer also kI [n, dI] and zI [n].  Each
    tensor has its own generator, drawn in fixed blocks of 4096 tokens, so any
    sub-range or subset of tensors is the same slice of the full sequence.
    """
    t1 = cfg.T if t1 is None else t1
    blk = 4096
    widths = {"kv": cfg.D, "kI": cfg.dI}
    out = {}
    def block(name, c):
        lo, hi = c * blk, min((c + 1) * blk, cfg.T)
        a, e = max(t0, lo) - lo, min(t1, hi) - lo
        r = rng_for(seed, cfg.name, name, b, c)
        if name in ("kv", "kI"):
            v = _act(cfg, r, (hi - lo, widths[name]))
        else:
            v = r.standard_normal(size=hi - lo, dtype=np.float32) * np.float32(cfg.z_std)
        return v[a:e]

    jobs = [(name, c) for name in parts if not (name in ("kI", "zI") and not cfg.dI)
            for c in range(t0 // blk, (t1 + blk - 1) // blk)]
    with _cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        res = list(ex.map(lambda jc: block(*jc), jobs))
    out = {}
    for (name, _), v in zip(jobs, res):
        out.setdefault(name, []).append(v)
    return {k: np.concatenate(v) for k, v in out.items()}


def gen_channel_logits(cfg: Config, b: int, width: int, t0: int = 0, t1: int | None = None,
                       seed: int = 0) -> np.ndarray:
    """Per-token, per-channel compression logits of sequence b, tokens [t0, t1):
    fp32 [n, width] ~ N(0, z_std^2), drawn in blocks of 4096 tokens like gen_tokens."""
    t1 = cfg.T if t1 is None else t1
    blk = 4096
    parts = []
    for c in range(t0 // blk, (t1 + blk - 1) // blk):
        lo, hi = c * blk, min((c + 1) * blk, cfg.T)
        r = rng_for(seed, cfg.name, "zc", width, b, c)
        v = r.standard_normal(size=(hi - lo, width), dtype=np.float32) * np.float32(cfg.z_std)
        parts.append(v[max(t0, lo) - lo:min(t1, hi) - lo])
    return np.concatenate(parts)


def gen_queries(cfg: Config, b: int, q0: int = 0, q1: int | None = None, seed: int = 0) -> dict:
    """Query-side tensors of sequence b, query rows [q0, q1).

    q [n, H, D], and with an indexer qI [n, HI, dI] and w [n, HI].
    """
    q1 = cfg.Tq if q1 is None else q1
    blk = 256

    def block(c):
        lo, hi = c * blk, min((c + 1) * blk, cfg.Tq)
        a, e = max(q0, lo) - lo, min(q1, hi) - lo
        r = rng_for(seed, cfg.name, "qry", b, c)
        got = {"q": _act(cfg, r, (hi - lo, cfg.H, cfg.D))[a:e]}
        if cfg.dI:
            got["qI"] = _act(cfg, r, (hi - lo, cfg.HI, cfg.dI), cfg.qI_dist)[a:e]
            got["w"] = r.uniform(0.0, 1.0, size=(hi - lo, cfg.HI)).astype(np.float32)[a:e]
        return got

    # blocks are independent generators: drawn in parallel, joined in order
    blocks = range(q0 // blk, (q1 + blk - 1) // blk)
    with _cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
        res = list(ex.map(block, blocks))
    return {k: np.concatenate([r[k] for r in res]) for k in res[0]} if res else {}
