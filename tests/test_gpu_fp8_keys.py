"""GPU parity of the FP4-query x FP8-key lightning indexer against the oracle.

FP8 indexer keys (E4M3 codes, a power-of-two scale per 32 channels) are
written by csa_compress_kv (CSA_FMT_FP8B32) and scored by csa_indexer_topk
against MXFP4 queries; the bar is the one every indexer test uses: key
bytes, top-k indices and scores bit for bit.  xmsumi.com DeepSeek-V4
article, section "算力与内存效率" (FP4 x FP8 at the FP8 rate); zcldvi.com
article (FP4 -> FP8 is lossless).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as wl
from exact import f32_rn, fma32
from gpu_common import dev, dev_bf16, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


def _fp8_keys(csa, oracle_mod, cfg, b, T, t0=0):
    toks = wl.gen_tokens(cfg, b, t0, T, parts=("kI", "zI"))
    sI = wl.gen_channel_scales(cfg)["sI"]
    kd = csa.compress_kv(dev_bf16(toks["kI"])[None], dev(toks["zI"])[None], dev(sI), cfg.m, csa.FMT_FP8B32, 0)
    kn = oracle_mod.compress_kv(widen(toks["kI"], cfg)[None], toks["zI"][None], sI, cfg.m, "fp8b32", 0)
    return kd, kn


@pytest.mark.parametrize("name,b,T", [("c2_csa_prefill_8k", 0, 8192), ("c2_csa_prefill_8k", 0, 8192 - 5),
                                      ("c5_hybrid_csa_decode_1m", 2, 1 << 20)])
def test_compress_fp8_keys_bitexact(csa, oracle_mod, name, b, T):
    cfg = wl.CONFIGS[name]
    (kc, ks), (okc, oks) = _fp8_keys(csa, oracle_mod, cfg, b, T)
    assert tuple(kc.shape) == (1, T // cfg.m, cfg.dI) and tuple(ks.shape) == (1, T // cfg.m, cfg.dI // 32)
    np.testing.assert_array_equal(kc.cpu().numpy(), okc)
    np.testing.assert_array_equal(ks.cpu().numpy(), oks)


def test_indexer_fp8_keys_prefill_sampled(csa, oracle_mod):
    cfg = wl.CONFIGS["c2_csa_prefill_8k"]
    (kd, ksd), kn = _fp8_keys(csa, oracle_mod, cfg, 0, cfg.T)
    qry = wl.gen_queries(cfg, 0)
    q_pos = np.arange(cfg.Tq, dtype=np.int64)[None]
    idx, sc = csa.indexer_topk(dev_bf16(qry["qI"])[None], dev(qry["w"])[None], kd, ksd, dev(q_pos), cfg.N,
                               cfg.m, cfg.k)
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    sel = np.unique(np.concatenate([np.arange(0, 12), np.arange(cfg.k * cfg.m - 8, cfg.k * cfg.m + 8),
                                    [cfg.Tq - 1], np.random.default_rng(43).choice(cfg.Tq, 200, replace=False)]))
    oidx, osc = oracle_mod.indexer_topk_fp8k(widen(qry["qI"], cfg)[sel][None], qry["w"][sel][None], kn,
                                             q_pos[:, sel], cfg.N, cfg.m, cfg.k)
    np.testing.assert_array_equal(idx[:, sel], oidx)
    np.testing.assert_array_equal(sc[:, sel].view(np.uint32), osc.view(np.uint32))


@pytest.mark.parametrize("name,B", [("c3_csa_decode_128k", 8), ("c5_hybrid_csa_decode_1m", 4)])
def test_indexer_fp8_keys_decode(csa, oracle_mod, name, B):
    """Decode rows at 128K (8 of the 32 sequences) and 1M context (all 4,
    Student-t indexer queries): every row bit for bit."""
    cfg = wl.CONFIGS[name]
    keys = [_fp8_keys(csa, oracle_mod, cfg, b, cfg.T) for b in range(B)]
    kd = torch.cat([k[0][0] for k in keys])
    ksd = torch.cat([k[0][1] for k in keys])
    kn = (np.concatenate([k[1][0] for k in keys]), np.concatenate([k[1][1] for k in keys]))
    qry = [wl.gen_queries(cfg, b) for b in range(B)]
    qI = np.stack([q["qI"] for q in qry])
    w = np.stack([q["w"] for q in qry])
    q_pos = np.full((B, 1), cfg.T - 1, np.int64)
    idx, sc = csa.indexer_topk(dev_bf16(qI), dev(w), kd, ksd, dev(q_pos), cfg.N, cfg.m, cfg.k)
    oidx, osc = oracle_mod.indexer_topk_fp8k(widen(qI, cfg), w, kn, q_pos, cfg.N, cfg.m, cfg.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), osc.view(np.uint32))


def _random_fp8_keys(rng, n, exps):
    """FP8 keys with random E4M3 codes (no NaN codes) and block scale bytes drawn from exps."""
    codes = rng.integers(0, 256, size=(n, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] ^= 1                     # 0x7F / 0xFF are NaN: never stored
    scales = rng.choice(np.array(exps, np.uint8), size=(n, 2))
    return codes, scales


def test_indexer_fp8_keys_wide_scale_spread(csa, oracle_mod):
    """Block scales far apart (the two block terms of a head up to 36 binades
    apart, the widest the oracle's 64-bit sum holds exactly), random E4M3 codes
    including subnormals and both signs, top-k of every visible entry (k = N)
    so that every score is compared, decode-shaped and prefill-shaped."""
    rng = np.random.default_rng(77)
    for B, Tq, N in ((2, 1, 3000), (1, 40, 700)):
        codes, scales = _random_fp8_keys(rng, B * N, list(range(127 - 12, 127 + 13)))
        qI = rng.standard_normal((B, Tq, 16, 64)).astype(np.float32)
        qI[..., 32:] *= np.float32(2.0 ** 11)
        qbits = wl.f32_to_bf16_bits(qI)
        w = rng.uniform(0.0, 1.0, (B, Tq, 16)).astype(np.float32)
        q_pos = np.tile(np.arange(N - Tq, N, dtype=np.int64), (B, 1))
        k = min(N, 4096)
        idx, sc = csa.indexer_topk(dev_bf16(qbits), dev(w), dev(codes.reshape(B, N, 64)),
                                   dev(scales.reshape(B, N, 2)), dev(q_pos), N, 1, k)
        oidx, osc = oracle_mod.indexer_topk_fp8k(wl.bf16_bits_to_f32(qbits), w,
                                                 (codes.reshape(B, N, 64), scales.reshape(B, N, 2)), q_pos, N, 1, k)
        np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
        np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), osc.view(np.uint32))


def test_indexer_fp8_keys_beyond_the_oracle_span(csa, oracle_mod):
    """Block terms 40 to 100 binades apart, and results in the fp32 subnormal
    range: the scores are checked against exact rational arithmetic (the
    oracle's 64-bit sum does not cover these spreads)."""
    rng = np.random.default_rng(78)
    N, HI = 64, 2
    codes, scales = _random_fp8_keys(rng, N, [127])
    scales[:, 0] = rng.integers(127 + 40, 127 + 100, size=N).astype(np.uint8)   # block 0 far above block 1
    scales[N // 2:, :] = scales[N // 2:, ::-1]                                  # ... or far below it
    # entries 0..7: E4M3 subnormal codes under the smallest scale: fp32-subnormal scores
    codes[:8] = (rng.integers(0, 8, size=(8, 64)) | (rng.integers(0, 2, size=(8, 64)) << 7)).astype(np.uint8)
    scales[:8] = 0
    qI = rng.standard_normal((1, 1, HI, 64)).astype(np.float32)
    qbits = wl.f32_to_bf16_bits(qI)
    w = np.ones((1, 1, HI), np.float32)
    q_pos = np.array([[N - 1]], np.int64)
    idx, sc = csa.indexer_topk(dev_bf16(qbits), dev(w), dev(codes[None]), dev(scales[None]), dev(q_pos), N, 1, N)
    idx, sc = idx.cpu().numpy()[0, 0], sc.cpu().numpy()[0, 0]
    qc, qs = oracle_mod.mxfp4_quant(wl.bf16_bits_to_f32(qbits)[0, 0])
    want = {}
    for j in range(N):
        s = np.float32(0.0)
        kv = oracle_mod.fp8b32_dequant(codes[j], scales[j])
        for h in range(HI):
            qv = oracle_mod.mxfp4_dequant(qc[h], qs[h])
            exact = sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qv, kv)), Fraction(0))
            d = _f32_rn_any(exact)
            s = fma32(w[0, 0, h], d if d > 0 else np.float32(0.0), s)
        want[j] = s
    got = {int(j): v for j, v in zip(idx, sc)}
    assert sorted(got) == list(range(N))
    for j in range(N):
        assert np.float32(got[j]).view(np.uint32) == np.float32(want[j]).view(np.uint32), j


def _f32_rn_any(x: Fraction) -> np.float32:
    """Nearest fp32 (ties to even) of an exact rational, subnormals and
    overflow included."""
    if x == 0:
        return np.float32(0.0)
    sub = Fraction(2) ** -149
    if abs(x) < Fraction(2) ** -126:
        q = x / sub
        n = q.numerator // q.denominator            # floor
        r = q - n
        if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
            n += 1
        v = np.float32(n) * np.float32(2.0 ** -126) * np.float32(2.0 ** -23)
        return v if n != 0 else (np.float32(-0.0) if x < 0 else np.float32(0.0))
    if abs(x) >= Fraction(2) ** 128:
        return np.float32(np.inf if x > 0 else -np.inf)
    return f32_rn(x)
