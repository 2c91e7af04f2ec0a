"""Pins of the oracle's FP4-query x FP8-key lightning indexer.

The key format (E4M3 codes, a power-of-two scale per 32 channels chosen so
that no element saturates) is checked against its rule and the E4M3 grid;
the head dot against an exact-rational emulation (tests/exact.py) of
"exact dot of the dequantised vectors, rounded once to fp32"; and the whole
top-k against the FP4 x FP4 path on keys that are MXFP4 values already
(zcldvi.com DeepSeek-V4 article: FP4 -> FP8 dequantisation is lossless, so
the two indexers must agree bit for bit there).
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import f32_rn, fma32


def _e4m3_grid(oracle_mod):
    return oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))


def test_fp8b32_scale_rule_and_grid(oracle_mod):
    rng = np.random.default_rng(1)
    v = rng.standard_normal((64, 64)).astype(np.float32)
    v *= np.ldexp(1.0, rng.integers(-30, 30, size=(64, 2))).repeat(32, axis=1).astype(np.float32)
    v[3, :32] = 0.0                                   # an all-zero block
    v[4, :32] = np.float32(448.0)                     # amax exactly 448 -> e = 0
    v[5, 32:] = np.float32(448.0 * 2.0 ** 7)          # -> e = 7
    codes, scales = oracle_mod.fp8b32_quant(v)
    assert codes.shape == (64, 64) and scales.shape == (64, 2)
    grid = _e4m3_grid(oracle_mod)
    for r in range(64):
        for b in range(2):
            blk = v[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            e = int(scales[r, b]) - 127
            if amax == 0:
                assert e == 0 and not np.any(grid[codes[r, 32 * b:32 * b + 32]])
                continue
            # the smallest e with amax / 2^e <= 448
            assert amax / 2.0 ** e <= 448 and amax / 2.0 ** (e - 1) > 448
            x = blk / 2.0 ** e
            got = grid[codes[r, 32 * b:32 * b + 32]]
            finite = grid[np.isfinite(grid)]
            for xi, gi in zip(x, got):   # nearest grid value (ties: either neighbour at equal distance)
                assert abs(gi - xi) == np.min(np.abs(finite - xi))
    assert scales[4, 0] == 127 and scales[5, 1] == 127 + 7


def test_fp8b32_keeps_grid_values(oracle_mod):
    """Values already of the form E4M3 x 2^e (with the block's max making e
    the chosen scale) come back unchanged."""
    rng = np.random.default_rng(2)
    grid = _e4m3_grid(oracle_mod)
    fin = grid[np.isfinite(grid) & (np.abs(grid) <= 448)]
    for e in (-20, -3, 0, 5, 40):
        blk = rng.choice(fin, (3, 32)) * 2.0 ** e
        blk[:, 0] = 448.0 * 2.0 ** e
        codes, scales = oracle_mod.fp8b32_quant(blk.astype(np.float32))
        np.testing.assert_array_equal(oracle_mod.fp8b32_dequant(codes, scales), blk)


def _exact_dot(oracle_mod, qc, qs, kc8, ks8):
    qv = oracle_mod.mxfp4_dequant(qc, qs)
    kv = oracle_mod.fp8b32_dequant(kc8, ks8)
    return f32_rn(sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qv, kv)), Fraction(0)))


def test_fp4q_fp8k_dot_is_exact_then_rounded(oracle_mod):
    rng = np.random.default_rng(3)
    L = oracle_mod.lib()
    for trial in range(300):
        q = rng.standard_normal(64).astype(np.float32)
        k = rng.standard_normal(64).astype(np.float32)
        # spreads between the two blocks, on either side (the dot's two terms
        # then need more than 24 bits together), and tiny elements that land
        # on E4M3 subnormals
        q[32:] *= np.float32(2.0 ** int(rng.integers(-12, 13)))
        k[32:] *= np.float32(2.0 ** int(rng.integers(-12, 13)))
        if trial % 3 == 0:
            k[rng.integers(0, 64, 8)] *= np.float32(2.0 ** -14)
        (qc,), (qs,) = oracle_mod.mxfp4_quant(q[None])
        kc8, ks8 = oracle_mod.fp8b32_quant(k)
        got = np.float32(L.orc_fp4q_fp8k_dot(qc.ctypes.data, qs.ctypes.data, kc8.ctypes.data, ks8.ctypes.data, 64))
        assert got == _exact_dot(oracle_mod, qc, qs, kc8, ks8), trial


def test_fp4_keys_give_the_fp4_indexer(oracle_mod):
    """Keys that are MXFP4 values already are stored losslessly in FP8, and the
    FP8-key indexer then returns the FP4 indexer's indices and scores."""
    rng = np.random.default_rng(4)
    B, T, m, HI, dI, k = 2, 96, 4, 8, 64, 10
    N = T // m
    kf = rng.standard_normal((B, N, dI)).astype(np.float32)
    kf[:, :, 32:] *= np.float32(8.0)
    kc4, ks4 = oracle_mod.mxfp4_quant(kf)
    k_vals = oracle_mod.mxfp4_dequant(kc4, ks4).astype(np.float32)
    kc8, ks8 = oracle_mod.fp8b32_quant(k_vals)
    np.testing.assert_array_equal(oracle_mod.fp8b32_dequant(kc8, ks8), k_vals)   # lossless
    qI = rng.standard_normal((B, T, HI, dI)).astype(np.float32)
    w = rng.uniform(0, 1, (B, T, HI)).astype(np.float32)
    q_pos = np.tile(np.arange(T, dtype=np.int64), (B, 1))
    i4, s4 = oracle_mod.indexer_topk(qI, w, (kc4, ks4), q_pos, N, m, k)
    i8, s8 = oracle_mod.indexer_topk_fp8k(qI, w, (kc8, ks8), q_pos, N, m, k)
    np.testing.assert_array_equal(i8, i4)
    np.testing.assert_array_equal(s8.view(np.uint32), s4.view(np.uint32))


def test_topk_fp8k_matches_exact_scores_and_sort(oracle_mod):
    rng = np.random.default_rng(5)
    B, T, m, HI, dI, k = 1, 40, 4, 3, 64, 6
    N = T // m
    kf = rng.standard_normal((B, N, dI)).astype(np.float32)
    kc8, ks8 = oracle_mod.fp8b32_quant(kf)
    qI = rng.standard_normal((B, T, HI, dI)).astype(np.float32)
    w = rng.uniform(0, 1, (B, T, HI)).astype(np.float32)
    q_pos = np.arange(T, dtype=np.int64)[None]
    idx, sc = oracle_mod.indexer_topk_fp8k(qI, w, (kc8, ks8), q_pos, N, m, k)
    for t in range(T):
        qc, qs = oracle_mod.mxfp4_quant(qI[0, t])
        nv = min(N, (t + 1) // m)
        scores = []
        for j in range(nv):
            s = np.float32(0.0)
            for h in range(HI):
                d = _exact_dot(oracle_mod, qc[h], qs[h], kc8[0, j], ks8[0, j])
                s = fma32(w[0, t, h], d if d > 0 else np.float32(0.0), s)
            scores.append((-float(s), j, s))
        scores.sort()
        want = [j for _, j, _ in scores[:k]] + [-1] * (k - min(k, nv))
        np.testing.assert_array_equal(idx[0, t], want)
        for r in range(min(k, nv)):
            assert sc[0, t, r] == scores[r][2]


def test_fp4q_fp8k_dot_rounds_once_at_a_tie(oracle_mod):
    """A dot whose exact value sits just above an fp32 tie: block 0 gives
    (2^25 + 2) 2^25 (a tie at 24 bits), block 1 adds 2^-10.  The one rounding
    goes up; rounding through an intermediate fp64 sum (61 bits needed) would
    lose the small term and round the tie to even instead."""
    q2 = np.zeros(64, np.int64)          # twice the E2M1 values
    k512 = np.zeros(64, np.int64)        # 512 times the E4M3 values
    q2[:16], k512[:16] = 12, 2 ** 17     # 16 x 12 x 2^17 = 3 x 2^23
    q2[16:24], k512[16:24] = 8, 2 ** 17  # 8 x 8 x 2^17 = 2^23
    q2[24], k512[24] = 1, 2              # + 2
    q2[32], k512[32] = 1, 1              # block 1: 1
    e2m1_code = {0: 0, 1: 1, 8: 6, 12: 7}
    e4m3_code = {0: 0x00, 1: 0x01, 2: 0x02, 2 ** 17: 0x78}
    qc = np.zeros(32, np.uint8)
    for i in range(64):
        qc[i // 2] |= np.uint8(e2m1_code[int(q2[i])] << (4 * (i & 1)))
    kc8 = np.array([e4m3_code[int(v)] for v in k512], np.uint8)
    qs = np.array([127, 127], np.uint8)
    ks8 = np.array([127 + 35, 127], np.uint8)            # block exponents 25 and -10
    got = np.float32(oracle_mod.lib().orc_fp4q_fp8k_dot(qc.ctypes.data, qs.ctypes.data, kc8.ctypes.data,
                                                        ks8.ctypes.data, 64))
    want = _exact_dot(oracle_mod, qc, qs, kc8, ks8)
    assert want == np.float32((2.0 ** 25 + 4) * 2.0 ** 25)
    assert got == want
