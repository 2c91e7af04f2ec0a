"""Pins of the oracle's lightning-indexer scores and top-k selection.

Scores are checked bit for bit against an exact-rational emulation of the
stated fp32 sequence (tests/exact.py), the selection against Python's sort on
(-score, index), and the visibility rule against its definition.
"""
from fractions import Fraction

import numpy as np
import pytest

from exact import f32_rn, fma32


def _score_fp4_exact(qc, qs, kc, ks, w):
    """sum_h fma(w_h, relu(RN(exact dot_h)), s) from the dequantised MXFP4 values."""
    from oracle import mxfp4_dequant
    s = np.float32(0.0)
    for h in range(qc.shape[0]):
        qv = mxfp4_dequant(qc[h], qs[h])
        kv = mxfp4_dequant(kc, ks)
        d = f32_rn(sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qv, kv)), Fraction(0)))
        r = d if d > 0 else np.float32(0.0)
        s = fma32(w[h], r, s)
    return s


def _score_f32_exact(q, k, w):
    s = np.float32(0.0)
    for h in range(q.shape[0]):
        d = np.float32(0.0)
        for i in range(q.shape[1]):
            d = fma32(q[h, i], k[i], d)
        r = d if d > 0 else np.float32(0.0)
        s = fma32(w[h], r, s)
    return s


def test_mxfp4_dot_is_exact_then_rounded(oracle_mod):
    rng = np.random.default_rng(20)
    L = oracle_mod.lib()
    for trial in range(300):
        spread = rng.integers(0, 12)
        v = rng.standard_normal((2, 64)).astype(np.float32)
        v[:, 32:] *= np.float32(2.0 ** (spread * (1 if trial % 2 else -1)))
        (qc, kc), (qs, ks) = oracle_mod.mxfp4_quant(v)
        got = L.orc_mxfp4_dot(qc.ctypes.data, qs.ctypes.data, kc.ctypes.data, ks.ctypes.data, 64)
        qv, kv = oracle_mod.mxfp4_dequant(qc, qs), oracle_mod.mxfp4_dequant(kc, ks)
        ref = f32_rn(sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qv, kv)), Fraction(0)))
        assert np.float32(got) == ref


def _visible(t, m, N):
    return min(N, max(0, (t + 1) // m))


@pytest.mark.parametrize("fp4", [False, True])
def test_topk_matches_exact_scores_and_sort(oracle_mod, fp4):
    rng = np.random.default_rng(21 + fp4)
    B, T, m, HI = 1, 48, 4, 4
    dI = 64 if fp4 else 32
    N = T // m
    qI = rng.standard_normal((B, T, HI, dI)).astype(np.float32)
    kf = rng.standard_normal((B, N, dI)).astype(np.float32)
    w = rng.uniform(0, 1, (B, T, HI)).astype(np.float32)
    q_pos = np.arange(T, dtype=np.int64)[None]
    keys = oracle_mod.mxfp4_quant(kf) if fp4 else kf
    k = N + 3                                   # k > |visible|: every candidate is returned
    idx, sc = oracle_mod.indexer_topk(qI, w, keys, q_pos, N, m, k)
    for t in range(0, T, 5):
        nv = _visible(t, m, N)
        if fp4:
            qc, qs = oracle_mod.mxfp4_quant(qI[0, t])
            exact = [_score_fp4_exact(qc, qs, keys[0][0, j], keys[1][0, j], w[0, t]) for j in range(nv)]
        else:
            exact = [_score_f32_exact(qI[0, t], kf[0, j], w[0, t]) for j in range(nv)]
        order = sorted(range(nv), key=lambda j: (-float(exact[j]), j))
        assert list(idx[0, t, :nv]) == order
        assert np.all(idx[0, t, nv:] == -1)
        np.testing.assert_array_equal(sc[0, t, :nv], np.array([exact[j] for j in order], np.float32))
        assert np.all(sc[0, t, :nv] >= 0)


def test_visibility_boundary(oracle_mod):
    """Entry j becomes a candidate exactly at t = (j + 1) m - 1."""
    rng = np.random.default_rng(23)
    m, N, HI, dI = 4, 8, 2, 32
    qI = rng.standard_normal((1, 40, HI, dI)).astype(np.float32)
    kf = rng.standard_normal((1, N, dI)).astype(np.float32)
    w = np.ones((1, 40, HI), np.float32)
    idx, _ = oracle_mod.indexer_topk(qI, w, kf, np.arange(40, dtype=np.int64)[None], N, m, N)
    for t in range(40):
        got = set(int(j) for j in idx[0, t] if j >= 0)
        assert got == {j for j in range(N) if (j + 1) * m - 1 <= t}


def test_ties_break_toward_lower_index(oracle_mod):
    """All-negative dots make every score +0: the lowest indices win, in order."""
    m, N, HI, dI = 4, 64, 2, 32
    qI = np.ones((1, 1, HI, dI), np.float32)
    kf = -np.ones((1, N, dI), np.float32)
    w = np.ones((1, 1, HI), np.float32)
    idx, sc = oracle_mod.indexer_topk(qI, w, kf, np.array([[10 ** 6]], np.int64), N, m, 16)
    assert list(idx[0, 0]) == list(range(16))
    assert np.all(sc == 0) and not np.any(np.signbit(sc))
    # a single positive key jumps to the front
    kf[0, 40] = 1.0
    idx, _ = oracle_mod.indexer_topk(qI, w, kf, np.array([[10 ** 6]], np.int64), N, m, 4)
    assert list(idx[0, 0]) == [40, 0, 1, 2]


def test_topk_truncates_in_score_order(oracle_mod):
    rng = np.random.default_rng(24)
    m, N, HI, dI, k = 4, 200, 4, 64, 17
    qI = rng.standard_normal((1, 3, HI, dI)).astype(np.float32)
    keys = oracle_mod.mxfp4_quant(rng.standard_normal((1, N, dI)).astype(np.float32))
    w = rng.uniform(0, 1, (1, 3, HI)).astype(np.float32)
    q_pos = np.array([[799, 500, 2]], np.int64)
    full, fs = oracle_mod.indexer_topk(qI, w, keys, q_pos, N, m, N)
    part, ps = oracle_mod.indexer_topk(qI, w, keys, q_pos, N, m, k)
    np.testing.assert_array_equal(part, full[..., :k])
    np.testing.assert_array_equal(ps, fs[..., :k])
    assert list(part[0, 2]) == [-1] * k          # t = 2 < m - 1 + 1: nothing visible
