"""Pins of the oracle's number formats, RoPE table and project exponential.

Every check compares the oracle with something other than itself: the OCP
format definitions enumerated independently, brute-force nearest-value search,
torch's float8 cast, numpy's fp64 cos/sin/exp and the figures the pages print.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e4m3_values():
    """All finite non-negative OCP E4M3 values by code, from the format definition."""
    vals = {}
    for code in range(128):
        e, m = code >> 3, code & 7
        if e == 15 and m == 7:
            continue  # NaN
        vals[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def test_e4m3_decode_table(oracle_mod):
    vals = _e4m3_values()
    dec = oracle_mod.e4m3_decode(np.arange(256))
    for code, v in vals.items():
        assert dec[code] == v
        assert dec[code | 0x80] == -v
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert max(vals.values()) == 448.0
    assert vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6


def _brute_nearest_e4m3(x):
    vals = _e4m3_values()
    codes = np.array(sorted(vals), dtype=np.int64)
    mags = np.array([vals[c] for c in codes])
    out = []
    for v in x:
        a = abs(v)
        if a >= 448.0:
            c = 0x7E
        else:
            d = np.abs(mags - a)
            best = np.flatnonzero(d == d.min())
            c = int(codes[best[0]]) if len(best) == 1 else int(codes[best][codes[best] % 2 == 0][0])
        out.append(c | (0x80 if math.copysign(1.0, v) < 0 else 0))
    return np.array(out, np.uint8)


def test_e4m3_encode_brute_force(oracle_mod):
    rng = np.random.default_rng(1)
    mags = np.array(sorted(_e4m3_values().values()))
    mids = (mags[1:] + mags[:-1]) / 2
    x = np.concatenate([
        mags, -mags, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
        rng.uniform(-500, 500, 2000), rng.standard_normal(2000) * 0.01,
        np.ldexp(rng.uniform(-1, 1, 2000), rng.integers(-12, 9, 2000)),
        [0.0, -0.0, 448.0, 449.0, 464.0, 1e30, -1e30, 2.0 ** -10, -(2.0 ** -10)],
    ])
    np.testing.assert_array_equal(oracle_mod.e4m3_encode(x), _brute_nearest_e4m3(x))


def test_e4m3_encode_matches_torch_cast(oracle_mod):
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(100000) * 50,
                        np.ldexp(rng.uniform(-1, 1, 100000), rng.integers(-14, 9, 100000))])
    x = x[np.abs(x) < 448].astype(np.float32)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle_mod.e4m3_encode(x.astype(np.float64)), t)


def test_e2m1_table_and_ties(oracle_mod):
    dec = oracle_mod.e2m1_decode(np.arange(16))
    np.testing.assert_array_equal(dec[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(dec[8:], -np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6]))
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "ocp_e2m1_ties.txt"))
            if ln.strip() and not ln.startswith("#")]
    for x, code, val in rows:
        c = oracle_mod.e2m1_encode([float(x)])[0]
        assert c == int(code), x
        assert oracle_mod.e2m1_decode([c])[0] == float(val)
        assert oracle_mod.e2m1_encode([-float(x)])[0] == int(code) | 8


def test_e2m1_encode_brute_force(oracle_mod):
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-8, 8, 20000), np.linspace(-7, 7, 561)])
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    exp = []
    for v in x:
        d = np.abs(mags - min(abs(v), 6.0))
        best = np.flatnonzero(d == d.min())
        c = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        exp.append(c | (8 if v < 0 or (v == 0 and math.copysign(1, v) < 0) else 0))
    np.testing.assert_array_equal(oracle_mod.e2m1_encode(x), np.array(exp, np.uint8))


def test_fp4_to_fp8_is_lossless(oracle_mod):
    """zcldvi.com article: dequantising FP4 to FP8 loses nothing (E4M3 has two
    more exponent bits than E2M1).  Every E2M1 value times a power-of-two block
    scale that lands in E4M3's range is itself an E4M3 value."""
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for k in range(-8, 7):
        v = e2 * 2.0 ** k
        v = v[(v == 0) | ((v >= 2.0 ** -9) & (v <= 448))]
        back = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(v))
        np.testing.assert_array_equal(back, v)


def test_sexp_accuracy(oracle_mod):
    x = np.concatenate([np.linspace(-87, 0, 200001), -np.logspace(-8, 1.9, 5000), [0.0, -0.0]])
    x = x.astype(np.float32)
    y = oracle_mod.sexp(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(y - ref) / ulp) <= 2.0
    assert oracle_mod.sexp(np.float32([0.0]))[0] == 1.0
    srt = np.argsort(x, kind="stable")
    assert np.all(np.diff(y[srt]) >= 0)
    assert oracle_mod.sexp(np.float32([-87.5, -100.0]))[0] == 0.0


def test_rope_table_against_numpy(oracle_mod):
    P, R, base = 4096, 64, 10000.0
    c, s = oracle_mod.rope_table(P, R, base)
    theta = base ** (-2.0 * np.arange(R // 2) / R)
    ang = np.arange(P)[:, None] * theta[None, :]
    for got, ref in ((c, np.cos(ang)), (s, np.sin(ang))):
        ulps = np.abs(got.astype(np.float64) - ref.astype(np.float32).astype(np.float64))
        ulps /= np.spacing(np.abs(ref).astype(np.float32).astype(np.float64) + 1e-30)
        assert ulps.max() <= 1.0
    # each pair rotation is orthonormal and p = 0 is the identity
    assert np.max(np.abs(c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2 - 1)) < 3e-7
    assert np.all(c[0] == 1) and np.all(s[0] == 0)


def test_rope_relative_position(oracle_mod):
    """Rotating q at t and k at u leaves q.k a function of t - u only."""
    P, R = 2048, 64
    c, s = oracle_mod.rope_table(P, R)
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(R), rng.standard_normal(R)

    def rot(v, p):
        x0, x1 = v[0::2], v[1::2]
        out = np.empty_like(v)
        out[0::2] = x0 * c[p] - x1 * s[p]
        out[1::2] = x0 * s[p] + x1 * c[p]
        return out
    d = [rot(q, t) @ rot(k, t - 37) for t in (37, 500, 1999)]
    assert np.ptp(d) < 1e-4 * np.abs(d).max()


def test_mixed_pack_layout_and_scales(oracle_mod):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 512)).astype(np.float32)
    v[3, 130] = 300.0          # large value in group 1 only
    v[4, :128] = 0.0           # empty group 0
    rows = oracle_mod.pack_mixed(v)
    assert rows.shape == (64, 592)
    scales = rows[:, 576:592].copy().view(np.float32)
    groups = [(0, 128), (128, 256), (256, 384), (384, 448)]
    for r in range(64):
        for g, (lo, hi) in enumerate(groups):
            amax = np.abs(v[r, lo:hi]).max()
            sc = float(scales[r, g])
            e = math.frexp(sc)[1] - 1
            assert sc == 2.0 ** e
            if amax == 0:
                assert sc == 1.0
                continue
            assert amax / sc <= 448 < amax / (sc / 2)          # smallest such power of two
            exp_codes = oracle_mod.e4m3_encode(v[r, lo:hi].astype(np.float64) / sc)
            np.testing.assert_array_equal(rows[r, lo:hi], exp_codes)
    # RoPE dims are bf16 (nearest-even), little endian, at bytes [448, 576)
    bf = torch.from_numpy(v[:, 448:]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(rows[:, 448:576].copy().view(np.uint16), bf)
    # only group 1 of row 3 has a changed scale relative to row-wise clean data
    assert scales[3, 1] > 4 * max(scales[3, 0], scales[3, 2])
    # dequantisation error bound: half an E4M3 step, relative 2^-4 for normals
    deq = oracle_mod.unpack_mixed(rows)
    nope = np.abs(deq[:, :448] - v[:, :448])
    tol = np.maximum(np.abs(v[:, :448]) * 2.0 ** -4, np.repeat(scales, [128, 128, 128, 64], axis=1) * 2.0 ** -10)
    assert np.all(nope <= tol + 1e-30)


def test_mxfp4_block_scale_rule(oracle_mod):
    rng = np.random.default_rng(6)
    v = (rng.standard_normal((200, 64)) * np.exp(rng.uniform(-6, 6, (200, 1)))).astype(np.float32)
    v[7, :32] = 0.0
    codes, scales = oracle_mod.mxfp4_quant(v)
    for r in range(200):
        for b in range(2):
            blk = v[r, 32 * b:32 * b + 32].astype(np.float64)
            amax = np.abs(blk).max()
            if amax == 0:
                assert scales[r, b] == 127
                continue
            X = 2.0 ** (math.floor(math.log2(amax)) - 2)
            assert scales[r, b] == int(round(math.log2(X))) + 127
            els = np.stack([codes[r] & 15, codes[r] >> 4], -1).reshape(-1)[32 * b:32 * b + 32]
            np.testing.assert_array_equal(els, oracle_mod.e2m1_encode(blk / X))
    deq = oracle_mod.mxfp4_dequant(codes, scales)
    assert np.all(np.abs(deq) <= np.repeat(np.ldexp(6.0, scales.astype(int) - 127), 32, -1))


def test_kv_cache_ratios_printed_on_pages():
    cfg = dict(ln.split()[:2] for ln in open(os.path.join(GOLDEN, "kv_cache_ratios.txt"))
               if ln.strip() and not ln.startswith("#"))
    gqa = float(cfg["gqa8_bf16_bytes_per_token"])
    row, idx_key = 592, 32 + 2               # mixed row; MXFP4 indexer key (64 dims)
    csa = row / 4 + idx_key / 4              # m = 4
    hca = row / 128                          # m' = 128
    ratio = (csa + hca) / 2 / gqa
    assert abs(ratio - float(cfg["about_two_percent"])) <= float(cfg["about_two_percent_abs_tolerance"])
    half = row / (512 * 2)
    assert abs(half - float(cfg["close_to_half"])) <= float(cfg["close_to_half_abs_tolerance"])
