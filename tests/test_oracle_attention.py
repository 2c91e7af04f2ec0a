"""Pins of the oracle's sparse (CSA) and dense (HCA) attention with the window.

* brute force: a dense masked attention over all entries and tokens at once,
  in numpy fp64, compared with the oracle's per-query key lists;
* m = 1, k = all, W = 0, s = 1 reduces CSA to exact causal MQA, checked with
  torch's scaled_dot_product_attention (fp64, is_causal) on rotated keys;
* with W > 0 the same case equals causal MQA where the last W keys count
  twice (logit + ln 2), again through scaled_dot_product_attention;
* k >= |visible| makes CSA equal HCA (dense over all visible entries), and
  the order of the selected indices does not matter.
"""
import math

import numpy as np
import pytest
import torch


def _rot64(v, c, s, inverse=False):
    x0, x1 = v[..., 0::2].astype(np.float64), v[..., 1::2].astype(np.float64)
    c, s = c.astype(np.float64), s.astype(np.float64)
    if inverse:
        s = -s
    out = np.empty(v.shape, np.float64)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def _dense_masked(q, q_pos, keys_e, keys_s, sel_mask, swa_pos0, W, scale, rope, R):
    """One big masked softmax over [entries ++ window tokens] per query."""
    B, Tq, H, D = q.shape
    out = np.zeros((B, Tq, H, D))
    for b in range(B):
        K = np.concatenate([keys_e[b], keys_s[b]], 0)
        Ne, Ts = keys_e.shape[1], keys_s.shape[1]
        for i in range(Tq):
            t = q_pos[b, i]
            u = swa_pos0[b] + np.arange(Ts)
            mask = np.concatenate([sel_mask[b, i], (u > t - W) & (u <= t)])
            if not mask.any():
                continue
            qr = q[b, i].astype(np.float64).copy()
            qr[:, D - R:] = _rot64(q[b, i, :, D - R:], rope[0][t], rope[1][t])
            lg = scale * qr @ K.T
            lg[:, ~mask] = -np.inf
            p = np.exp(lg - lg.max(1, keepdims=True))
            p /= p.sum(1, keepdims=True)
            o = p @ K
            o[:, D - R:] = _rot64(o[:, D - R:], rope[0][t], rope[1][t], inverse=True)
            out[b, i] = o
    return out


@pytest.mark.parametrize("fmt", ["f32", "mixed592"])
def test_sparse_matches_dense_masked_bruteforce(oracle_mod, fmt):
    rng = np.random.default_rng(30)
    B, T, m, H, R, W, k = 2, 64, 4, 4, 64, 8, 6
    D = 128 if fmt == "f32" else 512
    N = T // m
    rope = oracle_mod.rope_table(T, R)
    ent = rng.standard_normal((B, N, D)).astype(np.float32)
    tok = rng.standard_normal((B, T, D)).astype(np.float32)
    if fmt == "f32":
        cache, swa, f = ent, tok, oracle_mod.FMT_F32
        ke, ks = ent.astype(np.float64), tok.astype(np.float64)
    else:
        cache, swa, f = oracle_mod.pack_mixed(ent), oracle_mod.pack_mixed(tok), oracle_mod.FMT_MIXED592
        ke, ks = oracle_mod.unpack_mixed(cache), oracle_mod.unpack_mixed(swa)
    q = rng.standard_normal((B, T, H, D)).astype(np.float32)
    q_pos = np.tile(np.arange(T, dtype=np.int64), (B, 1))
    idx = np.full((B, T, k), -1, np.int32)
    sel = np.zeros((B, T, N), bool)
    for b in range(B):
        for t in range(T):
            nv = min(N, (t + 1) // m)
            pick = rng.permutation(nv)[:k]
            idx[b, t, :len(pick)] = pick
            sel[b, t, pick] = True
    scale = 1 / math.sqrt(D)
    swa_pos0 = np.zeros(B, np.int64)
    got, lse, bad = oracle_mod.attention(q, q_pos, cache, N, m, idx, swa, swa_pos0, W, scale, rope, R, f)
    ref = _dense_masked(q, q_pos, ke, ks, sel, swa_pos0, W, scale, rope, R)
    assert bad == 0
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def _rot_keys_f32(x, rope, R):
    """RoPE of each token at its own position, fp32 ops (what m = 1 compression stores)."""
    D = x.shape[-1]
    out = x.copy()
    c, s = rope[0][: x.shape[1]], rope[1][: x.shape[1]]
    x0, x1 = x[..., D - R::2], x[..., D - R + 1::2]
    out[..., D - R::2] = (x0 * c) - (x1 * s)
    out[..., D - R + 1::2] = (x0 * s) + (x1 * c)
    return out


@pytest.mark.parametrize("W", [0, 5])
def test_m1_all_keys_is_causal_mqa(oracle_mod, W):
    rng = np.random.default_rng(31)
    B, T, H, D, R = 1, 40, 3, 128, 64
    rope = oracle_mod.rope_table(T, R)
    x = rng.standard_normal((B, T, D)).astype(np.float32)
    z = rng.standard_normal((B, T)).astype(np.float32)
    ent = oracle_mod.compress(x, z, None, 1, R, rope=rope)           # m = 1, s = 1
    q = rng.standard_normal((B, T, H, D)).astype(np.float32)
    q_pos = np.arange(T, dtype=np.int64)[None]
    kI = rng.standard_normal((B, T, 32)).astype(np.float32)
    qI = rng.standard_normal((B, T, 2, 32)).astype(np.float32)
    w = rng.uniform(0, 1, (B, T, 2)).astype(np.float32)
    idx, _ = oracle_mod.indexer_topk(qI, w, kI, q_pos, T, 1, T)     # k = all
    scale = 1 / math.sqrt(D)
    got, _, bad = oracle_mod.attention(q, q_pos, ent, T, 1, idx, ent, np.zeros(1, np.int64), W,
                                       scale, rope, R, oracle_mod.FMT_F32)
    assert bad == 0
    # independent reference: rotate, then causal attention from torch
    kr = _rot_keys_f32(x, rope, R).astype(np.float64)
    qr = q.astype(np.float64).copy()
    qr[..., D - R:] = _rot64(q[..., D - R:], rope[0][:T][None, :, None], rope[1][:T][None, :, None])
    Q = torch.from_numpy(qr).permute(0, 2, 1, 3)
    K = torch.from_numpy(kr)[:, None].expand(B, H, T, D)
    if W == 0:
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, K, is_causal=True, scale=scale)
    else:
        tt = torch.arange(T)
        causal = tt[None, :] <= tt[:, None]
        win = causal & (tt[None, :] > tt[:, None] - W)
        zero = torch.zeros((), dtype=torch.float64)
        bias = (torch.where(causal, zero, torch.tensor(-math.inf, dtype=torch.float64))
                + torch.where(win, torch.tensor(math.log(2.0), dtype=torch.float64), zero))
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, K, attn_mask=bias, scale=scale)
    ref = o.permute(0, 2, 1, 3).numpy().copy()
    ref[..., D - R:] = _rot64(ref[..., D - R:], rope[0][:T][None, :, None], rope[1][:T][None, :, None],
                              inverse=True)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)


def test_full_selection_equals_dense_hca(oracle_mod):
    rng = np.random.default_rng(32)
    B, T, m, H, D, R, W = 2, 256, 8, 2, 512, 64, 16
    N = T // m
    rope = oracle_mod.rope_table(T, R)
    cache = oracle_mod.pack_mixed(rng.standard_normal((B, N, D)).astype(np.float32))
    swa = oracle_mod.pack_mixed(rng.standard_normal((B, T, D)).astype(np.float32))
    q = rng.standard_normal((B, T, H, D)).astype(np.float32)
    q_pos = np.tile(np.arange(T, dtype=np.int64), (B, 1))
    idx = np.full((B, T, N + 4), -1, np.int32)
    for t in range(T):
        nv = min(N, (t + 1) // m)
        idx[:, t, :nv] = rng.permutation(nv)
    args = (swa, np.zeros(B, np.int64), W, 1 / math.sqrt(D), rope, R, oracle_mod.FMT_MIXED592)
    sparse, l1, _ = oracle_mod.attention(q, q_pos, cache, N, m, idx, *args)
    dense, l2, _ = oracle_mod.attention(q, q_pos, cache, N, m, None, *args)
    np.testing.assert_allclose(sparse, dense, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_invalid_indices_skipped_and_counted(oracle_mod):
    rng = np.random.default_rng(33)
    B, T, m, H, D, R = 1, 32, 4, 2, 128, 64
    N = T // m
    rope = oracle_mod.rope_table(T, R)
    ent = rng.standard_normal((B, N, D)).astype(np.float32)
    q = rng.standard_normal((B, 1, H, D)).astype(np.float32)
    q_pos = np.array([[11]], np.int64)                 # entries 0..2 visible
    good = np.array([[[0, 2, -1, -1]]], np.int32)
    bad = np.array([[[0, 2, 3, 99]]], np.int32)        # 3 not yet visible, 99 >= N
    a = oracle_mod.attention(q, q_pos, ent, N, m, good, ent, np.zeros(1, np.int64), 0, 0.1, rope, R,
                             oracle_mod.FMT_F32)
    b = oracle_mod.attention(q, q_pos, ent, N, m, bad, ent, np.zeros(1, np.int64), 0, 0.1, rope, R,
                             oracle_mod.FMT_F32)
    np.testing.assert_array_equal(a[0], b[0])
    assert a[2] == 0 and b[2] == 2
    # no keys at all: zero output, lse = -inf
    none = np.full((1, 1, 4), -1, np.int32)
    o, l, _ = oracle_mod.attention(q, q_pos, ent, N, m, none, ent, np.zeros(1, np.int64), 0, 0.1,
                                   rope, R, oracle_mod.FMT_F32)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_single_key_returns_inverse_rotated_key(oracle_mod):
    """With one key the softmax weight is 1: o = RoPE^-1_t(kappa)."""
    rng = np.random.default_rng(34)
    D, R, m, t = 128, 64, 4, 13
    rope = oracle_mod.rope_table(32, R)
    ent = rng.standard_normal((1, 4, D)).astype(np.float32)
    q = rng.standard_normal((1, 1, 2, D)).astype(np.float32)
    o, _, _ = oracle_mod.attention(q, np.array([[t]], np.int64), ent, 4, m, np.array([[[1]]], np.int32),
                                   ent, np.zeros(1, np.int64), 0, 0.3, rope, R, oracle_mod.FMT_F32)
    exp = ent[0, 1].astype(np.float64).copy()
    exp[D - R:] = _rot64(ent[0, 1, D - R:], rope[0][t], rope[1][t], inverse=True)
    np.testing.assert_allclose(o[0, 0, 0], exp, atol=1e-12)
    np.testing.assert_allclose(o[0, 0, 1], exp, atol=1e-12)
