"""The one-launch decode attention (few query rows) against the oracle and
against the long-row path (CSA_ATTN_DECODE=0), through the C ABI.

Decode rows split their keys over many CTAs that merge their partial
softmax states in-kernel; these cases cover one row spread over the most
splits, rows whose splits are partly empty, rows without keys, sparse and
dense key lists, and an invalid index.  Outputs must match the oracle within
max|err| <= 1e-2 max|ref| (bf16 outputs, fp32 accumulation).
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_common import dev, dev_bf16, max_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


def _caches(oracle_mod, rng, B, N, Ts):
    cache = np.stack([oracle_mod.pack_mixed(rng.standard_normal((N, 512)).astype(np.float32)) for _ in range(B)])
    swa = np.stack([oracle_mod.pack_mixed(rng.standard_normal((Ts, 512)).astype(np.float32)) for _ in range(B)])
    return cache, swa


@pytest.mark.parametrize("B,N,m,k,W", [
    (1, 8192, 128, 0, 128),      # one row over ~130 splits (dense HCA)
    (4, 8192, 128, 0, 128),      # the 1M HCA decode shape
    (32, 8192, 4, 1024, 128),    # the CSA decode shape: 32 rows, k = 1024
    (3, 4096, 4, 300, 37),       # ragged tiles, few splits each
    (7, 2048, 4, 64, 0),         # one tile per row: most splits empty
])
def test_decode_attention_matches_oracle_and_long_row_path(csa, oracle_mod, monkeypatch, B, N, m, k, W):
    rng = np.random.default_rng(1000 + B + k)
    T = N * m
    Ts = 256
    rope_np, rope_dev = oracle_mod.rope_table(T + 1, 64), csa.rope_table(T + 1, 64)
    cache, swa = _caches(oracle_mod, rng, B, N, Ts)
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, 1, 64, 512)).astype(np.float32))
    q_pos = (T - 1 - rng.integers(0, 64, size=(B, 1))).astype(np.int64)
    pos0 = (q_pos[:, 0] - Ts + 1 + rng.integers(0, 32, size=B)).astype(np.int64)   # windows inside the buffer
    idx = None
    if k:
        idx = np.full((B, 1, k), -1, np.int32)
        for b in range(B):
            nv = min(N, (q_pos[b, 0] + 1) // m)
            sel = rng.permutation(nv)[:k - 3]
            idx[b, 0, :len(sel)] = sel                     # a few -1 pads at the end
    scale = 1 / math.sqrt(512)
    args = (dev_bf16(q), dev(q_pos), dev(cache), m)
    rest = (dev(swa), dev(pos0), W, scale, rope_dev)

    def run():
        ws = csa.Workspace()
        if k:
            o, l = csa.sparse_mqa(*args, dev(idx), *rest, lse=True, ws=ws)
        else:
            o, l = csa.hca_dense_attn(*args, *rest, lse=True, ws=ws)
        torch.cuda.synchronize()
        assert ws.flags() == 0
        return o.float().cpu().numpy(), l.cpu().numpy()

    got, glse = run()
    again, _ = run()
    np.testing.assert_array_equal(got, again)            # deterministic
    monkeypatch.setenv("CSA_ATTN_DECODE", "0")
    alt, _ = run()
    monkeypatch.delenv("CSA_ATTN_DECODE")
    ref, rlse, bad = oracle_mod.attention(wl.bf16_bits_to_f32(q), q_pos, cache, N, m, idx, swa, pos0, W, scale,
                                          rope_np, 64)
    assert bad == 0
    assert max_rel_err(got, ref) <= 1e-2, max_rel_err(got, ref)
    assert max_rel_err(alt, ref) <= 1e-2
    np.testing.assert_allclose(glse, rlse, rtol=0, atol=2e-2)


def test_decode_rows_without_keys_and_invalid_positions(csa, oracle_mod):
    """A batch where one row has no keys (position 0, no window) and one row's
    position has no RoPE row: zeros and -inf for them, the device-check flag
    for the bad position, the other rows unaffected."""
    rng = np.random.default_rng(2000)
    B, N, m, W, Ts = 4, 1024, 4, 16, 64
    T = N * m
    rope_np, rope_dev = oracle_mod.rope_table(T + 1, 64), csa.rope_table(T + 1, 64)
    cache, swa = _caches(oracle_mod, rng, B, N, Ts)
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, 1, 64, 512)).astype(np.float32))
    q_pos = np.array([[T - 1], [2], [T + 50], [T - 7]], np.int64)   # row 2: no RoPE row for it
    pos0 = np.array([T - Ts, 0, T - Ts, T - Ts], np.int64)
    idx = np.full((B, 1, 40), -1, np.int32)
    for b in (0, 3):
        idx[b, 0] = rng.permutation(N - 2)[:40]          # entries visible at both positions
    ws = csa.Workspace()
    out, lse = csa.sparse_mqa(dev_bf16(q), dev(q_pos), dev(cache), m, dev(idx), dev(swa), dev(pos0), W,
                              1 / math.sqrt(512), rope_dev, lse=True, ws=ws)
    torch.cuda.synchronize()
    assert ws.flags() & csa.FLAG_DEVICE_CHECK
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))
    good = [0, 3]
    ref, _, _ = oracle_mod.attention(wl.bf16_bits_to_f32(q[good]), q_pos[good], cache[good], N, m, idx[good],
                                     swa[good], pos0[good], W, 1 / math.sqrt(512), rope_np, 64)
    assert max_rel_err(out[good], ref) <= 1e-2
    # row 1 (t = 2): entries need 4 tokens, so only the window (tokens 0..2)
    ref1, _, _ = oracle_mod.attention(wl.bf16_bits_to_f32(q[1:2]), q_pos[1:2], cache[1:2], N, m, idx[1:2],
                                      swa[1:2], pos0[1:2], W, 1 / math.sqrt(512), rope_np, 64)
    assert max_rel_err(out[1:2], ref1) <= 1e-2


def test_decode_in_item_rescale(csa, oracle_mod):
    """100 rows (one split each: every tile of a row in one item) whose later
    key tiles carry much larger logits, so the running maxima grow tile by
    tile and O is rescaled in TMEM inside the item."""
    rng = np.random.default_rng(3000)
    B, N, m, k, W = 100, 1024, 4, 640, 0
    T = N * m
    rope_np, rope_dev = oracle_mod.rope_table(T + 1, 64), csa.rope_table(T + 1, 64)
    q32 = rng.standard_normal((1, 1, 64, 512)).astype(np.float32)
    dirn = q32[0, 0].mean(0)
    grow = np.linspace(0, 6, N).astype(np.float32)[:, None]
    ent = rng.standard_normal((N, 512)).astype(np.float32) + grow * dirn[None, :] / np.linalg.norm(dirn) * 8
    cache = np.broadcast_to(oracle_mod.pack_mixed(ent.astype(np.float32)), (B, N, 592)).copy()
    swa = np.zeros((B, 8, 592), np.uint8)
    q = np.broadcast_to(wl.f32_to_bf16_bits(q32), (B, 1, 64, 512)).copy()
    q_pos = np.full((B, 1), T - 1, np.int64)
    idx = np.broadcast_to(np.arange(N - k, N, dtype=np.int32), (B, 1, k)).copy()   # increasing logits
    pos0 = np.full(B, T - 8, np.int64)
    scale = 1 / math.sqrt(512)
    got = csa.sparse_mqa(dev_bf16(q), dev(q_pos), dev(cache), m, dev(idx), dev(swa), dev(pos0), W, scale,
                         rope_dev).float().cpu().numpy()
    ref, _, bad = oracle_mod.attention(wl.bf16_bits_to_f32(q[:1]), q_pos[:1], cache[:1], N, m, idx[:1], swa[:1],
                                       pos0[:1], W, scale, rope_np, 64)
    assert bad == 0
    for b in (0, 57, 99):
        assert max_rel_err(got[b:b + 1], ref) <= 1e-2


@pytest.mark.parametrize("B,k", [
    (2, 300),     # a few tiles per item: the items expand the cache rows themselves (masked slots)
    (40, 2000),   # many tiles per item: rows gathered ahead (invalid entries compacted away)
])
def test_decode_invalid_indices_scattered(csa, oracle_mod, B, k):
    """Selected lists with invalid indices (-1, past the cache, not yet
    visible) scattered through them, not only at the end: the oracle skips
    them; the kernels mask or compact them and set the device-check flag."""
    rng = np.random.default_rng(5000 + B)
    N, m, W, Ts = 4096, 4, 64, 128
    T = N * m
    rope_np, rope_dev = oracle_mod.rope_table(T + 1, 64), csa.rope_table(T + 1, 64)
    cache, swa = _caches(oracle_mod, rng, B, N, Ts)
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, 1, 64, 512)).astype(np.float32))
    q_pos = np.full((B, 1), T - 1 - 4 * 100, np.int64)          # entries >= 3996 not yet visible
    pos0 = (q_pos[:, 0] - Ts + 1).astype(np.int64)
    idx = np.stack([rng.permutation(N)[:k].astype(np.int32) for _ in range(B)])[:, None, :]
    bad = rng.random(idx.shape) < 0.1
    kinds = rng.integers(0, 3, size=idx.shape)
    idx = np.where(bad & (kinds == 0), -1, idx)
    idx = np.where(bad & (kinds == 1), N + 7, idx)                # past the cache
    idx = np.where(bad & (kinds == 2), N - 1, idx)                # not visible at q_pos
    idx = idx.astype(np.int32)
    ws = csa.Workspace()
    out, lse = csa.sparse_mqa(dev_bf16(q), dev(q_pos), dev(cache), m, dev(idx), dev(swa), dev(pos0), W,
                              1 / math.sqrt(512), rope_dev, lse=True, ws=ws)
    torch.cuda.synchronize()
    assert ws.flags() & csa.FLAG_DEVICE_CHECK
    ref, rlse, nbad = oracle_mod.attention(wl.bf16_bits_to_f32(q), q_pos, cache, N, m, idx, swa, pos0, W,
                                           1 / math.sqrt(512), rope_np, 64)
    assert nbad > 0
    got = out.float().cpu().numpy()
    assert max_rel_err(got, ref) <= 1e-2, max_rel_err(got, ref)
    np.testing.assert_allclose(lse.cpu().numpy(), rlse, rtol=0, atol=2e-2)
