"""GPU parity of every call against the CPU oracle, through the C ABI.

Bar: bit-exact compressed cache bytes, FP4 key bytes, top-k indices and
scores; attention outputs within max|err| <= 1e-2 max|ref| (bf16 out, fp32
accumulation) or 1e-5 (fp32 configuration).  Full-size runs use the launch
configuration of the benchmark and compare sampled query rows, which the
oracle computes one by one from its own cache and its own top-k.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_common import act_dev, dev, dev_bf16, max_rel_err, softmax_scale, tol, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


_ROPE = {}


def ropes(csa, oracle_mod, P):
    if P not in _ROPE:
        _ROPE.clear()
        _ROPE[P] = (oracle_mod.rope_table(P, 64), csa.rope_table(P, 64))
    return _ROPE[P]


# --------------------------------------------------------------------------
# compression and packing: bit-exact bytes
# --------------------------------------------------------------------------
COMPRESS_CASES = [
    # (config, sequence, tokens, m, pos0, part)
    ("c2_csa_prefill_8k", 0, 8192, 4, 0, "kv"),          # CSA cache, full size
    ("c2_csa_prefill_8k", 0, 8192 - 3, 4, 4096, "kv"),   # ragged tail, shifted positions
    ("c2_csa_prefill_8k", 0, 8192, 1, 0, "kv"),          # window (state) cache
    ("c2_csa_prefill_8k", 0, 8192, 4, 0, "kI"),          # FP4 indexer keys
    ("c4_hca_prefill_64k", 0, 65536, 128, 0, "kv"),      # HCA cache, full size
    ("c3_csa_decode_128k", 7, 131072, 4, 0, "kv"),       # one sequence of the 128K decode cache
    ("c5_hybrid_csa_decode_1m", 1, 1 << 20, 4, 0, "kI"),  # 1M-token FP4 keys
    ("c1_tiny_csa_prefill", 0, 512, 4, 0, "kv"),         # fp32 format
    ("c1_tiny_csa_prefill", 0, 512, 4, 0, "kI"),
    ("c1_tiny_csa_prefill", 0, 510, 1, 0, "kv"),
]


@pytest.mark.parametrize("name,b,T,m,pos0,part", COMPRESS_CASES)
def test_compress_bitexact(csa, oracle_mod, name, b, T, m, pos0, part):
    cfg = wl.CONFIGS[name]
    toks = wl.gen_tokens(cfg, b, 0, T, parts=(part, "z" if part == "kv" else "zI"))
    sc = wl.gen_channel_scales(cfg)
    x = toks[part]
    z = toks["z" if part == "kv" else "zI"]
    s = None if m == 1 else (sc["s"] if part == "kv" else sc["sI"])
    R = cfg.R if part == "kv" else 0
    if cfg.fp32:
        fmt, ofmt = csa.FMT_F32, "f32"
    elif part == "kv":
        fmt, ofmt = csa.FMT_MIXED592, "mixed592"
    else:
        fmt, ofmt = csa.FMT_MXFP4, "mxfp4"
    P = pos0 + T + 1
    rope_np, rope_dev = ropes(csa, oracle_mod, P)
    out = csa.compress_kv(act_dev(x, cfg)[None], dev(z)[None], None if s is None else dev(s), m, fmt,
                          R, rope_dev if R else None, pos0)
    ref = oracle_mod.compress_kv(widen(x, cfg)[None], z[None], s, m, ofmt, R, pos0, rope_np)
    if ofmt == "mxfp4":
        np.testing.assert_array_equal(out[0].cpu().numpy(), ref[0])
        np.testing.assert_array_equal(out[1].cpu().numpy(), ref[1])
    elif ofmt == "f32":
        np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    else:
        np.testing.assert_array_equal(out.cpu().numpy(), ref)


def test_pack_fp8_bf16_bitexact(csa, oracle_mod):
    rng = np.random.default_rng(40)
    v = (rng.standard_normal((5000, 512)) * np.exp(rng.uniform(-20, 12, (5000, 1)))).astype(np.float32)
    v[3, :128] = 0.0
    v[4, 5] = -0.0
    v[9, 100] = 1e30
    out = csa.kvcache_pack_fp8_bf16(dev(v))
    np.testing.assert_array_equal(out.cpu().numpy(), oracle_mod.pack_mixed(v))


# --------------------------------------------------------------------------
# indexer + top-k: bit-exact indices and scores
# --------------------------------------------------------------------------
def _keys(csa, oracle_mod, cfg, b, T):
    toks = wl.gen_tokens(cfg, b, 0, T, parts=("kI", "zI"))
    sI = wl.gen_channel_scales(cfg)["sI"]
    if cfg.fp32:
        kd = csa.compress_kv(dev(toks["kI"])[None], dev(toks["zI"])[None], dev(sI), cfg.m, csa.FMT_F32, 0)
        kn = oracle_mod.compress_kv(toks["kI"][None], toks["zI"][None], sI, cfg.m, "f32", 0)
        return (kd, None), kn
    kd = csa.compress_kv(act_dev(toks["kI"], cfg)[None], dev(toks["zI"])[None], dev(sI), cfg.m,
                         csa.FMT_MXFP4, 0)
    kn = oracle_mod.compress_kv(widen(toks["kI"], cfg)[None], toks["zI"][None], sI, cfg.m, "mxfp4", 0)
    return kd, kn


@pytest.mark.parametrize("name,rows", [("c1_tiny_csa_prefill", None), ("c2_csa_prefill_8k", 384)])
def test_indexer_topk_prefill(csa, oracle_mod, name, rows):
    cfg = wl.CONFIGS[name]
    (kd, ksd), kn = _keys(csa, oracle_mod, cfg, 0, cfg.T)
    qry = wl.gen_queries(cfg, 0)
    q_pos = np.arange(cfg.Tq, dtype=np.int64)[None]
    idx, sc = csa.indexer_topk(act_dev(qry["qI"], cfg)[None], dev(qry["w"])[None], kd, ksd, dev(q_pos),
                               cfg.N, cfg.m, cfg.k)
    idx, sc = idx.cpu().numpy(), sc.cpu().numpy()
    sel = np.arange(cfg.Tq) if rows is None else np.unique(np.concatenate([
        np.arange(0, 12), np.arange(cfg.k * cfg.m - 8, cfg.k * cfg.m + 8), [cfg.Tq - 1],
        np.random.default_rng(41).choice(cfg.Tq, rows, replace=False)]))
    oidx, osc = oracle_mod.indexer_topk(widen(qry["qI"], cfg)[sel][None], qry["w"][sel][None], kn,
                                        q_pos[:, sel], cfg.N, cfg.m, cfg.k)
    np.testing.assert_array_equal(idx[:, sel], oidx)
    np.testing.assert_array_equal(sc[:, sel], osc)


@pytest.mark.parametrize("name", ["c3_csa_decode_128k", "c5_hybrid_csa_decode_1m"])
def test_indexer_topk_decode_full(csa, oracle_mod, name):
    cfg = wl.CONFIGS[name]
    B = cfg.B
    keys_d = [_keys(csa, oracle_mod, cfg, b, cfg.T) for b in range(B)]
    kd = torch.cat([k[0][0] for k in keys_d])
    ksd = torch.cat([k[0][1] for k in keys_d])
    kn = (np.concatenate([k[1][0] for k in keys_d]), np.concatenate([k[1][1] for k in keys_d]))
    qry = [wl.gen_queries(cfg, b) for b in range(B)]
    qI = np.stack([q["qI"] for q in qry])
    w = np.stack([q["w"] for q in qry])
    q_pos = np.full((B, 1), cfg.T - 1, np.int64)
    idx, sc = csa.indexer_topk(act_dev(qI, cfg), dev(w), kd, ksd, dev(q_pos), cfg.N, cfg.m, cfg.k)
    oidx, osc = oracle_mod.indexer_topk(widen(qI, cfg), w, kn, q_pos, cfg.N, cfg.m, cfg.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    np.testing.assert_array_equal(sc.cpu().numpy(), osc)


# --------------------------------------------------------------------------
# whole CSA prefill pipeline: compress -> indexer/top-k -> sparse MQA
# --------------------------------------------------------------------------
def _prefill_pipeline(csa, oracle_mod, cfg, sample_rows):
    T = cfg.T
    toks = wl.gen_tokens(cfg, 0)
    sc = wl.gen_channel_scales(cfg)
    qry = wl.gen_queries(cfg, 0)
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    fmt = csa.FMT_F32 if cfg.fp32 else csa.FMT_MIXED592
    ofmt = "f32" if cfg.fp32 else "mixed592"
    kv_d, z_d = act_dev(toks["kv"], cfg)[None], dev(toks["z"])[None]
    cache = csa.compress_kv(kv_d, z_d, dev(sc["s"]), cfg.m, fmt, cfg.R, rope_dev)
    swa = csa.compress_kv(kv_d, z_d, None, 1, fmt, cfg.R, rope_dev)
    (kd, ksd), kn = _keys(csa, oracle_mod, cfg, 0, T)
    q_pos = np.arange(T, dtype=np.int64)[None]
    qpos_d = dev(q_pos)
    idx = csa.indexer_topk(act_dev(qry["qI"], cfg)[None], dev(qry["w"])[None], kd, ksd, qpos_d, cfg.N,
                           cfg.m, cfg.k, scores=False)
    out, lse = csa.sparse_mqa(act_dev(qry["q"], cfg)[None], qpos_d, cache, cfg.m, idx, swa,
                              dev(np.zeros(1, np.int64)), cfg.W, softmax_scale(cfg), rope_dev, cfg.R,
                              lse=True)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    # oracle from its own cache and its own top-k, on the sampled rows
    xw = widen(toks["kv"], cfg)[None]
    ocache = oracle_mod.compress_kv(xw, toks["z"][None], sc["s"], cfg.m, ofmt, cfg.R, 0, rope_np)
    oswa = oracle_mod.compress_kv(xw, toks["z"][None], None, 1, ofmt, cfg.R, 0, rope_np)
    rows = np.arange(T) if sample_rows is None else sample_rows
    oidx, _ = oracle_mod.indexer_topk(widen(qry["qI"], cfg)[rows][None], qry["w"][rows][None], kn,
                                      q_pos[:, rows], cfg.N, cfg.m, cfg.k)
    oout, olse, bad = oracle_mod.attention(widen(qry["q"], cfg)[rows][None], q_pos[:, rows], ocache,
                                           cfg.N, cfg.m, oidx, oswa, np.zeros(1, np.int64), cfg.W,
                                           softmax_scale(cfg), rope_np, cfg.R,
                                           oracle_mod.FMT_F32 if cfg.fp32 else oracle_mod.FMT_MIXED592)
    assert bad == 0
    return out[0, rows], lse[0, rows], oout[0], olse[0]


def test_csa_prefill_tiny_fp32_full(csa, oracle_mod):
    cfg = wl.CONFIGS["c1_tiny_csa_prefill"]
    got, glse, ref, rlse = _prefill_pipeline(csa, oracle_mod, cfg, None)
    assert max_rel_err(got, ref) <= tol(cfg)
    np.testing.assert_allclose(glse, rlse, rtol=0, atol=1e-4)


def test_csa_prefill_8k_sampled(csa, oracle_mod):
    cfg = wl.CONFIGS["c2_csa_prefill_8k"]
    rows = np.unique(np.concatenate([np.arange(0, 6), [127, 128, 129, 2046, 2047, 2048, 2051],
                                     np.random.default_rng(42).choice(cfg.T, 40, replace=False),
                                     [cfg.T - 1]]))
    got, glse, ref, rlse = _prefill_pipeline(csa, oracle_mod, cfg, rows)
    err = max_rel_err(got, ref)
    assert err <= tol(cfg), err
    np.testing.assert_allclose(glse, rlse, rtol=0, atol=2e-2)


# --------------------------------------------------------------------------
# decode: caches built from 128K / 1M tokens, sampled sequences checked
# --------------------------------------------------------------------------
def _decode_caches(csa, oracle_mod, cfg, oracle_seqs):
    """GPU caches for all B sequences; oracle caches for oracle_seqs."""
    T, W = cfg.T, cfg.W
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    sc = wl.gen_channel_scales(cfg)
    s_d = dev(sc["s"])
    cache = torch.empty((cfg.B, cfg.N, 592), dtype=torch.uint8, device="cuda")
    swa = torch.empty((cfg.B, W, 592), dtype=torch.uint8, device="cuda")
    ocache, oswa = {}, {}
    for b in range(cfg.B):
        toks = wl.gen_tokens(cfg, b, parts=("kv", "z"))
        kv_d, z_d = act_dev(toks["kv"], cfg)[None], dev(toks["z"])[None]
        csa.compress_kv(kv_d, z_d, s_d, cfg.m, csa.FMT_MIXED592, cfg.R, rope_dev, out=cache[b:b + 1])
        csa.compress_kv(kv_d[:, T - W:], z_d[:, T - W:], None, 1, csa.FMT_MIXED592, cfg.R, rope_dev,
                        pos0=T - W, out=swa[b:b + 1])
        if b in oracle_seqs:
            xw = widen(toks["kv"], cfg)[None]
            ocache[b] = oracle_mod.compress_kv(xw, toks["z"][None], sc["s"], cfg.m, "mixed592", cfg.R, 0,
                                               rope_np)
            oswa[b] = oracle_mod.compress_kv(xw[:, T - W:], toks["z"][None, T - W:], None, 1, "mixed592",
                                             cfg.R, T - W, rope_np)
        del kv_d, z_d
    return cache, swa, ocache, oswa, rope_np, rope_dev


@pytest.mark.parametrize("name", ["c3_csa_decode_128k", "c5_hybrid_csa_decode_1m",
                                  "c4_hca_decode_1m", "c5_hybrid_hca_decode_1m"])
def test_decode_sampled(csa, oracle_mod, name):
    cfg = wl.CONFIGS[name]
    B, T, W = cfg.B, cfg.T, cfg.W
    check = sorted({0, B // 3, (2 * B) // 3, B - 1})   # first, two middle and last sequences
    cache, swa, ocache, oswa, rope_np, rope_dev = _decode_caches(csa, oracle_mod, cfg, check)
    qry = [wl.gen_queries(cfg, b) for b in range(B)]
    q = np.stack([x["q"] for x in qry])
    q_pos = np.full((B, 1), T - 1, np.int64)
    pos0 = np.full(B, T - W, np.int64)
    if cfg.k:
        keys = [_keys(csa, oracle_mod, cfg, b, T) for b in range(B)]
        kd = torch.cat([k[0][0] for k in keys])
        ksd = torch.cat([k[0][1] for k in keys])
        qI = np.stack([x["qI"] for x in qry])
        w = np.stack([x["w"] for x in qry])
        idx = csa.indexer_topk(act_dev(qI, cfg), dev(w), kd, ksd, dev(q_pos), cfg.N, cfg.m, cfg.k,
                               scores=False)
        out = csa.sparse_mqa(act_dev(q, cfg), dev(q_pos), cache, cfg.m, idx, swa, dev(pos0), W,
                             softmax_scale(cfg), rope_dev, cfg.R)
    else:
        out = csa.hca_dense_attn(act_dev(q, cfg), dev(q_pos), cache, cfg.m, swa, dev(pos0), W,
                                 softmax_scale(cfg), rope_dev, cfg.R)
    out = out.float().cpu().numpy()
    for b in check:
        oidx = None
        if cfg.k:
            oidx, _ = oracle_mod.indexer_topk(widen(qI, cfg)[b:b + 1], w[b:b + 1], keys[b][1], q_pos[b:b + 1],
                                              cfg.N, cfg.m, cfg.k)
        ref, _, bad = oracle_mod.attention(widen(q, cfg)[b:b + 1], q_pos[b:b + 1], ocache[b], cfg.N, cfg.m,
                                           oidx, oswa[b], pos0[b:b + 1], W, softmax_scale(cfg), rope_np,
                                           cfg.R)
        assert bad == 0
        err = max_rel_err(out[b:b + 1], ref)
        assert err <= tol(cfg), (b, err)


# --------------------------------------------------------------------------
# properties: determinism, device checks, edge cases
# --------------------------------------------------------------------------
def _small_mixed(csa, oracle_mod, T=512, m=4, H=64, seed=50):
    rng = np.random.default_rng(seed)
    N = T // m
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    ent = rng.standard_normal((1, N, 512)).astype(np.float32)
    tok = rng.standard_normal((1, T, 512)).astype(np.float32)
    cache = oracle_mod.pack_mixed(ent)
    swa = oracle_mod.pack_mixed(tok)
    q = wl.f32_to_bf16_bits(rng.standard_normal((1, T, H, 512)).astype(np.float32))
    return rope_np, rope_dev, cache, swa, q, N


def test_attention_is_deterministic(csa, oracle_mod):
    rope_np, rope_dev, cache, swa, q, N = _small_mixed(csa, oracle_mod)
    T, m, k = 512, 4, 64
    rng = np.random.default_rng(51)
    idx = np.full((1, T, k), -1, np.int32)
    for t in range(T):
        nv = min(N, (t + 1) // m)
        p = rng.permutation(nv)[:k]
        idx[0, t, :len(p)] = p
    args = (dev(np.arange(T, dtype=np.int64)[None]), dev(cache), m, dev(idx), dev(swa),
            dev(np.zeros(1, np.int64)), 128, 1 / math.sqrt(512), rope_dev)
    from gpu_common import dev_bf16
    a = csa.sparse_mqa(dev_bf16(q), *args)
    b = csa.sparse_mqa(dev_bf16(q), *args)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_invalid_index_sets_device_check(csa, oracle_mod):
    rope_np, rope_dev, cache, swa, q, N = _small_mixed(csa, oracle_mod, T=64, H=64)
    from gpu_common import dev_bf16
    ws = csa.Workspace()
    q_pos = np.array([[40]], np.int64)
    good = np.array([[[0, 5, 9, -1]]], np.int32)
    bad = np.array([[[0, 5, 9, 10]]], np.int32)       # entry 10 covers tokens 40..43: not visible at 40
    qd = dev_bf16(q[:, 40:41])
    args = (dev(cache), 4)
    rest = (dev(swa), dev(np.zeros(1, np.int64)), 16, 0.05, rope_dev)
    o_good = csa.sparse_mqa(qd, dev(q_pos), *args, dev(good), *rest, ws=ws)
    assert ws.flags() == 0
    o_bad = csa.sparse_mqa(qd, dev(q_pos), *args, dev(bad), *rest, ws=ws)
    assert ws.flags() & csa.FLAG_DEVICE_CHECK
    assert torch.equal(o_good.view(torch.int16), o_bad.view(torch.int16))
    ws.reset()
    assert ws.flags() == 0


def test_no_keys_gives_zero(csa, oracle_mod):
    rope_np, rope_dev, cache, swa, q, N = _small_mixed(csa, oracle_mod, T=64, H=64)
    from gpu_common import dev_bf16
    none = np.full((1, 1, 8), -1, np.int32)
    out, lse = csa.sparse_mqa(dev_bf16(q[:, :1]), dev(np.array([[0]], np.int64)), dev(cache), 4, dev(none),
                              dev(swa), dev(np.zeros(1, np.int64)), 0, 0.05, rope_dev, lse=True)
    assert torch.all(out.float() == 0) and torch.all(torch.isinf(lse))


def test_hca_equals_sparse_with_all_entries(csa, oracle_mod):
    """k >= visible entries: the sparse call over all visible entries equals the dense call."""
    rope_np, rope_dev, cache, swa, q, N = _small_mixed(csa, oracle_mod, T=512, m=8, H=64)
    T, m = 512, 8
    idx = np.full((1, T, N), -1, np.int32)
    for t in range(T):
        nv = min(N, (t + 1) // m)
        idx[0, t, :nv] = np.arange(nv)
    from gpu_common import dev_bf16
    qp = dev(np.arange(T, dtype=np.int64)[None])
    rest = (dev(swa), dev(np.zeros(1, np.int64)), 32, 1 / math.sqrt(512), rope_dev)
    a = csa.sparse_mqa(dev_bf16(q), qp, dev(cache), m, dev(idx), *rest).float()
    b = csa.hca_dense_attn(dev_bf16(q), qp, dev(cache), m, *rest).float()
    assert float((a - b).abs().max()) <= 1e-2 * float(b.abs().max())


# --------------------------------------------------------------------------
# tensor-core attention: tile edges, rescale path, agreement with the CUDA-core kernel
# --------------------------------------------------------------------------
def _oracle_attn(oracle_mod, q, q_pos, cache, N, m, idx, swa, pos0, W, scale, rope_np):
    out, lse, bad = oracle_mod.attention(wl.bf16_bits_to_f32(q), q_pos, cache, N, m, idx, swa, pos0, W,
                                         scale, rope_np, 64)
    assert bad == 0
    return out, lse


@pytest.mark.parametrize("k,W", [(1, 0), (127, 1), (128, 0), (300, 37), (1024, 128), (4000, 128)])
def test_tc_tile_edges(csa, oracle_mod, k, W):
    """Key counts around the 128-key tile: empty tail, exact multiples, ragged."""
    from gpu_common import dev_bf16
    rng = np.random.default_rng(60 + k)
    T, m = 4 * 4096, 4
    N = T // m
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    cache = oracle_mod.pack_mixed(rng.standard_normal((1, N, 512)).astype(np.float32))
    swa = oracle_mod.pack_mixed(rng.standard_normal((1, 256, 512)).astype(np.float32))
    Tq = 6
    q = wl.f32_to_bf16_bits(rng.standard_normal((1, Tq, 64, 512)).astype(np.float32))
    q_pos = np.array([[T - 1, T - 2, 4 * k + 3, 200, 3, T - 100]], np.int64)
    pos0 = np.array([T - 256], np.int64)
    idx = np.full((1, Tq, k), -1, np.int32)
    for i, t in enumerate(q_pos[0]):
        nv = min(N, (t + 1) // m)
        p = rng.permutation(nv)[:k]
        idx[0, i, :len(p)] = p
    # window rows exist only for the last 256 positions: keep W-windows inside them
    q_pos_w = q_pos.copy()
    if W:
        q_pos_w[0] = np.maximum(q_pos[0], T - 256 + W)
        q_pos_w[0] = np.minimum(q_pos_w[0], T - 1)
    scale = 1 / math.sqrt(512)
    got = csa.sparse_mqa(dev_bf16(q), dev(q_pos_w), dev(cache), m, dev(idx), dev(swa), dev(pos0), W, scale,
                         rope_dev).float().cpu().numpy()
    ref, _ = _oracle_attn(oracle_mod, q, q_pos_w, cache, N, m, idx, swa, pos0, W, scale, rope_np)
    assert max_rel_err(got, ref) <= 1e-2


def test_tc_rescale_path(csa, oracle_mod):
    """Later key tiles with much larger logits force the lazy rescale of O."""
    from gpu_common import dev_bf16
    rng = np.random.default_rng(70)
    T, m, k = 4096, 4, 640
    N = T // m
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    q32 = rng.standard_normal((1, 1, 64, 512)).astype(np.float32)
    base = rng.standard_normal((1, N, 512)).astype(np.float32)
    # entries aligned with q (head-averaged) get growing weight: logits rise tile by tile
    dirn = q32[0, 0].mean(0)
    grow = np.linspace(0, 6, N).astype(np.float32)[None, :, None]
    ent = base + grow * dirn[None, None, :] / np.linalg.norm(dirn) * 8
    cache = oracle_mod.pack_mixed(ent.astype(np.float32))
    swa = oracle_mod.pack_mixed(rng.standard_normal((1, 128, 512)).astype(np.float32))
    q = wl.f32_to_bf16_bits(q32)
    q_pos = np.array([[T - 1]], np.int64)
    idx = np.arange(N - k, N, dtype=np.int32)[None, None, :]         # increasing logits
    pos0 = np.array([T - 128], np.int64)
    scale = 1 / math.sqrt(512)
    got, glse = csa.sparse_mqa(dev_bf16(q), dev(q_pos), dev(cache), m, dev(idx), dev(swa), dev(pos0), 128,
                               scale, rope_dev, lse=True)
    ref, rlse = _oracle_attn(oracle_mod, q, q_pos, cache, N, m, idx, swa, pos0, 128, scale, rope_np)
    assert max_rel_err(got.float().cpu().numpy(), ref) <= 1e-2
    np.testing.assert_allclose(glse.cpu().numpy(), rlse, rtol=0, atol=2e-2)


def test_simt_and_tc_kernels_agree(csa, oracle_mod, monkeypatch):
    from gpu_common import dev_bf16
    rope_np, rope_dev, cache, swa, q, N = _small_mixed(csa, oracle_mod, T=1024, m=4, H=64, seed=80)
    T, m, k = 1024, 4, 96
    rng = np.random.default_rng(81)
    idx = np.full((1, T, k), -1, np.int32)
    for t in range(T):
        nv = min(N, (t + 1) // m)
        p = rng.permutation(nv)[:k]
        idx[0, t, :len(p)] = p
    args = (dev(np.arange(T, dtype=np.int64)[None]), dev(cache), m, dev(idx), dev(swa),
            dev(np.zeros(1, np.int64)), 64, 1 / math.sqrt(512), rope_dev)
    tc = csa.sparse_mqa(dev_bf16(q), *args).float()
    monkeypatch.setenv("CSA_ATTN_IMPL", "simt")
    simt = csa.sparse_mqa(dev_bf16(q), *args).float()
    monkeypatch.delenv("CSA_ATTN_IMPL")
    rows = np.array([0, 1, 100, 511, 1023])
    ref, _ = _oracle_attn(oracle_mod, q[:, rows], np.arange(T, dtype=np.int64)[None][:, rows], cache, N, m,
                          idx[:, rows], swa, np.zeros(1, np.int64), 64, 1 / math.sqrt(512), rope_np)
    assert max_rel_err(tc.cpu().numpy()[:, rows], ref) <= 1e-2
    assert max_rel_err(simt.cpu().numpy()[:, rows], ref) <= 1e-2
    assert float((tc - simt).abs().max()) <= 1e-2 * float(simt.abs().max())


def test_tc_dequant_is_exact(csa, oracle_mod):
    """One selected key and no window: softmax weight 1, so the FP8 columns of
    the output are the dequantised key itself (bf16 of code x 2^e, exact)."""
    from gpu_common import dev_bf16
    rng = np.random.default_rng(90)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    exps = [-117, -60, -20, -9, -7, -1, 0, 3, 7, 8, 10]
    n = len(exps) * 2
    rows = np.zeros((1, n, 592), np.uint8)
    for r in range(n):
        rows[0, r, :448] = np.roll(np.resize(codes, 448), 37 * r)
        e = exps[r % len(exps)]
        sc = np.array([2.0 ** e, 2.0 ** (e - (r & 1)), 2.0 ** min(e + 1, 10), 2.0 ** e], np.float32)
        rows[0, r, 576:592] = sc.view(np.uint8)
        rows[0, r, 448:576] = wl.f32_to_bf16_bits(rng.standard_normal(64).astype(np.float32)).view(np.uint8)
    m, T = 1, n
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    q = wl.f32_to_bf16_bits(rng.standard_normal((1, n, 64, 512)).astype(np.float32))
    q_pos = np.arange(n, dtype=np.int64)[None]
    idx = np.arange(n, dtype=np.int32)[None, :, None]               # query r selects entry r only
    out = csa.sparse_mqa(dev_bf16(q), dev(q_pos), dev(rows), m, dev(idx), dev(rows), dev(np.zeros(1, np.int64)),
                         0, 0.05, rope_dev).float().cpu().numpy()
    want = oracle_mod.unpack_mixed(rows)[0, :, :448]
    for r in range(n):
        np.testing.assert_array_equal(out[0, r, :, :448], np.broadcast_to(want[r], (64, 448)))


# --------------------------------------------------------------------------
# indexer: FP8 tensor-core scoring against the exact integer (dp4a) kernel
# --------------------------------------------------------------------------
def _mxfp4_keys_random(rng, n, exps):
    """Random E2M1 codes (all 16) and E8M0 scale bytes drawn from `exps`."""
    codes = rng.integers(0, 256, size=(n, 32), dtype=np.uint8)
    scales = rng.choice(np.asarray(exps, np.uint8), size=(n, 2)).astype(np.uint8)
    return codes, scales


@pytest.mark.parametrize("B,Tq,N,m,key_exps,q_scale", [
    (2, 300, 700, 1, list(range(120, 135)), 1.0),      # ragged rows and entries, two sequences
    (1, 256, 256, 1, [0, 1, 2, 250, 254], 1e-30),      # block powers far outside [2^-100, 2^100]
    (1, 129, 64, 2, list(range(100, 160)), 3e4),       # one row past a 128-row tile; m = 2
])
def test_indexer_tc_scores_match_dp4a(csa, monkeypatch, B, Tq, N, m, key_exps, q_scale):
    """The FP8 tensor-core scores (exact block dots) equal the dp4a kernel's bit
    for bit: all visible scores, read back through a top-k of k = N."""
    rng = np.random.default_rng(7 + Tq + N)
    HI, dI = 16, 64
    codes, scales = _mxfp4_keys_random(rng, B * N, key_exps)
    kd = dev(codes.reshape(B, N, 32))
    ksd = dev(scales.reshape(B, N, 2))
    qI = (rng.standard_normal((B, Tq, HI, dI)) * q_scale).astype(np.float32)
    qI[:, :, 0, :32] = 0.0                                 # an all-zero block (exponent 0)
    qbits = wl.f32_to_bf16_bits(qI)
    w = rng.standard_normal((B, Tq, HI)).astype(np.float32)
    q_pos = np.tile(np.arange(Tq, dtype=np.int64), (B, 1)) + rng.integers(0, 3, size=(B, 1))
    args = (dev_bf16(qbits), dev(w), kd, ksd, dev(q_pos), N, m, N)
    idx_tc, sc_tc = csa.indexer_topk(*args)
    monkeypatch.setenv("CSA_INDEXER_IMPL", "dp4a")
    idx_dp, sc_dp = csa.indexer_topk(*args)
    monkeypatch.delenv("CSA_INDEXER_IMPL")
    np.testing.assert_array_equal(idx_tc.cpu().numpy(), idx_dp.cpu().numpy())
    np.testing.assert_array_equal(sc_tc.cpu().numpy().view(np.uint32), sc_dp.cpu().numpy().view(np.uint32))


def test_indexer_decode_scores_wide_scale_spread(csa, oracle_mod):
    """Decode-shaped scoring (one query row per sequence, N past the decode
    kernel's threshold) with block scales far apart, so the two block
    dots of a head meet both as one integer and through the two-product form
    (scale exponents up to ~33 apart);
    top-k of k = 4096 in two stages (chunk winners staged in shared memory)
    against the oracle, bit for bit.  Spreads stay where the oracle's fp64 dot
    is exact (13-bit block dots, shifts below 40)."""
    rng = np.random.default_rng(2024)
    B, N, HI, dI, k = 2, 9000, 16, 64, 4096
    codes, scales = _mxfp4_keys_random(rng, B * N, list(range(118, 143)))
    qI = rng.standard_normal((B, 1, HI, dI)).astype(np.float32)
    qI[:, :, 3, 32:] *= np.float32(2.0 ** 6)                 # one head's blocks 2^6 apart
    qbits = wl.f32_to_bf16_bits(qI)
    w = rng.uniform(0.0, 1.0, (B, 1, HI)).astype(np.float32)
    q_pos = np.array([[N - 1], [N - 700]], np.int64)          # the second row sees fewer entries
    idx, sc = csa.indexer_topk(dev_bf16(qbits), dev(w), dev(codes.reshape(B, N, 32)),
                               dev(scales.reshape(B, N, 2)), dev(q_pos), N, 1, k)
    oidx, osc = oracle_mod.indexer_topk(wl.bf16_bits_to_f32(qbits), w,
                                        (codes.reshape(B, N, 32), scales.reshape(B, N, 2)), q_pos, N, 1, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), osc.view(np.uint32))


@pytest.mark.parametrize("B,N,HI,key_exps,q_scale", [
    (2, 9000, 16, list(range(120, 135)), 1.0),          # ordinary scales (one-multiply epilogue)
    (1, 8192 + 77, 16, [0, 1, 2, 250, 254], 1e-30),     # powers far outside [2^-100, 2^100]
    (3, 8200, 12, list(range(100, 160)), 3e4),         # fewer heads than the MMA's 16 columns
])
def test_indexer_decode_tc_matches_dp4a(csa, monkeypatch, B, N, HI, key_exps, q_scale):
    """Decode scoring on the tensor cores (E2M1 operands straight from the
    stored codes) equals the integer decode kernel bit for bit: indices and
    scores of a top-4096 per row."""
    rng = np.random.default_rng(11 + N + HI)
    codes, scales = _mxfp4_keys_random(rng, B * N, key_exps)
    qI = (rng.standard_normal((B, 1, HI, 64)) * q_scale).astype(np.float32)
    qI[:, :, 0, :32] = 0.0                                 # an all-zero block (exponent 0)
    qbits = wl.f32_to_bf16_bits(qI)
    w = rng.standard_normal((B, 1, HI)).astype(np.float32)
    q_pos = (N - 1 - rng.integers(0, 300, size=(B, 1))).astype(np.int64)
    args = (dev_bf16(qbits), dev(w), dev(codes.reshape(B, N, 32)), dev(scales.reshape(B, N, 2)), dev(q_pos), N, 1,
            4096)
    idx_tc, sc_tc = csa.indexer_topk(*args)
    monkeypatch.setenv("CSA_INDEXER_IMPL", "dp4a")
    idx_dp, sc_dp = csa.indexer_topk(*args)
    monkeypatch.delenv("CSA_INDEXER_IMPL")
    np.testing.assert_array_equal(idx_tc.cpu().numpy(), idx_dp.cpu().numpy())
    np.testing.assert_array_equal(sc_tc.cpu().numpy().view(np.uint32), sc_dp.cpu().numpy().view(np.uint32))


def _pattern_with_positive_score(oracle_mod, rng, qbits, w):
    """32 random code bytes whose score at block scales 2^0 is positive."""
    q = wl.bf16_bits_to_f32(qbits)
    for _ in range(64):
        pat = rng.integers(0, 256, size=32, dtype=np.uint8)
        _, sc = oracle_mod.indexer_topk(q, w, (pat[None, None], np.full((1, 1, 2), 127, np.uint8)),
                                        np.zeros((1, 1), np.int64), 1, 1, 1)
        if sc[0, 0, 0] > 0:
            return pat
    raise AssertionError("no pattern with a positive score")


@pytest.mark.parametrize("N,k", [(20000, 1024), (20001, 1024), (20000, 2000)])   # odd N: copy-fed scorer
def test_indexer_decode_topk_equal_scores(csa, oracle_mod, N, k):
    """Decode rows (histogram top-k) whose scores repeat exactly, against the
    oracle bit for bit (equal scores by ascending index):
    row 0: 50 distinct entries repeated at random -- the sure and tie keys
    sorted together; row 1: one entry everywhere -- the threshold bin holds
    more than the tie list, selection over the whole row; row 2: 500 entries
    4x above 6000 equal ones above the rest -- too many sure and tie keys
    to sort at once, the ties selected first; row 3: fewer visible entries
    than k -- every one taken."""
    rng = np.random.default_rng(31337 + N)
    B, HI = 4, 16
    qI = rng.standard_normal((1, 1, HI, 64)).astype(np.float32)
    qbits = np.repeat(wl.f32_to_bf16_bits(qI), B, axis=0)
    w = np.repeat(rng.uniform(0.1, 1.0, (1, 1, HI)).astype(np.float32), B, axis=0)
    pat = _pattern_with_positive_score(oracle_mod, rng, qbits[:1], w[:1])
    codes = np.empty((B, N, 32), np.uint8)
    scales = np.empty((B, N, 2), np.uint8)
    pats, pscl = rng.integers(0, 256, size=(50, 32), dtype=np.uint8), rng.integers(124, 131, size=(50, 2))
    pick = rng.integers(0, 50, size=N)
    codes[0], scales[0] = pats[pick], pscl[pick]
    codes[1], scales[1] = pat, 127
    grp = rng.permutation(np.concatenate([np.full(500, 129), np.full(6000, 127), np.full(N - 6500, 124)]))
    codes[2], scales[2] = pat, grp[:, None]
    codes[3], scales[3] = _mxfp4_keys_random(rng, N, list(range(120, 135)))
    q_pos = np.array([[N - 1], [N - 1], [N - 1], [700]], np.int64)
    idx, sc = csa.indexer_topk(dev_bf16(qbits), dev(w), dev(codes), dev(scales), dev(q_pos), N, 1, k)
    oidx, osc = oracle_mod.indexer_topk(wl.bf16_bits_to_f32(qbits), w, (codes, scales), q_pos, N, 1, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    np.testing.assert_array_equal(sc.cpu().numpy().view(np.uint32), osc.view(np.uint32))
    assert len(set(osc[1, 0].tolist())) == 1 and list(oidx[1, 0]) == list(range(k))


# --------------------------------------------------------------------------
# per-channel compression logits: bit-exact bytes against the oracle
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,T,m,pos0,part,fmt", [
    ("c2_csa_prefill_8k", 8192 - 3, 4, 4096, "kv", "mixed592"),   # ragged tail, shifted positions
    ("c4_hca_prefill_64k", 16384 + 100, 128, 0, "kv", "mixed592"),  # HCA ratio
    ("c2_csa_prefill_8k", 4096, 1, 0, "kv", "mixed592"),           # m = 1: the tokens, scaled
    ("c2_csa_prefill_8k", 8192, 4, 0, "kI", "mxfp4"),              # FP4 indexer keys
    ("c1_tiny_csa_prefill", 510, 4, 0, "kv", "f32"),               # fp32 input and output
])
def test_compress_channel_logits_bitexact(csa, oracle_mod, name, T, m, pos0, part, fmt):
    cfg = wl.CONFIGS[name]
    toks = wl.gen_tokens(cfg, 0, 0, T, parts=(part,))
    x = toks[part]
    C = x.shape[1]
    zc = wl.gen_channel_logits(cfg, 0, C, 0, T)
    sc = wl.gen_channel_scales(cfg)
    s = sc["s"] if part == "kv" else sc["sI"]
    R = 64 if part == "kv" else 0
    rope_np, rope_dev = ropes(csa, oracle_mod, pos0 + T + 1)
    dfmt = {"mixed592": csa.FMT_MIXED592, "mxfp4": csa.FMT_MXFP4, "f32": csa.FMT_F32}[fmt]
    got = csa.compress_kv(act_dev(x, cfg)[None], dev(zc)[None], dev(s), m, dfmt, R, rope_dev if R else None,
                          pos0=pos0)
    ref = oracle_mod.compress_kv(widen(x, cfg)[None], zc[None], s, m, fmt, R, pos0, rope_np if R else None)
    if fmt == "mxfp4":
        np.testing.assert_array_equal(got[0].cpu().numpy(), ref[0])
        np.testing.assert_array_equal(got[1].cpu().numpy(), ref[1])
    elif fmt == "f32":
        np.testing.assert_array_equal(got.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    else:
        np.testing.assert_array_equal(got.cpu().numpy(), ref)


def test_compress_channel_logits_equal_channels_is_per_token(csa):
    """On the GPU too: logits repeated over channels store the per-token bytes."""
    cfg = wl.CONFIGS["c2_csa_prefill_8k"]
    toks = wl.gen_tokens(cfg, 0, 0, 2048, parts=("kv", "z"))
    x = act_dev(toks["kv"], cfg)[None]
    z = dev(toks["z"])[None]
    s = dev(wl.gen_channel_scales(cfg)["s"])
    rope = csa.rope_table(2049, 64)
    a = csa.compress_kv(x, z, s, 4, csa.FMT_MIXED592, 64, rope)
    b = csa.compress_kv(x, z[..., None].expand(1, 2048, 512).contiguous(), s, 4, csa.FMT_MIXED592, 64, rope)
    assert torch.equal(a, b)


# --------------------------------------------------------------------------
# chunked prefill against a resident cache (the 128K configuration's inputs)
# --------------------------------------------------------------------------
def test_chunked_prefill_equals_one_shot_and_oracle(csa, oracle_mod):
    """The first 16384 tokens of the 128K prefill in 4 chunks of 4096: the
    caches and the outputs equal one call over all tokens, byte for byte, and
    sampled rows of the last chunk match the oracle (its own caches and
    top-k) within the attention tolerance."""
    cfg = wl.CONFIGS["c2_csa_prefill_128k"]
    T, Tc, m = 16384, 4096, cfg.m
    toks = wl.gen_tokens(cfg, 0, 0, T)
    qry = wl.gen_queries(cfg, 0, 0, T)
    sc = wl.gen_channel_scales(cfg)
    rope_np, rope_dev = ropes(csa, oracle_mod, T + 1)
    kv, z = dev_bf16(toks["kv"])[None], dev(toks["z"])[None]
    kI, zI = dev_bf16(toks["kI"])[None], dev(toks["zI"])[None]
    s, sI = dev(sc["s"]), dev(sc["sI"])
    q, qI, w = dev_bf16(qry["q"])[None], dev_bf16(qry["qI"])[None], dev(qry["w"])[None]
    scale = softmax_scale(cfg)
    # one call over all tokens
    cache = csa.compress_kv(kv, z, s, m, csa.FMT_MIXED592, cfg.R, rope_dev)
    swa = csa.compress_kv(kv, z, None, 1, csa.FMT_MIXED592, cfg.R, rope_dev)
    kc, ks = csa.compress_kv(kI, zI, sI, m, csa.FMT_MXFP4, 0)
    q_pos = torch.arange(T, dtype=torch.int64, device="cuda")[None]
    idx = csa.indexer_topk(qI, w, kc, ks, q_pos, T // m, m, cfg.k, scores=False)
    out1 = csa.sparse_mqa(q, q_pos, cache, m, idx, swa, dev(np.zeros(1, np.int64)), cfg.W, scale, rope_dev, cfg.R)
    # the same in chunks
    cp = csa.ChunkedPrefill(T, m, cfg.k, cfg.W, rope_dev)
    out2 = torch.empty_like(q)
    for t0 in range(0, T, Tc):
        t1 = t0 + Tc
        cp.run(t0, t1, kv[:, t0:t1], z[:, t0:t1], kI[:, t0:t1], zI[:, t0:t1], s, sI, q[:, t0:t1], qI[:, t0:t1],
               w[:, t0:t1], scale, out=out2[:, t0:t1])
    torch.cuda.synchronize()
    assert torch.equal(cp.cache, cache) and torch.equal(cp.swa, swa)
    assert torch.equal(cp.kc, kc) and torch.equal(cp.ks, ks)
    assert torch.equal(out2, out1)
    # sampled rows of the last chunk against the oracle
    rows = np.array([T - Tc, T - Tc + 1, T - 1000, T - 129, T - 2, T - 1])
    xw = widen(toks["kv"], cfg)[None]
    ocache = oracle_mod.compress_kv(xw, toks["z"][None], sc["s"], m, "mixed592", cfg.R, 0, rope_np)
    oswa = oracle_mod.compress_kv(xw, toks["z"][None], None, 1, "mixed592", cfg.R, 0, rope_np)
    okeys = oracle_mod.compress_kv(widen(toks["kI"], cfg)[None], toks["zI"][None], sc["sI"], m, "mxfp4", 0)
    qp = np.arange(T, dtype=np.int64)[None]
    oidx, _ = oracle_mod.indexer_topk(widen(qry["qI"], cfg)[rows][None], qry["w"][rows][None], okeys,
                                      qp[:, rows], T // m, m, cfg.k)
    np.testing.assert_array_equal(idx[0, rows].cpu().numpy(), oidx[0])
    oout, _, bad = oracle_mod.attention(widen(qry["q"], cfg)[rows][None], qp[:, rows], ocache, T // m, m, oidx, oswa,
                                        np.zeros(1, np.int64), cfg.W, scale, rope_np, cfg.R,
                                        oracle_mod.FMT_MIXED592)
    assert bad == 0
    got = out2[0, rows].float().cpu().numpy()
    assert max_rel_err(got, oout[0]) <= tol(cfg)
