"""Parity at the full sizes of the two long prefill workloads (GPU vs oracle).

* HCA prefill of 1 x 65536 tokens at m' = 128 (512 entries), through
  hca_dense_attn with every query row in one call -- the plan the benchmark
  times (all cache and window rows expanded once, one work item per row);
  sampled rows against the oracle's dense attention over all visible
  entries plus the window.  xmsumi.com DeepSeek-V4 article, section
  "HCA（重度压缩注意力）"; "DeepSeek-V4 — MoE nyelvmodellek milliós
  kontextussal", section "Heavily Compressed Attention (HCA)".
* CSA prefill of 1 x 131072 tokens in query chunks of 8192 against caches
  that grow chunk by chunk (the benchmark's 128K configuration): in the last
  chunk every row has 30720 to 32768 candidate entries; sampled rows' top-k
  indices must equal the oracle's bit for bit and their attention rows match
  within the output tolerance.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_common import dev, dev_bf16, max_rel_err, softmax_scale, tol, widen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


def _ropes(csa, oracle_mod, P):
    rope_np = oracle_mod.rope_table(P, 64)
    rope_dev = csa.rope_table(P, 64)
    return rope_np, rope_dev


def test_hca_prefill_64k_sampled(csa, oracle_mod):
    cfg = wl.CONFIGS["c4_hca_prefill_64k"]
    T, m, W, N = cfg.T, cfg.m, cfg.W, cfg.N
    rope_np, rope_dev = _ropes(csa, oracle_mod, T + 1)
    sc = wl.gen_channel_scales(cfg)
    toks = wl.gen_tokens(cfg, 0, parts=("kv", "z"))
    kv_d, z_d = dev_bf16(toks["kv"])[None], dev(toks["z"])[None]
    cache = csa.compress_kv(kv_d, z_d, dev(sc["s"]), m, csa.FMT_MIXED592, cfg.R, rope_dev)
    swa = csa.compress_kv(kv_d, z_d, None, 1, csa.FMT_MIXED592, cfg.R, rope_dev)
    # the queries of all 65536 rows, generated and copied in slices
    q_d = torch.empty((1, T, cfg.H, cfg.D), dtype=torch.bfloat16, device="cuda")
    for t0 in range(0, T, 8192):
        q_d[0, t0:t0 + 8192] = dev_bf16(wl.gen_queries(cfg, 0, t0, t0 + 8192)["q"])
    q_pos = dev(np.arange(T, dtype=np.int64)[None])
    pos0 = dev(np.zeros(1, np.int64))
    out = csa.hca_dense_attn(q_d, q_pos, cache, m, swa, pos0, W, softmax_scale(cfg), rope_dev, cfg.R)
    rows = np.unique(np.concatenate([np.arange(0, 6), [127, 128, 129, 255, 256, 16383, 16384, 16385, 32767],
                                     np.random.default_rng(7).choice(T, 30, replace=False), [T - 1]]))
    assert rows.size >= 40
    got = out[0, torch.as_tensor(rows, device="cuda")].float().cpu().numpy()
    del q_d, out
    xw = widen(toks["kv"], cfg)[None]
    ocache = oracle_mod.compress_kv(xw, toks["z"][None], sc["s"], m, "mixed592", cfg.R, 0, rope_np)
    oswa = oracle_mod.compress_kv(xw, toks["z"][None], None, 1, "mixed592", cfg.R, 0, rope_np)
    q_rows = np.stack([wl.gen_queries(cfg, 0, int(r), int(r) + 1)["q"][0] for r in rows])
    ref, _, bad = oracle_mod.attention(widen(q_rows, cfg)[None], rows.astype(np.int64)[None], ocache, N, m, None,
                                       oswa, np.zeros(1, np.int64), W, softmax_scale(cfg), rope_np, cfg.R)
    assert bad == 0
    for i, r in enumerate(rows):   # each row on its own scale, then all together
        assert max_rel_err(got[i:i + 1], ref[0, i:i + 1]) <= tol(cfg), (r, max_rel_err(got[i:i + 1], ref[0, i:i + 1]))
    assert max_rel_err(got, ref[0]) <= tol(cfg)


def test_chunked_prefill_128k_last_chunk(csa, oracle_mod):
    cfg = wl.CONFIGS["c2_csa_prefill_128k"]
    T, Tc, m, W = cfg.T, 8192, cfg.m, cfg.W
    rope_np, rope_dev = _ropes(csa, oracle_mod, T + 1)
    sc = wl.gen_channel_scales(cfg)
    s_d, sI_d = dev(sc["s"]), dev(sc["sI"])
    scale = softmax_scale(cfg)
    cp = csa.ChunkedPrefill(T, m, cfg.k, W, rope_dev)
    last0 = T - Tc
    rows = np.unique(np.concatenate([[last0, last0 + 1, last0 + 2, T - 4096, T - 1000, T - 129, T - 128, T - 2,
                                      T - 1], last0 + np.random.default_rng(11).choice(Tc, 7, replace=False)]))
    for t0 in range(0, T, Tc):
        t1 = t0 + Tc
        toks = wl.gen_tokens(cfg, 0, t0, t1)
        qry = wl.gen_queries(cfg, 0, t0, t1)
        out = cp.run(t0, t1, dev_bf16(toks["kv"])[None], dev(toks["z"])[None], dev_bf16(toks["kI"])[None],
                     dev(toks["zI"])[None], s_d, sI_d, dev_bf16(qry["q"])[None], dev_bf16(qry["qI"])[None],
                     dev(qry["w"])[None], scale)
    sel = torch.as_tensor(rows - last0, device="cuda")
    got_idx = cp._idx[0, sel].cpu().numpy()
    got = out[0, sel].float().cpu().numpy()
    torch.cuda.synchronize()
    assert cp.ws_ix.flags() == 0 and cp.ws_attn.flags() == 0
    del out
    # the oracle over the whole sequence, for the sampled rows
    toks = wl.gen_tokens(cfg, 0)
    xw = widen(toks["kv"], cfg)[None]
    ocache = oracle_mod.compress_kv(xw, toks["z"][None], sc["s"], m, "mixed592", cfg.R, 0, rope_np)
    oswa = oracle_mod.compress_kv(xw[:, last0 - W:], toks["z"][None, last0 - W:], None, 1, "mixed592", cfg.R,
                                  last0 - W, rope_np)
    okeys = oracle_mod.compress_kv(widen(toks["kI"], cfg)[None], toks["zI"][None], sc["sI"], m, "mxfp4", 0)
    qr = [wl.gen_queries(cfg, 0, int(r), int(r) + 1) for r in rows]
    qp = rows.astype(np.int64)[None]
    oidx, _ = oracle_mod.indexer_topk(widen(np.stack([x["qI"][0] for x in qr]), cfg)[None],
                                      np.stack([x["w"][0] for x in qr])[None], okeys, qp, T // m, m, cfg.k)
    np.testing.assert_array_equal(got_idx, oidx[0])
    ref, _, bad = oracle_mod.attention(widen(np.stack([x["q"][0] for x in qr]), cfg)[None], qp, ocache, T // m, m,
                                       oidx, oswa, np.full(1, last0 - W, np.int64), W, scale, rope_np, cfg.R,
                                       oracle_mod.FMT_MIXED592)
    assert bad == 0
    assert max_rel_err(got, ref[0]) <= tol(cfg), max_rel_err(got, ref[0])
