"""Batch invariance: a sequence's results do not depend on the other sequences
of its batch ("DeepSeek-V4 — MoE nyelvmodellek milliós kontextussal",
section "Kommunikációs optimalizációk": batch-invariant, deterministic
kernels).

Held bit for bit by every step whose arithmetic is per sequence and per
entry: compressed cache bytes, indexer top-k indices and scores (decode rows
at 128K context: the tensor-core scorer, its histogram and the histogram
top-k), and prefill attention rows (one work item per query row).  Decode
attention is deterministic for a given batch size but splits each row's keys
over a number of CTAs that depends on how many rows share the GPU, so its
rounding may differ between batch sizes; that case is checked within the
output tolerance here.
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


def test_indexer_topk_and_keys_are_batch_invariant(csa):
    cfg = wl.CONFIGS["c3_csa_decode_128k"]
    B, T = 6, 65536   # 16384 entries per row: the histogram top-k path
    sI = dev(wl.gen_channel_scales(cfg)["sI"])
    toks = [wl.gen_tokens(cfg, b, 0, T, parts=("kI", "zI")) for b in range(B)]
    kI = torch.stack([dev_bf16(t["kI"]) for t in toks])
    zI = torch.stack([dev(t["zI"]) for t in toks])
    kc, ks = csa.compress_kv(kI, zI, sI, cfg.m, csa.FMT_MXFP4, 0)
    kc1, ks1 = csa.compress_kv(kI[3:4].contiguous(), zI[3:4].contiguous(), sI, cfg.m, csa.FMT_MXFP4, 0)
    assert torch.equal(kc[3:4], kc1) and torch.equal(ks[3:4], ks1)
    qry = [wl.gen_queries(cfg, b) for b in range(B)]
    qI = dev_bf16(np.stack([q["qI"] for q in qry]))
    w = dev(np.stack([q["w"] for q in qry]))
    N = T // cfg.m
    q_pos = torch.full((B, 1), T - 1, dtype=torch.int64, device="cuda")
    idx, sc = csa.indexer_topk(qI, w, kc, ks, q_pos, N, cfg.m, cfg.k)
    idx1, sc1 = csa.indexer_topk(qI[3:4].contiguous(), w[3:4].contiguous(), kc1, ks1, q_pos[3:4].contiguous(), N,
                                 cfg.m, cfg.k)
    assert torch.equal(idx[3:4], idx1)
    assert torch.equal(sc[3:4].view(torch.int32), sc1.view(torch.int32))


def test_prefill_attention_is_batch_invariant(csa, oracle_mod):
    rng = np.random.default_rng(4000)
    B, T, m, k, W = 2, 1024, 4, 96, 64
    N = T // m
    rope_dev = csa.rope_table(T + 1, 64)
    cache = np.stack([oracle_mod.pack_mixed(rng.standard_normal((N, 512)).astype(np.float32)) for _ in range(B)])
    swa = np.stack([oracle_mod.pack_mixed(rng.standard_normal((T, 512)).astype(np.float32)) for _ in range(B)])
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, T, 64, 512)).astype(np.float32))
    idx = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            nv = min(N, (t + 1) // m)
            p = rng.permutation(nv)[:k]
            idx[b, t, :len(p)] = p
    q_pos = np.tile(np.arange(T, dtype=np.int64), (B, 1))
    pos0 = np.zeros(B, np.int64)
    scale = 1 / math.sqrt(512)
    both = csa.sparse_mqa(dev_bf16(q), dev(q_pos), dev(cache), m, dev(idx), dev(swa), dev(pos0), W, scale, rope_dev)
    one = csa.sparse_mqa(dev_bf16(q[1:]), dev(q_pos[1:]), dev(cache[1:]), m, dev(idx[1:]), dev(swa[1:]),
                         dev(pos0[1:]), W, scale, rope_dev)
    assert torch.equal(both[1:].view(torch.int16), one.view(torch.int16))


def test_decode_attention_across_batch_sizes(csa, oracle_mod):
    """Sequence 5 alone and inside a batch of 32 (different split counts):
    equal within the output tolerance; each run is deterministic."""
    rng = np.random.default_rng(4100)
    B, N, m, k, W, Ts = 32, 4096, 4, 1024, 128, 256
    T = N * m
    rope_dev = csa.rope_table(T + 1, 64)
    cache = np.stack([oracle_mod.pack_mixed(rng.standard_normal((N, 512)).astype(np.float32)) for _ in range(B)])
    swa = np.stack([oracle_mod.pack_mixed(rng.standard_normal((Ts, 512)).astype(np.float32)) for _ in range(B)])
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, 1, 64, 512)).astype(np.float32))
    q_pos = np.full((B, 1), T - 1, np.int64)
    pos0 = np.full(B, T - Ts, np.int64)
    idx = np.stack([rng.permutation(N)[:k].astype(np.int32) for _ in range(B)])[:, None, :]
    scale = 1 / math.sqrt(512)
    args = lambda sl: (dev_bf16(q[sl]), dev(q_pos[sl]), dev(cache[sl]), m, dev(idx[sl]), dev(swa[sl]), dev(pos0[sl]),
                       W, scale, rope_dev)
    full = csa.sparse_mqa(*args(slice(0, B))).float()
    full2 = csa.sparse_mqa(*args(slice(0, B))).float()
    alone = csa.sparse_mqa(*args(slice(5, 6))).float()
    assert torch.equal(full, full2)
    err = float((full[5:6] - alone).abs().max()) / float(alone.abs().max())
    assert err <= 1e-2, err
