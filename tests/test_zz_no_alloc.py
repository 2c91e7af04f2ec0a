"""csa_indexer_topk_noalloc: the top-k call for callers that cannot allocate.

Some hosts (runtimes that plan all device memory up front and refuse later
allocations, plugins that get tensors but no allocator) cannot hand the
library a scratch workspace.  The no-allocation entry point keeps the score
scratch in a fixed device array inside the library.  This test calls it
through the C ABI twice in a row and checks that both calls return exactly
what the workspace-taking entry point returns (top-k indices and scores are
compared bit for bit, the bar every top-k test uses), and that an oversized
request is refused without a launch.

Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def test_noalloc_topk_matches_workspace_call():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as csa
    L = csa._lib.lib()

    # decode-shaped batch at 128K context (4 sequences) and a 2K prefill
    cases = []
    cfg = wl.CONFIGS["c3_csa_decode_128k"]
    B = 4
    keys, scales, qI, w = [], [], [], []
    sI = torch.from_numpy(wl.gen_channel_scales(cfg)["sI"]).cuda()
    for b in range(B):
        tok = wl.gen_tokens(cfg, b, parts=("kI", "zI"))
        kc, ks = csa.compress_kv(_bf16(tok["kI"])[None], torch.from_numpy(tok["zI"]).cuda()[None], sI,
                                 cfg.m, csa.FMT_MXFP4, 0)
        keys.append(kc)
        scales.append(ks)
        qry = wl.gen_queries(cfg, b)
        qI.append(qry["qI"])
        w.append(qry["w"])
    cases.append((torch.cat(keys), torch.cat(scales), _bf16(np.stack(qI)),
                  torch.from_numpy(np.stack(w)).cuda(),
                  torch.full((B, 1), cfg.T - 1, dtype=torch.int64, device="cuda"), cfg.N, cfg.m, cfg.k))
    cfg2 = wl.CONFIGS["c2_csa_prefill_8k"]
    T = 2048
    tok = wl.gen_tokens(cfg2, 0, 0, T, parts=("kI", "zI"))
    kc, ks = csa.compress_kv(_bf16(tok["kI"])[None], torch.from_numpy(tok["zI"]).cuda()[None],
                             torch.from_numpy(wl.gen_channel_scales(cfg2)["sI"]).cuda(), cfg2.m,
                             csa.FMT_MXFP4, 0)
    qry = wl.gen_queries(cfg2, 0, 0, T)
    cases.append((kc, ks, _bf16(qry["qI"])[None], torch.from_numpy(qry["w"]).cuda()[None],
                  torch.arange(T, dtype=torch.int64, device="cuda")[None], T // cfg2.m, cfg2.m, cfg2.k))

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for kc, ks, qI_d, w_d, qpos, N, m, k in cases:
        Bc, Tq, HI, dI = qI_d.shape
        ref_idx, ref_sc = csa.indexer_topk(qI_d, w_d, kc, ks, qpos, N, m, k)
        for _ in range(2):
            idx = torch.full((Bc, Tq, k), -7, dtype=torch.int32, device="cuda")
            sc = torch.full((Bc, Tq, k), 7.0, dtype=torch.float32, device="cuda")
            r = L.csa_indexer_topk_noalloc(_ptr(qI_d), csa.DTYPE_BF16, _ptr(w_d), _ptr(kc), _ptr(ks),
                                           csa.FMT_MXFP4, _ptr(qpos), Bc, Tq, HI, dI, N, m, k, _ptr(idx),
                                           _ptr(sc), stream)
            assert r == 0, L.csa_last_error()
            torch.cuda.synchronize()
            assert torch.equal(idx, ref_idx)
            assert torch.equal(sc.view(torch.int32), ref_sc.view(torch.int32))

    # exactly the scratch's 4,194,304 scores (the last 2048 rows of the 8K
    # prefill against all 2048 entries) fill it and still match; one row
    # more is refused before any launch
    T8 = cfg2.T
    tok = wl.gen_tokens(cfg2, 0, 0, T8, parts=("kI", "zI"))
    kc8, ks8 = csa.compress_kv(_bf16(tok["kI"])[None], torch.from_numpy(tok["zI"]).cuda()[None],
                               torch.from_numpy(wl.gen_channel_scales(cfg2)["sI"]).cuda(), cfg2.m,
                               csa.FMT_MXFP4, 0)
    qry = wl.gen_queries(cfg2, 0, T8 - 2049, T8)
    N8 = T8 // cfg2.m
    for Tq in (2048, 2049):
        qI_d = _bf16(qry["qI"][2049 - Tq:])[None]
        w_d = torch.from_numpy(qry["w"][2049 - Tq:]).cuda()[None]
        qpos = torch.arange(T8 - Tq, T8, dtype=torch.int64, device="cuda")[None]
        idx = torch.full((1, Tq, cfg2.k), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((1, Tq, cfg2.k), 7.0, dtype=torch.float32, device="cuda")
        r = L.csa_indexer_topk_noalloc(_ptr(qI_d), csa.DTYPE_BF16, _ptr(w_d), _ptr(kc8), _ptr(ks8),
                                       csa.FMT_MXFP4, _ptr(qpos), 1, Tq, 16, 64, N8, cfg2.m, cfg2.k, _ptr(idx),
                                       _ptr(sc), stream)
        if Tq * N8 <= 4194304:
            assert r == 0, L.csa_last_error()
            ref_idx, ref_sc = csa.indexer_topk(qI_d, w_d, kc8, ks8, qpos, N8, cfg2.m, cfg2.k)
            torch.cuda.synchronize()
            assert torch.equal(idx, ref_idx)
            assert torch.equal(sc.view(torch.int32), ref_sc.view(torch.int32))
        else:
            assert r == -2 and b"16 MiB" in L.csa_last_error()

    # more scores than the built-in scratch holds: refused before any launch
    kc, ks, qI_d, w_d, qpos, N, m, k = cases[0]
    idx = torch.empty((1, 8192, 16), dtype=torch.int32, device="cuda")
    r = L.csa_indexer_topk_noalloc(_ptr(qI_d), csa.DTYPE_BF16, _ptr(w_d), _ptr(kc), _ptr(ks),
                                   csa.FMT_MXFP4, _ptr(qpos), 1, 8192, 16, 64, 1024, 4, 16, _ptr(idx),
                                   None, stream)
    assert r == -2
    assert b"16 MiB" in L.csa_last_error()
