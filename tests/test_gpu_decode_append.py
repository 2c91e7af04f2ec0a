"""Decode-time cache maintenance (csa_decode_append) against block compression.

Appending tokens 0 .. T-1 one call at a time must leave exactly the bytes
csa_compress_kv stores for the whole sequence: the compressed entries, the
MXFP4 indexer keys and the window rows (which also moves down the buffer as it
fills).  The CSA entries are also compared with the oracle directly.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_common import dev, dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


@pytest.mark.parametrize("m,T,with_keys", [(4, 300, True), (128, 400, False), (1, 70, True)])
def test_decode_append_matches_block_compression(csa, oracle_mod, m, T, with_keys):
    B, W, Ts, C, CI = 2, 32, 64, 512, 64
    rng = np.random.default_rng(1000 + m)
    kv_bits = wl.f32_to_bf16_bits(rng.standard_normal((B, T, C)).astype(np.float32))
    z = (0.5 * rng.standard_normal((B, T))).astype(np.float32)
    kI_bits = wl.f32_to_bf16_bits(rng.standard_normal((B, T, CI)).astype(np.float32))
    zI = (0.5 * rng.standard_normal((B, T))).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    sI = rng.uniform(0.5, 1.5, CI).astype(np.float32)
    kv_d, kI_d = dev_bf16(kv_bits), dev_bf16(kI_bits)
    z_d, zI_d, s_d, sI_d = dev(z), dev(zI), dev(s), dev(sI)
    rope = csa.rope_table(T + 1, 64)
    nmax = T // m
    lc = csa.LayerCache(B, nmax, m, W, Ts, CI=CI if with_keys else 0)
    for t in range(T):
        tp = torch.full((B,), t, dtype=torch.int64, device="cuda")
        if with_keys:
            csa.decode_append(lc, kv_d[:, t].contiguous(), z_d[:, t].contiguous(), tp, rope,
                              kI_d[:, t].contiguous(), zI_d[:, t].contiguous(), s_d, sI_d)
        else:
            csa.decode_append(lc, kv_d[:, t].contiguous(), z_d[:, t].contiguous(), tp, rope, s=s_d)
    torch.cuda.synchronize()
    ref = csa.compress_kv(kv_d, z_d, s_d, m, csa.FMT_MIXED592, 64, rope)
    np.testing.assert_array_equal(lc.cache.cpu().numpy(), ref[:, :nmax].cpu().numpy())
    if with_keys:
        kc, ks = csa.compress_kv(kI_d, zI_d, sI_d, m, csa.FMT_MXFP4, 0)
        np.testing.assert_array_equal(lc.kI_codes.cpu().numpy(), kc.cpu().numpy())
        np.testing.assert_array_equal(lc.kI_scales.cpu().numpy(), ks.cpu().numpy())
    # the window cache holds tokens swa_pos0 .. T-1 from row 0: at least the
    # last W and at most Ts of them (a slide keeps W - 1 rows and adds one)
    p0 = lc.swa_pos0.cpu().numpy()
    assert (p0 == p0[0]).all() and max(0, T - Ts) <= p0[0] <= max(0, T - W)
    p0 = int(p0[0])
    win = csa.compress_kv(kv_d[:, p0:].contiguous(), z_d[:, p0:].contiguous(), None, 1, csa.FMT_MIXED592, 64,
                          rope, pos0=p0)
    np.testing.assert_array_equal(lc.swa[:, :T - p0].cpu().numpy(), win.cpu().numpy())
    # the oracle's bytes for sequence 0's entries
    x0 = wl.bf16_bits_to_f32(kv_bits[:1])
    oc = oracle_mod.compress_kv(x0, z[:1], s, m, "mixed592", 64, 0, oracle_mod.rope_table(T + 1, 64))
    np.testing.assert_array_equal(lc.cache[:1].cpu().numpy(), oc[:, :nmax])


def test_decode_append_rejects_bad_shapes(csa):
    lc = csa.LayerCache(1, 4, 4, 32, 40)   # Ts < 2 W
    kv = torch.zeros((1, 512), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(1, dtype=torch.float32, device="cuda")
    tp = torch.zeros(1, dtype=torch.int64, device="cuda")
    with pytest.raises(csa.CsaError):
        csa.decode_append(lc, kv, z, tp, csa.rope_table(8, 64))
