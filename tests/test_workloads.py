"""The seeded input generators (workloads.py) on CPU.

Any slice of a sequence must regenerate exactly (the benchmarks and the
sampled parity checks generate chunks and single rows on their own), the
configurations must hold the sizes the workloads name, and the drawn values
must have the stated distributions.
"""
import numpy as np
import pytest

import workloads as wl


@pytest.mark.parametrize("name", ["c2_csa_prefill_8k", "c2_csa_prefill_128k", "c3_csa_decode_128k"])
def test_token_slices_regenerate(name):
    cfg = wl.CONFIGS[name]
    full = wl.gen_tokens(cfg, 1, 0, 12000)
    for t0, t1 in ((0, 1), (4095, 4097), (5000, 12000), (8191, 8193)):
        part = wl.gen_tokens(cfg, 1, t0, t1)
        for key in full:
            np.testing.assert_array_equal(part[key], full[key][t0:t1])


def test_query_slices_and_channel_logits_regenerate():
    cfg = wl.CONFIGS["c2_csa_prefill_8k"]
    full = wl.gen_queries(cfg, 0, 0, 700)
    part = wl.gen_queries(cfg, 0, 255, 513)
    for key in full:
        np.testing.assert_array_equal(part[key], full[key][255:513])
    zc = wl.gen_channel_logits(cfg, 0, 512, 0, 8000)
    np.testing.assert_array_equal(wl.gen_channel_logits(cfg, 0, 512, 4000, 4200), zc[4000:4200])
    assert zc.shape == (8000, 512) and zc.dtype == np.float32


def test_sequences_and_seeds_differ():
    cfg = wl.CONFIGS["c3_csa_decode_128k"]
    a = wl.gen_tokens(cfg, 0, 0, 64, parts=("kv",))["kv"]
    b = wl.gen_tokens(cfg, 1, 0, 64, parts=("kv",))["kv"]
    c = wl.gen_tokens(cfg, 0, 0, 64, seed=1, parts=("kv",))["kv"]
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_configuration_sizes():
    c = wl.CONFIGS
    assert (c["c2_csa_prefill_8k"].T, c["c2_csa_prefill_8k"].N, c["c2_csa_prefill_8k"].k) == (8192, 2048, 512)
    assert (c["c3_csa_decode_128k"].B, c["c3_csa_decode_128k"].N, c["c3_csa_decode_128k"].k) == (32, 32768, 1024)
    assert (c["c4_hca_prefill_64k"].N, c["c4_hca_decode_1m"].N, c["c4_hca_decode_1m"].B) == (512, 8192, 16)
    assert (c["c5_hybrid_csa_decode_1m"].N, c["c5_hybrid_hca_decode_1m"].N) == (262144, 8192)
    assert c["c2_csa_prefill_128k"].N == 32768
    for cfg in c.values():
        if not cfg.fp32:
            assert (cfg.H, cfg.D, cfg.R, cfg.W) == (64, 512, 64, 128)


def test_value_distributions():
    cfg = wl.CONFIGS["c2_csa_prefill_8k"]
    t = wl.gen_tokens(cfg, 0, 0, 8192)
    kv = wl.bf16_bits_to_f32(t["kv"]).astype(np.float64)
    assert abs(kv.mean()) < 0.01 and abs(kv.std() - 1.0) < 0.01          # N(0, 1), bf16-rounded
    assert abs(t["z"].std() - 0.5) < 0.02                                  # logits N(0, 0.5^2)
    q = wl.gen_queries(cfg, 0, 0, 256)
    assert q["w"].min() >= 0.0 and q["w"].max() <= 1.0                     # head weights U(0, 1)
    sc = wl.gen_channel_scales(cfg)
    assert sc["s"].min() >= 0.5 and sc["s"].max() <= 1.5                   # channel scales U(0.5, 1.5)
    qt = wl.gen_queries(wl.CONFIGS["c5_hybrid_csa_decode_1m"], 0, 0, 1)["qI"]
    qn = wl.gen_queries(wl.CONFIGS["c3_csa_decode_128k"], 0, 0, 1)["qI"]
    assert qt.shape == qn.shape == (1, 16, 64)
