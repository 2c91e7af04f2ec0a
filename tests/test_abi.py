"""C-ABI boundary checks that need no GPU.

* every function declared in include/csa_b300.h is exported by libcsa_b300.so;
* the host RoPE table of the library equals the oracle's bit for bit (both
  evaluate cos/sin in fp64 and round to fp32);
* argument validation answers INVALID_ARG / UNSUPPORTED before anything is
  launched.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def csa():
    from long_context_sparse_29_b300 import build
    build.build()
    import long_context_sparse_29_b300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "csa_b300.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_five_calls():
    names = _declared()
    for n in ("csa_compress_kv", "csa_indexer_topk", "csa_sparse_mqa", "hca_dense_attn",
              "kvcache_pack_fp8_bf16"):
        assert n in names


def test_every_declared_symbol_is_exported(csa):
    L = ctypes.CDLL(csa._lib.SO_PATH)
    for name in _declared():
        assert hasattr(L, name), name
    assert set(_declared()) <= set(csa._lib.SIGNATURES)


def test_rope_table_matches_oracle_bitwise(csa, oracle_mod):
    for P, R, base in ((4096, 64, 10000.0), (257, 32, 500.0)):
        c = np.empty((P, R // 2), np.float32)
        s = np.empty((P, R // 2), np.float32)
        csa._lib.check(csa._lib.lib().csa_rope_table(P, R, base, c.ctypes.data, s.ctypes.data))
        oc, os_ = oracle_mod.rope_table(P, R, base)
        np.testing.assert_array_equal(c.view(np.uint32), oc.view(np.uint32))
        np.testing.assert_array_equal(s.view(np.uint32), os_.view(np.uint32))


def test_rope_table_far_positions_match_oracle(csa, oracle_mod):
    # positions near 1M, where the fp64 angle is large
    P, R = (1 << 20) + 8, 64
    c = np.empty((P, R // 2), np.float32)
    s = np.empty((P, R // 2), np.float32)
    csa._lib.check(csa._lib.lib().csa_rope_table(P, R, 10000.0, c.ctypes.data, s.ctypes.data))
    oc, os_ = oracle_mod.rope_table(P, R)
    np.testing.assert_array_equal(c, oc)
    np.testing.assert_array_equal(s, os_)


def test_validation_errors_before_launch(csa):
    L = csa._lib.lib()
    # NULL pointers with work to do
    r = L.csa_compress_kv(None, 1, None, None, None, None, 0, 0, 1, 8, 512, 64, 4, 1, None, None, None)
    assert r == -1 and b"NULL" in L.csa_last_error()
    # pos0 not a multiple of m
    r = L.csa_compress_kv(None, 1, None, None, None, None, 0, 2, 1, 8, 512, 64, 4, 1, None, None, None)
    assert r == -1
    # mixed rows need C = 512, R = 64
    r = L.csa_compress_kv(ctypes.c_void_p(16), 1, ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                          ctypes.c_void_p(16), 100, 0, 1, 8, 256, 64, 4, 1, ctypes.c_void_p(16), None, None)
    assert r == -2
    # m > 128
    r = L.csa_compress_kv(None, 1, None, None, None, None, 0, 0, 1, 1024, 512, 64, 256, 1, None, None, None)
    assert r == -2
    # top-k limits
    r = L.csa_indexer_topk(None, 1, None, None, None, 2, None, 1, 1, 16, 64, 8, 4, 5000, None, None,
                           None, 0, None)
    assert r == -2
    r = L.csa_indexer_topk(None, 1, None, None, None, 0, None, 1, 1, 16, 64, 8, 4, 16, None, None,
                           None, 0, None)
    assert r == -2        # bf16 queries need MXFP4 keys
    # attention: bf16 queries need the mixed cache and D = 512
    r = L.csa_sparse_mqa(None, 1, None, 1, 1, 64, 128, 64, 1, None, 8, 4, None, 4, None, None, 0, 0,
                         0.1, None, None, 1, None, None, None, 0, None)
    assert r == -1        # NULL pointers are reported first
    ws = ctypes.c_void_p(256)
    r = L.csa_sparse_mqa(ctypes.c_void_p(16), 1, ctypes.c_void_p(16), 1, 1, 64, 128, 64, 1,
                         ctypes.c_void_p(16), 8, 4, ctypes.c_void_p(16), 4, None, None, 0, 0, 0.1,
                         ctypes.c_void_p(16), ctypes.c_void_p(16), 1, ctypes.c_void_p(16), None, ws,
                         1 << 20, None)
    assert r == -2
    assert L.csa_workspace_size(99, 1, 1, 1, 1, 1, 1, 1, 0) == -1
    assert L.csa_workspace_size(1, 1, 8, 2048, 512, 0, 0, 0, 0) >= 256 + 8 * 2048 * 4


def test_binding_requires_cuda_tensors(csa):
    import torch
    x = torch.zeros(1, 8, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        csa.compress_kv(x, torch.zeros(1, 8), None, 4, csa.FMT_MIXED592, 64)


def test_decode_append_and_channel_logits_validation(csa):
    """Every case is refused on the host (or has nothing to do): no launch."""
    L = csa._lib.lib()
    P = ctypes.c_void_p
    ok16 = P(16)   # stand-in pointers, never dereferenced: each call below fails validation first

    def append(kv=ok16, kI=None, C=512, R=64, CI=0, m=4, B=1, Ts=64, W=32, nmax=4):
        return L.csa_decode_append(kv, ok16, kI, ok16 if kI else None, None, None, ok16, ok16, 100, ok16, B, C, R,
                                   CI, m, ok16, ok16, ok16 if kI else None, ok16 if kI else None, ok16, nmax,
                                   ok16 if kI else None, ok16 if kI else None, ok16, Ts, W, ok16, None)

    assert append(m=0) == -1 and b"bad sizes" in L.csa_last_error()
    assert append(m=129) == -1
    assert append(C=256) == -2
    assert append(R=32) == -2
    assert append(kI=ok16, CI=48) == -2
    assert append(Ts=40, W=32) == -1 and b"Ts" in L.csa_last_error()
    assert append(kv=None) == -1 and b"NULL" in L.csa_last_error()
    assert append(kv=P(24)) == -1 and b"aligned" in L.csa_last_error()
    assert append(kv=None, B=0) == 0      # nothing to append
    r = L.csa_compress_kv_channel_logits(None, 1, None, None, None, None, 0, 0, 1, 8, 512, 64, 4, 1, None, None,
                                         None)
    assert r == -1 and b"csa_compress_kv_channel_logits" in L.csa_last_error()
    r = L.csa_compress_kv_channel_logits(None, 1, None, None, None, None, 0, 0, 1, 1024, 512, 64, 256, 1, None,
                                         None, None)
    assert r == -2


def test_missing_library_fails_loudly(monkeypatch):
    """No fallback: with the CUDA library absent, the first call raises."""
    from long_context_sparse_29_b300 import _lib
    monkeypatch.setattr(_lib, "SO_PATH", os.path.join(ROOT, "no_such_dir", "libcsa_b300.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.lib()


def test_calls_with_nothing_to_do_return_ok(csa):
    """Empty work is not an error and launches nothing: no complete block, no
    queries, no sequences.  (Pointers are NULL; the workspace pointer is
    only checked for alignment, never used.)"""
    L = csa._lib.lib()
    ws = ctypes.c_void_p(256)
    # T < m: no complete block
    assert L.csa_compress_kv(None, 1, None, None, None, None, 0, 0, 1, 3, 512, 64, 4, 1, None, None, None) == 0
    assert L.csa_compress_kv_channel_logits(None, 1, None, None, None, None, 0, 0, 1, 3, 512, 64, 4, 1, None,
                                            None, None) == 0
    # no queries
    assert L.csa_indexer_topk(None, 1, None, None, None, 2, None, 1, 0, 16, 64, 2048, 4, 512, None, None, None,
                              0, None) == 0
    assert L.csa_sparse_mqa(None, 1, None, 1, 0, 64, 512, 64, 1, None, 0, 4, None, 0, None, None, 0, 0, 0.1,
                            None, None, 1, None, None, ws, 1 << 20, None) == 0
    # no sequences
    assert L.hca_dense_attn(None, 1, None, 0, 5, 64, 512, 64, 1, None, 0, 128, None, None, 0, 0, 0.1, None, None,
                            1, None, None, ws, 1 << 20, None) == 0
