"""Pins of the oracle's block compression (CSA m=4, HCA m'=128) and its RoPE.

Checks against closed forms (m = 1 is the identity; equal logits give the
mean), an independent fp64 softmax-weighted sum, and an independent numpy
fp32 rotation at the block's last token position.
"""
import numpy as np
import pytest


def _rot32(v, cos_row, sin_row):
    """fp32 rotation of interleaved pairs, one rounding per product and sum."""
    x0, x1 = v[..., 0::2].astype(np.float32), v[..., 1::2].astype(np.float32)
    out = np.empty(v.shape, np.float32)
    out[..., 0::2] = (x0 * cos_row) - (x1 * sin_row)
    out[..., 1::2] = (x0 * sin_row) + (x1 * cos_row)
    return out


@pytest.fixture(scope="module")
def rope(oracle_mod):
    return oracle_mod.rope_table(4096, 64)


def test_m1_is_identity(oracle_mod):
    rng = np.random.default_rng(10)
    x = rng.standard_normal((2, 37, 96)).astype(np.float32)
    z = rng.standard_normal((2, 37)).astype(np.float32)
    s = rng.uniform(0.5, 1.5, 96).astype(np.float32)
    np.testing.assert_array_equal(oracle_mod.compress(x, z, None, 1, 0), x)
    np.testing.assert_array_equal(oracle_mod.compress(x, z, s, 1, 0), x * s)


@pytest.mark.parametrize("m", [1, 4, 128])
def test_rope_at_block_last_token(oracle_mod, rope, m):
    rng = np.random.default_rng(11)
    T, C, R, pos0 = 3 * m + (m - 1), 128, 64, 2 * m
    x = rng.standard_normal((1, T, C)).astype(np.float32)
    z = rng.standard_normal((1, T)).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    plain = oracle_mod.compress(x, z, s, m, 0)
    rot = oracle_mod.compress(x, z, s, m, R, pos0=pos0, rope=rope)
    N = T // m
    assert rot.shape == (1, N, C) and N == 3          # the incomplete tail block is dropped
    np.testing.assert_array_equal(rot[..., :C - R], plain[..., :C - R])
    for j in range(N):
        p = pos0 + j * m + m - 1
        np.testing.assert_array_equal(rot[0, j, C - R:], _rot32(plain[0, j, C - R:], rope[0][p], rope[1][p]))


@pytest.mark.parametrize("m", [2, 4, 128])
def test_equal_logits_give_scaled_mean(oracle_mod, m):
    rng = np.random.default_rng(12)
    x = rng.integers(-8, 9, size=(1, 4 * m, 64)).astype(np.float32)
    z = np.full((1, 4 * m), 0.3, np.float32)
    s = rng.uniform(0.5, 1.5, 64).astype(np.float32)
    got = oracle_mod.compress(x, z, s, m, 0)
    mean = x.reshape(1, 4, m, 64).astype(np.float64).mean(axis=2)   # exact: small ints / 2^k
    np.testing.assert_array_equal(got, (mean.astype(np.float32) * s))


@pytest.mark.parametrize("m", [4, 128])
def test_matches_fp64_softmax_weighted_sum(oracle_mod, m):
    rng = np.random.default_rng(13)
    T, C = 8 * m, 64
    x = rng.standard_normal((2, T, C)).astype(np.float32)
    z = (rng.standard_normal((2, T)) * 2).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    got = oracle_mod.compress(x, z, s, m, 0).astype(np.float64)
    zz = z.reshape(2, -1, m).astype(np.float64)
    a = np.exp(zz - zz.max(-1, keepdims=True))
    a /= a.sum(-1, keepdims=True)
    xx = x.reshape(2, -1, m, C).astype(np.float64)
    ref = np.einsum("bnm,bnmc->bnc", a, xx) * s
    bound = (np.einsum("bnm,bnmc->bnc", a, np.abs(xx)) * s) * (m + 8) * 2.0 ** -23
    assert np.all(np.abs(got - ref) <= bound)


def test_weights_sum_to_one(oracle_mod):
    rng = np.random.default_rng(14)
    for m in (4, 128):
        z = (rng.standard_normal((1, 16 * m)) * 3).astype(np.float32)
        got = oracle_mod.compress(np.ones((1, 16 * m, 8), np.float32), z, None, m, 0)
        assert np.all(np.abs(got - 1.0) <= m * 2.0 ** -23 * 2)


# --------------------------------------------------------------------------
# per-channel compression logits (z [B, T, C])
# --------------------------------------------------------------------------
@pytest.mark.parametrize("m", [1, 4, 128])
def test_channel_logits_equal_across_channels_is_per_token(oracle_mod, rope, m):
    """Logits that do not vary over channels reduce to the per-token operator,
    bit for bit (RoPE included)."""
    rng = np.random.default_rng(20 + m)
    T, C = 3 * m + 1, 128
    x = rng.standard_normal((2, T, C)).astype(np.float32)
    z = (rng.standard_normal((2, T)) * 1.5).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    per_tok = oracle_mod.compress(x, z, s, m, 64, pos0=5, rope=rope)
    per_ch = oracle_mod.compress(x, np.repeat(z[..., None], C, axis=2), s, m, 64, pos0=5, rope=rope)
    np.testing.assert_array_equal(per_ch, per_tok)


def test_channel_logits_one_hot_and_equal(oracle_mod):
    """Channel c whose logits put all weight on token i_c gives s_c x_{i_c, c}
    exactly; a channel with equal logits gives s_c times the block mean."""
    rng = np.random.default_rng(30)
    m, C = 4, 64
    x = rng.integers(-8, 9, size=(1, 2 * m, C)).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    z = np.full((1, 2 * m, C), -60.0, np.float32)      # sexp(-120) = 0: weight exactly 0
    pick = rng.integers(0, m, size=(2, C))
    for j in range(2):
        for c in range(C // 2):
            z[0, j * m + pick[j, c], c] = 60.0
    z[0, :, C // 2:] = 0.25                            # equal logits in the upper half of the channels
    got = oracle_mod.compress(x, z, s, m, 0)
    for j in range(2):
        for c in range(C // 2):
            assert got[0, j, c] == np.float32(x[0, j * m + pick[j, c], c] * s[c])
    mean = x.reshape(1, 2, m, C).astype(np.float64).mean(axis=2)[..., C // 2:]
    np.testing.assert_array_equal(got[..., C // 2:], mean.astype(np.float32) * s[C // 2:])


def test_channel_logits_permute_with_channels(oracle_mod):
    """Channels do not interact (no RoPE): permuting the channels of x, z and
    s permutes the output the same way."""
    rng = np.random.default_rng(31)
    m, T, C = 4, 40, 96
    x = rng.standard_normal((1, T, C)).astype(np.float32)
    z = rng.standard_normal((1, T, C)).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    perm = rng.permutation(C)
    a = oracle_mod.compress(x, z, s, m, 0)
    b = oracle_mod.compress(x[..., perm], z[..., perm], s[perm], m, 0)
    np.testing.assert_array_equal(b, a[..., perm])


@pytest.mark.parametrize("m", [4, 128])
def test_channel_logits_match_fp64(oracle_mod, m):
    """Against an fp64 per-channel softmax-weighted sum, within the rounding
    bound of the fp32 sequence."""
    rng = np.random.default_rng(32 + m)
    T, C = 6 * m, 64
    x = rng.standard_normal((2, T, C)).astype(np.float32)
    z = (rng.standard_normal((2, T, C)) * 2).astype(np.float32)
    s = rng.uniform(0.5, 1.5, C).astype(np.float32)
    got = oracle_mod.compress(x, z, s, m, 0).astype(np.float64)
    zz = z.reshape(2, -1, m, C).astype(np.float64)
    a = np.exp(zz - zz.max(2, keepdims=True))
    a /= a.sum(2, keepdims=True)
    xx = x.reshape(2, -1, m, C).astype(np.float64)
    ref = (a * xx).sum(2) * s
    bound = ((a * np.abs(xx)).sum(2) * s) * (m + 8) * 2.0 ** -23
    assert np.all(np.abs(got - ref) <= bound)
