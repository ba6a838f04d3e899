"""Pins of the oracle's per-channel pooling (CPU only).

The compressor variant with one logit per raw token and channel ("DeepSeek-V4
논문 읽기: 백만 토큰 컨텍스트를 저렴하게", section "Compressed Sparse Attention (CSA)"
step 1: m consecutive entries merged into one; the merge weights here are a
softmax over the block's tokens taken separately for every channel).  Pinned
to things other than itself:
  * logits equal across channels reduce it to the per-token pooling, bit for
    bit (the same float64 operations in the same order);
  * a brute force in another formulation (scipy's softmax over the token axis
    of a [m, d] block, then a column sum);
  * closed forms: m = 1 is the identity; adding a per-channel constant to a
    block's logits changes nothing; every output lies between its channel's
    smallest and largest input; one dominant logit picks its token's value.
A transposed softmax (over channels instead of tokens), a dropped max shift
or a wrong row index fails one of them.
"""
from __future__ import annotations

import numpy as np
from scipy.special import softmax

import oracle


def draw(seed: int, R: int, d: int):
    g = np.random.default_rng(seed)
    x = g.standard_normal((R, d)).astype(np.float32)
    z = g.standard_normal((R, d))
    return x, z


def test_equal_logits_reduce_to_the_per_token_pooling():
    x, zt = draw(1, 64, 24)[0], np.random.default_rng(2).standard_normal(64)
    z = np.repeat(zt[:, None], 24, axis=1)
    for m in (1, 3, 4, 8, 16):
        nb = 64 // m
        got = oracle.compress_channels(x, z, m, 0, nb, "f64")
        want = oracle.compress(x, zt, m, 0, nb, "f64")
        np.testing.assert_array_equal(got, want)


def test_matches_a_brute_force_softmax_over_tokens():
    R, d = 96, 16
    x, z = draw(3, R, d)
    for m, lo, hi in ((4, 0, 24), (8, 2, 9), (128 // 8, 1, 5)):
        got = oracle.compress_channels(x, z, m, lo, hi, "f64")
        for j in range(lo, hi):
            rows = np.arange(j * m, (j + 1) * m) % R
            w = softmax(z[rows], axis=0)                   # [m, d]: over tokens, per channel
            want = (w * x[rows].astype(np.float64)).sum(axis=0)
            np.testing.assert_allclose(got[j - lo], want, rtol=1e-13, atol=1e-15)


def test_ring_rows_wrap_modulo_R():
    """Block j reads raw positions j*m .. j*m+m-1 from ring rows p mod R."""
    R, d, m = 32, 8, 4
    x, z = draw(4, R, d)
    j = 11                                                 # positions 44..47 -> rows 12..15
    got = oracle.compress_channels(x, z, m, j, j + 1, "f64")
    want = oracle.compress_channels(x[12:16], z[12:16], m, 0, 1, "f64")
    np.testing.assert_array_equal(got, want)


def test_closed_forms():
    R, d = 64, 12
    x, z = draw(5, R, d)
    xd = x.astype(np.float64)
    # m = 1: each block is one token with weight 1
    np.testing.assert_array_equal(oracle.compress_channels(x, z, 1, 0, R, "f64"), xd)
    # shift invariance: a per-channel constant added to every logit of a block
    m = 8
    z2 = z + np.linspace(-3.0, 5.0, d)[None, :]
    np.testing.assert_allclose(oracle.compress_channels(x, z2, m, 0, R // m, "f64"),
                               oracle.compress_channels(x, z, m, 0, R // m, "f64"),
                               rtol=1e-13, atol=1e-15)
    # convex combination: each output within its channel's block range
    out = oracle.compress_channels(x, z, m, 0, R // m, "f64")
    blocks = xd.reshape(R // m, m, d)
    assert np.all(out >= blocks.min(axis=1) - 1e-15) and np.all(out <= blocks.max(axis=1) + 1e-15)
    # one dominant logit per channel picks that token's value
    zd = np.zeros((R, d))
    pick = np.arange(d) % m
    for c in range(d):
        zd[pick[c]::m, c] = 800.0
    out = oracle.compress_channels(x, zd, m, 0, R // m, "f64")
    np.testing.assert_allclose(out, blocks[:, pick, np.arange(d)], rtol=0, atol=1e-300)


def test_storage_rounding_matches_the_per_token_call():
    """The f32 and bf16 roundings are the per-token pooling's (same helper
    semantics): equal logits give equal stored values."""
    x, zt = draw(6, 32, 8)[0], np.random.default_rng(7).standard_normal(32)
    z = np.repeat(zt[:, None], 8, axis=1)
    for store in ("f32", "bf16"):
        np.testing.assert_array_equal(oracle.compress_channels(x, z, 4, 0, 8, store),
                                      oracle.compress(x, zt, 4, 0, 8, store))
