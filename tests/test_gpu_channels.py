"""GPU parity of sa_compress_channels, the compressor variant with one pooling
logit per raw token and channel, against the oracle's definition.

Every pooled row is within one unit in the last place of the storage type
plus the fp32 evaluation bound of the oracle's float64 value (the bound of
the per-token pooling: the weights of one channel sum to 1 as there); rows
outside the closed blocks are untouched.  Cases: decode (one block per
sequence, some sequences closing none, ring rows wrapping), the HCA block
size m' = 128, a prefill chunk pooling every block, f32 storage, equal logits
across channels (which reduce it to the per-token pooling), and a block range
that overflows the cache.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host
from test_gpu_parity import check_cache, pool_bound

pytestmark = pytest.mark.gpu


def sa():
    import sparse_attention_27_b300 as m
    return m


def run(store, B, R, d, m, N_cap, lo, hi, seed=11, z=None):
    x = synth.normal(seed, "xch", (B, R, d), store)
    if z is None:
        z = synth.normal(seed, "zch", (B, R, d), "f32")
    x_c = synth.normal(seed, "xch_c", (B, N_cap, d), store)        # prior cache contents
    code = sa().SA_BF16 if store == "bf16" else sa().SA_F32
    xc_d = dev(x_c)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    max_blocks = int(max(1, (hi - lo).max()))
    sa().sa_compress_channels(code, B, d, m, dev(x), dev(z), R, dev(lo), dev(hi), max_blocks, xc_d,
                              N_cap, err=err)
    torch.cuda.synchronize()
    return x, z, x_c, host(xc_d), int(err.item())


def check(store, x, z, x_c, got, m, lo, hi):
    B = x.shape[0]
    for b in range(B):
        l, h = int(lo[b]), int(hi[b])
        if h > l:
            ref = oracle.compress_channels(x[b], z[b], m, l, h, store)
            check_cache(got[b, l:h], ref, store, f"seq {b}", pool_bound(x[b], m, l, h))
        keep = np.ones(got.shape[1], dtype=bool)
        keep[l:h] = False
        np.testing.assert_array_equal(got[b, keep], x_c[b, keep])


@pytest.mark.parametrize("store", ["bf16", "f32"])
def test_decode_blocks_with_ring_wrap(store):
    """One block per sequence at positions whose rows wrap around the ring;
    one sequence closes no block this step."""
    B, R, d, m, N_cap = 5, 64, 128, 4, 512
    hi = np.array([10, 100, 511, 17, 250], dtype=np.int32)
    lo = hi - np.array([1, 1, 1, 0, 1], dtype=np.int32)
    x, z, x_c, got, err = run(store, B, R, d, m, N_cap, lo, hi)
    assert err == 0
    check(store, x, z, x_c, got, m, lo, hi)


def test_hca_block_size_and_prefill_chunk():
    B, R, d = 2, 1024, 128
    lo = np.array([3, 0], dtype=np.int32)
    hi = np.array([4, 8], dtype=np.int32)                   # m' = 128: one block, then eight
    x, z, x_c, got, err = run("bf16", B, R, d, 128, 8, lo, hi, seed=12)
    assert err == 0
    check("bf16", x, z, x_c, got, 128, lo, hi)
    R, m = 4096, 4                                          # a prefill chunk: every block
    lo = np.array([0], dtype=np.int32)
    hi = np.array([R // m], dtype=np.int32)
    x, z, x_c, got, err = run("bf16", 1, R, 64, m, R // m, lo, hi, seed=13)
    assert err == 0
    check("bf16", x, z, x_c, got, m, lo, hi)


def test_equal_logits_give_the_per_token_pooling():
    """Logits equal across channels: within the same bound of the per-token
    oracle, as csa_compress's rows are."""
    B, R, d, m = 3, 64, 128, 4
    zt = synth.normal(14, "zt", (B, R), "f32")
    z = np.repeat(zt[:, :, None], d, axis=2).astype(np.float32)
    hi = np.array([5, 9, 16], dtype=np.int32)
    lo = hi - 1
    x, _, x_c, got, err = run("bf16", B, R, d, m, 64, lo, hi, seed=14, z=z)
    assert err == 0
    for b in range(B):
        ref = oracle.compress(x[b], zt[b], m, int(lo[b]), int(hi[b]), "bf16")
        check_cache(got[b, lo[b]:hi[b]], ref, "bf16", f"seq {b}",
                    pool_bound(x[b], m, int(lo[b]), int(hi[b])))


def test_block_outside_the_cache_is_reported_and_skipped():
    B, R, d, m, N_cap = 2, 64, 64, 4, 8
    lo = np.array([7, 8], dtype=np.int32)                    # sequence 1's block 8 >= N_cap
    hi = np.array([8, 9], dtype=np.int32)
    x, z, x_c, got, err = run("bf16", B, R, d, m, N_cap, lo, hi, seed=15)
    assert err == 1 << sa().SA_ERR_BOUNDS
    check("bf16", x[:1], z[:1], x_c[:1], got[:1], m, lo[:1], hi[:1])
    np.testing.assert_array_equal(got[1], x_c[1])
