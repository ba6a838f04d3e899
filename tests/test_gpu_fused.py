"""GPU parity of csa_decode, the CSA layer of one decode step in one launch,
through the C ABI.

csa_decode must give the results of the three calls it fuses (csa_compress,
csa_index_topk, csa_attend) on the same inputs:
  * the cache rows it pools are bit-identical to csa_compress's (the same
    fp32 evaluation order), and every other cache row is untouched;
  * idx is bit-identical to csa_index_topk's (the same scores, the same
    exact top-k), which the staged tests check against the oracle;
  * idx is a valid top-k of the float64 oracle's scores, and equal to the
    oracle's selection on inputs whose scores fp32 computes exactly;
  * O and LSE are within 2e-2 (bf16 inputs, fp32 accumulation) of the
    oracle's on every row whose selection equals the oracle's (all rows on
    the exact-score inputs).
Shapes cover several tiles per CTA with a ragged last tile, rows whose
visible entries are all selected (n <= k), rows where no block closes, very
early positions (no compressed entry, a short window), k = 0 (window only),
fewer heads than the MMA's 64, a NaN row, rows whose k-th largest score
falls outside the top-k's relative bin window, and the full 128K and 1M
decode workloads.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_inputs import exact_scores
from gpu_util import host, make_step
from test_gpu_parity import check_topk_valid

pytestmark = pytest.mark.gpu
TOL = 2e-2


def sa():
    import sparse_attention_27_b300 as m
    return m


def run_both(w, x, o_dtype="f32"):
    """(unfused step, fused step) after one pass each on the same inputs."""
    ref = make_step(w, x, o_dtype=o_dtype)
    ref.csa()
    fus = make_step(w, x, o_dtype=o_dtype)
    assert fus.fused_ok()
    fus.csa_fused()
    torch.cuda.synchronize()
    return ref, fus


def check_fused(w, x, expect_err=0, o_dtype="f32", exact=False):
    """csa_decode against the three calls (caches and idx bit-identical) and
    against the oracle: idx a valid top-k of the oracle's scores (equal to
    the oracle's selection when the scores are exact), O and LSE within the
    tolerance on every row whose selection equals the oracle's."""
    ref, fus = run_both(w, x, o_dtype)
    assert ref.device_errors() == expect_err and fus.device_errors() == expect_err, (
        ref.device_errors(), fus.device_errors())
    for name in ("k_c", "v_c", "ik_c"):
        np.testing.assert_array_equal(host(fus.x[name]), host(ref.x[name]), err_msg=name)
    idx = host(fus.idx).reshape(w.B, w.k)
    np.testing.assert_array_equal(idx, host(ref.idx).reshape(w.B, w.k))
    orc = oracle.reference(w, x)
    same = np.array([np.array_equal(idx[b], orc["idx"][b]) for b in range(w.B)])
    if exact:
        assert same.all(), np.nonzero(~same)
    else:
        nan_rows = np.array([np.isnan(orc["scores"][b]).any() for b in range(w.B)])
        ok = ~nan_rows
        if ok.any() and w.k > 0:
            rec = check_topk_valid(idx[ok], orc["scores"][ok], orc["nvis"][ok], w.k)
            assert rec >= 0.99, rec
    o = host(fus.o)
    if o.dtype == np.uint16:
        o = synth.bf16_bits_to_f32(o)
    o = o.reshape(w.B, w.H, w.d).astype(np.float64)
    lse = host(fus.lse).reshape(w.B, w.H)
    rows = np.nonzero(same)[0]
    assert len(rows) > 0
    fin = np.isfinite(orc["lse"][rows])
    assert np.array_equal(np.isfinite(lse[rows]), fin)
    err_o = float(np.abs(o[rows] - orc["o"][rows]).max())
    err_l = float(np.abs(lse[rows][fin] - orc["lse"][rows][fin]).max()) if fin.any() else 0.0
    assert err_o <= TOL and err_l <= TOL, (err_o, err_l)
    return dict(o_err=err_o, lse_err=err_l, idx=idx, rows_compared=len(rows))


@pytest.mark.parametrize("L,B,k", [(20003, 3, 256), (8192, 8, 2048), (4100, 2, 64),
                                   (70000, 1, 64), (60003, 5, 1000)])
def test_fused_decode_matches_the_three_calls(L, B, k):
    w = synth.Workload("fdec", "decode", B=B, L=L, T=1, R=128, k=k, x8=True)
    x = synth.make_inputs(w)
    check_fused(w, x)
    check_fused(w, exact_scores(w, x), exact=True)


def test_fused_decode_mixed_positions_and_closing_blocks():
    """Each sequence at its own position: some close a block this step, some
    do not (empty block range), some are so early that no compressed entry is
    visible and the window is short."""
    w = synth.Workload("fmix", "decode", B=8, L=12000, T=1, R=128, k=256, x8=True)
    x = synth.make_inputs(w)
    pos = np.array([11999, 11998, 3, 0, 1024 * 4 - 1, 1024 * 4, 2, 6003], dtype=np.int32)
    x["q_pos"] = pos.reshape(w.B, 1)
    closes = (pos + 1) % w.m == 0
    x["blk_hi"] = ((pos + 1) // w.m).astype(np.int32)
    x["blk_lo"] = (x["blk_hi"] - closes).astype(np.int32)
    x["hblk_hi"] = ((pos + 1) // w.m2).astype(np.int32)
    x["hblk_lo"] = x["hblk_hi"].copy()
    check_fused(w, x)
    check_fused(w, exact_scores(w, x), exact=True)


def test_fused_decode_window_only_and_fewer_heads():
    w = synth.Workload("fwin", "decode", B=3, L=3000, T=1, R=128, H=40, k=0, W=100)
    check_fused(w, synth.make_inputs(w))
    w2 = synth.Workload("fh", "decode", B=4, L=9001, T=1, R=256, H=16, k=300, W=200)
    check_fused(w2, synth.make_inputs(w2), o_dtype="bf16")


def test_fused_decode_nan_row_rejected_like_the_three_calls():
    """A NaN head weight in one sequence makes every score of that row NaN
    (a NaN indexer query would not: the ReLU maps a NaN product to 0): both
    paths reject that row (idx all -1, SA_ERR_NAN) and attend its window only;
    the other rows are unaffected."""
    w = synth.Workload("fnan", "decode", B=3, L=20003, T=1, R=128, k=256, x8=True)
    x = synth.make_inputs(w)
    x["w_idx"] = x["w_idx"].copy()
    x["w_idx"][1, 0, 5] = np.nan
    r = check_fused(w, x, expect_err=1 << sa().SA_ERR_NAN)
    assert np.all(r["idx"][1] == -1) and np.all(r["idx"][[0, 2]] >= 0)


@pytest.mark.parametrize("case", ["sample_far_above", "top_bin_lists", "top_bin_overflow"])
def test_fused_topk_relative_bins_end_bins(case):
    """The fused top-k bins keys relative to the largest key of each CTA's
    first score tile (1024 bins per octave, 6 octaves below that sample to 2
    above); keys outside the window share an end bin, which the exact select
    handles without the bins' shared prefix.  Indexer key rows scaled by 2^10
    put the k-th largest key there: in the bottom bin (a few huge rows in the
    sampled tiles, k past them: the bin overflows the lists, cluster-wide
    radix passes), in the top bin with ~3000 keys (listed, exact select over
    the union) and with ~5000 (overflow).  idx must stay bit-identical to
    csa_index_topk's and a valid top-k of the oracle's scores."""
    w = synth.Workload("frel", "decode", B=4, L=65536, T=1, R=128,
                       k=256 if case == "sample_far_above" else 2048, x8=True)
    x = synth.make_inputs(w)
    g = np.random.default_rng(5)
    tiles = w.ncap // 128
    for b in range(w.B):
        if case == "sample_far_above":          # 4 rows in every 8th tile (each CTA's first)
            rows = np.concatenate([t * 128 + g.choice(128, 4, replace=False)
                                   for t in range(0, tiles, 8)])
        else:                                   # rows outside every 8th tile
            cand = np.array([j for j in range(w.ncap - 8) if (j // 128) % 8 != 0])
            rows = g.choice(cand, 3000 if case == "top_bin_lists" else 5000, replace=False)
        synth.scale_rows(x["ik_c"][b], np.sort(rows), 1024.0, "bf16")
    check_fused(w, x)


@pytest.mark.parametrize("name", ["decode128k", "decode1m"])
def test_fused_decode_full_size(name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    check_fused(w, x, o_dtype="bf16")
    check_fused(w, exact_scores(w, x), o_dtype="bf16", exact=True)


def test_fused_decode_host_validation():
    m = sa()
    x = torch.empty(4096, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(8, dtype=torch.int32, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    args = dict(q=x, q_idx=x, w=f, q_pos=i, k_raw=x, v_raw=x, ik_raw=x, z=f, R=128, blk_lo=i,
                blk_hi=i, max_blocks=1, k_c=x, v_c=x, ik_c=x, N_cap=16, idx=i, o=x, lse=f)
    with pytest.raises(m.SaError) as e:        # head dim 64: not this kernel's shape
        m.csa_decode(1, 64, 64, 64, 64, 4, 8, 16, 0.1, **args)
    assert e.value.status == m.SA_ERR_UNSUPPORTED
    with pytest.raises(m.SaError) as e:        # misaligned queries
        m.csa_decode(1, 64, 128, 64, 64, 4, 8, 16, 0.1, **dict(args, q=x[1:]))
    assert e.value.status == m.SA_ERR_INVALID_ARG
    with pytest.raises(m.SaError) as e:        # window longer than the ring
        m.csa_decode(1, 64, 128, 64, 64, 4, 8, 200, 0.1, **args)
    assert e.value.status == m.SA_ERR_INVALID_ARG
