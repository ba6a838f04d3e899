"""GPU parity of sa_decode_step, both layers of one decode step in one
persistent launch, through the C ABI.

sa_decode_step must give the results of the separate calls (csa_compress,
csa_index_topk, csa_attend, hca_compress_attend) on the same inputs:
  * every cache row it pools (CSA K, V, indexer key; HCA K, V) is
    bit-identical to the separate calls' (the same fp32 evaluation order),
    and every other cache row is untouched;
  * idx is bit-identical to csa_index_topk's (the same scores, the same
    exact top-k), and equal to the float64 oracle's selection on inputs whose
    scores fp32 computes exactly (tests/exact_inputs.py);
  * O, LSE (CSA) and HO, HLSE (HCA) are within 2e-2 (bf16 inputs, fp32
    accumulation) of the oracle's on every row whose selection equals the
    oracle's.
Shapes cover several score items per row with a ragged last tile, rows whose
visible entries are all selected (n <= k), rows where no block closes, very
early positions (no compressed entry, a short window), k = 0 (window only),
fewer heads than the MMA's 64, a NaN row, a batch much larger than the SM
count (items of many rows in flight at once) and the full 128K decode.
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
CACHES = ("k_c", "v_c", "ik_c", "hk_c", "hv_c")


def sa():
    import sparse_attention_27_b300 as m
    return m


def run_both(w, x, o_dtype="f32"):
    """(separate calls, one sa_decode_step) after one pass each on the same
    inputs."""
    ref = make_step(w, x, o_dtype=o_dtype)
    ref.run()
    one = make_step(w, x, o_dtype=o_dtype)
    assert one.step_ok()
    one.decode_step()
    torch.cuda.synchronize()
    return ref, one


def as_f64(t):
    a = host(t)
    if a.dtype == np.uint16:
        a = synth.bf16_bits_to_f32(a)
    return a.astype(np.float64)


def check_step(w, x, expect_err=0, o_dtype="f32", exact=False):
    """sa_decode_step against the separate calls (caches and idx
    bit-identical) and against the oracle (idx a valid top-k of its scores,
    equal to its selection when the scores are exact; O, LSE, HO, HLSE within
    the tolerance on rows whose selection equals the oracle's)."""
    ref, one = run_both(w, x, o_dtype)
    assert ref.device_errors() == expect_err and one.device_errors() == expect_err, (
        ref.device_errors(), one.device_errors())
    for name in CACHES:
        np.testing.assert_array_equal(host(one.x[name]), host(ref.x[name]), err_msg=name)
    idx = host(one.idx).reshape(w.B, w.k)
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
    errs = {}
    for o_name, l_name, rows in (("o", "lse", np.nonzero(same)[0]),
                                 ("ho", "hlse", np.arange(w.B))):
        o = as_f64(getattr(one, o_name)).reshape(w.B, w.H, w.d)
        lse = host(getattr(one, l_name)).reshape(w.B, w.H)
        ro = orc[o_name].reshape(w.B, w.H, w.d)
        rl = orc[l_name].reshape(w.B, w.H)
        assert len(rows) > 0
        fin = np.isfinite(rl[rows])
        assert np.array_equal(np.isfinite(lse[rows]), fin), l_name
        err_o = float(np.abs(o[rows] - ro[rows]).max())
        err_l = float(np.abs(lse[rows][fin] - rl[rows][fin]).max()) if fin.any() else 0.0
        assert err_o <= TOL and err_l <= TOL, (o_name, err_o, err_l)
        errs[o_name] = (err_o, err_l)
    return dict(errs=errs, idx=idx)


@pytest.mark.parametrize("L,B,k", [(20003, 3, 256), (8192, 8, 2048), (4100, 2, 64),
                                   (70000, 1, 64), (60003, 5, 1000)])
def test_decode_step_matches_the_separate_calls(L, B, k):
    w = synth.Workload("sdec", "decode", B=B, L=L, T=1, R=128, k=k, x8=True)
    x = synth.make_inputs(w)
    check_step(w, x)
    check_step(w, exact_scores(w, x), exact=True)


def test_decode_step_mixed_positions_and_closing_blocks():
    """Each sequence at its own position: some close a CSA block this step,
    one closes an HCA block, some close none, some are so early that no
    compressed entry is visible and the window is short."""
    w = synth.Workload("smix", "decode", B=8, L=12000, T=1, R=128, k=256, x8=True)
    x = synth.make_inputs(w)
    pos = np.array([11999, 11998, 3, 0, 1024 * 4 - 1, 1024 * 4, 2, 6003], dtype=np.int32)
    x["q_pos"] = pos.reshape(w.B, 1)
    for lo, hi, m in (("blk_lo", "blk_hi", w.m), ("hblk_lo", "hblk_hi", w.m2)):
        closes = (pos + 1) % m == 0
        x[hi] = ((pos + 1) // m).astype(np.int32)
        x[lo] = (x[hi] - closes).astype(np.int32)
    check_step(w, x)
    check_step(w, exact_scores(w, x), exact=True)


def test_decode_step_window_only_and_fewer_heads():
    w = synth.Workload("swin", "decode", B=3, L=3000, T=1, R=128, H=40, k=0, W=100)
    check_step(w, synth.make_inputs(w))
    w2 = synth.Workload("sh", "decode", B=4, L=9001, T=1, R=256, H=16, k=300, W=200)
    check_step(w2, synth.make_inputs(w2), o_dtype="bf16")


def test_decode_step_many_rows_in_flight():
    """B = 300 sequences of 4096 tokens: far more items than SMs, so the
    top-k and attention of early rows run while later rows are scored."""
    w = synth.Workload("smany", "decode", B=300, L=4096, T=1, R=128, k=512, x8=True)
    x = synth.make_inputs(w)
    check_step(w, exact_scores(w, x), o_dtype="bf16", exact=True)


def test_decode_step_nan_row_rejected_like_the_separate_calls():
    """A NaN head weight in one sequence makes every score of that row NaN:
    both paths reject that row (idx all -1, SA_ERR_NAN) and attend its window
    only; the other rows and the HCA layer are unaffected."""
    w = synth.Workload("snan", "decode", B=3, L=20003, T=1, R=128, k=256, x8=True)
    x = synth.make_inputs(w)
    x["w_idx"] = x["w_idx"].copy()
    x["w_idx"][1, 0, 5] = np.nan
    r = check_step(w, x, expect_err=1 << sa().SA_ERR_NAN)
    assert np.all(r["idx"][1] == -1) and np.all(r["idx"][[0, 2]] >= 0)


def test_decode_step_full_size():
    w = synth.WORKLOADS["decode128k"]
    x = synth.make_inputs(w)
    check_step(w, x, o_dtype="bf16")
    check_step(w, exact_scores(w, x), o_dtype="bf16", exact=True)


def test_decode_step_repeated_calls_reuse_the_workspace():
    """Two calls on one workspace give the same results: the call zeroes its
    counters on the stream each time."""
    w = synth.Workload("srep", "decode", B=6, L=20000, T=1, R=128, k=512, x8=True)
    x = exact_scores(w, synth.make_inputs(w))
    one = make_step(w, x, o_dtype="bf16")
    one.decode_step()
    torch.cuda.synchronize()
    first = {n: host(getattr(one, n)).copy() for n in ("idx", "o", "lse", "ho", "hlse")}
    one.decode_step()
    torch.cuda.synchronize()
    assert one.device_errors() == 0
    for n, v in first.items():
        np.testing.assert_array_equal(host(getattr(one, n)), v, err_msg=n)


def test_decode_step_host_validation():
    m = sa()
    x = torch.empty(1 << 16, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(8, dtype=torch.int32, device="cuda")
    f = torch.zeros(256, dtype=torch.float32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    args = dict(q=x, q_idx=x, w=f, q_hca=x, q_pos=i, k_raw=x, v_raw=x, ik_raw=x, z=f, hk_raw=x,
                hv_raw=x, hz=f, R=128, blk_lo=i, blk_hi=i, max_blocks=1, hblk_lo=i, hblk_hi=i,
                max_blocks2=1, k_c=x, v_c=x, ik_c=x, N_cap=16, hk_c=x, hv_c=x, N2_cap=4, idx=i,
                o=x, lse=f, ho=x, hlse=f, ws=ws)
    with pytest.raises(m.SaError) as e:        # head dim 64: not this kernel's shape
        m.sa_decode_step(1, 64, 64, 64, 64, 4, 8, 16, 128, 0.1, **args)
    assert e.value.status == m.SA_ERR_UNSUPPORTED
    with pytest.raises(m.SaError) as e:        # rows longer than one CTA's key space
        m.sa_decode_step(1, 64, 128, 64, 64, 4, 8, 16, 128, 0.1, **dict(args, N_cap=40000))
    assert e.value.status == m.SA_ERR_UNSUPPORTED
    with pytest.raises(m.SaError) as e:        # misaligned queries
        m.sa_decode_step(1, 64, 128, 64, 64, 4, 8, 16, 128, 0.1, **dict(args, q=x[1:]))
    assert e.value.status == m.SA_ERR_INVALID_ARG
    with pytest.raises(m.SaError) as e:        # workspace too small
        m.sa_decode_step(1, 64, 128, 64, 64, 4, 8, 16, 128, 0.1, **dict(args, ws=ws[:256]))
    assert e.value.status == m.SA_ERR_INVALID_ARG
