"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs.

Stages are compared one kernel at a time.  Where a later stage needs an
intermediate, the oracle's intermediate is uploaded to the GPU (never the
other way round):
  * compression  -- GPU caches vs oracle caches (bf16: <= 1 ulp, >= 99.9% exact;
                    f32: 1e-6 relative);
  * scores       -- GPU scores from the oracle's compressed indexer keys vs
                    oracle scores: max_j |s - s_ref| / max_j |s_ref| <= 1e-4 per row;
  * top-k        -- bit-exact on the same fp32 score arrays (drawn by synth);
                    on GPU-computed scores, a valid top-k of the oracle scores
                    up to the score tolerance;
  * attention    -- GPU csa_attend fed the oracle's idx vs oracle O/LSE:
                    max abs 2e-2 (bf16 inputs, fp32 accumulation), 1e-5 (fp32);
  * HCA          -- same tolerances.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, make_step

pytestmark = pytest.mark.gpu

TOL_ATT = {"bf16": 2e-2, "f32": 1e-5}
TOL_SCORE = 1e-4


def sa():
    import sparse_attention_27_b300 as m
    return m


def exact_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Doubles that are bf16 values -> bf16 bit patterns (exact)."""
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def to_store(x: np.ndarray, store: str) -> np.ndarray:
    return exact_bf16_bits(x) if store == "bf16" else x.astype(np.float32)


def bf16_ulp_diff(a_bits: np.ndarray, b_f64: np.ndarray) -> np.ndarray:
    b_bits = exact_bf16_bits(b_f64).astype(np.int32)
    a = a_bits.astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b_bits & 0x8000, -(b_bits & 0x7FFF), b_bits)
    return np.abs(a - b)


def pool_bound(x_ring: np.ndarray, m: int, lo: int, hi: int) -> np.ndarray:
    """Error bound of an fp32 evaluation of a softmax-pooled block, per output
    element: (m + 3) * 2^-24 * max_i |x_i| (weights summing to 1, each with a
    few ulps of error, m fp32 multiply-adds)."""
    R = x_ring.shape[0]
    pos = np.arange(lo * m, hi * m) % R
    xb = oracle.to_f64(x_ring[pos]).reshape(hi - lo, m, -1)
    return (m + 3) * 2.0 ** -24 * np.abs(xb).max(axis=1)


def check_cache(gpu: np.ndarray, ref: np.ndarray, store: str, what: str, bound: np.ndarray):
    """GPU cache rows vs the oracle's (rounded to the storage type): within one
    unit of the storage type's last place plus the fp32 evaluation bound."""
    if store == "bf16":
        g = ((gpu.astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    else:
        g = gpu.astype(np.float64)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 23)
    err = np.abs(g - ref)
    ok = err <= ulp + bound
    assert ok.all(), f"{what}: worst excess {(err - ulp - bound).max()}"
    return float((err == 0).mean())


def check_scores(gpu: np.ndarray, ref: np.ndarray, nvis: np.ndarray):
    worst = 0.0
    for r in range(ref.shape[0]):
        n = int(nvis[r])
        if n == 0:
            continue
        den = np.abs(ref[r, :n]).max()
        err = np.abs(gpu[r, :n].astype(np.float64) - ref[r, :n]).max()
        worst = max(worst, err / den if den > 0 else err)
    assert worst <= TOL_SCORE, f"score rel err {worst}"
    return worst


def check_topk_valid(idx: np.ndarray, s_ref: np.ndarray, nvis: np.ndarray, k: int):
    """idx is a valid top-k of s_ref up to the score tolerance; returns recall
    against the oracle's exact selection."""
    ref_idx, _ = oracle.topk(s_ref, nvis, k)
    hits = tot = 0
    for r in range(idx.shape[0]):
        n = int(nvis[r]); take = min(k, n)
        sel = idx[r, :take]
        assert np.all(idx[r, take:] == -1)
        assert np.all(np.diff(sel) > 0) and (take == 0 or (sel[0] >= 0 and sel[-1] < n))
        if 0 < take < n:
            tol = TOL_SCORE * np.abs(s_ref[r, :n]).max()
            chosen = np.zeros(n, bool); chosen[sel] = True
            assert s_ref[r, :n][chosen].min() >= s_ref[r, :n][~chosen].max() - 2 * tol
        hits += len(np.intersect1d(sel, ref_idx[r, :take]))
        tot += take
    return hits / max(tot, 1)


def run_staged(w: synth.Workload, x: dict, rows=None):
    """Full GPU pass plus the staged comparisons; returns a dict of metrics."""
    torch.cuda.synchronize()
    step = make_step(w, x)
    D = step.D
    scores = torch.full((w.B, w.T, w.ncap), float("nan"), dtype=torch.float32, device="cuda")
    step.compress_csa()
    step.index_topk(scores_out=scores)
    step.attend_csa()
    step.hca()
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    rows = np.arange(w.B * w.T) if rows is None else np.asarray(rows)
    caches = oracle.compress_all(w, x)
    ref = oracle.reference(w, x, rows=rows, caches=caches)
    out = {}
    # --- compression: only the blocks compressed this pass
    istore = "f32" if w.indexer == "f32" else "bf16"
    exact = []
    for b in range(w.B):
        lo, hi = int(x["blk_lo"][b]), int(x["blk_hi"][b])
        if hi > lo:
            for name, raw, store in (("k_c", "k_raw", w.dtype), ("v_c", "v_raw", w.dtype),
                                     ("ik_c", "ik_raw", istore)):
                exact.append(check_cache(host(step.x[name][b, lo:hi]), caches[name][b, lo:hi],
                                         store, name, pool_bound(x[raw][b], w.m, lo, hi)))
        lo, hi = int(x["hblk_lo"][b]), int(x["hblk_hi"][b])
        if hi > lo:
            for name, raw in (("hk_c", "hk_raw"), ("hv_c", "hv_raw")):
                exact.append(check_cache(host(step.x[name][b, lo:hi]), caches[name][b, lo:hi],
                                         w.dtype, name, pool_bound(x[raw][b], w.m2, lo, hi)))
    out["cache_exact_frac"] = float(np.mean(exact)) if exact else 1.0
    # --- scores from the oracle's indexer keys (same inputs on both sides)
    step.x["ik_c"].copy_(dev(to_store(caches["ik_c"], istore)))
    scores2 = torch.full_like(scores, float("nan"))
    step.index_topk(scores_out=scores2)
    torch.cuda.synchronize()
    s_gpu = host(scores2.reshape(w.B * w.T, w.ncap)[torch.from_numpy(rows).cuda()])
    out["score_err"] = check_scores(s_gpu, ref["scores"], ref["nvis"])
    # --- top-k on GPU scores: valid w.r.t. oracle scores, recall vs oracle's selection
    idx_gpu = host(step.idx).reshape(w.B * w.T, w.k)[rows]
    out["recall"] = check_topk_valid(idx_gpu, ref["scores"], ref["nvis"], w.k)
    # --- attention fed the oracle's idx, caches restored to the GPU's own
    idx_ref_full = np.full((w.B * w.T, w.k), -1, dtype=np.int32)
    idx_ref_full[rows] = ref["idx"]
    step.attend_csa(idx=dev(idx_ref_full.reshape(w.B, w.T, w.k)))
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    o = host(step.o).reshape(w.B * w.T, w.H, w.d)[rows]
    lse = host(step.lse).reshape(w.B * w.T, w.H)[rows]
    tol = TOL_ATT[w.dtype]
    out["o_err"] = float(np.abs(o - ref["o"]).max())
    fin = np.isfinite(ref["lse"])
    assert np.array_equal(np.isfinite(lse), fin)
    out["lse_err"] = float(np.abs(lse[fin] - ref["lse"][fin]).max()) if fin.any() else 0.0
    assert out["o_err"] <= tol and out["lse_err"] <= tol, out
    ho = host(step.ho).reshape(w.B * w.T, w.H, w.d)[rows]
    hlse = host(step.hlse).reshape(w.B * w.T, w.H)[rows]
    out["ho_err"] = float(np.abs(ho - ref["ho"]).max())
    fin = np.isfinite(ref["hlse"])
    assert np.array_equal(np.isfinite(hlse), fin)
    out["hlse_err"] = float(np.abs(hlse[fin] - ref["hlse"][fin]).max()) if fin.any() else 0.0
    assert out["ho_err"] <= tol and out["hlse_err"] <= tol, out
    return out


# ---------------------------------------------------------------- small cases

def test_tiny_f32_full_path():
    w = synth.WORKLOADS["tiny"]
    r = run_staged(w, synth.make_inputs(w))
    assert r["recall"] >= 0.99, r


@pytest.mark.parametrize("L,B,k", [(20003, 3, 256), (8192, 2, 2048), (4100, 1, 64)])
def test_decode_bf16_small(L, B, k):
    w = synth.Workload("dec", "decode", B=B, L=L, T=1, R=128, k=k, x8=True)
    r = run_staged(w, synth.make_inputs(w))
    assert r["recall"] >= 0.99, r


@pytest.mark.parametrize("L,k,W", [(1000, 64, 128), (777, 100, 5), (520, 16, 0)])
def test_prefill_bf16_small(L, k, W):
    w = synth.Workload("pre", "prefill", B=1, L=L, T=L, k=k, W=W, x8=True)
    r = run_staged(w, synth.make_inputs(w))
    assert r["recall"] >= 0.98, r


def test_prefill_bf16_deep_pipeline():
    """A prefill chunk with enough query rows (3000 items a launch) for the
    attention kernel's deep shape (one CTA per SM, six K/V stages, four
    producer warps); raw key rows scaled by 2^band over 8 bands of position,
    so that the pooled key rows and the window rows of later queries carry
    larger logits and key lists cross rescale bands mid-item.  Every row is
    compared with the oracle."""
    w = synth.Workload("preD", "prefill", B=1, L=3000, T=3000, k=256, W=128, x8=True)
    x = synth.make_inputs(w)
    R = x["k_raw"].shape[1]
    for band in range(1, 8):
        rows = np.arange(band * R // 8, (band + 1) * R // 8)
        synth.scale_rows(x["k_raw"][0], rows, float(2 ** band), w.dtype)
    r = run_staged(w, x)
    assert r["recall"] >= 0.98, r


@pytest.mark.parametrize("H", [1, 16, 40])
def test_decode_bf16_fewer_heads(H):
    w = synth.Workload("decH", "decode", B=3, L=3000, T=1, R=128, H=H, k=300, W=100, m2=16)
    run_staged(w, synth.make_inputs(w))


def test_decode_bf16_logit_bands_force_rescales():
    """Compressed key rows are scaled by 2^band over 8 bands of cache index, so
    logits grow along every key list: an item whose tiles cross a band boundary
    from band 4 up must raise its running max by more than the online softmax's
    rescale threshold (32 log2 units) mid-item and rescale O.  The shape keeps
    items several tiles long (16 rows, 34 CSA tiles and 65 HCA tiles per row)."""
    w = synth.Workload("decB", "decode", B=16, L=65536, T=1, R=256, k=2048, W=128, m2=16)
    x = synth.make_inputs(w)
    for b in range(w.B):
        for band in range(1, 8):
            rows = np.arange(band * w.ncap // 8, (band + 1) * w.ncap // 8)
            synth.scale_rows(x["k_c"][b], rows, float(2 ** band), w.dtype)
            rows2 = np.arange(band * w.ncap2 // 8, (band + 1) * w.ncap2 // 8)
            synth.scale_rows(x["hk_c"][b], rows2, float(2 ** band), w.dtype)
    run_staged(w, x)


def test_decode_bf16_one_row_many_splits():
    """One query row: the HCA list (4375 rows + window, 71 tiles) is split one
    tile per CTA, 71 partials merged by merge_splits_kernel in one row; the
    staged check runs the CSA attention twice on one workspace.  Two runs
    agree exactly."""
    w = synth.Workload("dec1", "decode", B=1, L=70000, T=1, R=128, k=64, W=128, m2=16)
    x = synth.make_inputs(w)
    r1 = run_staged(w, x)
    r2 = run_staged(w, x)
    assert r1["o_err"] == r2["o_err"] and r1["ho_err"] == r2["ho_err"], (r1, r2)


def test_prefill_f32_multi_sequence_ragged():
    w = synth.Workload("pre32", "prefill", B=2, L=301, T=150, H=5, HI=3, dI=32, d=64, m=4, k=7,
                       W=9, m2=16, dtype="f32", indexer="f32")
    run_staged(w, synth.make_inputs(w))


# --------------------------------------------------------------- top-k exact

def _topk_case(kind: str, rows: int, ncap: int, seed: int):
    g = np.random.default_rng(seed)
    if kind == "ties":
        s = g.integers(0, 4, (rows, ncap)).astype(np.float32)
    elif kind == "negzero":
        s = np.where(g.random((rows, ncap)) < 0.5, np.float32(-0.0), np.float32(0.0))
        s[:, ::5] = 1.0
    elif kind == "relu":
        s = np.maximum(g.standard_normal((rows, ncap)), 0).astype(np.float32)
    elif kind == "wide":        # magnitudes over 60 decades, with infinities
        s = (g.standard_normal((rows, ncap)) * 10.0 ** g.uniform(-30, 30, (rows, ncap)))
        s = s.astype(np.float32)
        s[:, 3::97] = np.inf
        s[:, 5::89] = -np.inf
    else:
        s = g.standard_normal((rows, ncap)).astype(np.float32)
    return s


@pytest.mark.parametrize("kind", ["random", "ties", "negzero", "relu", "wide"])
@pytest.mark.parametrize("ncap,k", [(1024, 64), (32768, 2048), (262144, 2048), (5000, 4999),
                                    (16384, 2048), (12000, 1000)])
def test_topk_bit_exact_same_scores(kind, ncap, k):
    m = 4
    rows = 6
    s = _topk_case(kind, rows, ncap, ncap + k)
    # positions: n = ncap, ncap-1, k, k+1, k-1, 1
    nv = np.array([ncap, ncap - 1, min(k, ncap), min(k + 1, ncap), max(k - 1, 0), 1])
    q_pos = (nv * m - 1).astype(np.int32)
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa().csa_index_topk(sa().SA_F32, rows, 1, 1, 1, m, k, None, None, None, None, None, ncap,
                        dev(q_pos), idx, scores_in=dev(s), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want, bad = oracle.topk(s.astype(np.float64), nv, k)
    assert bad == 0
    np.testing.assert_array_equal(host(idx), want)


@pytest.mark.parametrize("kind", ["random", "ties", "wide"])
def test_topk_bit_exact_many_long_rows(kind):
    """More rows than fit one cluster per SM pair: one CTA per row of 20000."""
    m, rows, ncap, k = 4, 100, 20000, 2048
    s = _topk_case(kind, rows, ncap, 7)
    nv = np.random.default_rng(8).integers(k - 5, ncap + 1, rows)
    q_pos = (nv * m - 1).astype(np.int32)
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa().csa_index_topk(sa().SA_F32, rows, 1, 1, 1, m, k, None, None, None, None, None, ncap,
                        dev(q_pos), idx, scores_in=dev(s), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want, bad = oracle.topk(s.astype(np.float64), nv, k)
    assert bad == 0
    np.testing.assert_array_equal(host(idx), want)


def test_topk_nan_row_rejected():
    rows, ncap, k = 3, 4096, 100
    s = np.random.default_rng(1).standard_normal((rows, ncap)).astype(np.float32)
    s[1, 1234] = np.nan
    q_pos = np.full(rows, ncap * 4 - 1, dtype=np.int32)
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sa().csa_index_topk(sa().SA_F32, rows, 1, 1, 1, 4, k, None, None, None, None, None, ncap,
                        dev(q_pos), idx, scores_in=dev(s), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & (1 << sa().SA_ERR_NAN)
    got = host(idx)
    assert np.all(got[1] == -1)
    want, bad = oracle.topk(s.astype(np.float64), np.full(rows, ncap), k)
    np.testing.assert_array_equal(got[[0, 2]], want[[0, 2]])


# --------------------------------------------------------- merge and errors

def test_attn_merge_matches_oracle():
    g = np.random.default_rng(2)
    rows, d, n = 300, 128, 3
    O = g.standard_normal((n, rows, d)).astype(np.float32)
    L = (g.standard_normal((n, rows)) * 3).astype(np.float32)
    L[1, ::7] = -np.inf
    L[:, 5] = -np.inf
    o = torch.empty((rows, d), dtype=torch.float32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    sa().attn_merge([dev(O[i]) for i in range(n)], [dev(L[i]) for i in range(n)], o, lse)
    torch.cuda.synchronize()
    Om, Lm = oracle.merge(O.astype(np.float64), L.astype(np.float64))
    np.testing.assert_allclose(host(o), Om, atol=1e-5, rtol=1e-5)
    fin = np.isfinite(Lm)
    assert np.array_equal(np.isfinite(host(lse)), fin)
    np.testing.assert_allclose(host(lse)[fin], Lm[fin], atol=1e-5)
    assert np.all(host(o)[5] == 0)


def test_out_of_range_index_reported_not_faulted():
    w = synth.Workload("dec", "decode", B=2, L=4096, T=1, R=128, k=64)
    x = synth.make_inputs(w)
    step = make_step(w, x)
    bad = np.tile(np.arange(64, dtype=np.int32), (2, 1, 1))
    bad[0, 0, 3] = w.ncap + 5           # beyond the visible blocks
    bad[1, 0, 7] = -7                    # negative, not the -1 padding
    step.attend_csa(idx=dev(bad))
    torch.cuda.synchronize()
    assert step.device_errors() & (1 << sa().SA_ERR_BOUNDS)
    assert np.all(np.isfinite(host(step.o)))


def test_host_validation_rejects_bad_arguments():
    m = sa()
    with pytest.raises(m.SaError) as e:
        m.csa_compress(9, 9, 1, 128, 64, 4, None, None, None, None, 128, None, None, 1, None, None,
                       None, None, 10)
    assert e.value.status == m.SA_ERR_INVALID_ARG
    x = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.SaError):   # misaligned q
        m.csa_attend(m.SA_BF16, 1, 1, 64, 128, 4, 8, 8, 0.1, x[1:], x, x, x, 4, x, x, x, 8,
                     x, x)


def test_two_stream_schedule_matches_one_stream():
    """HybridStep.run_two_streams (the bench's schedule: the indexer split into a
    score call and a top-k call, the HCA layer on a second stream after the
    scores) gives bit-identical outputs to HybridStep.run on one stream."""
    w = synth.Workload("sched", "decode", B=8, L=20003, T=1, R=128, k=256, W=128, x8=True)
    x = synth.make_inputs(w)
    one = make_step(w, x)
    one.run()
    two = make_step(w, x)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    two.run_two_streams(s1, s2)
    torch.cuda.synchronize()
    assert one.device_errors() == 0 and two.device_errors() == 0
    for name in ("idx", "o", "lse", "ho", "hlse"):
        np.testing.assert_array_equal(host(getattr(two, name)), host(getattr(one, name)),
                                      err_msg=name)


# ----------------------------------------------------------- full-size cases

def test_decode128k_full_size():
    w = synth.WORKLOADS["decode128k"]
    r = run_staged(w, synth.make_inputs(w))
    assert r["recall"] >= 0.99, r


def test_decode1m_full_size():
    w = synth.WORKLOADS["decode1m"]
    r = run_staged(w, synth.make_inputs(w))
    assert r["recall"] >= 0.99, r


def test_prefill64k_full_size_sampled_rows():
    w = synth.WORKLOADS["prefill64k"]
    x = synth.make_inputs(w)
    g = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(w.T - 128, w.T),
                                     g.choice(w.T, 512, replace=False)]))
    r = run_staged(w, x, rows=rows)
    assert r["recall"] >= 0.99, r


@pytest.mark.parametrize("L,B,k,m2", [(20003, 3, 256, 128), (70000, 1, 64, 16)])
def test_bf16_output_is_the_rounded_f32_output(L, B, k, m2):
    """csa_attend and hca_compress_attend with a bf16 O: the same kernels and
    splits as with an f32 O, rounded to nearest-even at the store, so the
    bf16 output is bit-identical to the f32 output rounded to bf16, and
    within 2e-2 of the oracle (the second shape splits the HCA row over many
    CTAs, so the rounding happens in the split merge)."""
    w = synth.Workload("decO", "decode", B=B, L=L, T=1, R=128, k=k, m2=m2, x8=True)
    x = synth.make_inputs(w)
    f32 = make_step(w, x)
    f32.run()
    b16 = make_step(w, x, o_dtype="bf16")
    b16.run()
    torch.cuda.synchronize()
    assert f32.device_errors() == 0 and b16.device_errors() == 0
    np.testing.assert_array_equal(host(b16.idx), host(f32.idx))
    for name in ("o", "ho"):
        want = host(getattr(f32, name).to(torch.bfloat16))
        np.testing.assert_array_equal(host(getattr(b16, name)), want, err_msg=name)
    for name in ("lse", "hlse"):
        np.testing.assert_array_equal(host(getattr(b16, name)), host(getattr(f32, name)))
    ref = oracle.reference(w, x)
    same = [b for b in range(w.B) if np.array_equal(host(b16.idx)[b, 0], ref["idx"][b])]
    o = synth.bf16_bits_to_f32(host(b16.o)).reshape(ref["o"].shape).astype(np.float64)
    ho = synth.bf16_bits_to_f32(host(b16.ho)).reshape(ref["ho"].shape).astype(np.float64)
    if same:
        assert np.abs(o[same] - ref["o"][same]).max() <= TOL_ATT["bf16"]
    assert np.abs(ho - ref["ho"]).max() <= TOL_ATT["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_attend_ignores_minus_one_inside_the_selection(dtype):
    """A -1 inside the first min(k, n) slots of idx (a rejected row is all
    -1) names no key: csa_attend must leave it out of the softmax, as the
    oracle's key multiset does, on the tensor-core (bf16) and CUDA-core
    (f32) kernels alike.  Holes in every other row, a whole row of -1 in
    one."""
    # (fp32: no x8 rows, whose large logits are outside the 1e-5 regime of the
    # fp32 configuration)
    w = synth.Workload("holes", "decode", B=4, L=20003, T=1, R=128, k=256, x8=dtype == "bf16",
                       dtype=dtype, indexer=dtype)
    x = synth.make_inputs(w)
    ref = oracle.reference(w, x)
    idx = ref["idx"].copy()
    idx[0, ::3] = -1
    idx[2, 100:180] = -1
    idx[3, :] = -1
    step = make_step(w, x)
    step.compress_csa()
    step.attend_csa(idx=dev(idx.reshape(w.B, 1, w.k)))
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    caches = oracle.compress_all(w, x)
    keys, vals = zip(*[oracle.csa_keys(b, w.L - 1, idx[b], caches["k_c"], caches["v_c"],
                                       x["k_raw"], x["v_raw"], w.W) for b in range(w.B)])
    o_ref, lse_ref = oracle.attend(x["q"].reshape(w.B, w.H, w.d), list(keys), list(vals),
                                   w.sm_scale)
    o = host(step.o).reshape(w.B, w.H, w.d)
    lse = host(step.lse).reshape(w.B, w.H)
    tol = TOL_ATT[dtype]
    assert np.abs(o - o_ref).max() <= tol and np.abs(lse - lse_ref).max() <= tol
