"""Pins for the float64 oracle, against things other than itself: hand-worked
fixtures (tests/golden), a brute-force restatement in another formulation,
library routines the special cases reduce to (torch's bf16 conversion and
scaled-dot-product attention), and invariants of the definitions."""
import json
import os
import zlib

import numpy as np
import pytest
import torch

import bruteforce as bf
import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ rounding

def test_round_bf16_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),       # subnormals
        (rng.standard_normal(2000) * 3e38).astype(np.float32),        # near overflow
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0, 3.0e38], np.float32),
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to(x.astype(np.float64), "bf16")
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------- compress

def test_compress_golden():
    g = _gold("compress_block.json")
    x = np.array(g["x"], dtype=np.float64)
    z = np.array(g["z"])
    got = oracle.compress(x, z, g["m"], 0, 3, "f64")
    np.testing.assert_allclose(got, np.array(g["expected"]), atol=g["tolerance"], rtol=0)


@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_compress_vs_bruteforce(m):
    rng = np.random.default_rng(m)
    L, d = 64, 12
    x = rng.standard_normal((L, d))
    z = rng.standard_normal(L) * 3
    want = bf.pooling_matrix(L, m, z) @ x
    got = oracle.compress(x, z, m, 0, L // m, "f64")
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)


def test_compress_ring_and_range():
    # blocks [3, 7) of a ring of 16 rows holding positions 16..31 (p mod 16)
    rng = np.random.default_rng(3)
    m, R, d = 4, 16, 5
    pos_x = rng.standard_normal((64, d))
    pos_z = rng.standard_normal(64)
    ring_x = np.zeros((R, d)); ring_z = np.zeros(R)
    for p in range(16, 32):
        ring_x[p % R] = pos_x[p]; ring_z[p % R] = pos_z[p]
    got = oracle.compress(ring_x, ring_z, m, 4, 8, "f64")
    want = bf.pooling_matrix(64, m, pos_z)[4:8] @ pos_x
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=0)


def test_compress_invariants_and_rounding():
    rng = np.random.default_rng(4)
    m, d = 4, 64
    x = rng.standard_normal((4096, d)) * 5
    z = rng.standard_normal(4096) * 4
    c = oracle.compress(x, z, m, 0, 1024, "f64")
    xb = x.reshape(1024, m, d)
    assert np.all(c <= xb.max(axis=1) + 1e-12) and np.all(c >= xb.min(axis=1) - 1e-12)
    ones = oracle.compress(np.ones((4096, d)), z, m, 0, 1024, "f64")
    np.testing.assert_allclose(ones, 1.0, atol=1e-14)
    cb = oracle.compress(x, z, m, 0, 1024, "bf16")
    np.testing.assert_array_equal(cb, oracle.round_to(c, "bf16"))
    cf = oracle.compress(x, z, m, 0, 1024, "f32")
    np.testing.assert_array_equal(cf, c.astype(np.float32).astype(np.float64))


# -------------------------------------------------------------- scores

def test_scores_golden():
    g = _gold("index_scores.json")
    q = np.array(g["q"])[None]
    w = np.array(g["w"])[None]
    keys = np.array(g["keys"])[None]
    s = oracle.index_scores(q, w, keys, np.array([0]), np.array([4]))
    np.testing.assert_allclose(s[0], g["expected"], atol=g["tolerance"], rtol=0)
    idx, bad = oracle.topk(s, np.array([4]), 2)
    assert bad == 0 and idx[0].tolist() == g["topk2_expected"]


def test_scores_vs_bruteforce_and_causality():
    rng = np.random.default_rng(5)
    rows, HI, dI, n = 7, 5, 16, 40
    q = rng.standard_normal((rows, HI, dI))
    w = rng.random((rows, HI))
    ik = rng.standard_normal((1, n, dI))
    nvis = np.array([0, 1, 5, 17, 39, 40, 23])
    s = oracle.index_scores(q, w, ik, np.zeros(rows, np.int64), nvis)
    want = bf.scores(q, w, ik[0], nvis)
    fin = np.isfinite(want)
    np.testing.assert_array_equal(np.isfinite(s), fin)
    np.testing.assert_allclose(s[fin], want[fin], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- top-k

def _check_topk_invariants(s, nvis, k, idx):
    for r in range(s.shape[0]):
        n = int(nvis[r]); take = min(k, n)
        sel = idx[r][:take]
        assert np.all(idx[r][take:] == -1)
        assert np.all(np.diff(sel) > 0) and (take == 0 or (sel[0] >= 0 and sel[-1] < n))
        if 0 < take < n:
            chosen = np.zeros(n, bool); chosen[sel] = True
            lo = s[r, :n][chosen].min(); hi = s[r, :n][~chosen].max()
            assert lo >= hi
            # at the threshold the lowest indices win
            tie_sel = np.where(chosen & (s[r, :n] == lo))[0]
            tie_uns = np.where(~chosen & (s[r, :n] == lo))[0]
            if len(tie_sel) and len(tie_uns):
                assert tie_sel.max() < tie_uns.min()


@pytest.mark.parametrize("case", ["random", "ties", "zeros", "negzero", "short"])
def test_topk_vs_bruteforce(case):
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    rows, n, k = 9, 300, 37
    if case == "random":
        s = rng.standard_normal((rows, n))
    elif case == "ties":
        s = rng.integers(0, 4, (rows, n)).astype(np.float64)
    elif case == "zeros":
        s = np.where(rng.random((rows, n)) < 0.7, 0.0, rng.random((rows, n)))
    elif case == "negzero":
        s = np.where(rng.random((rows, n)) < 0.5, -0.0, 0.0)
        s[:, ::7] = 1.0
    else:
        s = rng.standard_normal((rows, n))
    nvis = rng.integers(0, n + 1, rows) if case == "short" else np.full(rows, n)
    nvis[0] = 0
    nvis[1] = min(nvis[1], k - 1)
    idx, bad = oracle.topk(s, nvis, k)
    assert bad == 0
    np.testing.assert_array_equal(idx, bf.topk(s, nvis, k))
    _check_topk_invariants(s, nvis, k, idx)


def test_topk_scale_invariance_and_nan():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 3, 8)); w = rng.random((4, 3))
    ik = rng.standard_normal((1, 50, 8)); nv = np.full(4, 50)
    s1 = oracle.index_scores(q, w, ik, np.zeros(4, np.int64), nv)
    s2 = oracle.index_scores(q, w * 7.5, ik, np.zeros(4, np.int64), nv)
    np.testing.assert_array_equal(oracle.topk(s1, nv, 10)[0], oracle.topk(s2, nv, 10)[0])
    s1[2, 5] = np.nan
    idx, bad = oracle.topk(s1, nv, 10)
    assert bad == 1 and np.all(idx[2] == -1)


# ----------------------------------------------------------- attention

def _sdpa(q, k, v, mask, scale):
    """torch scaled_dot_product_attention, fp64 CPU. q [rows,H,d], k/v [n,d]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]          # [1,H,rows,d]
    kt = torch.from_numpy(k)[None, None].expand(1, q.shape[1], -1, -1)
    vt = torch.from_numpy(v)[None, None].expand(1, q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask)[None, None], scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def _tiny(**kw):
    base = dict(mode="prefill", B=1, L=64, T=64, H=3, d=16, HI=2, dI=8, m=4, k=5, W=6, m2=8,
                dtype="f64", indexer="f64")
    base.update(kw)
    return synth.Workload("t", **base)


def test_csa_m1_full_topk_no_window_is_causal_mqa():
    w = _tiny(m=1, k=64, W=0)
    x = synth.make_inputs(w)
    r = oracle.reference(w, x)
    L = w.L
    q = x["q"].reshape(L, w.H, w.d).astype(np.float64)
    K = x["k_raw"][0].astype(np.float64); V = x["v_raw"][0].astype(np.float64)
    mask = np.tril(np.ones((L, L), bool))
    np.testing.assert_allclose(r["k_c"][0], K, atol=0)     # m=1 pooling weight is exactly 1
    np.testing.assert_allclose(r["o"], _sdpa(q, K, V, mask, w.sm_scale), atol=1e-12)


def test_hca_m1_no_window_is_dense_causal_attention():
    w = _tiny(m2=1, W=0)
    x = synth.make_inputs(w)
    r = oracle.reference(w, x)
    L = w.L
    q = x["q_hca"].reshape(L, w.H, w.d).astype(np.float64)
    K = x["hk_raw"][0].astype(np.float64); V = x["hv_raw"][0].astype(np.float64)
    mask = np.tril(np.ones((L, L), bool))
    np.testing.assert_allclose(r["ho"], _sdpa(q, K, V, mask, w.sm_scale), atol=1e-12)


def test_csa_k0_is_sliding_window_attention():
    w = _tiny(k=0, W=5)
    x = synth.make_inputs(w)
    r = oracle.reference(w, x)
    L = w.L
    q = x["q"].reshape(L, w.H, w.d).astype(np.float64)
    K = x["k_raw"][0].astype(np.float64); V = x["v_raw"][0].astype(np.float64)
    i = np.arange(L)
    mask = (i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - 5)
    np.testing.assert_allclose(r["o"], _sdpa(q, K, V, mask, w.sm_scale), atol=1e-12)


@pytest.mark.parametrize("m,m2,k,W", [(4, 8, 5, 6), (2, 16, 3, 1), (4, 8, 100, 0), (1, 1, 1, 5)])
def test_path_vs_bruteforce(m, m2, k, W):
    w = _tiny(m=m, m2=m2, k=k, W=W, L=48, T=48)
    x = synth.make_inputs(w)
    r = oracle.reference(w, x)
    t = x["q_pos"][0]
    X, V, Ik, z = (x[n][0].astype(np.float64) for n in ("k_raw", "v_raw", "ik_raw", "z"))
    q = x["q"][0].astype(np.float64); qI = x["q_idx"][0].astype(np.float64)
    wI = x["w_idx"][0].astype(np.float64)
    Kc, Vc, IkC, s, idx, O, lse = bf.csa(q, qI, wI, t, X, V, Ik, z, m, k, W, w.sm_scale)
    np.testing.assert_allclose(r["k_c"][0], Kc, atol=1e-12)
    np.testing.assert_allclose(r["ik_c"][0], IkC, atol=1e-12)
    fin = np.isfinite(s)
    np.testing.assert_allclose(r["scores"][fin], s[fin], rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(r["idx"], idx)
    np.testing.assert_allclose(r["o"], O, atol=1e-12)
    np.testing.assert_allclose(r["lse"], lse, atol=1e-12)
    hq = x["q_hca"][0].astype(np.float64)
    hX, hV, hz = (x[n][0].astype(np.float64) for n in ("hk_raw", "hv_raw", "hz"))
    hKc, hVc, hO, hlse = bf.hca(hq, t, hX, hV, hz, m2, W, w.sm_scale)
    np.testing.assert_allclose(r["hk_c"][0], hKc, atol=1e-12)
    np.testing.assert_allclose(r["ho"], hO, atol=1e-12)
    np.testing.assert_allclose(r["hlse"], hlse, atol=1e-12)
    # empty key set (first positions with W=0 and no complete block) -> O=0, LSE=-inf
    if W == 0:
        assert np.all(r["lse"][0] == -np.inf) and np.all(r["o"][0] == 0)


def test_attention_output_in_value_range():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((5, 4, 16))
    keys = [rng.standard_normal((n, 16)) * 3 for n in (1, 2, 17, 100, 9)]
    vals = [rng.standard_normal((n, 16)) for n in (1, 2, 17, 100, 9)]
    O, lse = oracle.attend(q, keys, vals, 0.25)
    for r in range(5):
        assert np.all(O[r] <= vals[r].max(0) + 1e-12) and np.all(O[r] >= vals[r].min(0) - 1e-12)
    np.testing.assert_allclose(O[0], np.broadcast_to(vals[0][0], (4, 16)), atol=1e-15)


# --------------------------------------------------------------- merge

def test_merge_split_invariance_and_identity():
    rng = np.random.default_rng(9)
    H, d, n = 4, 16, 60
    q = rng.standard_normal((1, H, d))
    K = rng.standard_normal((n, d)); V = rng.standard_normal((n, d))
    O, lse = oracle.attend(q, [K], [V], 0.3)
    cuts = [0, 7, 8, 33, 60]
    Ops, lps = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.attend(q, [K[a:b]], [V[a:b]], 0.3)
        Ops.append(o.reshape(H, d)); lps.append(l.reshape(H))
    Ops.append(np.zeros((H, d))); lps.append(np.full(H, -np.inf))   # empty part
    Om, lm = oracle.merge(np.stack(Ops), np.stack(lps))
    np.testing.assert_allclose(Om, O.reshape(H, d), atol=1e-13)
    np.testing.assert_allclose(lm, lse.reshape(H), atol=1e-13)
    Oe, le = oracle.merge(np.zeros((2, 3, d)), np.full((2, 3), -np.inf))
    assert np.all(Oe == 0) and np.all(le == -np.inf)


# --------------------------------------------------------------- MXFP4

def test_mxfp4_golden():
    g = _gold("mxfp4_blocks.json")
    x = np.array(g["blocks"], dtype=np.float64)
    codes, scales = oracle.mxfp4_quantize(x)
    assert scales.reshape(-1).tolist() == g["expected_scales"]
    assert codes.tolist() == g["expected_codes"]


def test_mxfp4_grid_roundtrip():
    rng = np.random.default_rng(10)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    x = grid[rng.integers(0, 8, (200, 32))] * np.where(rng.random((200, 32)) < .5, -1, 1)
    x[:, 0] = 6.0                                   # amax 6 -> exponent 0 before scaling
    e = rng.integers(-20, 20, 200)
    x = x * np.exp2(e)[:, None]
    codes, scales = oracle.mxfp4_quantize(x)
    np.testing.assert_array_equal(scales[:, 0].astype(int) - 127, e)
    np.testing.assert_array_equal(oracle.mxfp4_dequantize(codes, scales), x)


def test_mxfp4_error_bound():
    # |x - deq(q(x))| <= half the e2m1 spacing at the element's magnitude, or saturation error
    rng = np.random.default_rng(11)
    x = rng.standard_normal((500, 64))
    codes, scales = oracle.mxfp4_quantize(x)
    y = oracle.mxfp4_dequantize(codes, scales)
    e = (scales.astype(int) - 127).repeat(32, axis=1)
    u = np.abs(x) / np.exp2(e)
    assert np.all(u < 8)                           # amax / 2^e < 8 by the scale rule
    spacing = np.where(u < 2, 0.5, np.where(u < 4, 1.0, 2.0))
    err = np.abs(x - y) / np.exp2(e)
    assert np.all(err <= np.maximum(spacing / 2, u - 6) + 1e-12)


def test_mxfp4_row_exponent_spread_of_the_128k_draws():
    """The MXFP4 kernel folds each block's scale into e4m3 as 2^(e_b - e_row),
    e_row the larger of the row's two block exponents; that is exact while
    e_row - e_b <= 8 (e4m3's smallest subnormal is 2^-9).  On the 128K decode
    workload's own indexer draws (keys and queries; the x8 rows scale a whole
    row and leave the spread unchanged) no row is beyond that, so the kernel's
    only rounding there is its fp32 accumulation."""
    w = synth.WORKLOADS["mxfp4"]
    worst = 0
    for name, shape in (("ik_c", (w.B, w.ncap, w.dI)), ("q_idx", (w.B, w.T, w.HI, w.dI))):
        x = synth.normal(w.seed, name, shape, "bf16").reshape(-1, 2048, w.dI)
        for chunk in x:
            _, scales = oracle.mxfp4_quantize(chunk)
            e = scales.astype(int).reshape(-1, w.dI // 32)
            worst = max(worst, int((e.max(axis=1) - e.min(axis=1)).max()))
    print(f"largest block-exponent spread within a row: {worst}")
    assert worst <= 8


def test_e2m1_grid_scaled_down_is_exact_in_e4m3_up_to_shift_8():
    """The bound behind the MXFP4 -> FP8 fold: every e2m1 value times 2^-s is
    an e4m3 value for s = 0..8, and not every one is at s = 9.  e4m3 as in the
    OCP 8-bit floating point spec: bias 7, three mantissa bits, subnormals at
    exponent field 0, no infinities, S.1111.111 the only NaNs; enumerated from
    all 256 codes."""
    vals = set()
    for b in range(256):
        sign = -1.0 if b & 0x80 else 1.0
        e, m = (b >> 3) & 0xF, b & 7
        if e == 15 and m == 7:
            continue                                     # NaN
        v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.add(sign * v)
    assert max(vals) == 448.0 and min(v for v in vals if v > 0) == 2.0 ** -9
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for s in range(9):
        for c in grid:
            assert c * 2.0 ** -s in vals and -c * 2.0 ** -s in vals, (c, s)
    assert 0.5 * 2.0 ** -9 not in vals                   # first loss at s = 9
