"""GPU parity of the low-precision (MXFP4) indexer path against the float64
oracle.

Source: "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈", section "오픈소스 MoE 인프라:
MegaMoE와 TileLang" -- the indexer QK path is stored in FP4 (MXFP4) and
dequantised to FP8 without loss, with the top-k selector keeping 99.7% of the
KV entries.

* quantiser     -- the library's MXFP4 codes and scales are bit-exact with the
                   oracle's on the same bf16 values (integer results decided
                   from the same bf16 inputs by the same OCP MX rule);
* scores        -- GPU scores from the oracle's MXFP4 operands against the
                   oracle's double-precision scores of the dequantised values:
                   max_j |s - s_ref| / max_j |s_ref| per row (reported; gated
                   at the bf16 path's 1e-4 when the tensor core's fp8
                   accumulation allows it);
* top-k         -- a valid top-k of the oracle's MXFP4 scores up to that error;
* recall        -- against the oracle's selection from double-precision scores
                   of the unquantised bf16 operands: a property of 4-bit
                   rounding on this data, not of the kernel, so it is reported
                   with only a low alarm floor (0.75);
* attention     -- the CSA attention given the MXFP4 selection is unchanged
                   (2e-2 against the oracle on the same indices).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, make_step

pytestmark = pytest.mark.gpu

TOL_SCORE_MX = 1e-4


def sa():
    import sparse_attention_27_b300 as m
    return m


def _quantize_gpu(x_bits: np.ndarray):
    m = sa()
    x = dev(x_bits)
    codes = torch.empty(x.numel() // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.numel() // 32, dtype=torch.uint8, device="cuda")
    m.sa_mxfp4_quantize(x, codes, scales)
    torch.cuda.synchronize()
    return host(codes), host(scales)


def test_quantizer_bit_exact_on_draws_and_edges():
    g = np.random.default_rng(5)
    draws = synth.normal(0, "q_idx", (64, 64, 64), "bf16").reshape(-1)
    # hand-picked blocks: ties between grid points, saturation, tiny, zero, -0
    edge = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.1, -6, 7, 0, -0.5, 1, 4, -3] +
                    [0.0] * 16 + [3e-39, -1e-38] + [0.0] * 30 + [-0.0] * 32 +
                    list(g.standard_normal(32) * 1e30), dtype=np.float32)
    x = np.concatenate([draws, synth.f32_to_bf16_bits(edge)])
    codes, scales = _quantize_gpu(x)
    want_c, want_s = oracle.mxfp4_quantize(x.reshape(-1, 32))
    np.testing.assert_array_equal(scales, want_s.reshape(-1))
    np.testing.assert_array_equal(codes, want_c.reshape(-1))


def _mx_case(B: int, L: int, k: int):
    w = synth.Workload("mx", "decode", B=B, L=L, T=1, R=128, k=k, x8=True, indexer="mxfp4")
    return w, synth.make_inputs(w)


def _row_rel_err(gpu, ref, nvis):
    worst = 0.0
    for r in range(ref.shape[0]):
        n = int(nvis[r])
        den = np.abs(ref[r, :n]).max()
        err = np.abs(gpu[r, :n].astype(np.float64) - ref[r, :n]).max()
        worst = max(worst, err / den if den > 0 else err)
    return worst


@pytest.mark.parametrize("B,L,k", [(4, 20000, 256), (32, 131072, 2048)])
def test_mxfp4_indexer_scores_topk_recall(B, L, k):
    w, x = _mx_case(B, L, k)
    step = make_step(w, x)
    rows = np.arange(w.B * w.T)
    # --- the whole CSA indexer path on the GPU: compress (MXFP4 key out),
    # quantise the queries, score, select
    step.compress_csa()
    step.index_topk()
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    caches = oracle.compress_all(w, x)
    kc_ref, ks_ref = oracle.mxfp4_quantize(caches["ik_c"])
    kc_gpu, ks_gpu = host(step.x["ik_c"]), host(step.x["ik_c_scales"])
    new = np.zeros(w.ncap, bool)
    new[int(x["blk_lo"][0]):int(x["blk_hi"][0])] = True
    # drawn cache rows: bit-exact; the block compressed this step: its pooled
    # bf16 value may differ by one ulp, so compare dequantised values
    np.testing.assert_array_equal(ks_gpu[:, ~new], ks_ref[:, ~new])
    np.testing.assert_array_equal(kc_gpu[:, ~new], kc_ref[:, ~new])
    dq_gpu = oracle.mxfp4_dequantize(kc_gpu[:, new], ks_gpu[:, new])
    dq_ref = oracle.mxfp4_dequantize(kc_ref[:, new], ks_ref[:, new])
    step_size = 2.0 ** (ks_ref[:, new].astype(np.float64) - 127)     # one e2m1 step <= 2^e
    assert np.all(np.abs(dq_gpu - dq_ref).reshape(step_size.shape[:2] + (-1,)).max(-1)
                  <= step_size.max(-1))
    qc_ref, qs_ref = oracle.mxfp4_quantize(x["q_idx"].reshape(w.B * w.T, w.HI, w.dI))
    np.testing.assert_array_equal(host(step.q_scales).reshape(qs_ref.shape), qs_ref)
    np.testing.assert_array_equal(host(step.q_codes).reshape(qc_ref.shape), qc_ref)
    # --- scores from the oracle's MXFP4 operands (same inputs on both sides)
    step.x["ik_c"].copy_(dev(kc_ref))
    step.x["ik_c_scales"].copy_(dev(ks_ref))
    ref = oracle.reference(w, x, rows=rows, caches=dict(caches, ik_c_mx=(kc_ref, ks_ref)))
    scores = torch.full((w.B, w.T, w.ncap), float("nan"), dtype=torch.float32, device="cuda")
    step.index_topk(scores_out=scores)
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    s_gpu = host(scores).reshape(w.B * w.T, w.ncap)
    err = _row_rel_err(s_gpu, ref["scores"], ref["nvis"])
    print(f"MXFP4 score rel err {err:.3e}")
    assert err <= TOL_SCORE_MX, err
    # --- top-k on the GPU scores: valid with respect to the oracle's scores
    idx = host(step.idx).reshape(w.B * w.T, w.k)
    for r in rows:
        n = int(ref["nvis"][r]); take = min(w.k, n)
        sel = idx[r, :take]
        assert np.all(np.diff(sel) > 0) and sel[0] >= 0 and sel[-1] < n
        chosen = np.zeros(n, bool); chosen[sel] = True
        tol = 2 * TOL_SCORE_MX * np.abs(ref["scores"][r, :n]).max()
        assert ref["scores"][r, :n][chosen].min() >= ref["scores"][r, :n][~chosen].max() - tol
    # --- recall against the selection from the unquantised bf16 operands
    s_full = oracle.index_scores(x["q_idx"].reshape(w.B * w.T, w.HI, w.dI),
                                 x["w_idx"].reshape(w.B * w.T, w.HI).astype(np.float64),
                                 caches["ik_c"], rows // w.T, ref["nvis"])
    idx_full, _ = oracle.topk(s_full, ref["nvis"], w.k)
    hits = sum(len(np.intersect1d(idx[r], idx_full[r])) for r in rows)
    recall = hits / (len(rows) * w.k)
    print(f"MXFP4 top-{w.k} recall vs bf16 selection: {recall:.4f}")
    assert recall >= 0.75, recall
    # --- CSA attention given the MXFP4 selection is the unchanged attention
    step.x["ik_c"].copy_(dev(kc_gpu))
    step.x["ik_c_scales"].copy_(dev(ks_gpu))
    step.attend_csa()
    torch.cuda.synchronize()
    keys, vals = zip(*[oracle.csa_keys(b, int(x["q_pos"][b, 0]), idx[b], caches["k_c"],
                                       caches["v_c"], x["k_raw"], x["v_raw"], w.W)
                       for b in range(w.B)])
    o_ref, _ = oracle.attend(x["q"].reshape(w.B, w.H, w.d), list(keys), list(vals), w.sm_scale)
    o = host(step.o).reshape(o_ref.shape)
    assert float(np.abs(o - o_ref).max()) <= 2e-2


@pytest.mark.parametrize("B,L", [(2, 1184), (1, 4128)])
def test_mxfp4_prefill_scores(B, L):
    """The four-queries-per-group kernel (prefill): causal limits cut groups
    and chunks mid-tile and the last tile is ragged (N_cap = 296 = 2 tiles + 40
    rows; 1032 = 8 tiles + 8 rows).  Scores on the oracle's MXFP4 operands,
    every fifth query row, against the oracle's double-precision scores of the
    dequantised values."""
    w = synth.Workload("mxpre", "prefill", B=B, L=L, T=L, k=64, W=128, indexer="mxfp4")
    x = synth.make_inputs(w)
    step = make_step(w, x)
    step.compress_csa()
    caches = oracle.compress_all(w, x)
    kc_ref, ks_ref = oracle.mxfp4_quantize(caches["ik_c"])
    step.x["ik_c"].copy_(dev(kc_ref))
    step.x["ik_c_scales"].copy_(dev(ks_ref))
    scores = torch.full((w.B, w.T, w.ncap), float("nan"), dtype=torch.float32, device="cuda")
    step.index_topk(scores_out=scores)
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    rows = np.arange(0, w.B * w.T, 5)
    ref = oracle.reference(w, x, rows=rows, caches=dict(caches, ik_c_mx=(kc_ref, ks_ref)))
    s_gpu = host(scores).reshape(w.B * w.T, w.ncap)[rows]
    vis = ref["nvis"] > 0
    assert vis.sum() > 0.9 * len(rows)
    err = _row_rel_err(s_gpu[vis], ref["scores"][vis], ref["nvis"][vis])
    print(f"MXFP4 prefill score rel err {err:.3e}")
    assert err <= TOL_SCORE_MX, err
