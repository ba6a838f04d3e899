"""Pins of the oracle's backward pass (CPU only).

The backward of one pass treats the top-k selection as a constant mask (the
pages: "EP 95. DeepSeek-V4 논문 읽기 — 노정석", IDEAS -- top-k selection is not
differentiable) and the caches' storage rounding as the identity.  It is
pinned to things other than itself:
  * central finite differences of a float64 forward built from the oracle's
    forward steps with the selection frozen, for every input the gradient
    reaches: queries, raw K/V and pooling logits (through the window and the
    pooling of the pass's blocks) and cache rows (decode);
  * torch autograd of a dense masked attention written independently, for
    the attention part;
  * special cases: block size 1 makes the pooling the identity (raw
    gradient = cache gradient, logit gradient 0); the indexer gets none.
"""
from __future__ import annotations

import types

import numpy as np
import pytest
import torch

import oracle
import synth


def f64_workload(mode, B, L, T, **kw):
    """A small workload stored in float64 (no rounding anywhere): the shape
    fields of synth.Workload, and its inputs drawn as float32 and widened."""
    w = synth.Workload("fd", mode, B=B, L=L, T=T, dtype="f32", indexer="f32", **kw)
    x = synth.make_inputs(w)
    x = {k: (v.astype(np.float64) if v.dtype == np.float32 else v) for k, v in x.items()}
    fields = {f: getattr(w, f) for f in ("name", "mode", "B", "L", "T", "H", "d", "HI", "dI",
                                        "m", "k", "W", "m2", "R", "x8", "seed")}
    v = types.SimpleNamespace(**fields, dtype="f64", indexer="f64")
    v.ring, v.sm_scale = w.ring, w.sm_scale
    v.ncap, v.ncap2, v.rows = w.ncap, w.ncap2, w.rows
    return v, x


def forward_loss(w, x, idx, dO, dhO):
    """sum(dO * O) + sum(dhO * hO) with the selection fixed to ``idx``, from
    the oracle's forward steps in float64."""
    caches = oracle.compress_all(w, x)
    pos = x["q_pos"].reshape(-1)
    keys, vals, hk, hv = [], [], [], []
    for r in range(w.B * w.T):
        b, t = r // w.T, int(pos[r])
        K, V = oracle.csa_keys(b, t, idx[r], caches["k_c"], caches["v_c"], x["k_raw"],
                               x["v_raw"], w.W)
        keys.append(K); vals.append(V)
        K, V = oracle.hca_keys(b, t, w.m2, caches["hk_c"], caches["hv_c"], x["hk_raw"],
                               x["hv_raw"], w.W)
        hk.append(K); hv.append(V)
    O, _ = oracle.attend(x["q"].reshape(w.B * w.T, w.H, w.d), keys, vals, w.sm_scale)
    hO, _ = oracle.attend(x["q_hca"].reshape(w.B * w.T, w.H, w.d), hk, hv, w.sm_scale)
    return float((dO.reshape(O.shape) * O).sum() + (dhO.reshape(hO.shape) * hO).sum())


def grads_and_fd(w, x, names, n_probe=40, h=1e-6, seed=0):
    g = np.random.default_rng(seed)
    dO = g.standard_normal((w.B, w.T, w.H, w.d))
    dhO = g.standard_normal((w.B, w.T, w.H, w.d))
    fwd = oracle.reference(w, x)
    idx = fwd["idx"]
    an = oracle.reference_backward(w, x, dO, dhO, fwd)
    key = {"q": "dq", "q_hca": "dq_hca", "k_raw": "dk_raw", "v_raw": "dv_raw", "z": "dz",
           "hk_raw": "dhk_raw", "hv_raw": "dhv_raw", "hz": "dhz", "k_c": "dk_c",
           "v_c": "dv_c", "hk_c": "dhk_c", "hv_c": "dhv_c"}
    worst = {}
    pooled = {"k_c": ("blk_lo", "blk_hi"), "v_c": ("blk_lo", "blk_hi"),
              "hk_c": ("hblk_lo", "hblk_hi"), "hv_c": ("hblk_lo", "hblk_hi")}
    for n in names:
        a = x[n]
        flat = a.reshape(-1)
        cand = np.arange(flat.size)
        if n in pooled:
            # a cache row pooled in this pass is overwritten, so its input value
            # has no influence; its gradient (as attended) reaches the raw rows
            # through the pooling, which the raw-row probes check
            lo_n, hi_n = pooled[n]
            rowi = (cand // a.shape[-1]) % a.shape[-2]
            seq = cand // (a.shape[-1] * a.shape[-2])
            cand = cand[~((rowi >= x[lo_n][seq]) & (rowi < x[hi_n][seq]))]
        probes = g.choice(cand, size=min(n_probe, cand.size), replace=False)
        err, scale = 0.0, np.abs(an[key[n]]).max() + 1e-300
        for i in probes:
            old = flat[i]
            flat[i] = old + h
            lp = forward_loss(w, x, idx, dO, dhO)
            flat[i] = old - h
            lm = forward_loss(w, x, idx, dO, dhO)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            err = max(err, abs(fd - an[key[n]].reshape(-1)[i]))
        worst[n] = err / scale
    return worst, an


def test_backward_matches_finite_differences_prefill():
    """Every position a query; all blocks are pooled in the pass, so the raw
    K/V and the logits get gradient through both the window and the pooling."""
    w, x = f64_workload("prefill", B=1, L=48, T=48, H=3, d=8, HI=2, dI=4, m=4, k=3, W=5, m2=8)
    worst, _ = grads_and_fd(w, x, ["q", "q_hca", "k_raw", "v_raw", "z", "hk_raw", "hv_raw",
                                   "hz"])
    for n, e in worst.items():
        assert e < 1e-6, (n, e)


def test_backward_matches_finite_differences_decode():
    """Given caches: the gradient reaches the attended cache rows directly,
    and the block the token closes through its pooling."""
    w, x = f64_workload("decode", B=2, L=160, T=1, H=2, d=8, HI=2, dI=4, m=4, k=6, W=7, m2=16,
                        R=32)
    worst, an = grads_and_fd(w, x, ["q", "k_c", "v_c", "hk_c", "hv_c", "k_raw", "v_raw", "z",
                                    "hz"])
    for n, e in worst.items():
        assert e < 1e-6, (n, e)
    # only the selected cache rows (and the closed block) have gradient
    fwd = oracle.reference(w, x)
    for b in range(w.B):
        sel = set(fwd["idx"][b][fwd["idx"][b] >= 0].tolist())
        nz = set(np.nonzero(np.abs(an["dk_c"][b]).sum(1))[0].tolist())
        assert nz <= sel


def test_attention_backward_matches_torch_autograd():
    """Per key entry: dK, dV and dq of a dense masked softmax attention built
    in torch float64 and differentiated by autograd."""
    g = np.random.default_rng(3)
    rows, H, d = 5, 4, 16
    n = [7, 1, 0, 12, 3]
    q = g.standard_normal((rows, H, d))
    keys = [g.standard_normal((k, d)) for k in n]
    vals = [g.standard_normal((k, d)) for k in n]
    dO = g.standard_normal((rows, H, d))
    scale = 0.3
    dq, dK, dV, off = oracle.attend_backward(q, keys, vals, dO, scale)
    for r in range(rows):
        tq = torch.tensor(q[r], requires_grad=True)
        if n[r] == 0:
            assert np.all(dq[r] == 0)
            continue
        tk = torch.tensor(keys[r], requires_grad=True)
        tv = torch.tensor(vals[r], requires_grad=True)
        att = torch.softmax(scale * tq @ tk.T, dim=-1)
        (att @ tv * torch.tensor(dO[r])).sum().backward()
        np.testing.assert_allclose(dq[r], tq.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dK[off[r]:off[r + 1]], tk.grad.numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dV[off[r]:off[r + 1]], tv.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_block_size_one_pooling_is_the_identity():
    """m = 1: each block is one raw row with weight 1, so the pooling passes
    the cache gradient to the raw row unchanged and the logit gets none."""
    g = np.random.default_rng(5)
    X = g.standard_normal((9, 6))
    z = g.standard_normal(9)
    dXc = g.standard_normal((9, 6))
    dX, dz = oracle.compress_backward(X, z, 1, 0, 9, dXc)
    np.testing.assert_array_equal(dX, dXc)
    np.testing.assert_array_equal(dz, np.zeros(9))


def test_pooling_backward_equal_logits_is_the_mean_gradient():
    """Equal logits: weights 1/m, so every raw row gets dXc/m, and the logit
    gradient is (X_i - mean) . dXc / m, which sums to 0 over the block."""
    g = np.random.default_rng(6)
    m, d = 4, 5
    X = g.standard_normal((m, d))
    dXc = g.standard_normal((1, d))
    dX, dz = oracle.compress_backward(X, np.zeros(m), m, 0, 1, dXc)
    np.testing.assert_allclose(dX, np.tile(dXc / m, (m, 1)), rtol=1e-15)
    want = ((X - X.mean(0)) @ dXc[0]) / m
    np.testing.assert_allclose(dz, want, rtol=1e-12, atol=1e-15)
    assert abs(dz.sum()) < 1e-14
