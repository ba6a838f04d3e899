"""GPU parity of the backward pass (csa_attend_backward, hca_attend_backward,
sa_compress_backward through the C ABI) against the float64 oracle's
reference_backward, whose own pins are in test_oracle_backward.py.

The oracle's caches, selection, O and LSE are uploaded to the GPU (never the
other way round), so both sides differentiate the same function; the GPU computes
in fp32 from the same stored inputs.  Gate: every gradient tensor within
1e-4 of the largest magnitude of the oracle's (fp32 accumulation over a few
thousand terms, added in an unfixed order by atomics).  Shapes: the tiny
fp32 configuration (queries at the end of a 4K sequence), a bf16 prefill
with a ragged last tile and a short window, a bf16 decode at 20K context
with its block-closing step, and an HCA block of 16.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, make_step
from test_gpu_parity import to_store

pytestmark = pytest.mark.gpu
TOL = 1e-4


def run_backward(w, x, seed=11):
    ref = oracle.reference(w, x)
    dO = synth.normal(seed, "dO", (w.B, w.T, w.H, w.d), "f32")
    dhO = synth.normal(seed, "dhO", (w.B, w.T, w.H, w.d), "f32")
    g_ref = oracle.reference_backward(w, x, dO.astype(np.float64), dhO.astype(np.float64), ref)
    step = make_step(w, x, o_dtype="f32")
    for n in ("k_c", "v_c", "hk_c", "hv_c"):     # the oracle's cache rows, as stored
        step.x[n].copy_(dev(to_store(ref[n], w.dtype)))
    up = lambda a: dev(np.ascontiguousarray(a, dtype=np.float32).reshape(w.B, w.T, *a.shape[1:]))
    g = step.backward(dev(dO), dev(dhO), idx=dev(ref["idx"].reshape(w.B, w.T, w.k)),
                      o=up(ref["o"]), lse=up(ref["lse"]), ho=up(ref["ho"]), hlse=up(ref["hlse"]))
    torch.cuda.synchronize()
    assert step.device_errors() == 0
    worst = {}
    for n, gr in g_ref.items():
        got = host(g[n]).astype(np.float64).reshape(gr.shape)
        scale = np.abs(gr).max()
        err = np.abs(got - gr).max()
        worst[n] = err / scale if scale > 0 else err
        assert worst[n] <= TOL, (n, worst[n], scale)
    return worst


def test_backward_tiny_f32():
    w = synth.WORKLOADS["tiny"]
    run_backward(w, synth.make_inputs(w))


@pytest.mark.parametrize("L,k,W", [(777, 100, 5), (1000, 64, 128)])
def test_backward_prefill_bf16(L, k, W):
    w = synth.Workload("bwp", "prefill", B=1, L=L, T=L, k=k, W=W, m2=16, x8=True)
    run_backward(w, synth.make_inputs(w))


def test_backward_decode_bf16():
    w = synth.Workload("bwd", "decode", B=3, L=20003, T=1, R=128, k=256, x8=True)
    x = synth.make_inputs(w)
    run_backward(w, x)
