"""Inputs whose indexer scores fp32 computes exactly, for tests that need the
GPU's selection to equal the oracle's row for row."""
from __future__ import annotations

import numpy as np

import synth


def exact_scores(w, x, seed=0):
    """``x`` with indexer operands whose scores fp32 and float64 both compute
    exactly: queries and keys are integers in [-2, 2], head weights are
    multiples of 1/8, and the pooling logits are zero, so a pooled indexer key
    is a mean of m integers (a multiple of 1/4 for m = 4).  Every product and
    partial sum is then a small multiple of 1/32 and the scores are equal on
    both sides -- with many ties, so the lowest-index rule decides a lot of
    selections.  Arrays absent from ``x`` (the caches of a prefill) stay
    absent."""
    x = dict(x)
    for name in ("q_idx", "ik_c", "ik_raw"):
        if name in x:
            x[name] = synth.integers(seed, "x" + name, x[name].shape, -2, 2, "bf16")
    x["w_idx"] = synth.dyadic(seed, "xw_idx", x["w_idx"].shape, 8, 8)
    x["z"] = np.zeros_like(x["z"])
    return x
