"""csa_index_topk_noalloc, the indexer + top-k entry point for callers that
cannot give the library scratch memory (engines that own all device memory
and pass only inputs and outputs, plugins barred from side allocations,
decode loops that cannot pay for cudaMalloc).  Its scores live in a fixed
device array inside the library instead of a caller workspace.

The GPU test checks that, called through the C ABI, it selects exactly the
indices csa_index_topk selects on the same inputs, on two calls in a row
with different shapes and inputs (the second call reuses the array the first
one filled, with a different row stride), and that a call leaves the
device's free memory unchanged.  Index sets are integer results of the same kernels, so the
comparison is exact.  This file is named to be collected last."""
from __future__ import annotations

import ctypes
from dataclasses import replace

import numpy as np
import pytest

import synth


def _inputs(w, seed_shift: int):
    import torch
    from gpu_util import dev
    x = synth.make_inputs(replace(w, seed=w.seed + seed_shift))
    t = {n: dev(x[n]) for n in ("q_idx", "w_idx", "ik_c", "q_pos")}
    t["idx"] = torch.full((w.B, w.T, w.k), -7, dtype=torch.int32, device="cuda")
    return t


def _with_workspace(m, w, t):
    import torch
    ws_bytes = m.csa_index_topk_workspace_bytes(w.B, w.T, w.ncap, w.k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    idx = torch.full_like(t["idx"], -7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.csa_index_topk(m.SA_BF16, w.B, w.T, w.HI, w.dI, w.m, w.k, t["q_idx"], None, t["w_idx"],
                     t["ik_c"], None, w.ncap, t["q_pos"], idx, ws=ws, ws_bytes=ws_bytes, err=err)
    return idx, err


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice():
    """Two calls in a row with different shapes: the second has fewer entries
    per sequence (a shorter row stride in the shared score array) and a
    shorter causal range than the first, so a top-k that read a score left in
    the array by the first call would select differently.  Each call's
    indices must equal csa_index_topk's on a fresh workspace, and the second
    call must not change the device's free memory."""
    import torch
    import sparse_attention_27_b300 as m
    from gpu_util import host
    lib = ctypes.CDLL(m.LIB_PATH)
    assert hasattr(lib, "csa_index_topk_noalloc")
    # 8 sequences at 128K context (32768 entries each), then 5 at 100003
    # tokens (25000 entries): both within the array's 2,097,152 scores
    cases = [synth.Workload("noalloc", "decode", B=8, L=131072, T=1, R=128, x8=True),
             synth.Workload("noalloc2", "decode", B=5, L=100003, T=1, R=128, x8=True)]
    for i, w in enumerate(cases):
        assert w.B * w.T * w.ncap <= m.NOALLOC_MAX_SCORES
        t = _inputs(w, i)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        m.csa_index_topk_noalloc(m.SA_BF16, w.B, w.T, w.HI, w.dI, w.m, w.k, t["q_idx"], None,
                                 t["w_idx"], t["ik_c"], None, w.ncap, t["q_pos"], t["idx"],
                                 err=err)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if i > 0:      # the first call may load the library's device code
            assert free_after == free_before, (free_before, free_after)
        want, err_ref = _with_workspace(m, w, t)
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and int(err_ref.item()) == 0
        got = host(t["idx"])
        np.testing.assert_array_equal(got, host(want))
        assert np.all(got[:, :, : w.k] >= 0)


def test_noalloc_rejects_sizes_beyond_its_array():
    """Host-side check, made before any CUDA call (also runs without a GPU)."""
    import sparse_attention_27_b300 as m
    big = m.NOALLOC_MAX_SCORES // 32768 + 1      # sequences of 32768 entries
    with pytest.raises(m.SaError) as e:
        m.csa_index_topk_noalloc(m.SA_BF16, big, 1, 64, 64, 4, 2048, 16, None, 16, 16, None,
                                 32768, 16, 16, stream=0)
    assert e.value.status == m.SA_ERR_UNSUPPORTED
