"""GPU parity of the path across steps: the cache split of "DeepSeek-V4 논문
읽기: 백만 토큰 컨텍스트를 저렴하게", section "KV Cache 관리: 저장 구조까지
변경" -- compressed caches, a sliding-window ring, and a tail of tokens not
yet compressed -- kept up to date by the library's own calls, step after step.

* Decode, many steps in a row (the separate calls, csa_decode, and
  sa_decode_step): each step writes its token into ring row
  t mod R of every layer's per-token arrays, compresses the CSA block the
  token closes (every m = 4 steps) and the HCA block (every m' = 128 steps),
  and attends.  The float64 oracle keeps its own caches, compressed from the
  same seeded tokens, and every step's selection, O and LSE, and every newly
  closed cache row, are compared with it.
* Prefill in two chunks: the second chunk's queries run on the caches the
  first chunk's compressors wrote (blocks from blk_lo > 0 on, queries from
  t0 > 0 on, the block straddling the chunk boundary completed by the second
  chunk), against the oracle's one-piece prefill of the whole sequence.

The indexer operands are exact-score inputs (tests/exact_inputs.py), so the
GPU's selection equals the oracle's row for row at every step.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth
from exact_inputs import exact_scores
from gpu_util import dev, host, make_step
from test_gpu_parity import TOL_ATT, check_cache, exact_bf16_bits, pool_bound

pytestmark = pytest.mark.gpu

RING = {"k_raw": "k_c", "v_raw": "v_c", "ik_raw": "ik_c"}


def sa_lib():
    import sparse_attention_27_b300 as m
    return m
PER_TOKEN = ("k_raw", "v_raw", "ik_raw", "z", "hk_raw", "hv_raw", "hz")
PER_STEP = ("q", "q_hca", "q_idx", "w_idx")


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def draw_token(w, s: int, seed: int = 7) -> dict:
    """The raw arrays of step s's new token (one per sequence): K, V, the
    indexer key (integers, for exact scores) and zero CSA pooling logits
    (equal weights), the HCA layer's K, V and random logits."""
    B = w.B
    return {"k_raw": synth.normal(seed, f"k_raw@{s}", (B, w.d), "bf16"),
            "v_raw": synth.normal(seed, f"v_raw@{s}", (B, w.d), "bf16"),
            "ik_raw": synth.integers(seed, f"ik_raw@{s}", (B, w.dI), -2, 2, "bf16"),
            "z": np.zeros(B, dtype=np.float32),
            "hk_raw": synth.normal(seed, f"hk_raw@{s}", (B, w.d), "bf16"),
            "hv_raw": synth.normal(seed, f"hv_raw@{s}", (B, w.d), "bf16"),
            "hz": synth.normal(seed, f"hz@{s}", (B,), "f32")}


def draw_queries(w, s: int, seed: int = 7) -> dict:
    B, H, d = w.B, w.H, w.d
    return {"q": synth.normal(seed, f"q@{s}", (B, 1, H, d), "bf16"),
            "q_hca": synth.normal(seed, f"q_hca@{s}", (B, 1, H, d), "bf16"),
            "q_idx": synth.integers(seed, f"q_idx@{s}", (B, 1, w.HI, w.dI), -2, 2, "bf16"),
            "w_idx": synth.dyadic(seed, f"w_idx@{s}", (B, 1, w.HI), 8, 8)}


def block_range(t: int, m: int, B: int):
    hi = (t + 1) // m
    lo = hi - 1 if (t + 1) % m == 0 else hi
    return np.full(B, lo, dtype=np.int32), np.full(B, hi, dtype=np.int32)


@pytest.mark.parametrize("mode", ["fused", "split", "step"])
def test_decode_steps_advance_the_rings_and_close_blocks(mode):
    """260 consecutive decode steps of 4 sequences from position 15875: 65
    CSA blocks and 2 HCA blocks close on the way (at t = 15999 and 16127).
    The step runs as csa_decode + hca_compress_attend (fused), as the
    separate calls (split) or as one sa_decode_step (step)."""
    S, t0 = 260, 15875
    w = synth.Workload("steps", "decode", B=4, L=t0 + S + 1, T=1, R=256, k=256, W=128)
    x = exact_scores(w, synth.make_inputs(w))
    x["q_pos"] = np.full((w.B, 1), t0, dtype=np.int32)
    x["blk_lo"], x["blk_hi"] = block_range(t0, w.m, w.B)
    x["hblk_lo"], x["hblk_hi"] = block_range(t0, w.m2, w.B)
    x["blk_hi"] = x["blk_lo"].copy()             # the state before the first step
    x["hblk_hi"] = x["hblk_lo"].copy()
    step = make_step(w, x, o_dtype="f32")
    step.D.max_blocks = step.D.max_blocks2 = 1
    # the oracle's caches, in storage form; only blocks < n_c(t0) hold history
    ref_c = {n: x[n].copy() for n in ("k_c", "v_c", "ik_c", "hk_c", "hv_c")}
    closed_csa = closed_hca = 0
    for s in range(1, S + 1):
        t = t0 + s
        tok, qs = draw_token(w, s), draw_queries(w, s)
        slot = t % w.R
        for n in PER_TOKEN:                      # the oracle's rings: row t mod R
            x[n][:, slot] = tok[n]
        x["q_pos"] = np.full((w.B, 1), t, dtype=np.int32)
        step.x["q_pos"].copy_(dev(x["q_pos"]))
        # the library's rings: one sa_ring_write for every per-token array
        sa_lib().sa_ring_write(w.B, w.R, step.x["q_pos"], [step.x[n] for n in PER_TOKEN],
                               [dev(tok[n]) for n in PER_TOKEN], err=step.err)
        for n in PER_STEP:
            x[n] = qs[n]
            step.x[n].copy_(dev(qs[n]))
        x["blk_lo"], x["blk_hi"] = block_range(t, w.m, w.B)
        x["hblk_lo"], x["hblk_hi"] = block_range(t, w.m2, w.B)
        for n in ("q_pos", "blk_lo", "blk_hi", "hblk_lo", "hblk_hi"):
            step.x[n].copy_(dev(x[n]))
        # the GPU step
        if mode == "step":
            step.decode_step()
        else:
            if mode == "fused":
                step.csa_fused()
            else:
                step.csa()
            step.hca()
        torch.cuda.synchronize()
        assert step.device_errors() == 0, (s, step.device_errors())
        # the oracle's step on its own caches
        xo = dict(x, **ref_c)
        ref = oracle.reference(w, xo)
        idx = host(step.idx).reshape(w.B, w.k)
        np.testing.assert_array_equal(idx, ref["idx"], err_msg=f"step {s}")
        for a, b_, r in (("o", "lse", ("o", "lse")), ("ho", "hlse", ("ho", "hlse"))):
            o = host(getattr(step, a)).reshape(ref[r[0]].shape)
            lse = host(getattr(step, b_)).reshape(ref[r[1]].shape)
            assert np.abs(o - ref[r[0]]).max() <= TOL_ATT["bf16"], (s, a)
            assert np.abs(lse - ref[r[1]]).max() <= TOL_ATT["bf16"], (s, b_)
        # newly closed blocks: GPU rows against the oracle's, then the oracle
        # keeps its own rows (rounded to bf16) as its history
        lo, hi = int(x["blk_lo"][0]), int(x["blk_hi"][0])
        if hi > lo:
            closed_csa += 1
            for n, raw in (("k_c", "k_raw"), ("v_c", "v_raw"), ("ik_c", "ik_raw")):
                for b in range(w.B):
                    check_cache(host(step.x[n][b, lo:hi]), ref[n][b, lo:hi], "bf16", n,
                                pool_bound(x[raw][b], w.m, lo, hi))
                ref_c[n][:, lo:hi] = exact_bf16_bits(ref[n][:, lo:hi])
            np.testing.assert_array_equal(host(step.x["ik_c"][:, lo:hi]), ref_c["ik_c"][:, lo:hi])
        lo, hi = int(x["hblk_lo"][0]), int(x["hblk_hi"][0])
        if hi > lo:
            closed_hca += 1
            for n, raw in (("hk_c", "hk_raw"), ("hv_c", "hv_raw")):
                for b in range(w.B):
                    check_cache(host(step.x[n][b, lo:hi]), ref[n][b, lo:hi], "bf16", n,
                                pool_bound(x[raw][b], w.m2, lo, hi))
                ref_c[n][:, lo:hi] = exact_bf16_bits(ref[n][:, lo:hi])
    assert closed_csa == 65 and closed_hca == 2, (closed_csa, closed_hca)


def _chunk(x: dict, lo: int, hi: int, w) -> dict:
    """The inputs of queries [lo, hi) of a one-sequence prefill: their
    queries and positions, and the blocks that close inside the chunk."""
    c = dict(x)
    for n in ("q", "q_hca", "q_idx", "w_idx", "q_pos"):
        c[n] = np.ascontiguousarray(x[n][:, lo:hi])
    c["blk_lo"] = np.array([lo // w.m], dtype=np.int32)
    c["blk_hi"] = np.array([hi // w.m], dtype=np.int32)
    c["hblk_lo"] = np.array([lo // w.m2], dtype=np.int32)
    c["hblk_hi"] = np.array([hi // w.m2], dtype=np.int32)
    return c


@pytest.mark.parametrize("L,t0", [(1500, 701), (2048, 1024)])
def test_prefill_second_chunk_on_the_first_chunks_caches(L, t0):
    """The chunk boundary t0 = 701 falls inside a CSA block (700..703) and an
    HCA block (640..767), which the second chunk's compressors complete;
    t0 = 1024 falls on a boundary of both."""
    w = synth.Workload("chunks", "prefill", B=1, L=L, T=L, k=64, W=128, x8=True)
    x = exact_scores(w, synth.make_inputs(w))
    x1, x2 = _chunk(x, 0, t0, w), _chunk(x, t0, L, w)
    s1 = make_step(replace(w, T=t0), x1)
    s1.run()
    s2 = make_step(replace(w, T=L - t0), x2)
    for n in ("k_c", "v_c", "ik_c", "hk_c", "hv_c"):      # the caches the first chunk wrote
        s2.x[n] = s1.x[n]
    s2.run()
    torch.cuda.synchronize()
    assert s1.device_errors() == 0 and s2.device_errors() == 0
    rows = np.arange(t0, L)
    ref = oracle.reference(w, x, rows=rows)
    np.testing.assert_array_equal(host(s2.idx).reshape(L - t0, w.k), ref["idx"])
    for a, r in (("o", "o"), ("lse", "lse"), ("ho", "ho"), ("hlse", "hlse")):
        got = host(getattr(s2, a)).reshape(ref[r].shape)
        fin = np.isfinite(ref[r])
        assert np.array_equal(np.isfinite(got), fin), a
        assert np.abs(got[fin] - ref[r][fin]).max() <= TOL_ATT["bf16"], a
    # every cache row, written by either chunk, against the one-piece prefill
    for n, raw, m in (("k_c", "k_raw", w.m), ("v_c", "v_raw", w.m), ("ik_c", "ik_raw", w.m),
                      ("hk_c", "hk_raw", w.m2), ("hv_c", "hv_raw", w.m2)):
        nb = L // m
        check_cache(host(s2.x[n][0, :nb]), ref[n][0, :nb], "bf16", n,
                    pool_bound(x[raw][0], m, 0, nb))


def test_ring_write_puts_each_token_in_row_t_mod_R():
    """sa_ring_write: row b of each array lands in ring row pos[b] mod R of
    its ring, bit for bit; every other ring row is untouched; a negative
    position is reported (SA_ERR_BOUNDS) and its rows are skipped."""
    m = sa_lib()
    B, R = 5, 12
    g = torch.Generator(device="cuda").manual_seed(3)
    rings = [torch.randn(B, R, 128, device="cuda", generator=g).to(torch.bfloat16),
             torch.randn(B, R, 64, device="cuda", generator=g).to(torch.bfloat16),
             torch.randn(B, R, device="cuda", generator=g)]
    rows = [torch.randn(B, 128, device="cuda", generator=g).to(torch.bfloat16),
            torch.randn(B, 64, device="cuda", generator=g).to(torch.bfloat16),
            torch.randn(B, device="cuda", generator=g)]
    pos = torch.tensor([0, 11, 12, 37, -1], dtype=torch.int32, device="cuda")
    before = [r.clone() for r in rings]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.sa_ring_write(B, R, pos, rings, rows, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1 << m.SA_ERR_BOUNDS
    for ring, row, old in zip(rings, rows, before):
        want = old.clone()
        for b, p_ in enumerate(pos.tolist()):
            if p_ >= 0:
                want[b, p_ % R] = row[b]
        assert torch.equal(ring.view(torch.uint8) if ring.dtype != torch.float32 else ring.view(torch.int32),
                           want.view(torch.uint8) if want.dtype != torch.float32 else want.view(torch.int32))
    with pytest.raises(m.SaError) as e:       # a row size that is not a multiple of 4 bytes
        m.sa_ring_write(B, R, pos, [rings[0][..., :1]], [rows[0][:, :1]])
    assert e.value.status == m.SA_ERR_INVALID_ARG
