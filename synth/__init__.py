"""Seeded synthetic inputs for the CSA + HCA hot path.

This module only draws random numbers and stores them in the path's storage
formats (float32, bfloat16 bit patterns in uint16, int32 positions).  It holds
none of the method's arithmetic: no compression, scoring, selection,
attention or quantisation.  Both the CUDA path's tests and the float64 oracle
take their inputs from here and nowhere else.

Drawing: numpy PCG64.  Large arrays are drawn in fixed chunks of 2^22 values;
chunk c of tensor ``name`` comes from ``PCG64(SeedSequence([seed, crc32(name)]))
.jumped(c)``, so every value is fixed by (seed, name, shape) alone and chunks can
be drawn by several threads.  bfloat16 values are float32 draws rounded to
nearest, ties to even.

Workloads (the pages' long-context settings; the pages measure on long-context
retrieval suites that are not reproduced here, so these seeded draws stand in
for them):

* ``tiny``      -- 1 sequence, L=4096, 16 query heads, fp32, CSA m=4 k=64,
                   indexer 4 heads, window 128, HCA m'=128, 256 query
                   positions at the end of the sequence.
* ``decode128k`` -- batch 32, one new token each at position 131071, 64 heads,
                   bf16 caches, CSA m=4 k=2048 W=128, indexer 64 heads,
                   HCA m'=128 (1024 entries); 1% of compressed key rows x8.
* ``prefill64k`` -- 1 sequence of 65536 tokens, all positions queried.
* ``decode1m``   -- batch 4 at position 1048578 (262144 CSA entries, 8192 HCA
                   entries, a 3-token tail); no x8 rows.
* ``mxfp4``      -- the decode128k draws; the indexer operands are later
                   stored as MXFP4 by each side's own quantiser.
"""
from __future__ import annotations

import math
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

CHUNK = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "decode" (caches given, one query per sequence) or "prefill"
    B: int               # sequences
    L: int               # tokens whose KV exists (decode: query position is L-1)
    T: int               # queries per sequence
    H: int = 64          # query heads (one shared KV head)
    d: int = 128         # head dim
    HI: int = 64         # indexer heads
    dI: int = 64         # indexer dim
    m: int = 4           # CSA block
    k: int = 2048        # CSA top-k
    W: int = 128         # sliding window
    m2: int = 128        # HCA block
    R: int = 0           # raw ring rows (0: identity layout R = L)
    dtype: str = "bf16"  # storage type of K/V/q ("bf16" or "f32")
    x8: bool = False     # 1% of compressed key rows (or blocks) scaled by 8
    indexer: str = "bf16"  # "bf16", "f32" or "mxfp4"
    seed: int = 0

    @property
    def ring(self) -> int:
        return self.R if self.R else self.L

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def ncap(self) -> int:
        return self.L // self.m

    @property
    def ncap2(self) -> int:
        return self.L // self.m2

    @property
    def rows(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "tiny": Workload("tiny", "prefill", B=1, L=4096, T=256, H=16, HI=4, k=64,
                     dtype="f32", indexer="f32"),
    "decode128k": Workload("decode128k", "decode", B=32, L=131072, T=1, R=128, x8=True),
    "prefill64k": Workload("prefill64k", "prefill", B=1, L=65536, T=65536, x8=True),
    "decode1m": Workload("decode1m", "decode", B=4, L=1048579, T=1, R=128),
    "mxfp4": Workload("mxfp4", "decode", B=32, L=131072, T=1, R=128, x8=True,
                      indexer="mxfp4"),
}


def workload(name: str, **over) -> Workload:
    """A named workload, optionally with fields overridden (small test cases)."""
    w = WORKLOADS[name] if name in WORKLOADS else Workload(name, **over)
    return replace(w, **over) if name in WORKLOADS and over else w


# ------------------------------------------------------------------ drawing

def _gen(seed: int, name: str, chunk: int) -> np.random.Generator:
    ss = np.random.SeedSequence([seed, zlib.crc32(name.encode())])
    return np.random.Generator(np.random.PCG64(ss).jumped(chunk))


def _draw(seed: int, name: str, n: int, kind: str) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)

    def fill(c: int) -> None:
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        g = _gen(seed, name, c)
        if kind == "normal":
            g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        else:
            g.random(hi - lo, dtype=np.float32, out=out[lo:hi])

    nch = (n + CHUNK - 1) // CHUNK
    if nch <= 1:
        for c in range(nch):
            fill(c)
    else:
        with ThreadPoolExecutor(max_workers=min(16, nch)) as ex:
            list(ex.map(fill, range(nch)))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit pattern (uint16), round to nearest, ties to even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(seed: int, name: str, shape, store: str) -> np.ndarray:
    """N(0,1) draws of ``shape`` stored as float32 or bfloat16 bits."""
    x = _draw(seed, name, int(np.prod(shape)), "normal").reshape(shape)
    return f32_to_bf16_bits(x) if store == "bf16" else x


def uniform(seed: int, name: str, shape) -> np.ndarray:
    return _draw(seed, name, int(np.prod(shape)), "uniform").reshape(shape)


def integers(seed: int, name: str, shape, lo: int, hi: int, store: str) -> np.ndarray:
    """Uniform integers in [lo, hi] of ``shape``, stored as float32 or
    bfloat16 bits (exact for |value| <= 256)."""
    g = _gen(seed, name, 0)
    x = g.integers(lo, hi + 1, size=shape).astype(np.float32)
    return f32_to_bf16_bits(x) if store == "bf16" else x


def dyadic(seed: int, name: str, shape, num_hi: int, den: int) -> np.ndarray:
    """Uniform values j / den, j in [0, num_hi], of ``shape`` as float32."""
    g = _gen(seed, name, 0)
    return (g.integers(0, num_hi + 1, size=shape).astype(np.float32) / np.float32(den))


def choose_rows(seed: int, name: str, n: int, count: int) -> np.ndarray:
    """``count`` distinct indices in [0, n), sorted."""
    g = _gen(seed, name, 0)
    return np.sort(g.choice(n, size=count, replace=False))


def scale_rows(a: np.ndarray, rows: np.ndarray, factor: float, store: str) -> None:
    """Multiply rows (second-to-last axis) of one sequence's array by a power of two."""
    if store == "bf16":
        v = bf16_bits_to_f32(a[rows]) * np.float32(factor)
        a[rows] = f32_to_bf16_bits(v)
    else:
        a[rows] *= np.float32(factor)


# ------------------------------------------------------------- workloads

def make_inputs(w: Workload) -> dict:
    """All inputs of one decode step / prefill chunk of ``w`` as numpy arrays.

    Keys (bf16 arrays are uint16 bit patterns; layouts row-major):
      q_pos [B,T] int32          query positions (0-based)
      q [B,T,H,d], q_hca [B,T,H,d]   queries of the CSA and the HCA layer
      q_idx [B,T,HI,dI], w_idx [B,T,HI] f32   indexer queries and head weights
      CSA layer raw ring:  k_raw, v_raw [B,R,d], ik_raw [B,R,dI], z [B,R] f32
      HCA layer raw ring:  hk_raw, hv_raw [B,R,d], hz [B,R] f32
      decode only (caches given): k_c, v_c [B,ncap,d], ik_c [B,ncap,dI],
                                  hk_c, hv_c [B,ncap2,d]
      blk_lo, blk_hi [B] int32 (CSA blocks this step compresses)
      hblk_lo, hblk_hi [B] int32 (HCA blocks this step compresses)
    Raw position p lives in ring row p mod R.
    """
    s, st = w.seed, w.dtype
    ist = "bf16" if w.indexer in ("bf16", "mxfp4") else "f32"
    R = w.ring
    x = {}
    if w.mode == "decode":
        t = w.L - 1
        x["q_pos"] = np.full((w.B, w.T), t, dtype=np.int32)
    else:
        t0 = w.L - w.T
        x["q_pos"] = np.broadcast_to(np.arange(t0, w.L, dtype=np.int32), (w.B, w.T)).copy()
    x["q"] = normal(s, "q", (w.B, w.T, w.H, w.d), st)
    x["q_hca"] = normal(s, "q_hca", (w.B, w.T, w.H, w.d), st)
    x["q_idx"] = normal(s, "q_idx", (w.B, w.T, w.HI, w.dI), ist)
    x["w_idx"] = uniform(s, "w_idx", (w.B, w.T, w.HI))
    x["k_raw"] = normal(s, "k_raw", (w.B, R, w.d), st)
    x["v_raw"] = normal(s, "v_raw", (w.B, R, w.d), st)
    x["ik_raw"] = normal(s, "ik_raw", (w.B, R, w.dI), ist)
    x["z"] = normal(s, "z", (w.B, R), "f32")
    x["hk_raw"] = normal(s, "hk_raw", (w.B, R, w.d), st)
    x["hv_raw"] = normal(s, "hv_raw", (w.B, R, w.d), st)
    x["hz"] = normal(s, "hz", (w.B, R), "f32")
    if w.mode == "decode":
        x["k_c"] = normal(s, "k_c", (w.B, w.ncap, w.d), st)
        x["v_c"] = normal(s, "v_c", (w.B, w.ncap, w.d), st)
        x["ik_c"] = normal(s, "ik_c", (w.B, w.ncap, w.dI), ist)
        x["hk_c"] = normal(s, "hk_c", (w.B, w.ncap2, w.d), st)
        x["hv_c"] = normal(s, "hv_c", (w.B, w.ncap2, w.d), st)
        if w.x8:
            cnt = w.ncap // 100
            for b in range(w.B):
                rows = choose_rows(s, f"x8_{b}", w.ncap, cnt)
                scale_rows(x["k_c"][b], rows, 8.0, st)
                scale_rows(x["ik_c"][b], rows, 8.0, ist)
        t = w.L - 1
        closes = (t + 1) % w.m == 0
        x["blk_lo"] = np.full(w.B, (t + 1) // w.m - (1 if closes else 0), dtype=np.int32)
        x["blk_hi"] = np.full(w.B, (t + 1) // w.m, dtype=np.int32)
        closes2 = (t + 1) % w.m2 == 0
        x["hblk_lo"] = np.full(w.B, (t + 1) // w.m2 - (1 if closes2 else 0), dtype=np.int32)
        x["hblk_hi"] = np.full(w.B, (t + 1) // w.m2, dtype=np.int32)
    else:
        if w.x8:
            nblk = w.L // w.m
            cnt = nblk // 100
            for b in range(w.B):
                blocks = choose_rows(s, f"x8_{b}", nblk, cnt)
                rows = (blocks[:, None] * w.m + np.arange(w.m)[None, :]).reshape(-1)
                scale_rows(x["k_raw"][b], rows, 8.0, st)
                scale_rows(x["ik_raw"][b], rows, 8.0, ist)
        x["blk_lo"] = np.zeros(w.B, dtype=np.int32)
        x["blk_hi"] = np.full(w.B, w.L // w.m, dtype=np.int32)
        x["hblk_lo"] = np.zeros(w.B, dtype=np.int32)
        x["hblk_hi"] = np.full(w.B, w.L // w.m2, dtype=np.int32)
    return x
