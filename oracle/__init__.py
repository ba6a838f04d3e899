"""Float64 CPU oracle for the CSA + HCA hot path (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (``sparse_attention_27_b300``) never
imports it, and this package never imports the product path: the two share
no code.  Inputs come from ``synth``.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one OpenMP
parallel-for over independent rows).  This module converts stored inputs to
double exactly, maps raw positions to ring rows (position p lives in row
p mod R), assembles each query's key multiset, and calls the C definitions in
the order the pages give them:

    compress  ->  indexer scores  ->  per-query top-k  ->  attention (CSA)
    compress  ->  dense attention over all compressed rows (HCA)

Sources (page title, section):
  "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈" -- "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)"
  "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게" -- "Compressed Sparse Attention
      (CSA)", "Heavily Compressed Attention (HCA)", "KV Cache 관리: 저장 구조까지 변경"
  "EP 95. DeepSeek-V4 논문 읽기 — 노정석" -- IDEAS (1/4 compression, lightning indexer, MQA)
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_ip = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.orc_round_bf16.argtypes = [C.c_double]
            L.orc_round_bf16.restype = C.c_double
            L.orc_compress.argtypes = [C.c_int64, C.c_int, C.c_int, _dp, _dp, C.c_int, _dp]
            L.orc_compress_channels.argtypes = [C.c_int64, C.c_int, C.c_int, _dp, _dp, C.c_int,
                                                _dp]
            L.orc_index_scores.argtypes = [C.c_int64, C.c_int, C.c_int, _dp, _dp, _dp, C.c_int64,
                                           _ip, _ip, _dp]
            L.orc_topk.argtypes = [C.c_int64, C.c_int64, _dp, _ip, C.c_int, _i32p]
            L.orc_topk.restype = C.c_int64
            L.orc_attend.argtypes = [C.c_int64, C.c_int, C.c_int, C.c_double, _dp, _ip, _dp, _dp,
                                     _dp, _dp]
            L.orc_merge.argtypes = [C.c_int, C.c_int64, C.c_int, _dp, _dp, _dp, _dp]
            L.orc_mxfp4_quantize.argtypes = [C.c_int64, _dp, _u8p, _u8p]
            L.orc_mxfp4_dequantize.argtypes = [C.c_int64, _u8p, _u8p, _dp]
            L.orc_attend_backward.argtypes = [C.c_int64, C.c_int, C.c_int, C.c_double, _dp, _ip,
                                              _dp, _dp, _dp, _dp, _dp, _dp]
            L.orc_compress_backward.argtypes = [C.c_int64, C.c_int, C.c_int, _dp, _dp, _dp, _dp,
                                                _dp]
            _lib = L
    return _lib


# ----------------------------------------------------------- conversions

def to_f64(a: np.ndarray) -> np.ndarray:
    """Stored value -> double, exactly.  uint16 arrays are bfloat16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def round_to(x: np.ndarray, store: str) -> np.ndarray:
    """Round doubles to the storage type, returned as doubles."""
    if store == "f32":
        return x.astype(np.float32).astype(np.float64)
    if store == "bf16":
        f = np.vectorize(lib().orc_round_bf16, otypes=[np.float64])
        return f(x)
    return x


def _c(a, dt=np.float64):
    return np.ascontiguousarray(a, dtype=dt)


# ------------------------------------------------------ step definitions

def compress(x_ring: np.ndarray, z_ring: np.ndarray, m: int, blk_lo: int, blk_hi: int,
             store: str) -> np.ndarray:
    """Softmax-pooled blocks [blk_lo, blk_hi) of one sequence.

    x_ring [R, d] (stored values), z_ring [R] pooling logits.  Block j covers raw
    positions j*m .. j*m+m-1, found in ring rows p mod R.  Returns doubles
    rounded to ``store`` ("f32", "bf16" or "f64").
    """
    R, d = x_ring.shape
    nb = blk_hi - blk_lo
    if nb <= 0:
        return np.zeros((0, d))
    pos = (np.arange(blk_lo * m, blk_hi * m) % R)
    X = _c(to_f64(x_ring)[pos])
    Z = _c(np.asarray(z_ring, dtype=np.float64)[pos])
    out = np.empty((nb, d))
    mode = {"f64": 0, "f32": 1, "bf16": 2}[store]
    lib().orc_compress(nb, m, d, X, Z, mode, out)
    return out


def compress_channels(x_ring: np.ndarray, z_ring: np.ndarray, m: int, blk_lo: int,
                      blk_hi: int, store: str) -> np.ndarray:
    """Per-channel softmax-pooled blocks [blk_lo, blk_hi) of one sequence:
    x_ring and z_ring [R, d] (one logit per raw token and channel).  Block j
    covers raw positions j*m .. j*m+m-1, found in ring rows p mod R.  Returns
    doubles rounded to ``store`` ("f32", "bf16" or "f64")."""
    R, d = x_ring.shape
    nb = blk_hi - blk_lo
    if nb <= 0:
        return np.zeros((0, d))
    pos = (np.arange(blk_lo * m, blk_hi * m) % R)
    X = _c(to_f64(x_ring)[pos])
    Z = _c(np.asarray(z_ring, dtype=np.float64)[pos])
    out = np.empty((nb, d))
    mode = {"f64": 0, "f32": 1, "bf16": 2}[store]
    lib().orc_compress_channels(nb, m, d, X, Z, mode, out)
    return out


def n_visible(t: np.ndarray, m: int) -> np.ndarray:
    """Complete blocks visible to a query at position t: floor((t+1)/m)."""
    return (np.asarray(t, dtype=np.int64) + 1) // m


def index_scores(q_idx: np.ndarray, w_idx: np.ndarray, ik_c: np.ndarray, seq: np.ndarray,
                 nvis: np.ndarray) -> np.ndarray:
    """s[r, j] = sum_h w[r,h] * max(0, q_I[r,h,:] . Ik_c[seq[r], j, :]), j < nvis[r].

    q_idx [rows, HI, dI], w_idx [rows, HI], ik_c [nseq, ncap, dI] (doubles or
    stored values).  Entries j >= nvis[r] are -inf.
    """
    rows, HI, dI = q_idx.shape
    ncap = ik_c.shape[1]
    s = np.empty((rows, ncap))
    lib().orc_index_scores(rows, HI, dI, _c(to_f64(q_idx)), _c(w_idx), _c(to_f64(ik_c)), ncap,
                           _c(seq, np.int64), _c(nvis, np.int64), s)
    return s


def topk(scores: np.ndarray, n: np.ndarray, k: int):
    """Per-row top-k (score desc, index asc), output ascending with -1 padding.

    Returns (idx [rows, k] int32, number of rows rejected for NaN scores)."""
    rows, ld = scores.shape
    idx = np.empty((rows, k), dtype=np.int32)
    bad = lib().orc_topk(rows, ld, _c(scores), _c(n, np.int64), k, idx)
    return idx, int(bad)


def attend(q: np.ndarray, keys: list, values: list, scale: float):
    """MQA over an explicit key multiset per row.

    q [rows, H, d]; keys[r], values[r] are [n_r, d] arrays.  Returns (O, LSE)."""
    rows, H, d = q.shape
    off = np.zeros(rows + 1, dtype=np.int64)
    off[1:] = np.cumsum([len(k) for k in keys])
    K = _c(np.concatenate([to_f64(k).reshape(-1, d) for k in keys]) if off[-1] else np.zeros((1, d)))
    V = _c(np.concatenate([to_f64(v).reshape(-1, d) for v in values]) if off[-1] else np.zeros((1, d)))
    O = np.empty((rows, H, d))
    lse = np.empty((rows, H))
    lib().orc_attend(rows, H, d, scale, _c(to_f64(q)), off, K, V, O, lse)
    return O, lse


def merge(O_parts: np.ndarray, lse_parts: np.ndarray):
    """Exact merge of partials: O_parts [n, rows, d], lse_parts [n, rows]."""
    n, rows, d = O_parts.shape
    O = np.empty((rows, d))
    lse = np.empty(rows)
    lib().orc_merge(n, rows, d, _c(O_parts), _c(lse_parts), O, lse)
    return O, lse


def mxfp4_quantize(x: np.ndarray):
    """MXFP4 along the last axis (a multiple of 32): returns (codes uint8
    [..., n/2], scales uint8 [..., n/32])."""
    x = to_f64(x)
    shp = x.shape
    assert shp[-1] % 32 == 0
    nblk = int(np.prod(shp)) // 32
    codes = np.empty(nblk * 16, dtype=np.uint8)
    scales = np.empty(nblk, dtype=np.uint8)
    lib().orc_mxfp4_quantize(nblk, _c(x.reshape(-1)), codes, scales)
    return codes.reshape(shp[:-1] + (shp[-1] // 2,)), scales.reshape(shp[:-1] + (shp[-1] // 32,))


def mxfp4_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    nblk = scales.size
    x = np.empty(nblk * 32)
    lib().orc_mxfp4_dequantize(nblk, _c(codes.reshape(-1), np.uint8), _c(scales.reshape(-1), np.uint8), x)
    return x.reshape(scales.shape[:-1] + (scales.shape[-1] * 32,))


def window_positions(t: int, W: int) -> np.ndarray:
    """Raw positions of the sliding window of a query at t: max(0, t-W+1) .. t."""
    return np.arange(max(0, t - W + 1), t + 1)


def csa_keys(b: int, t: int, idx_row: np.ndarray, k_c, v_c, k_raw, v_raw, W: int):
    """Key multiset of one CSA query: selected compressed rows plus the window."""
    R = k_raw.shape[1]
    sel = idx_row[idx_row >= 0]
    win = window_positions(t, W) % R
    K = np.concatenate([to_f64(k_c[b][sel]), to_f64(k_raw[b][win])])
    V = np.concatenate([to_f64(v_c[b][sel]), to_f64(v_raw[b][win])])
    return K, V


def hca_keys(b: int, t: int, m2: int, hk_c, hv_c, hk_raw, hv_raw, W: int):
    """Key multiset of one HCA query: every visible compressed row plus the window."""
    R = hk_raw.shape[1]
    nh = (t + 1) // m2
    win = window_positions(t, W) % R
    K = np.concatenate([to_f64(hk_c[b][:nh]), to_f64(hk_raw[b][win])])
    V = np.concatenate([to_f64(hv_c[b][:nh]), to_f64(hv_raw[b][win])])
    return K, V


# ---------------------------------------------------------- whole path

def reference(w, x: dict, rows=None, caches: dict | None = None) -> dict:
    """The whole hot path for one decode step / prefill chunk, on query rows
    ``rows`` (flat b*T + t indices; default all).

    ``w`` is a ``synth.Workload``, ``x`` its inputs.  Steps:
      1. compress this step's CSA blocks (K, V, indexer keys) and HCA blocks
         (K, V) into copies of the caches (decode) or new caches (prefill);
      2. indexer scores of every visible compressed entry;
      3. top-k per query;
      4. CSA attention over selected rows + window;
      5. HCA attention over all visible HCA rows + window.
    ``caches`` may pass already-compressed caches (keys k_c, v_c, ik_c, hk_c,
    hv_c as doubles or stored values) to skip step 1.
    Returns dict with k_c, v_c, ik_c, hk_c, hv_c (stored-type doubles),
    scores [n,ncap], idx [n,k], o [n,H,d], lse [n,H], ho, hlse.
    """
    B, T = w.B, w.T
    store = w.dtype
    istore = "bf16" if w.indexer in ("bf16", "mxfp4") else w.indexer
    rows = np.arange(B * T) if rows is None else np.asarray(rows)
    if caches is None:
        caches = compress_all(w, x)
    k_c, v_c, ik_c, hk_c, hv_c = (caches[n] for n in ("k_c", "v_c", "ik_c", "hk_c", "hv_c"))
    bs, ts = rows // T, rows % T
    tpos = x["q_pos"].reshape(-1)[rows].astype(np.int64)
    nvis = n_visible(tpos, w.m)
    q_idx = x["q_idx"].reshape(B * T, w.HI, w.dI)[rows]
    w_idx = x["w_idx"].reshape(B * T, w.HI)[rows]
    if w.indexer == "mxfp4":
        qc, qs = mxfp4_quantize(q_idx)
        q_idx_v = mxfp4_dequantize(qc, qs)
        kc_, ks_ = caches["ik_c_mx"] if "ik_c_mx" in caches else mxfp4_quantize(ik_c)
        ik_v = mxfp4_dequantize(kc_, ks_)
    else:
        q_idx_v, ik_v = to_f64(q_idx), ik_c
    scores = index_scores(q_idx_v, w_idx.astype(np.float64), ik_v, bs, nvis)
    idx, bad = topk(scores, nvis, w.k)
    q = x["q"].reshape(B * T, w.H, w.d)[rows]
    keys, vals = zip(*[csa_keys(b, t, idx[i], k_c, v_c, x["k_raw"], x["v_raw"], w.W)
                       for i, (b, t) in enumerate(zip(bs, tpos))]) if len(rows) else ([], [])
    o, lse = attend(q, list(keys), list(vals), w.sm_scale)
    qh = x["q_hca"].reshape(B * T, w.H, w.d)[rows]
    hkeys, hvals = zip(*[hca_keys(b, t, w.m2, hk_c, hv_c, x["hk_raw"], x["hv_raw"], w.W)
                         for b, t in zip(bs, tpos)]) if len(rows) else ([], [])
    ho, hlse = attend(qh, list(hkeys), list(hvals), w.sm_scale)
    return dict(caches, scores=scores, idx=idx, nan_rows=bad, o=o, lse=lse, ho=ho, hlse=hlse,
                rows=rows, nvis=nvis)


def compress_all(w, x: dict) -> dict:
    """Step 1 of ``reference``: the caches after this step's compression."""
    store = w.dtype
    istore = "bf16" if w.indexer in ("bf16", "mxfp4") else w.indexer
    out = {}
    if w.mode == "decode":
        k_c, v_c, ik_c = to_f64(x["k_c"]), to_f64(x["v_c"]), to_f64(x["ik_c"])
        hk_c, hv_c = to_f64(x["hk_c"]), to_f64(x["hv_c"])
    else:
        k_c = np.zeros((w.B, w.ncap, w.d)); v_c = np.zeros_like(k_c)
        ik_c = np.zeros((w.B, w.ncap, w.dI))
        hk_c = np.zeros((w.B, w.ncap2, w.d)); hv_c = np.zeros_like(hk_c)
    for b in range(w.B):
        lo, hi = int(x["blk_lo"][b]), int(x["blk_hi"][b])
        if hi > lo:
            k_c[b, lo:hi] = compress(x["k_raw"][b], x["z"][b], w.m, lo, hi, store)
            v_c[b, lo:hi] = compress(x["v_raw"][b], x["z"][b], w.m, lo, hi, store)
            ik_c[b, lo:hi] = compress(x["ik_raw"][b], x["z"][b], w.m, lo, hi, istore)
        lo, hi = int(x["hblk_lo"][b]), int(x["hblk_hi"][b])
        if hi > lo:
            hk_c[b, lo:hi] = compress(x["hk_raw"][b], x["hz"][b], w.m2, lo, hi, store)
            hv_c[b, lo:hi] = compress(x["hv_raw"][b], x["hz"][b], w.m2, lo, hi, store)
    out.update(k_c=k_c, v_c=v_c, ik_c=ik_c, hk_c=hk_c, hv_c=hv_c)
    return out


# --------------------------------------------------------------- backward
# The gradient of one pass for a loss whose gradient with respect to the
# attention outputs is given (dO for the CSA layer, dhO for the HCA layer).
# The top-k selection is a constant mask ("EP 95. DeepSeek-V4 논문 읽기 — 노정석",
# IDEAS: top-k selection is not differentiable), so the indexer (its queries,
# weights and keys) gets no gradient; the gradient flows to the queries, to
# the attended cache rows and window rows, and through the pooling of the
# blocks compressed in this pass to the raw rows and their pooling logits.
# The storage rounding of the caches is taken as the identity.

def attend_backward(q: np.ndarray, keys: list, values: list, dO: np.ndarray, scale: float):
    """Gradient of ``attend`` for dL/dO = dO: (dq [rows,H,d], dK [n_total,d],
    dV [n_total,d]) with dK, dV per entry of the concatenated key multisets."""
    rows, H, d = q.shape
    off = np.zeros(rows + 1, dtype=np.int64)
    off[1:] = np.cumsum([len(k) for k in keys])
    n = int(off[-1])
    K = _c(np.concatenate([to_f64(k).reshape(-1, d) for k in keys]) if n else np.zeros((1, d)))
    V = _c(np.concatenate([to_f64(v).reshape(-1, d) for v in values]) if n else np.zeros((1, d)))
    dq = np.empty((rows, H, d))
    dK = np.empty((max(n, 1), d))
    dV = np.empty((max(n, 1), d))
    lib().orc_attend_backward(rows, H, d, scale, _c(to_f64(q)), off, K, V, _c(dO), dq, dK, dV)
    return dq, dK[:n], dV[:n], off


def compress_backward(x_ring: np.ndarray, z_ring: np.ndarray, m: int, blk_lo: int,
                      blk_hi: int, dXc: np.ndarray):
    """Gradient of ``compress`` (unrounded) for blocks [blk_lo, blk_hi):
    (dX [nb*m, d] of raw positions blk_lo*m .., dz [nb*m])."""
    R, d = x_ring.shape
    nb = blk_hi - blk_lo
    pos = np.arange(blk_lo * m, blk_hi * m) % R
    X = _c(to_f64(x_ring)[pos])
    Z = _c(np.asarray(z_ring, dtype=np.float64)[pos])
    dX = np.empty((nb * m, d))
    dz = np.zeros(nb * m)
    if nb > 0:
        lib().orc_compress_backward(nb, m, d, X, Z, _c(dXc), dX, dz)
    return dX, dz


def reference_backward(w, x: dict, dO: np.ndarray, dhO: np.ndarray, fwd: dict | None = None):
    """Gradients of one pass (all query rows) for dL/dO = dO [B,T,H,d] (CSA
    layer) and dL/dhO = dhO (HCA layer), given the forward ``fwd`` (from
    ``reference``; computed if None).  Returns dq, dq_hca [B,T,H,d]; dk_c,
    dv_c [B,ncap,d] and dhk_c, dhv_c [B,ncap2,d] (cache rows as attended);
    dk_raw, dv_raw, dhk_raw, dhv_raw [B,R,d] (window rows plus the pooling of
    this pass's blocks); dz, dhz [B,R]."""
    B, T, H, d = w.B, w.T, w.H, w.d
    R = w.ring
    if fwd is None:
        fwd = reference(w, x)
    out = {}
    pos = x["q_pos"].reshape(-1).astype(np.int64)
    rows = np.arange(B * T)
    for layer in ("csa", "hca"):
        hca = layer == "hca"
        qn, kc_n, vc_n, kr_n, vr_n = (("q_hca", "hk_c", "hv_c", "hk_raw", "hv_raw") if hca else
                                      ("q", "k_c", "v_c", "k_raw", "v_raw"))
        kc, vc = fwd[kc_n], fwd[vc_n]
        keys, vals, src = [], [], []
        for r in rows:
            b, t = int(r // T), int(pos[r])
            win = window_positions(t, w.W) % R
            if hca:
                sel = np.arange((t + 1) // w.m2)
                K, V = hca_keys(b, t, w.m2, kc, vc, x[kr_n], x[vr_n], w.W)
            else:
                sel = fwd["idx"][r][fwd["idx"][r] >= 0]
                K, V = csa_keys(b, t, fwd["idx"][r], kc, vc, x[kr_n], x[vr_n], w.W)
            keys.append(K)
            vals.append(V)
            src.append((b, sel, win))
        g = (dhO if hca else dO).reshape(B * T, H, d).astype(np.float64)
        dq, dK, dV, off = attend_backward(x[qn].reshape(B * T, H, d), keys, vals, g, w.sm_scale)
        dkc = np.zeros(kc.shape)
        dvc = np.zeros(vc.shape)
        dkr = np.zeros((B, R, d))
        dvr = np.zeros((B, R, d))
        for r, (b, sel, win) in enumerate(src):
            o = off[r]
            ns = len(sel)
            np.add.at(dkc[b], sel, dK[o:o + ns])
            np.add.at(dvc[b], sel, dV[o:o + ns])
            np.add.at(dkr[b], win, dK[o + ns:off[r + 1]])
            np.add.at(dvr[b], win, dV[o + ns:off[r + 1]])
        # the pooling of this pass's blocks: cache-row gradients to raw rows
        m = w.m2 if hca else w.m
        zn = "hz" if hca else "z"
        lo_n, hi_n = ("hblk_lo", "hblk_hi") if hca else ("blk_lo", "blk_hi")
        dz = np.zeros((B, R))
        for b in range(B):
            lo, hi = int(x[lo_n][b]), int(x[hi_n][b])
            if hi <= lo:
                continue
            rr = np.arange(lo * m, hi * m) % R
            for src_n, dc, dr in ((kr_n, dkc, dkr), (vr_n, dvc, dvr)):
                dX, dzp = compress_backward(x[src_n][b], x[zn][b], m, lo, hi, dc[b, lo:hi])
                np.add.at(dr[b], rr, dX)
                np.add.at(dz[b], rr, dzp)
        pre = "h" if hca else ""
        out["dq_hca" if hca else "dq"] = dq.reshape(B, T, H, d)
        out[f"d{pre}k_c"], out[f"d{pre}v_c"] = dkc, dvc
        out[f"d{pre}k_raw"], out[f"d{pre}v_raw"] = dkr, dvr
        out["dhz" if hca else "dz"] = dz
    return out
