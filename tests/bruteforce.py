"""Brute-force restatement of the path for tiny inputs, written apart from the
oracle and in a different formulation, to pin it:

* compression as one dense pooling matrix P [n_blocks, L] applied to X;
* indexer scores by an einsum over heads;
* top-k by a full lexicographic sort of (-score, index);
* attention over the concatenated key matrix [compressed rows; raw rows] with
  an additive 0 / -inf mask, softmax by scipy's logsumexp.

numpy / scipy only.  Used by the CPU tests, never by the product path.
"""
from __future__ import annotations

import numpy as np
from scipy.special import logsumexp


def bf16_to_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def pooling_matrix(L: int, m: int, z: np.ndarray) -> np.ndarray:
    """P[j, p] = softmax weight of raw position p inside block j (0 elsewhere)."""
    nb = L // m
    P = np.zeros((nb, L))
    for j in range(nb):
        zz = z[j * m:(j + 1) * m].astype(np.float64)
        e = np.exp(zz - zz.max())
        P[j, j * m:(j + 1) * m] = e / e.sum()
    return P


def scores(qI: np.ndarray, w: np.ndarray, IkC: np.ndarray, nvis: np.ndarray) -> np.ndarray:
    """qI [rows,HI,dI], w [rows,HI], IkC [n,dI] (one sequence)."""
    dots = np.einsum("rhc,jc->rhj", qI, IkC)
    s = np.einsum("rh,rhj->rj", w, np.maximum(dots, 0.0))
    n = IkC.shape[0]
    mask = np.arange(n)[None, :] >= np.asarray(nvis)[:, None]
    s[mask] = -np.inf
    return s


def topk(s: np.ndarray, nvis: np.ndarray, k: int) -> np.ndarray:
    rows, n = s.shape
    out = np.full((rows, k), -1, dtype=np.int32)
    for r in range(rows):
        nv = int(nvis[r])
        cand = np.arange(nv)
        order = np.lexsort((cand, -s[r, :nv]))   # primary: -score, secondary: index
        pick = np.sort(cand[order[:min(k, nv)]])
        out[r, :len(pick)] = pick
    return out


def attention_masked(q: np.ndarray, Kall: np.ndarray, Vall: np.ndarray, mask: np.ndarray,
                     scale: float):
    """q [rows,H,d]; Kall/Vall [n,d]; mask [rows,n] bool (True = attended).
    A key may appear several times in Kall (multiset)."""
    lg = scale * np.einsum("rhd,nd->rhn", q, Kall)
    lg = np.where(mask[:, None, :], lg, -np.inf)
    lse = logsumexp(lg, axis=-1)
    empty = ~mask.any(axis=1)
    lse[empty] = -np.inf
    p = np.exp(lg - np.where(np.isfinite(lse), lse, 0.0)[..., None])
    p[empty] = 0.0
    O = np.einsum("rhn,nd->rhd", p, Vall)
    return O, lse


def csa(q, qI, w, t, X, V, Ik, z, m, k, W, scale, store=None):
    """Whole CSA for one sequence with raw arrays X,V [L,d], Ik [L,dI], logits z [L].
    Returns (Kc, Vc, IkC, s, idx, O, lse)."""
    L = X.shape[0]
    P = pooling_matrix(L, m, z)
    Kc, Vc, IkC = P @ X, P @ V, P @ Ik
    if store is not None:
        Kc, Vc, IkC = store(Kc), store(Vc), store(IkC)
    nvis = (np.asarray(t) + 1) // m
    s = scores(qI, w, IkC, nvis)
    idx = topk(s, nvis, k)
    n = Kc.shape[0]
    Kall = np.concatenate([Kc, X])
    Vall = np.concatenate([Vc, V])
    mask = np.zeros((len(t), n + L), dtype=bool)
    for r, tt in enumerate(t):
        sel = idx[r][idx[r] >= 0]
        mask[r, sel] = True
        lo = max(0, tt - W + 1)
        mask[r, n + lo:n + tt + 1] = True
    O, lse = attention_masked(q, Kall, Vall, mask, scale)
    return Kc, Vc, IkC, s, idx, O, lse


def hca(q, t, X, V, z, m2, W, scale, store=None):
    L = X.shape[0]
    P = pooling_matrix(L, m2, z)
    Kc, Vc = P @ X, P @ V
    if store is not None:
        Kc, Vc = store(Kc), store(Vc)
    n = Kc.shape[0]
    Kall = np.concatenate([Kc, X])
    Vall = np.concatenate([Vc, V])
    mask = np.zeros((len(t), n + L), dtype=bool)
    for r, tt in enumerate(t):
        mask[r, :(tt + 1) // m2] = True
        lo = max(0, tt - W + 1)
        mask[r, n + lo:n + tt + 1] = True
    O, lse = attention_masked(q, Kall, Vall, mask, scale)
    return Kc, Vc, O, lse
