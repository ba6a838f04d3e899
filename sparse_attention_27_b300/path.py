"""One pass of the hybrid compressed attention hot path through the C ABI.

``HybridStep`` owns the output buffers and scratch of one decode step (or
prefill chunk) and issues, in order, the library calls of the two layer
kinds:

  CSA layer:  csa_compress -> csa_index_topk -> csa_attend
              (or csa_decode, the same layer in one launch, for one query
              per sequence)
  HCA layer:  hca_compress_attend

(CSA and HCA are different layers, interleaved in the model -- "오픈소스 LLM의
새 이정표: DeepSeek-V4 시리즈", section "기존의 벽을 허문 아키텍처: 하이브리드 압축
어텐션" -- so their outputs are not merged with each other; each layer has its
own caches and sliding window.)  torch is used only to allocate device memory
and to provide streams; all arithmetic runs in libsa27's kernels.

Tensor names (device tensors, layouts row-major):
  q, q_hca [B,T,H,d]; q_idx [B,T,HI,dI] (bf16 also for the MXFP4 indexer:
  each pass quantises it to MXFP4 codes + scales before scoring);
  w_idx [B,T,HI] f32; q_pos [B,T] int32;
  k_raw, v_raw [B,R,d]; ik_raw [B,R,dI]; z [B,R] f32 (CSA layer ring);
  hk_raw, hv_raw [B,R,d]; hz [B,R] f32 (HCA layer ring);
  k_c, v_c [B,ncap,d]; ik_c [B,ncap,dI] (MXFP4: ik_c = codes [B,ncap,dI/2] u8
  and ik_c_scales [B,ncap,dI/32] u8);
  hk_c, hv_c [B,ncap2,d];
  blk_lo, blk_hi, hblk_lo, hblk_hi [B] int32 (blocks compressed this pass).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (SA_BF16, SA_F32, SA_MXFP4, csa_attend, csa_attend_backward,
               csa_attend_workspace_bytes, csa_compress, csa_decode, csa_index_topk,
               csa_index_topk_workspace_bytes, hca_attend_backward, hca_compress_attend,
               hca_compress_attend_workspace_bytes, sa_compress_backward, sa_decode_step,
               sa_decode_step_workspace_bytes, sa_mxfp4_quantize)

_CODES = {"f32": SA_F32, "bf16": SA_BF16, "mxfp4": SA_MXFP4}


@dataclass
class Dims:
    B: int
    T: int
    H: int
    d: int
    HI: int
    dI: int
    m: int
    k: int
    W: int
    m2: int
    R: int
    ncap: int
    ncap2: int
    dtype: str          # "bf16" or "f32" (K/V/q storage)
    indexer: str        # "bf16", "f32" or "mxfp4"
    sm_scale: float
    max_blocks: int     # bound on CSA blocks compressed per sequence this pass
    max_blocks2: int    # bound on HCA blocks compressed per sequence this pass
    o_dtype: str = "f32"  # attention output O of both layers: "f32" or "bf16"


class HybridStep:
    def __init__(self, dims: Dims, x: dict, device="cuda"):
        self.D, self.x = dims, x
        D = dims
        rows = D.B * D.T
        dev = torch.device(device)
        self.idx = torch.empty((D.B, D.T, D.k), dtype=torch.int32, device=dev)
        odt = torch.bfloat16 if D.o_dtype == "bf16" else torch.float32
        self.o = torch.empty((D.B, D.T, D.H, D.d), dtype=odt, device=dev)
        self.lse = torch.empty((D.B, D.T, D.H), dtype=torch.float32, device=dev)
        self.ho = torch.empty_like(self.o)
        self.hlse = torch.empty_like(self.lse)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        dt = _CODES[D.dtype]
        self.ws_index = csa_index_topk_workspace_bytes(D.B, D.T, D.ncap, D.k)
        self.ws_attend = csa_attend_workspace_bytes(dt, D.B, D.T, D.H, D.d, D.k, D.W)
        self.ws_hca = hca_compress_attend_workspace_bytes(dt, D.B, D.T, D.H, D.d, D.ncap2, D.W)
        self.ws_a = torch.empty(max(self.ws_index, 256), dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(max(self.ws_attend, 256), dtype=torch.uint8, device=dev)
        self.ws_c = torch.empty(max(self.ws_hca, 256), dtype=torch.uint8, device=dev)
        self.scores = None
        self.ws_step = None
        if D.indexer == "mxfp4":
            self.q_codes = torch.empty((D.B, D.T, D.HI, D.dI // 2), dtype=torch.uint8, device=dev)
            self.q_scales = torch.empty((D.B, D.T, D.HI, D.dI // 32), dtype=torch.uint8,
                                        device=dev)
        assert rows > 0

    # -------------------------------------------------------------- layers
    def compress_csa(self, stream=None):
        D, x = self.D, self.x
        csa_compress(_CODES[D.dtype], _CODES[D.indexer], D.B, D.d, D.dI, D.m, x["k_raw"],
                     x["v_raw"], x["ik_raw"], x["z"], D.R, x["blk_lo"], x["blk_hi"], D.max_blocks,
                     x["k_c"], x["v_c"], x["ik_c"], x.get("ik_c_scales"), D.ncap, err=self.err,
                     stream=stream)

    def index_topk(self, stream=None, scores_out=None, scores_in=None):
        D, x = self.D, self.x
        q, q_scales = x["q_idx"], None
        if D.indexer == "mxfp4" and scores_in is None:
            sa_mxfp4_quantize(x["q_idx"], self.q_codes, self.q_scales, stream=stream)
            q, q_scales = self.q_codes, self.q_scales
        csa_index_topk(_CODES[D.indexer], D.B, D.T, D.HI, D.dI, D.m, D.k, q,
                       q_scales, x["w_idx"], x["ik_c"], x.get("ik_c_scales"), D.ncap,
                       x["q_pos"], self.idx, scores_out=scores_out, scores_in=scores_in,
                       ws=self.ws_a, ws_bytes=self.ws_a.numel(), err=self.err, stream=stream)

    def index_topk_split(self, stream, scored):
        """index_topk as two calls on ``stream``: the indexer scores into the
        workspace (top-k size 0), event ``scored``, then the top-k from those
        scores -- the same two kernels, with a point in between that another
        stream can wait for."""
        D, x = self.D, self.x
        sc = self.ws_a[: D.B * D.T * D.ncap * 4].view(torch.float32)
        q, q_scales = x["q_idx"], None
        if D.indexer == "mxfp4":
            sa_mxfp4_quantize(x["q_idx"], self.q_codes, self.q_scales, stream=stream)
            q, q_scales = self.q_codes, self.q_scales
        csa_index_topk(_CODES[D.indexer], D.B, D.T, D.HI, D.dI, D.m, 0, q, q_scales, x["w_idx"],
                       x["ik_c"], x.get("ik_c_scales"), D.ncap, x["q_pos"], None,
                       scores_out=sc, err=self.err, stream=stream)
        scored.record(stream)
        csa_index_topk(_CODES[D.indexer], D.B, D.T, D.HI, D.dI, D.m, D.k, None, None, None, None,
                       None, D.ncap, x["q_pos"], self.idx, scores_in=sc, err=self.err,
                       stream=stream)

    def attend_csa(self, stream=None, idx=None):
        D, x = self.D, self.x
        csa_attend(_CODES[D.dtype], D.B, D.T, D.H, D.d, D.m, D.k, D.W, D.sm_scale, x["q"],
                   x["q_pos"], x["k_c"], x["v_c"], D.ncap, self.idx if idx is None else idx,
                   x["k_raw"], x["v_raw"], D.R, self.o, self.lse, ws=self.ws_b,
                   ws_bytes=self.ws_b.numel(), err=self.err, stream=stream)

    def hca(self, stream=None):
        D, x = self.D, self.x
        hca_compress_attend(_CODES[D.dtype], D.B, D.T, D.H, D.d, D.m2, D.W, D.sm_scale, x["q_hca"],
                            x["q_pos"], x["hk_raw"], x["hv_raw"], x["hz"], D.R, x["hblk_lo"],
                            x["hblk_hi"], D.max_blocks2, x["hk_c"], x["hv_c"], D.ncap2, self.ho,
                            self.hlse, ws=self.ws_c, ws_bytes=self.ws_c.numel(), err=self.err,
                            stream=stream)

    def csa(self, stream=None):
        self.compress_csa(stream)
        self.index_topk(stream)
        self.attend_csa(stream)

    def fused_ok(self) -> bool:
        """Whether csa_decode takes this pass: one bf16 query per sequence
        with the bf16 indexer, 64 x 64 indexer heads, head dim 128."""
        D = self.D
        return (D.T == 1 and D.dtype == "bf16" and D.indexer == "bf16" and D.HI == 64 and
                D.dI == 64 and D.d == 128 and D.H <= 64)

    def csa_fused(self, stream=None):
        """The CSA layer in one launch (csa_decode): compress the blocks this
        pass closes, index, top-k and attend."""
        D, x = self.D, self.x
        csa_decode(D.B, D.H, D.d, D.HI, D.dI, D.m, D.k, D.W, D.sm_scale, x["q"], x["q_idx"],
                   x["w_idx"], x["q_pos"], x["k_raw"], x["v_raw"], x["ik_raw"], x["z"], D.R,
                   x["blk_lo"], x["blk_hi"], D.max_blocks, x["k_c"], x["v_c"], x["ik_c"], D.ncap,
                   self.idx, self.o, self.lse, err=self.err, stream=stream)

    def step_ok(self) -> bool:
        """Whether sa_decode_step takes this pass: csa_decode's shapes, rows
        of at most 32768 compressed entries, blocks of at most 128 rows."""
        D = self.D
        return (self.fused_ok() and D.m <= 128 and D.m2 <= 128 and
                sa_decode_step_workspace_bytes(D.B, D.H, D.ncap, D.k, D.W, D.ncap2) > 0)

    def decode_step(self, stream=None):
        """Both layers of the pass in one launch (sa_decode_step)."""
        D, x = self.D, self.x
        if self.ws_step is None:
            n = sa_decode_step_workspace_bytes(D.B, D.H, D.ncap, D.k, D.W, D.ncap2)
            self.ws_step = torch.empty(max(n, 256), dtype=torch.uint8, device=self.o.device)
        sa_decode_step(D.B, D.H, D.d, D.HI, D.dI, D.m, D.k, D.W, D.m2, D.sm_scale, x["q"],
                       x["q_idx"], x["w_idx"], x["q_hca"], x["q_pos"], x["k_raw"], x["v_raw"],
                       x["ik_raw"], x["z"], x["hk_raw"], x["hv_raw"], x["hz"], D.R, x["blk_lo"],
                       x["blk_hi"], D.max_blocks, x["hblk_lo"], x["hblk_hi"], D.max_blocks2,
                       x["k_c"], x["v_c"], x["ik_c"], D.ncap, x["hk_c"], x["hv_c"], D.ncap2,
                       self.idx, self.o, self.lse, self.ho, self.hlse, self.ws_step,
                       err=self.err, stream=stream)

    def run(self, stream=None):
        """The whole pass on one stream."""
        self.csa(stream)
        self.hca(stream)

    def run_two_streams(self, s_csa: torch.cuda.Stream, s_hca: torch.cuda.Stream):
        """The CSA and HCA layers on two streams (they share no buffer).  The
        HCA layer starts once the CSA indexer's scores are written: the score
        kernel, the step's largest HBM stream, then has the GPU to itself, and
        HCA overlaps the top-k and the CSA attention."""
        cur = torch.cuda.current_stream()
        ev = torch.cuda.Event()
        ev.record(cur)
        s_csa.wait_event(ev)
        s_hca.wait_event(ev)
        self.compress_csa(s_csa)
        scored = torch.cuda.Event()
        self.index_topk_split(s_csa, scored)
        self.attend_csa(s_csa)
        s_hca.wait_event(scored)
        self.hca(s_hca)
        e1, e2 = torch.cuda.Event(), torch.cuda.Event()
        e1.record(s_csa)
        e2.record(s_hca)
        cur.wait_event(e1)
        cur.wait_event(e2)

    def run_fused_two_streams(self, s_csa: torch.cuda.Stream, s_hca: torch.cuda.Stream):
        """The CSA layer in one launch (csa_decode) on one stream and the HCA
        layer on another, both starting at once (they share no buffer)."""
        cur = torch.cuda.current_stream()
        ev = torch.cuda.Event()
        ev.record(cur)
        s_csa.wait_event(ev)
        s_hca.wait_event(ev)
        self.csa_fused(s_csa)
        self.hca(s_hca)
        e1, e2 = torch.cuda.Event(), torch.cuda.Event()
        e1.record(s_csa)
        e2.record(s_hca)
        cur.wait_event(e1)
        cur.wait_event(e2)

    def backward(self, dout, dhout, idx=None, o=None, lse=None, ho=None, hlse=None,
                 stream=None) -> dict:
        """Gradients of this pass for dL/dO = dout and dL/dhO = dhout (f32
        [B,T,H,d]), the selection (idx, default this pass's) held fixed.  The
        forward's O and LSE default to this pass's outputs (o_dtype "f32").
        Returns fresh f32 tensors: dq, dq_hca; dk_c, dv_c, dhk_c, dhv_c (cache
        rows as attended); dk_raw, dv_raw, dhk_raw, dhv_raw (window rows and
        the pooling of this pass's blocks); dz, dhz."""
        D, x = self.D, self.x
        dt = _CODES[D.dtype]
        dev = self.o.device
        f = lambda shape: torch.zeros(shape, dtype=torch.float32, device=dev)
        g = {"dq": f((D.B, D.T, D.H, D.d)), "dq_hca": f((D.B, D.T, D.H, D.d)),
             "dk_c": f((D.B, D.ncap, D.d)), "dv_c": f((D.B, D.ncap, D.d)),
             "dhk_c": f((D.B, D.ncap2, D.d)), "dhv_c": f((D.B, D.ncap2, D.d)),
             "dk_raw": f((D.B, D.R, D.d)), "dv_raw": f((D.B, D.R, D.d)),
             "dhk_raw": f((D.B, D.R, D.d)), "dhv_raw": f((D.B, D.R, D.d)),
             "dz": f((D.B, D.R)), "dhz": f((D.B, D.R))}
        o = self.o if o is None else o
        lse = self.lse if lse is None else lse
        ho = self.ho if ho is None else ho
        hlse = self.hlse if hlse is None else hlse
        csa_attend_backward(dt, D.B, D.T, D.H, D.d, D.m, D.k, D.W, D.sm_scale, x["q"], x["q_pos"],
                            x["k_c"], x["v_c"], D.ncap, self.idx if idx is None else idx,
                            x["k_raw"], x["v_raw"], D.R, o, lse, dout, g["dq"], g["dk_c"],
                            g["dv_c"], g["dk_raw"], g["dv_raw"], err=self.err, stream=stream)
        hca_attend_backward(dt, D.B, D.T, D.H, D.d, D.m2, D.W, D.sm_scale, x["q_hca"],
                            x["q_pos"], x["hk_c"], x["hv_c"], D.ncap2, x["hk_raw"], x["hv_raw"],
                            D.R, ho, hlse, dhout, g["dq_hca"], g["dhk_c"], g["dhv_c"],
                            g["dhk_raw"], g["dhv_raw"], err=self.err, stream=stream)
        sa_compress_backward(dt, D.B, D.d, D.m, x["k_raw"], x["v_raw"], x["z"], D.R, x["blk_lo"],
                             x["blk_hi"], D.max_blocks, g["dk_c"], g["dv_c"], D.ncap,
                             g["dk_raw"], g["dv_raw"], g["dz"], err=self.err, stream=stream)
        sa_compress_backward(dt, D.B, D.d, D.m2, x["hk_raw"], x["hv_raw"], x["hz"], D.R,
                             x["hblk_lo"], x["hblk_hi"], D.max_blocks2, g["dhk_c"], g["dhv_c"],
                             D.ncap2, g["dhk_raw"], g["dhv_raw"], g["dhz"], err=self.err,
                             stream=stream)
        return g

    def device_errors(self) -> int:
        return int(self.err.item())


# ------------------------------------------------------------ host arrays
# Helpers that upload one pass's inputs, given as numpy arrays in the
# storage formats of the C ABI (bf16 as uint16 bit patterns, f32, int32),
# and build the HybridStep that runs them.  ``w`` is any object with the
# shape fields of a workload (B, T, H, d, HI, dI, m, k, W, m2, ring, ncap,
# ncap2, dtype, indexer, sm_scale, mode).

def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy -> device tensor; uint16 arrays are bfloat16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    """device tensor -> numpy; bfloat16 comes back as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def dims_from(w, x: dict, o_dtype: str = "f32") -> Dims:
    """The Dims of one pass: shapes from ``w``, compression bounds from the
    block ranges in ``x``."""
    return Dims(o_dtype=o_dtype, B=w.B, T=w.T, H=w.H, d=w.d, HI=w.HI, dI=w.dI, m=w.m, k=w.k, W=w.W, m2=w.m2,
                R=w.ring, ncap=w.ncap, ncap2=w.ncap2, dtype=w.dtype, indexer=w.indexer,
                sm_scale=w.sm_scale,
                max_blocks=int((x["blk_hi"] - x["blk_lo"]).max()),
                max_blocks2=int((x["hblk_hi"] - x["hblk_lo"]).max()))


def device_inputs(w, x: dict, device="cuda") -> dict:
    """Every array of ``x`` on the device.  An MXFP4 indexer keeps its key
    cache as codes and scales, written by the library's quantiser from the
    given bf16 cache (or zero for a prefill, whose compressor writes them).
    A prefill gets zeroed caches for its compressors to fill."""
    from . import sa_mxfp4_quantize
    t = {k: to_device(v, device) for k, v in x.items()}
    if w.indexer == "mxfp4":
        ik = t.pop("ik_c", None)
        codes = torch.zeros((w.B, w.ncap, w.dI // 2), dtype=torch.uint8, device=device)
        scales = torch.zeros((w.B, w.ncap, w.dI // 32), dtype=torch.uint8, device=device)
        if ik is not None:
            sa_mxfp4_quantize(ik, codes, scales)
        t["ik_c"], t["ik_c_scales"] = codes, scales
    if w.mode == "prefill":
        cdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        idt = torch.bfloat16 if w.indexer in ("bf16", "mxfp4") else torch.float32
        t["k_c"] = torch.zeros((w.B, w.ncap, w.d), dtype=cdt, device=device)
        t["v_c"] = torch.zeros_like(t["k_c"])
        if w.indexer != "mxfp4":
            t["ik_c"] = torch.zeros((w.B, w.ncap, w.dI), dtype=idt, device=device)
        t["hk_c"] = torch.zeros((w.B, w.ncap2, w.d), dtype=cdt, device=device)
        t["hv_c"] = torch.zeros_like(t["hk_c"])
    return t


def step_from(w, x: dict, device="cuda", o_dtype: str = "f32") -> HybridStep:
    """A HybridStep over ``x`` uploaded to ``device``, with attention outputs
    in ``o_dtype``."""
    return HybridStep(dims_from(w, x, o_dtype), device_inputs(w, x, device), device)
