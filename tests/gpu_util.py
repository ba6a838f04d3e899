"""Helpers for the GPU tests: move synth inputs to the device and run the
path through the C ABI (sparse_attention_27_b300), then bring results back as
numpy for comparison with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import synth


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy -> device tensor; uint16 arrays are bfloat16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    """device tensor -> numpy; bfloat16 comes back as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def dims_of(w: synth.Workload, x: dict):
    from sparse_attention_27_b300.path import Dims
    return Dims(B=w.B, T=w.T, H=w.H, d=w.d, HI=w.HI, dI=w.dI, m=w.m, k=w.k, W=w.W, m2=w.m2,
                R=w.ring, ncap=w.ncap, ncap2=w.ncap2, dtype=w.dtype, indexer=w.indexer,
                sm_scale=w.sm_scale,
                max_blocks=int((x["blk_hi"] - x["blk_lo"]).max()),
                max_blocks2=int((x["hblk_hi"] - x["hblk_lo"]).max()))


def device_inputs(w: synth.Workload, x: dict, device="cuda") -> dict:
    t = {k: dev(v, device) for k, v in x.items()}
    if w.indexer == "mxfp4":
        # the indexer key cache is stored as MXFP4: quantise the drawn bf16 cache
        # with the library's quantiser (prefill: empty cache, written by compress)
        import sparse_attention_27_b300 as sa
        ik = t.pop("ik_c", None)
        codes = torch.zeros((w.B, w.ncap, w.dI // 2), dtype=torch.uint8, device=device)
        scales = torch.zeros((w.B, w.ncap, w.dI // 32), dtype=torch.uint8, device=device)
        if ik is not None:
            sa.sa_mxfp4_quantize(ik, codes, scales)
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


def make_step(w: synth.Workload, x: dict, device="cuda"):
    from sparse_attention_27_b300.path import HybridStep
    return HybridStep(dims_of(w, x), device_inputs(w, x, device), device)
