"""Benchmark: CSA + HCA decode query-tokens/s at 128K context on B300.

One step = one decode token for each of the 32 sequences through one CSA
layer (compress the block the token closes, indexer scores, top-k 2048,
sparse attention over the selected rows + a 128-token window) and one HCA
layer (compress the closing 128-token block, dense attention over all 1024
HCA rows + the window), on synthetic seeded inputs of the 128K decode shape.
The two layers run on two streams (they share no data) inside one captured
CUDA graph.  Before every timed step, outside the timed interval, L2 is
flushed by a 512 MiB write and then a 256 MiB read (the read writes back the
flush's dirty lines, so the step starts from a clean L2 that holds none of its
inputs); each step is timed with CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode128k|decode1m]

Prints one JSON line.  Multi-GPU (torchrun): every rank runs its own batch of
32 sequences (weak scaling, no data-path collective); time = max over ranks.
``--impl reference`` times the float64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA+HCA decode query-tokens/s at 128K and 1M ctx; HBM GB/s vs peak"
UNIT = "query-tokens/s"
WORKLOAD = "decode128k"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# Sources of the dominant kernel; the ncu DRAM traffic recorded in
# profiles/traffic.txt is reported only while these files hash to the value
# recorded with it (a changed kernel has no valid traffic figure).
SCORE_SOURCES = ["sparse_attention_27_b300/csrc/score_tc.cu", "sparse_attention_27_b300/csrc/common.cuh",
                 "sparse_attention_27_b300/csrc/kernels.cuh"]
FUSED_SOURCES = ["sparse_attention_27_b300/csrc/decode_fused.cu",
                 "sparse_attention_27_b300/csrc/common.cuh", "sparse_attention_27_b300/csrc/kernels.cuh",
                 "sparse_attention_27_b300/csrc/topk_dev.cuh",
                 "sparse_attention_27_b300/csrc/compress_dev.cuh"]
STEP_SOURCES = ["sparse_attention_27_b300/csrc/decode_step.cu",
                "sparse_attention_27_b300/csrc/common.cuh", "sparse_attention_27_b300/csrc/kernels.cuh",
                "sparse_attention_27_b300/csrc/topk_dev.cuh",
                "sparse_attention_27_b300/csrc/compress_dev.cuh"]
MX_SOURCES = ["sparse_attention_27_b300/csrc/score_mx.cu", "sparse_attention_27_b300/csrc/common.cuh",
              "sparse_attention_27_b300/csrc/kernels.cuh", "sparse_attention_27_b300/csrc/score_jobs.cuh"]


def source_hash(files) -> str:
    import hashlib
    h = hashlib.sha1()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, files, alg_bytes: int):
    """(bytes per launch, capture note) from profiles/traffic.txt, or (None, why).

    A capture of another workload of the same kernel is scaled to this one by
    the algorithmic bytes the two launches move (the kernel reads each byte
    once, so its traffic grows in proportion)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    cur = source_hash(files)
    try:
        for line in open(path):
            f = line.split()
            if len(f) >= 4 and not line.startswith("#") and f[0] == kernel:
                if f[1] != cur:
                    return None, "kernel changed since the ncu capture"
                dram, cap_alg, note = int(f[2]), int(f[3]), " ".join(f[4:])
                if cap_alg == alg_bytes:
                    return dram, note
                return (round(dram * alg_bytes / cap_alg),
                        f"scaled by algorithmic bytes {alg_bytes}/{cap_alg} from: {note}")
    except OSError:
        pass
    return None, "no ncu capture recorded"


def max_over_ranks(v: float, device=None) -> float:
    """The largest v over the ranks of the default process group (v itself
    without one): the only collective of a multi-GPU run, which shards the
    decode batch with no exchange on the data path."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def graph_kernels(graph, cudart) -> list:
    """Function names of the kernel nodes of a captured (not yet instantiated)
    CUDA graph, read back through the runtime's graph API."""
    ct = ctypes

    class KernelNodeParams(ct.Structure):
        _fields_ = [("func", ct.c_void_p), ("grid", ct.c_uint * 3), ("block", ct.c_uint * 3),
                    ("smem", ct.c_uint), ("params", ct.c_void_p), ("extra", ct.c_void_p)]

    n = ct.c_size_t(0)
    if cudart.cudaGraphGetNodes(ct.c_void_p(graph), None, ct.byref(n)) != 0:
        raise RuntimeError("cudaGraphGetNodes failed")
    nodes = (ct.c_void_p * n.value)()
    cudart.cudaGraphGetNodes(ct.c_void_p(graph), nodes, ct.byref(n))
    names = []
    for nd in nodes:
        kind = ct.c_int(-1)
        cudart.cudaGraphNodeGetType(ct.c_void_p(nd), ct.byref(kind))
        if kind.value != 0:                      # cudaGraphNodeTypeKernel
            continue
        prm = KernelNodeParams()
        name = ct.c_char_p()
        if (cudart.cudaGraphKernelNodeGetParams(ct.c_void_p(nd), ct.byref(prm)) == 0 and
                cudart.cudaFuncGetName(ct.byref(name), ct.c_void_p(prm.func)) == 0 and name.value):
            names.append(name.value.decode(errors="replace"))
        else:
            names.append("?")
    return names


def algorithmic_bytes(w, o_bytes: int = 4) -> dict:
    """Minimum bytes one decode step must move (each needed row read once);
    the attention output O is written in elements of ``o_bytes``."""
    e = 2  # bf16
    if w.indexer == "mxfp4":        # e2m1 codes + one e8m0 scale per 32, keys and queries
        row = w.dI // 2 + w.dI // 32
        per_seq_index = w.ncap * row + w.HI * row + w.HI * 4
    else:
        per_seq_index = w.ncap * w.dI * e + w.HI * w.dI * e + w.HI * 4
    per_seq_csa = (per_seq_index + w.k * 2 * w.d * e + w.W * 2 * w.d * e + w.H * w.d * e
                   + w.k * 4 + w.H * w.d * o_bytes + w.H * 4)
    per_seq_hca = (w.ncap2 * 2 * w.d * e + w.W * 2 * w.d * e + w.H * w.d * e
                   + w.H * w.d * o_bytes + w.H * 4)
    return dict(index=per_seq_index * w.B, csa=per_seq_csa * w.B, hca=per_seq_hca * w.B,
                step=(per_seq_csa + per_seq_hca) * w.B)


def prefill_pairs(w, pos) -> dict:
    """(query, key) pairs of a prefill chunk, from its query positions: indexer
    scores over the visible compressed entries; CSA attention over the
    selected entries plus the window; HCA attention over every visible HCA
    entry plus the window."""
    import numpy as np
    t = np.asarray(pos, dtype=np.int64).reshape(-1)
    nc = (t + 1) // w.m
    nh = (t + 1) // w.m2
    win = np.minimum(w.W, t + 1)
    return dict(index=int(nc.sum()), csa=int((np.minimum(w.k, nc) + win).sum()),
                hca=int((nh + win).sum()))


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1800.0, "fallback"


def prefill_calls(steps: int, warmup: int, device: int = 0) -> dict:
    """Per-call times of the 64K prefill chunk (every position a query) and
    the tensor throughput of its contractions: indexer 2*HI*dI flops per
    score, attention 4*H*d per (query, key) pair (QK and PV).  The calls read
    GB-sized operands, far beyond L2, so no flush is needed between them.
    Each call is timed alone with CUDA events on the current stream, median
    of ``steps`` after ``warmup`` untimed calls."""
    import torch
    import synth
    from sparse_attention_27_b300.path import step_from
    import sparse_attention_27_b300 as sa
    w = synth.WORKLOADS["prefill64k"]
    x = synth.make_inputs(w)
    step = step_from(w, x, o_dtype="bf16")
    D = step.D
    sc = torch.empty((w.B, w.T, w.ncap), dtype=torch.float32, device="cuda")

    def timeit(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    with Clocks(device) as clk:
        ms = {"compress_csa": timeit(step.compress_csa)}
        ms["score"] = timeit(lambda: sa.csa_index_topk(
            sa.SA_BF16, D.B, D.T, D.HI, D.dI, D.m, 0, step.x["q_idx"], None, step.x["w_idx"],
            step.x["ik_c"], None, D.ncap, step.x["q_pos"], None, scores_out=sc))
        ms["topk"] = timeit(lambda: sa.csa_index_topk(
            sa.SA_BF16, D.B, D.T, D.HI, D.dI, D.m, D.k, None, None, None, None, None, D.ncap,
            step.x["q_pos"], step.idx, scores_in=sc))
        ms["attend_csa"] = timeit(step.attend_csa)
        ms["hca"] = timeit(step.hca)
    pairs = prefill_pairs(w, x["q_pos"])
    flops = {"score": pairs["index"] * 2 * w.HI * w.dI,
             "attend_csa": pairs["csa"] * 4 * w.H * w.d, "hca": pairs["hca"] * 4 * w.H * w.d}
    peak, peak_kind = bf16_peak()
    tf = {k: flops[k] / (ms[k] * 1e-3) / 1e12 for k in flops}
    errs = step.device_errors()
    total = sum(ms.values())
    out = {"workload": "prefill64k", "tokens": w.B * w.T, "steps": steps, "warmup": warmup,
           "ms": ms, "chunk_ms": total, "tokens_per_s": w.B * w.T / (total * 1e-3),
           "pairs": pairs, "tflop": {k: v / 1e12 for k, v in flops.items()}, "tflops": tf,
           "frac_of_bf16_peak": {k: v / peak for k, v in tf.items()},
           "bf16_peak_tflops": peak, "peak_source": peak_kind, "device_errors": errs,
           "clocks": clk.summary(),
           "note": "each call timed alone (CUDA events, median); O in bf16"}
    del step, sc, x
    torch.cuda.empty_cache()
    return out


def run_prefill_calls(args) -> None:
    print(json.dumps({"mode": "prefill-calls", **prefill_calls(args.steps, args.warmup)}),
          flush=True)


def fp32_alu_peak(device: int = 0) -> float:
    """fp32 CUDA-core peak in TFLOP/s: SMs x 128 fp32 lanes x 2 (FMA) x the
    SM clock's maximum (NVML), the bound of the backward's CUDA-core kernels."""
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = Clocks(device).max_mhz or 2032.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def backward_pairs(w, pos) -> dict:
    """(query, key) pairs of the backward's attention: CSA selected + window,
    HCA visible + window (as prefill_pairs)."""
    return prefill_pairs(w, pos)


def backward_calls(steps: int, warmup: int, device: int = 0) -> dict:
    """Time the backward of one pass -- csa_attend_backward,
    hca_attend_backward and the two sa_compress_backward calls -- at the 128K
    decode shape (32 rows) and on a 4096-token prefill chunk.  Flops: 10*H*d
    per (query, key) pair (S, dP, dq, dK and dV products)."""
    import torch
    import synth
    from sparse_attention_27_b300.path import step_from
    out = {}
    peak = fp32_alu_peak(device)
    for name, w in (("decode128k", synth.WORKLOADS["decode128k"]),
                    ("prefill4k", synth.Workload("prefill4k", "prefill", B=1, L=4096, T=4096,
                                                  x8=True))):
        x = synth.make_inputs(w)
        step = step_from(w, x, o_dtype="f32")
        step.run()
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        dO = torch.randn(step.o.shape, device="cuda", generator=g)
        dhO = torch.randn(step.o.shape, device="cuda", generator=g)
        for _ in range(warmup):
            step.backward(dO, dhO)
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step.backward(dO, dhO)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        pairs = backward_pairs(w, x["q_pos"])
        flop = (pairs["csa"] + pairs["hca"]) * 10 * w.H * w.d
        tf = flop / (ms * 1e-3) / 1e12
        out[name] = {"ms": ms, "tflop": flop / 1e12, "tflops": tf,
                     "roofline": {"bound": "alu", "achieved": tf, "peak": peak,
                                  "unit": "TFLOP/s", "frac": tf / peak,
                                  "peak_source": "SMs x 128 fp32 lanes x 2 x max SM clock"},
                     "device_errors": step.device_errors()}
        del step, x
        torch.cuda.empty_cache()
    out["note"] = ("backward of one pass (selection fixed): attention of both layers and the "
                   "pooling; fp32 CUDA-core kernels; gradient buffers allocated and zeroed "
                   "inside the timed call")
    return out


class Clocks:
    """SM clock and clock-event reasons sampled every ~2 ms by a background
    thread while the timed region runs, read through NVML (the driver's
    libnvidia-ml.so.1, via ctypes; reading only, no setting is changed)."""

    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, device: int):
        import ctypes
        import torch
        self.samples = []
        self.max_mhz = None
        self.h = None
        self.why = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device)
            u = str(props.uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            if nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) != 0:
                bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
                if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                    raise RuntimeError("no NVML handle for " + u + " / " + bus)
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.nv, self.h, self.ct = nv, h, ctypes
        except Exception as e:  # no NVML: report no samples, and why
            self.h = None
            self.why = str(e)

    def _loop(self):
        ct, nv = self.ct, self.nv
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop.is_set():
            if (nv.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0 and
                    nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ct.byref(rs)) == 0):
                self.samples.append((float(clk.value),
                                     [n for n, bit in self.REASONS.items() if rs.value & bit]))
            self.stop.wait(0.002)

    def __enter__(self):
        import threading
        self.stop = threading.Event()
        self.t = None
        if self.h is not None:
            self.t = threading.Thread(target=self._loop, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        self.stop.set()
        if self.t:
            self.t.join()

    def summary(self) -> dict:
        sm = [m for m, _ in self.samples]
        reasons = sorted({n for _, rs in self.samples for n in rs})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(sm)}
        if self.why:
            out["unavailable"] = self.why
        return out


def load_cudart():
    """The CUDA runtime library, for the graph API calls of graph_kernels."""
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    raise RuntimeError("libcudart not found")


class PipelinedIO:
    """End-to-end decode steps from pinned host memory, over three buffer sets.

    Three HybridSteps (buffer sets 0, 1, 2) share the caches and rings; each has
    its own per-step inputs -- q, q_hca, q_idx, w_idx, q_pos and the new
    token's ring rows (staged) -- in one device buffer filled by one copy from
    one pinned host buffer, and its own outputs (o, lse, ho, hlse) in one
    device buffer read back by one copy.  ``record`` captures n consecutive
    steps: while step k computes, step k + 1's inputs are already in place and
    step k - 1's outputs go out on a copy stream; a set's refill and readout
    have two steps' time before the set is used again.  Each step first writes its
    token into ring row t mod R of every layer's per-token arrays
    (sa_ring_write, one launch) on the CSA stream, before either layer runs.
    Every step's copies are inside the timed region."""

    IN = ["q", "q_hca", "q_idx", "w_idx", "q_pos"]
    RING = {"csa": ["k_raw", "v_raw", "ik_raw", "z"], "hca": ["hk_raw", "hv_raw", "hz"]}
    OUT = ["o", "lse", "ho", "hlse"]

    SETS = 3

    def __init__(self, w, x, mode: str):
        import numpy as np
        import torch
        from sparse_attention_27_b300.path import HybridStep, step_from
        self.mode = mode
        base = step_from(w, x, o_dtype="bf16")
        dev = base.o.device
        slot = (w.L - 1) % w.ring
        ring_names = self.RING["csa"] + self.RING["hca"]
        self.steps, self.d_in, self.h_in, self.d_out, self.h_out, self.staged = [], [], [], [], [], []
        for p in range(self.SETS):
            xs = dict(base.x)
            tens = [base.x[n] for n in self.IN] + [base.x[n][:, slot] for n in ring_names]
            buf, views = self._carve(tens, dev)
            for n, v in zip(self.IN, views[:len(self.IN)]):
                v.copy_(base.x[n])
                xs[n] = v
            staged = dict(zip(ring_names, views[len(self.IN):]))
            for n, v in staged.items():
                v.copy_(base.x[n][:, slot])
            st = base if p == 0 else HybridStep(base.D, xs, dev)
            if p == 0:
                for n in self.IN:
                    st.x[n] = xs[n]
            outs = [getattr(st, n) for n in self.OUT]
            obuf, oviews = self._carve(outs, dev)
            for n, v in zip(self.OUT, oviews):
                setattr(st, n, v)
            hbuf = torch.empty(buf.numel(), dtype=torch.uint8, pin_memory=True)
            hbuf.copy_(buf.cpu())
            self.steps.append(st)
            self.d_in.append(buf)
            self.h_in.append(hbuf)
            self.staged.append(staged)
            self.d_out.append(obuf)
            self.h_out.append(torch.empty(obuf.numel(), dtype=torch.uint8, pin_memory=True))
        self.slot = slot
        self.h2d_bytes = self.d_in[0].numel()
        self.d2h_bytes = self.d_out[0].numel()
        self.copies = 2

    @staticmethod
    def _carve(tensors, dev):
        import torch
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, device=dev)
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for o, t in zip(offs, tensors)]
        return buf, views

    def _compute(self, p, s_csa, s_hca):
        """Step p on the layer streams, scheduled as in the device-timed step
        (step: one sa_decode_step launch; fused: both layers at once; split:
        HCA after the CSA scores), after one sa_ring_write puts the step's
        new token into every ring."""
        import torch
        import sparse_attention_27_b300 as sa
        st = self.steps[p]
        names = self.RING["csa"] + self.RING["hca"]
        sa.sa_ring_write(st.D.B, st.D.R, st.x["q_pos"], [st.x[n] for n in names],
                         [self.staged[p][n] for n in names], err=st.err, stream=s_csa)
        if self.mode == "step":
            st.decode_step(s_csa)
            return
        ring = torch.cuda.Event()
        ring.record(s_csa)
        s_hca.wait_event(ring)
        if self.mode == "fused":
            st.csa_fused(s_csa)
            st.hca(s_hca)
        else:
            st.compress_csa(s_csa)
            scored = torch.cuda.Event()
            st.index_topk_split(s_csa, scored)
            st.attend_csa(s_csa)
            s_hca.wait_event(scored)
            st.hca(s_hca)

    def record(self, s_csa, s_hca, s_cp, s_out, n: int = 4):
        """n consecutive steps over the buffer sets (step k uses set k mod
        SETS).  The compute streams wait on each other directly: step k's
        CSA stream (its ring write, then the CSA layer) after step k - 1's HCA
        layer, step k's HCA stream after step k's ring write.  A step's inputs
        were copied in while the step before it ran; its outputs go out while
        the next one runs; its set is refilled from pinned memory for step
        k + SETS (or the next replay) once it is done, and step k + SETS writes
        the set's outputs only after they have gone out."""
        import torch
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        for s_ in (s_csa, s_hca, s_cp, s_out):
            s_.wait_event(start)
        in_ev = [None] * self.SETS                # inputs of set p in place
        out_ev = [None] * self.SETS               # outputs of set p copied out
        hca_done = None                           # the previous step's HCA layer
        for k in range(n):
            p = k % self.SETS
            for e in (in_ev[p], out_ev[p], hca_done):
                if e is not None:
                    s_csa.wait_event(e)
            self._compute(p, s_csa, s_hca)
            e1, e2 = torch.cuda.Event(), torch.cuda.Event()
            e1.record(s_csa)
            e2.record(s_hca)
            hca_done = e2
            s_out.wait_event(e1)
            s_out.wait_event(e2)
            with torch.cuda.stream(s_out):        # this step's outputs while the next runs
                self.h_out[p].copy_(self.d_out[p], non_blocking=True)
            out_ev[p] = torch.cuda.Event()
            out_ev[p].record(s_out)
            s_cp.wait_event(e1)
            s_cp.wait_event(e2)
            with torch.cuda.stream(s_cp):         # refill this set for step k + SETS
                self.d_in[p].copy_(self.h_in[p], non_blocking=True)
            in_ev[p] = torch.cuda.Event()
            in_ev[p].record(s_cp)
        j1, j2, j3 = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        j1.record(s_out)
        j2.record(s_cp)
        j3.record(s_csa)
        for e in (j1, j2, j3):
            cur.wait_event(e)


def cpu_baseline(w, x, seqs: int) -> dict:
    """The float64 oracle, as it stands, on ``seqs`` sequences of the same step."""
    import numpy as np
    import oracle
    import synth
    import dataclasses
    sub = dataclasses.replace(w, B=seqs)
    xs = {k: (v[:seqs] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == w.B else v)
          for k, v in x.items()}
    t0 = time.perf_counter()
    oracle.reference(sub, xs)
    dt = time.perf_counter() - t0
    out = {"value": seqs * sub.T / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
           "sample": f"{seqs} of {w.B} sequences of one {w.name} step (full CSA+HCA path, "
                     f"float64, OpenMP over query rows), {dt:.2f} s"}
    # the same on one core, on a smaller sample (OpenMP of the loaded oracle)
    try:
        gomp = ctypes.CDLL("libgomp.so.1")
        n1 = max(1, seqs // 16)
        sub1 = dataclasses.replace(w, B=n1)
        xs1 = {k: (v[:n1] if isinstance(v, np.ndarray) and v.ndim >= 1 and v.shape[0] == w.B
                   else v) for k, v in x.items()}
        gomp.omp_set_num_threads(1)
        t0 = time.perf_counter()
        oracle.reference(sub1, xs1)
        dt1 = time.perf_counter() - t0
        gomp.omp_set_num_threads(os.cpu_count())
        out["one_core"] = {"value": n1 * sub1.T / dt1, "sample": f"{n1} sequences, {dt1:.2f} s"}
    except OSError:
        pass
    return out


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    w = synth.WORKLOADS[WORKLOAD]
    x = synth.make_inputs(w)
    seqs = 4
    for _ in range(args.warmup):
        cpu_baseline(w, x, seqs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_baseline(w, x, seqs)
    dt = time.perf_counter() - t0
    v = seqs * args.steps / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sequences_per_step": seqs},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{seqs} of {w.B} sequences per step"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def decode_measure(w, steps: int, warmup: int, rank: int, world: int, local: int,
                   e2e: bool = True, schedule: str = "auto") -> dict:
    """Time the decode step of workload ``w`` (inputs already resident in HBM):
    the whole step (one CUDA graph, CSA and HCA on two streams), the
    dominant kernel alone (the indexer scoring call as a one-node graph) and
    the step end to end (inputs from pinned host memory, outputs back).  L2 is
    flushed before every timed replay; every replay is timed with CUDA events
    on the launching stream.  ``schedule``: "step" runs both layers as one
    sa_decode_step launch; "fused" runs the CSA layer as one csa_decode launch
    and the HCA layer on a second stream; "split" runs csa_compress, the
    indexer's score and top-k calls and csa_attend, HCA on a second stream;
    "auto" takes the fused one where csa_decode fills the GPU, else the split
    one (the measured faster schedules).
    Returns the measurement as a dict."""
    import torch
    import synth
    import sparse_attention_27_b300 as sa
    from sparse_attention_27_b300.path import step_from

    x = synth.make_inputs(w)
    step = step_from(w, x, o_dtype="bf16")
    cudart = load_cudart()
    s_csa, s_hca = torch.cuda.Stream(), torch.cuda.Stream()
    # auto: the fused CSA layer (one cluster of CTAs per sequence) where the
    # batch fills most of the GPU with clusters (measured at 128K, B = 32:
    # 99.8 us a step, against 112.2 us for the separate calls and 121.7 us
    # for the whole step in one sa_decode_step launch); with few sequences
    # (1M, B = 4) the clusters leave most SMs idle and the separate calls are
    # faster (86 vs 125 us)
    if schedule == "auto":
        mode = "fused" if step.fused_ok() and w.B >= 16 else "split"
    else:
        mode = schedule
    fused = mode == "fused"
    if mode == "step":
        run_step = lambda s_csa, s_hca: step.decode_step()      # on the current stream
    else:
        run_step = step.run_fused_two_streams if fused else step.run_two_streams
    for _ in range(2):              # outside the graph: sets kernel attributes, loads modules
        run_step(s_csa, s_hca)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph(keep_graph=True)
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        run_step(s_csa, s_hca)
    # the step's kernel launches: the captured graph's kernel nodes (the step
    # issues only library calls and event edges, so every kernel node is ours)
    kernels = graph_kernels(g.raw_cuda_graph(), cudart)
    g.instantiate()
    torch.cuda.synchronize()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    sweep = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")   # 256 MiB, summed in place

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            flush.zero_()              # evict: a write larger than L2 ...
            sweep.sum()                # ... then a read, so the step starts with clean lines
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        ms = timed(g.replay, steps)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(sum(ms), device="cuda")
    ms_sorted = sorted(ms)
    pct = lambda q: ms_sorted[min(len(ms_sorted) - 1, int(q * len(ms_sorted)))]
    errs = step.device_errors()
    value = world * w.B * w.T * steps / (total_ms / 1e3)

    # ---- dominant kernel alone: the fused CSA layer (csa_decode), or the
    # indexer's scoring call (csa_index_topk with k = 0) of the split schedule
    D = step.D
    sc = torch.empty((w.B, w.T, w.ncap), dtype=torch.float32, device="cuda")
    mx = w.indexer == "mxfp4"

    def score_only():
        if mode == "step":
            step.decode_step()
            return
        if fused:
            step.csa_fused()
            return
        if mx:   # the step has already quantised this token's indexer queries
            sa.csa_index_topk(sa.SA_MXFP4, D.B, D.T, D.HI, D.dI, D.m, 0, step.q_codes,
                              step.q_scales, step.x["w_idx"], step.x["ik_c"],
                              step.x["ik_c_scales"], D.ncap, step.x["q_pos"], None, scores_out=sc)
        else:
            sa.csa_index_topk(sa.SA_BF16, D.B, D.T, D.HI, D.dI, D.m, 0, step.x["q_idx"], None,
                              step.x["w_idx"], step.x["ik_c"], None, D.ncap, step.x["q_pos"],
                              None, scores_out=sc)
    for _ in range(3):
        score_only()
    torch.cuda.synchronize()
    g_score = torch.cuda.CUDAGraph()       # replayed, so host launch work is not timed
    with torch.cuda.graph(g_score, stream=cap):
        score_only()
    for _ in range(3):
        g_score.replay()
    k_ms = timed(g_score.replay, steps)
    k_avg = sum(k_ms) / len(k_ms)
    ab = algorithmic_bytes(w, o_bytes=2)
    peak, peak_kind = peaks()
    k_bytes = ab["step"] if mode == "step" else ab["csa"] if fused else ab["index"]
    achieved = k_bytes / (k_avg / 1e3) / 1e9
    score_kernel = ("decode_step_kernel" if mode == "step" else
                    "csa_decode_kernel" if fused else
                    "score_mx_kernel" if mx else "score_tc_kernel")
    k_call = ("sa_decode_step, both layers, counter memset + kernel" if mode == "step" else
              "csa_decode, the whole CSA layer, one-node graph" if fused else
              "csa_index_topk scores, k=0, one-node graph")
    traffic, traffic_note = recorded_traffic(
        score_kernel, STEP_SOURCES if mode == "step" else FUSED_SOURCES if fused else
        MX_SOURCES if mx else SCORE_SOURCES, k_bytes)
    step_gbs = ab["step"] / (total_ms / steps / 1e3) / 1e9

    # ---- end to end: each step's inputs from pinned host memory, its
    # outputs back to pinned host memory, sixteen steps per graph, three buffer sets
    e2e_out = None
    if e2e:
        pio = PipelinedIO(w, x, mode)
        s_cp, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        # sixteen steps per graph: the L2 flush before each timed replay leaves
        # the first host-to-device copy after it several times slower than the
        # rest (measured 106-118 against 29 us for 1.36 MB), a cost a decode
        # loop pays once, not every step
        per_graph = 16
        for _ in range(2):
            pio.record(s_csa, s_hca, s_cp, s_out, per_graph)
        torch.cuda.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e, stream=cap):
            pio.record(s_csa, s_hca, s_cp, s_out, per_graph)
        for _ in range(3):
            g_e2e.replay()
        e_ms = timed(g_e2e.replay, max(1, steps // per_graph))
        e_total = max_over_ranks(sum(e_ms), device="cuda")
        n_steps = per_graph * max(1, steps // per_graph)
        e2e_out = {"value": world * w.B * w.T * n_steps / (e_total / 1e3), "unit": UNIT,
                   "h2d_bytes_per_step": pio.h2d_bytes, "d2h_bytes_per_step": pio.d2h_bytes,
                   "copies_per_step": pio.copies, "steps": n_steps,
                   "note": "pinned host buffers; each step one copy of its inputs in (q, q_hca, "
                           "q_idx, w, positions, the new ring rows) and one of its outputs (O in "
                           "bf16, LSE) out, and one sa_ring_write of its token into the rings; "
                           "three buffer sets, sixteen steps per graph (L2 flushed before each "
                           "graph): a step's inputs arrive "
                           "while the step before it runs, its outputs leave while the next one "
                           "runs, and a set is reused two steps after it was freed"}
        del pio
    out = {
        "value": value, "ms_per_step": total_ms / steps,
        "config": {"workload": w.name, "batch": w.B, "context": w.L, "heads": w.H,
                   "head_dim": w.d, "m": w.m, "top_k": w.k, "window": w.W, "m2": w.m2,
                   "indexer_heads": w.HI, "indexer": w.indexer, "o_dtype": "bf16",
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed step: a 512 MiB write, then a 256 MiB read",
                   "schedule": mode,
                   "graph": ("one CUDA graph per step: a counter memset and one "
                             "sa_decode_step launch for both layers" if mode == "step" else
                             "one CUDA graph per step, the CSA layer as one csa_decode launch "
                             "and the HCA layer on two streams, both from the start" if fused
                             else "one CUDA graph per step, CSA and HCA on two streams, HCA "
                                  "after the CSA scores")},
        "step_algorithmic_bytes": ab["step"], "step_gbs": step_gbs,
        "step_frac_of_hbm": step_gbs / peak,
        "roofline": {"kernel": f"{score_kernel} ({k_call})",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": traffic, "traffic_source": traffic_note,
                     "avg_launch_ms": k_avg, "algorithmic_bytes_per_launch": k_bytes},
        "e2e": e2e_out, "gpu_launches": len(kernels) * steps,
        "step_ms": {"p10": pct(0.10), "median": statistics.median(ms), "p90": pct(0.90)},
        "kernels_per_step": len(kernels), "kernels": sorted(set(kernels)),
        "device_errors": errs, "clocks": clk.summary(),
    }
    return out, x


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--schedule", default="auto", choices=["auto", "step", "fused", "split"],
                    help="both layers as one sa_decode_step launch (step), the CSA layer as one "
                         "csa_decode launch (fused) or as its separate calls (split); auto: "
                         "fused where csa_decode fills the GPU, else split")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the headline workload (no 1M decode and 64K prefill objects)")
    ap.add_argument("--prefill-calls", action="store_true",
                    help="instead of the decode step: per-call times and TFLOP/s of the 64K "
                         "prefill chunk")
    ap.add_argument("--workload", default=WORKLOAD, choices=["decode128k", "decode1m", "mxfp4"],
                    help="decode at 128K (B=32, the default), at 1M (B=4), or at 128K with "
                         "the MXFP4 indexer")
    args = ap.parse_args()
    globals()["WORKLOAD"] = args.workload
    if args.impl == "reference":
        run_reference(args)
        return
    if args.prefill_calls:
        run_prefill_calls(args)
        return
    assert args.warmup >= 3

    import dataclasses
    import torch
    import torch.distributed as dist
    import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    w = synth.WORKLOADS[WORKLOAD]
    if world > 1:                   # every rank decodes its own sequences (seeded by rank)
        w = dataclasses.replace(w, seed=rank)
    head, x = decode_measure(w, args.steps, args.warmup, rank, world, local,
                             schedule=args.schedule)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, x, seqs=w.B)
    del x
    torch.cuda.empty_cache()

    # the metric's second context (1M decode) and the prefill contractions, on
    # the default run only (rank 0 of a single-GPU run)
    extra = {}
    if WORKLOAD == "decode128k" and world == 1 and not args.no_extra:
        w1 = synth.WORKLOADS["decode1m"]
        m1, x1 = decode_measure(w1, args.steps, args.warmup, rank, world, local,
                                schedule=args.schedule)
        if not args.no_cpu_baseline:
            m1["cpu_baseline"] = cpu_baseline(w1, x1, seqs=w1.B)
        del x1
        torch.cuda.empty_cache()
        extra["decode1m"] = m1
        extra["prefill64k"] = prefill_calls(steps=3, warmup=1, device=local)
        extra["backward"] = backward_calls(steps=5, warmup=2, device=local)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": head["config"],
        }
        for k_ in ("step_algorithmic_bytes", "step_gbs", "step_frac_of_hbm", "roofline", "e2e",
                   "gpu_launches", "step_ms", "kernels_per_step", "kernels", "device_errors",
                   "clocks"):
            line[k_] = head[k_]
        line["cpu_baseline"] = cpu
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
