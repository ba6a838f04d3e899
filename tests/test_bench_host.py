"""Host logic of bench.py on the CPU: the clock sampler's decoding of NVML
clock-event reasons and its summary (against a fake NVML that only answers the
two read queries the sampler makes), the recorded-traffic lookup and its
scaling between workloads, and the algorithmic byte counts against the figures
worked out from the workload definitions."""
from __future__ import annotations

import ctypes
import os
import time

import pytest

import bench
import synth


class FakeNVML:
    """Answers nvmlDeviceGetClockInfo / nvmlDeviceGetCurrentClocksEventReasons
    from fixed lists, cycling."""

    def __init__(self, clocks, reasons):
        self.clocks, self.reasons, self.i = clocks, reasons, 0

    def nvmlDeviceGetClockInfo(self, h, kind, ptr):
        ptr._obj.value = self.clocks[self.i % len(self.clocks)]
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, ptr):
        ptr._obj.value = self.reasons[self.i % len(self.reasons)]
        self.i += 1
        return 0


def _sampler(fake) -> bench.Clocks:
    c = bench.Clocks.__new__(bench.Clocks)
    c.samples, c.max_mhz, c.why = [], 2032.0, None
    c.nv, c.h, c.ct = fake, object(), ctypes
    return c


def test_clock_sampler_decodes_reasons_and_takes_the_median():
    fake = FakeNVML([2032, 1980, 2032], [0x0, 0x4, 0x4 | 0x40])
    with _sampler(fake) as c:
        deadline = time.time() + 5
        while len(c.samples) < 9 and time.time() < deadline:
            time.sleep(0.005)
    s = c.summary()
    assert s["samples"] >= 9
    assert s["sm_mhz"] == 2032.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert "unavailable" not in s


def test_clock_sampler_without_nvml_reports_why():
    c = bench.Clocks.__new__(bench.Clocks)
    c.samples, c.max_mhz, c.why, c.h = [], None, "no NVML here", None
    with c:
        pass
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["unavailable"] == "no NVML here"


def test_recorded_traffic_exact_scaled_and_stale(monkeypatch):
    kernel, files = "score_tc_kernel", bench.SCORE_SOURCES
    cur = bench.source_hash(files)
    dram, note = bench.recorded_traffic(kernel, files, 134488064)
    if dram is None:
        pytest.skip("score_tc_kernel sources changed since the recorded capture")
    line = [l.split() for l in open(os.path.join(bench.ROOT, "profiles", "traffic.txt"))
            if l.split() and l.split()[0] == kernel][0]
    recorded = int(line[2])
    assert dram == recorded and "decode128k" in note
    half, note2 = bench.recorded_traffic(kernel, files, 134488064 // 2)
    assert half == round(recorded / 2) and note2.startswith("scaled by algorithmic bytes")
    monkeypatch.setattr(bench, "source_hash", lambda f: "0" * 16 if f is files else cur)
    stale, why = bench.recorded_traffic(kernel, files, 134488064)
    assert stale is None and "changed" in why


def test_algorithmic_bytes_of_the_workloads():
    # 128K decode, per sequence: indexer keys 32768 x 64 bf16 + q_I + w; the
    # CSA gather of 2048 selected K/V rows and the 128-row window (512 B each);
    # q, idx, O (f32) and LSE; HCA: 1024 compressed K/V rows + window + q, O, LSE
    per_index = 32768 * 128 + 64 * 128 + 64 * 4
    per_csa = per_index + 2048 * 512 + 128 * 512 + 64 * 256 + 2048 * 4 + 64 * 512 + 64 * 4
    per_hca = 1024 * 512 + 128 * 512 + 64 * 256 + 64 * 512 + 64 * 4
    ab = bench.algorithmic_bytes(synth.WORKLOADS["decode128k"])
    assert ab["index"] == 32 * per_index
    assert ab["step"] == 32 * (per_csa + per_hca)
    # MXFP4 indexer: 34 bytes per 64-element row (32 of codes, 2 of scales),
    # 3.76x fewer indexer bytes than bf16
    mx = bench.algorithmic_bytes(synth.WORKLOADS["mxfp4"])
    assert mx["index"] == 32 * (32768 * 34 + 64 * 34 + 64 * 4)
    assert abs(ab["index"] / mx["index"] - 3.76) < 0.01
    # 1M decode: 262144 indexer rows per sequence dominate
    m1 = bench.algorithmic_bytes(synth.WORKLOADS["decode1m"])
    assert m1["index"] == 4 * (262144 * 128 + 64 * 128 + 64 * 4)
    # O written in bf16: 64 x 128 x 2 bytes fewer per layer and sequence
    ab16 = bench.algorithmic_bytes(synth.WORKLOADS["decode128k"], o_bytes=2)
    assert ab16["index"] == ab["index"]
    assert ab["step"] - ab16["step"] == 32 * 2 * 64 * 128 * 2


def test_prefill_pairs_of_the_64k_chunk():
    """The 64K prefill chunk (t = 0..65535, m = 4, m' = 128, k = 2048, W = 128):
    536,854,528 indexer scores, 134,207,552 CSA and 25,125,440 HCA
    (query, key) pairs -- 4.40, 4.40 and 0.82 TFLOP at 8192 and 32768 flops
    per score and pair."""
    import numpy as np
    w = synth.WORKLOADS["prefill64k"]
    p = bench.prefill_pairs(w, np.arange(65536))
    assert p == {"index": 536854528, "csa": 134207552, "hca": 25125440}
    assert round(p["index"] * 2 * w.HI * w.dI / 1e12, 2) == 4.40
    assert round(p["csa"] * 4 * w.H * w.d / 1e12, 2) == 4.40
    assert round(p["hca"] * 4 * w.H * w.d / 1e12, 2) == 0.82
