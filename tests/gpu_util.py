"""Helpers for the GPU tests: the package's upload helpers under short
names (numpy <-> device, a HybridStep over a synth workload's inputs)."""
from __future__ import annotations

from sparse_attention_27_b300.path import (device_inputs, dims_from, step_from, to_device,
                                           to_host)

dev = to_device
host = to_host
dims_of = dims_from
make_step = step_from

__all__ = ["dev", "host", "dims_of", "device_inputs", "make_step"]
