"""Helpers of the GPU parity tests: seeded inputs on both sides, tolerance checks.

Inputs for the oracle are always drawn on the CPU by synth.py; the device gets
either the same arrays uploaded or the same values drawn by synth_gpu (checked
equal in test_gpu_synth).  No expected value comes from the CUDA path.
"""
from __future__ import annotations

import numpy as np
import torch

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

# f32 outputs and states: |gpu - oracle| <= ATOL + RTOL * |oracle|
RTOL, ATOL = 1e-4, 1e-5


def assert_close(got, ref, what, rtol=RTOL, atol=ATOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    excess = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    bad = int((excess > 0).sum())
    assert bad == 0, f"{what}: {bad} elements out of tolerance, worst excess {excess.max():.3e}"


def to_dev(x: np.ndarray, bf16_bits: bool = False) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    if bf16_bits:
        t = t.view(torch.bfloat16)
    return t.cuda()


def rows_to_dev(rows: dict, bf16: bool) -> dict:
    return {n: to_dev(a, bf16) for n, a in rows.items()}


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def small_case(w: synth.Workload):
    """Initial state, ring and conv weights of a workload on the CPU (all units)."""
    return synth.all_state(w), synth.all_ring(w), synth.all_conv_w(w)


def layer_state(state, ring, conv_w) -> kb.LayerState:
    return kb.LayerState(to_dev(state), to_dev(ring), to_dev(conv_w))


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int32), b.view(torch.int32))
