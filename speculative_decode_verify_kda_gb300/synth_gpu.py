"""Device-side fill of the seeded synthetic inputs (same values as synth.py).

Large workloads (up to ~2 GB of raw rows per round) are drawn directly into
device tensors by ``libkda_synth.so``; every element equals the one synth.py
draws for the same tensor key and flat index.  Input preparation only: none of
the method's arithmetic is here.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import synth

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libkda_synth.so")
D = synth.D
_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the package libraries first")
        L = ctypes.CDLL(LIB_PATH)
        for fn in (L.synth_fill_normal, L.synth_fill_uniform):
            fn.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_float, ctypes.c_int,
                           ctypes.c_void_p, ctypes.c_void_p]
            fn.restype = ctypes.c_int
        _lib = L
    return _lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def fill_normal(t: torch.Tensor, key: int, start: int = 0, sigma: float = 1.0) -> torch.Tensor:
    assert t.is_cuda and t.is_contiguous() and t.dtype in (torch.float32, torch.bfloat16)
    rc = lib().synth_fill_normal(key, start, t.numel(), sigma, int(t.dtype == torch.bfloat16),
                                 ctypes.c_void_p(t.data_ptr()), _stream())
    if rc:
        raise RuntimeError("synth_fill_normal launch failed")
    return t


def fill_uniform(t: torch.Tensor, key: int, start: int = 0, half_width: float = 0.5) -> torch.Tensor:
    assert t.is_cuda and t.is_contiguous() and t.dtype in (torch.float32, torch.bfloat16)
    rc = lib().synth_fill_uniform(key, start, t.numel(), half_width, int(t.dtype == torch.bfloat16),
                                  ctypes.c_void_p(t.data_ptr()), _stream())
    if rc:
        raise RuntimeError("synth_fill_uniform launch failed")
    return t


def row_dtype(w: synth.Workload):
    return torch.bfloat16 if w.bf16 else torch.float32


def rows(w: synth.Workload, round_idx: int, device="cuda") -> dict:
    """Raw rows of one round on the device: q,k,v,g [L][B][T][H][128], beta [L][B][T][H]."""
    out = {}
    for name in synth.ROW_TENSORS:
        shape = (w.L, w.B, w.T, w.H) + ((D,) if name != "beta" else ())
        t = torch.empty(shape, dtype=row_dtype(w), device=device)
        out[name] = fill_normal(t, synth.tensor_key(w.seed, name, round_idx))
    return out


def state(w: synth.Workload, device="cuda") -> torch.Tensor:
    t = torch.empty((w.L, w.B, w.H, D, D), dtype=torch.float32, device=device)
    return fill_normal(t, synth.tensor_key(w.seed, "state"), 0, w.state_sigma)


def ring(w: synth.Workload, device="cuda") -> torch.Tensor:
    t = torch.empty((w.L, w.B, w.H, 3, 3, D), dtype=torch.float32, device=device)
    return fill_normal(t, synth.tensor_key(w.seed, "ring"), 0, w.ring_sigma)


def conv_w(w: synth.Workload, device="cuda") -> torch.Tensor:
    t = torch.empty((w.L, w.H, 3, D, 4), dtype=torch.float32, device=device)
    return fill_uniform(t, synth.tensor_key(w.seed, "conv_w"), 0, w.conv_half_width)


def logits(w: synth.Workload, round_idx: int, device="cuda") -> torch.Tensor:
    """Logits [B][T][V] of synth.logits: normal draws, bf16 for bf16 workloads."""
    t = torch.empty((w.B, w.T, w.V), dtype=row_dtype(w), device=device)
    return fill_normal(t, synth.tensor_key(w.seed, "logits", round_idx))


def logit_argmax(lg: torch.Tensor) -> torch.Tensor:
    """The argmax of each row of lg [..][V], the lowest index winning ties (input
    preparation: the value V - i of a maximal element i is unique, so their maximum
    names the first maximal index)."""
    V = int(lg.shape[-1])
    m = lg.amax(-1, keepdim=True)
    rev = torch.arange(V, 0, -1, device=lg.device, dtype=torch.int32)
    return V - torch.where(lg == m, rev, torch.zeros_like(rev)).amax(-1).to(torch.int64)


def drafts(w: synth.Workload, round_idx: int, device="cuda", lg: torch.Tensor | None = None
           ) -> tuple[torch.Tensor, list]:
    """Drafts int32 [B][T-1] that accept exactly the round's target j per session: the
    argmax of the round's logits (lg, or drawn here) up to j, then a different token."""
    j = synth.accept_targets(w, round_idx)
    if lg is None:
        lg = logits(w, round_idx, device)
    vam = logit_argmax(lg).cpu().numpy()
    d = synth.drafts_for(vam, j, w.V)
    return torch.as_tensor(d, device=device), [int(x) for x in j]
