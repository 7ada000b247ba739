"""spec_accept_noalloc: greedy accept for callers that cannot allocate device memory.

Some users of this library cannot call cudaMalloc when they accept a round: their
device memory is handed out up front by a fixed arena, or their host path must not
allocate or free because those calls can synchronise the device.  For them the
library keeps the accept's partial results in a fixed array of its own.

These tests call it through the C ABI (ctypes on libkda_spec.so) and compare it
with spec_accept and with the CPU oracle on the same inputs, on two calls in a row
with different inputs, so a stale array from the first call cannot hide behind the
second.  The file sorts last so that a run stopping at the first failure has run
everything else first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from libs import ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

NOALLOC_SCRATCH_BYTES = 1 << 20


def _noalloc_fn():
    ensure_built()
    L = kb.lib()
    fn = L.spec_accept_noalloc
    vp, ci = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp]
    fn.restype = ci
    return L, fn


def test_noalloc_rejects_oversized_problem_before_any_launch():
    L, fn = _noalloc_fn()
    B, T, V = 1000, 15, 32768  # 1000 * 15 * 8 slices * 16 B = 1.9 MB > 1 MiB
    assert L.spec_accept_scratch_bytes(B, T, V) > NOALLOC_SCRATCH_BYTES
    rc = fn(0x10000, kb.BF16, B, T, V, 0x10000, None, None, None, None, None)
    assert rc == kb.EINVAL
    assert b"above its fixed 1048576" in L.kda_last_error()


@pytest.mark.gpu
def test_noalloc_matches_spec_accept_and_oracle_twice_in_a_row(orc):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    L, fn = _noalloc_fn()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [synth.Workload("na1", L=1, B=24, H=1, T=15, bf16=True, V=32768, rounds=1, seed=0xA11C, accept="skewed"),
             synth.Workload("na2", L=1, B=7, H=1, T=8, bf16=False, V=1003, rounds=1, seed=0xA11D, accept="uniform")]
    for w in cases:
        lg = synth.logits(w, 0)
        if w.name == "na2":
            lg[3, 1, 17] = np.nan  # a NaN row in session 3: reached only if drafts match row 0
        jt = synth.accept_targets(w, 0)
        d = synth.drafts_for(synth.logit_argmax(w, 0), jt, w.V)
        logits = torch.from_numpy(lg)
        logits = (logits.view(torch.bfloat16) if w.bf16 else logits).cuda()
        drafts = torch.from_numpy(d).cuda()
        # the existing entry point
        st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        j_ref, b_ref, k_ref = kb.spec_accept(logits, drafts, dev_status=st_ref)
        # no-allocation entry point
        out = torch.full((3, w.B), -7, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = fn(logits.data_ptr(), kb.BF16 if w.bf16 else kb.F32, w.B, w.T, w.V, drafts.data_ptr(),
                out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), st.data_ptr(), stream)
        assert rc == kb.OK, L.kda_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out[0], j_ref) and torch.equal(out[1], b_ref) and torch.equal(out[2], k_ref)
        assert int(st[0]) == int(st_ref[0])
        if w.name == "na1":
            assert [int(x) for x in out[0].cpu()] == [int(x) for x in jt]
        # the oracle on the same rows: j and bonus per session, a NaN row reached gives
        # bonus -1 and the device status bit
        got = out.cpu().numpy()
        nan_seen = False
        for b in range(w.B):
            jr, br, _, rc = orc.accept(lg[b], d[b])
            assert (int(got[0, b]), int(got[1, b]), int(got[2, b])) == (jr, br, jr + 1), (w.name, b)
            nan_seen |= rc == 2
        assert bool(int(st[0]) & kb.ST_NAN) == nan_seen
