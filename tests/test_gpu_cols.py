"""GPU: column-stash rollback (the vLLM-style alternative the pages weigh against
snapshot + replay, glm_spec.rs module doc, ROLLBACK).  Its verify leaves the same bits
as kda_verify_scan, every column holds the state and ring after its row, and its
rollback (a copy of the kept column) equals snapshot + replay bit for bit."""
from __future__ import annotations

import pytest
import torch

from gpu_util import bits_equal, layer_state, rows_to_dev, small_case
from libs import ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu

W = synth.Workload("cols", L=2, B=5, H=6, T=7, bf16=True, V=64, rounds=1, seed=141, accept="uniform")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def test_verify_cols_state_out_and_columns():
    state0, ring0, cw = small_case(W)
    rows = rows_to_dev(synth.all_rows(W, 0), W.bf16)
    a = layer_state(state0, ring0, cw)
    out_a = torch.empty((W.L, W.B, W.T, W.H, 128), device="cuda")
    kb.kda_verify_scan(a, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], out=out_a)
    c = layer_state(state0, ring0, cw)
    out_c = torch.empty_like(out_a)
    cols = kb.ColStash(c, W.T)
    kb.kda_verify_scan_cols(c, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], cols, out=out_c)
    torch.cuda.synchronize()
    assert bits_equal(a.state, c.state) and bits_equal(a.conv_ring, c.conv_ring) and bits_equal(out_a, out_c)
    for t in range(W.T):
        r = layer_state(state0, ring0, cw)
        sl = {n: x[:, :, :t + 1].contiguous() for n, x in rows.items()}
        kb.kda_verify_scan(r, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"])
        torch.cuda.synchronize()
        assert bits_equal(cols.state_cols[:, :, :, t], r.state), t
        assert bits_equal(cols.ring_cols[:, :, :, t], r.conv_ring), t


@pytest.mark.parametrize("mem", ["host", "device"])
def test_rollback_cols_equals_snapshot_replay(mem):
    state0, ring0, cw = small_case(W)
    rows = rows_to_dev(synth.all_rows(W, 0), W.bf16)
    for shift in range(W.T):
        keep = [((b + shift) % W.T) + 1 for b in range(W.B)]
        k_arg = keep if mem == "host" else torch.tensor(keep, dtype=torch.int32, device="cuda")
        a = layer_state(state0, ring0, cw)
        stash = kb.Stash(a)
        kb.kda_verify_scan(a, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], stash=stash)
        kb.kda_rollback(a, stash, k_arg)
        c = layer_state(state0, ring0, cw)
        cols = kb.ColStash(c, W.T)
        kb.kda_verify_scan_cols(c, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], cols)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        kb.kda_rollback_cols(c, cols, k_arg, dev_status=status)
        torch.cuda.synchronize()
        assert int(status[0]) == 0
        assert bits_equal(a.state, c.state), (shift, keep)
        assert bits_equal(a.conv_ring, c.conv_ring), (shift, keep)


def test_rollback_cols_bad_device_keep():
    state0, ring0, cw = small_case(W)
    rows = rows_to_dev(synth.all_rows(W, 0), W.bf16)
    c = layer_state(state0, ring0, cw)
    cols = kb.ColStash(c, W.T)
    kb.kda_verify_scan_cols(c, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], cols)
    after = c.state.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kb.kda_rollback_cols(c, cols, torch.tensor([0, 8, 7, 7, 7], dtype=torch.int32, device="cuda"), dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & kb.ST_BADKEEP
    assert bits_equal(c.state, after)
