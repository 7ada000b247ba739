"""GPU: a round issued per layer (as a model issues it) and a round replayed from a
CUDA graph give the same bits as the one-launch round.

Per-layer issue: one kda_verify_scan per layer over that layer's views, then
spec_accept, then one kda_rollback over all layers from the snapshots the per-layer
calls wrote (glm_spec.rs module doc, VERIFY-ROW BATCHING: one launch per layer per
round).  CUDA-graph replay of whole rounds is the launch amortisation the pages use
for their batched snapshot and verify rounds.
"""
from __future__ import annotations

import pytest
import torch

from gpu_util import bits_equal, layer_state, rows_to_dev, small_case, to_dev
from libs import ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu

W = synth.Workload("pl", L=5, B=3, H=12, T=8, bf16=True, V=700, rounds=4, seed=91, accept="uniform")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def _round_inputs(w, r):
    rows = synth.all_rows(w, r)
    lg = synth.logits(w, r)
    d = synth.drafts_for(synth.logit_argmax(w, r), synth.accept_targets(w, r), w.V)
    return rows, lg, d


class _Case:
    """A layer state with its stash, fixed input buffers, outputs and a plan."""

    def __init__(self, w, plan_cls, stream=None):
        state0, ring0, cw = small_case(w)
        self.st = layer_state(state0, ring0, cw)
        self.stash = kb.Stash(self.st)
        rows, lg, d = _round_inputs(w, 0)
        self.rows = rows_to_dev(rows, w.bf16)
        self.lg = to_dev(lg, w.bf16)
        self.d = to_dev(d)
        self.out = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device="cuda")
        self.j = torch.empty(w.B, dtype=torch.int32, device="cuda")
        self.bonus = torch.empty_like(self.j)
        self.keep = torch.empty_like(self.j)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scratch = torch.empty(kb.spec_accept_scratch_bytes(w.B, w.T, w.V), dtype=torch.uint8, device="cuda")
        self.plan = plan_cls(self.st, self.rows, self.out, self.stash, self.lg, self.d, self.j, self.bonus,
                             self.keep, self.status, self.scratch, stream)

    def load(self, w, r):
        rows, lg, d = _round_inputs(w, r)
        for n, x in rows_to_dev(rows, w.bf16).items():
            self.rows[n].copy_(x)
        self.lg.copy_(to_dev(lg, w.bf16))
        self.d.copy_(to_dev(d))

    def same_as(self, other) -> bool:
        return all(bits_equal(x, y) for x, y in (
            (self.st.state, other.st.state), (self.st.conv_ring, other.st.conv_ring), (self.out, other.out),
            (self.stash.state_snap, other.stash.state_snap), (self.stash.ring_snap, other.stash.ring_snap),
        )) and torch.equal(self.j, other.j) and torch.equal(self.keep, other.keep) \
            and torch.equal(self.bonus, other.bonus)


def test_per_layer_round_equals_one_launch_round():
    a = _Case(W, kb.RoundPlan)
    b = _Case(W, kb.LayerRoundPlan)
    for r in range(W.rounds):
        a.load(W, r)
        b.load(W, r)
        a.plan()
        b.plan()
        torch.cuda.synchronize()
        assert [int(x) for x in a.j.cpu()] == list(synth.accept_targets(W, r))
        assert b.same_as(a), f"round {r}"
        assert int(a.status[0]) == 0 and int(b.status[0]) == 0


def test_graph_replayed_rounds_equal_eager_rounds():
    side = torch.cuda.Stream()
    a = _Case(W, kb.LayerRoundPlan)
    with torch.cuda.stream(side):
        b = _Case(W, kb.LayerRoundPlan, side)
    torch.cuda.synchronize()
    # round 0 eagerly on both (for b it is also the warm-up before capture)
    a.plan()
    with torch.cuda.stream(side):
        b.plan()
    torch.cuda.synchronize()
    b.plan.capture()
    for r in range(1, W.rounds):
        a.load(W, r)
        b.load(W, r)
        torch.cuda.synchronize()
        a.plan()
        b.plan.replay()
        torch.cuda.synchronize()
        assert b.same_as(a), f"round {r}"
    assert int(b.status[0]) == 0


def test_capture_needs_a_side_stream():
    a = _Case(synth.Workload("c", L=2, B=1, H=2, T=3, bf16=False, V=50, rounds=1, seed=92, accept="uniform"),
              kb.LayerRoundPlan)
    with pytest.raises(ValueError):
        a.plan.capture()
