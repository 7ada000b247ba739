"""GPU: ping-pong rounds (kda_verify_scan_pingpong) give the same bits as in-place
rounds with a copied snapshot, leave the pre-round buffers untouched, and match the
oracle.

A ping-pong round reads the committed state from one buffer and writes the next
state into the other; the buffer it read is the round's snapshot (glm_spec.rs,
ROLLBACK and the Glm5VerifyCkpt doc: one snapshot per layer per round, taken before
row 0), so no snapshot copy is made.  kda_rollback then replays the kept rows from it.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import assert_close, bits_equal, host, layer_state, rows_to_dev, small_case, to_dev
from libs import ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu

W = synth.Workload("pp", L=3, B=4, H=10, T=8, bf16=True, V=900, rounds=5, seed=0x9919, accept="uniform")
WV = synth.Workload("ppv", L=2, B=5, H=6, T=15, bf16=False, V=300, rounds=4, seed=0x9920, accept="uniform")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def _inputs(w, r):
    rows = synth.all_rows(w, r)
    keep = [j + 1 for j in synth.accept_targets(w, r)]
    return rows_to_dev(rows, w.bf16), keep


def test_pingpong_rounds_equal_in_place_rounds():
    state0, ring0, cw = small_case(W)
    a = layer_state(state0, ring0, cw)  # in place, snapshot copied by the verify
    stash = kb.Stash(a)
    b = layer_state(state0, ring0, cw)  # ping-pong
    pp = kb.PingPong(b)
    out_a = torch.empty((W.L, W.B, W.T, W.H, 128), dtype=torch.float32, device="cuda")
    out_b = torch.full_like(out_a, float("nan"))
    for r in range(W.rounds):
        rows, keep = _inputs(W, r)
        if r == W.rounds - 1:
            keep = [W.T] * W.B  # a round that keeps every row: nothing to roll back
        pre_state, pre_ring = pp.state().clone(), pp.ring().clone()
        kb.kda_verify_scan(a, *(rows[n] for n in ("q", "k", "v", "g", "beta")), out=out_a, stash=stash)
        kb.kda_verify_scan_pingpong(pp, *(rows[n] for n in ("q", "k", "v", "g", "beta")), out=out_b)
        torch.cuda.synchronize()
        # verify: outputs and post-round state agree; the pre-round buffers are untouched
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        assert bits_equal(a.state, pp.state()) and bits_equal(a.conv_ring, pp.ring()), f"round {r}: verify state"
        assert bits_equal(pp.states[pp.last], pre_state) and bits_equal(pp.rings[pp.last], pre_ring)
        assert bits_equal(stash.state_snap, pre_state) and bits_equal(stash.ring_snap, pre_ring)
        kb.kda_rollback(a, stash, keep)
        kb.kda_rollback_pingpong(pp, keep)
        torch.cuda.synchronize()
        assert bits_equal(a.state, pp.state()) and bits_equal(a.conv_ring, pp.ring()), f"round {r}: committed state"


def test_pingpong_matches_the_oracle(orc):
    w = synth.Workload("ppo", L=1, B=2, H=3, T=6, bf16=True, V=64, rounds=1, seed=0x9921, accept="uniform")
    state0, ring0, cw = small_case(w)
    pp = kb.PingPong(layer_state(state0, ring0, cw))
    rows_np = synth.all_rows(w, 0)
    rows = rows_to_dev(rows_np, w.bf16)
    out = torch.empty((1, w.B, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    keep = [3, w.T]
    kb.kda_verify_scan_pingpong(pp, *(rows[n] for n in ("q", "k", "v", "g", "beta")), out=out)
    kb.kda_rollback_pingpong(pp, torch.tensor(keep, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    for b in range(w.B):
        u = {n: rows_np[n][0, b] for n in rows_np}
        args = (u["q"], u["k"], u["v"], u["g"], u["beta"], cw[0])
        s_T, r_T, o = orc.verify(*args, ring0[0, b], state0[0, b])
        s_k, r_k = orc.rollback(keep[b], *args, ring0[0, b], state0[0, b], r_T, s_T)
        assert_close(host(out[0, b]), o, f"outputs of session {b}")
        assert_close(host(pp.state()[0, b]), s_k, f"state of session {b}")
        assert np.array_equal(host(pp.ring()[0, b]), r_k), f"ring of session {b}"


@pytest.mark.parametrize("mem", ["host", "device"])
def test_pingpong_per_session_rows_equal_in_place(mem):
    state0, ring0, cw = small_case(WV)
    a = layer_state(state0, ring0, cw)
    stash = kb.Stash(a)
    pp = kb.PingPong(layer_state(state0, ring0, cw))
    out_a = torch.zeros((WV.L, WV.B, WV.T, WV.H, 128), dtype=torch.float32, device="cuda")
    out_b = torch.zeros_like(out_a)
    g = np.random.default_rng(7)
    for r in range(WV.rounds):
        rows, _ = _inputs(WV, r)
        t_rows = [int(x) for x in g.integers(1, WV.T + 1, WV.B)]
        keep = [int(g.integers(1, t + 1)) for t in t_rows]
        tr = t_rows if mem == "host" else torch.tensor(t_rows, dtype=torch.int32, device="cuda")
        kp = keep if mem == "host" else torch.tensor(keep, dtype=torch.int32, device="cuda")
        x = [rows[n] for n in ("q", "k", "v", "g", "beta")]
        kb.kda_verify_scan_var(a, *x, tr, out=out_a, stash=stash)
        kb.kda_verify_scan_pingpong(pp, *x, out=out_b, t_rows=tr)
        torch.cuda.synchronize()
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        assert bits_equal(a.state, pp.state()) and bits_equal(a.conv_ring, pp.ring()), f"round {r}: verify state"
        kb.kda_rollback_var(a, stash, tr, kp)
        kb.kda_rollback_pingpong(pp, kp, t_rows=tr)
        torch.cuda.synchronize()
        assert bits_equal(a.state, pp.state()) and bits_equal(a.conv_ring, pp.ring()), f"round {r}: committed"


def _plan_case(w, plan_cls, stream=None):
    state0, ring0, cw = small_case(w)
    st = layer_state(state0, ring0, cw)
    rows, _ = _inputs(w, 0)
    lg = to_dev(synth.logits(w, 0), w.bf16)
    d = to_dev(synth.drafts_for(synth.logit_argmax(w, 0), synth.accept_targets(w, 0), w.V))
    out = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    j, bonus, keep = (torch.empty(w.B, dtype=torch.int32, device="cuda") for _ in range(3))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(kb.spec_accept_scratch_bytes(w.B, w.T, w.V), dtype=torch.uint8, device="cuda")
    if plan_cls is kb.RoundPlan:
        holder = kb.Stash(st)
        plan = kb.RoundPlan(st, rows, out, holder, lg, d, j, bonus, keep, status, scratch, stream)
        committed = lambda: (st.state, st.conv_ring)  # noqa: E731
    else:
        holder = kb.PingPong(st)
        plan = kb.PingPongRoundPlan(holder, rows, out, lg, d, j, bonus, keep, status, scratch, stream)
        committed = lambda: (holder.state(), holder.ring())  # noqa: E731
    return dict(rows=rows, lg=lg, d=d, out=out, j=j, status=status, plan=plan, committed=committed, holder=holder)


def _load(case, w, r):
    rows, _ = _inputs(w, r)
    for n, x in rows.items():
        case["rows"][n].copy_(x)
    case["lg"].copy_(to_dev(synth.logits(w, r), w.bf16))
    case["d"].copy_(to_dev(synth.drafts_for(synth.logit_argmax(w, r), synth.accept_targets(w, r), w.V)))


def test_pingpong_plan_eager_and_graph_equal_round_plan():
    side = torch.cuda.Stream()
    a = _plan_case(W, kb.RoundPlan)
    b = _plan_case(W, kb.PingPongRoundPlan)
    with torch.cuda.stream(side):
        c = _plan_case(W, kb.PingPongRoundPlan, side)
    torch.cuda.synchronize()
    # rounds 0 and 1 eagerly everywhere (for c also the warm-up of both parities)
    for r in range(W.rounds):
        for x in (a, b, c):
            _load(x, W, r)
        torch.cuda.synchronize()
        a["plan"]()
        b["plan"]()
        if r < 2:
            with torch.cuda.stream(side):
                c["plan"]()
            if r == 1:
                torch.cuda.synchronize()
                c["plan"].capture()
        else:
            c["plan"].replay()
        torch.cuda.synchronize()
        assert [int(x) for x in a["j"].cpu()] == list(synth.accept_targets(W, r))
        sa, ra = a["committed"]()
        for x in (b, c):
            sb, rb = x["committed"]()
            assert bits_equal(sa, sb) and bits_equal(ra, rb), f"round {r}: committed state"
            assert bits_equal(a["out"], x["out"]) and torch.equal(a["j"], x["j"]), f"round {r}: outputs"
            assert int(x["status"][0]) == 0
