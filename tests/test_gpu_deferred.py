"""GPU: a round whose verify first applies the previous round's accept
(kda_verify_scan_deferred) gives the same bits as the previous round's kda_rollback
followed by a ping-pong verify, and matches the oracle.

The rollback (glm_spec.rs, glm5_verify_rollback: restore the per-round snapshot and
replay rows 0..keep-1) is the same replay; it runs inside the next round's launch, so
the state crosses HBM once per round instead of twice for a session that rolls back.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import assert_close, bits_equal, host, layer_state, rows_to_dev, small_case
from libs import ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def _rounds(L, B, H, Ts, bf16, seed):
    """Raw rows of consecutive rounds with the given row counts (one workload per T)."""
    out = []
    for r, T in enumerate(Ts):
        w = synth.Workload(f"d{T}", L=L, B=B, H=H, T=T, bf16=bf16, V=64, rounds=r + 1, seed=seed + 7 * T,
                           accept="uniform")
        out.append(synth.all_rows(w, r))
    return out


def _keeps(B, Ts, seed):
    """Per round and session a keep in 1..T, with full keeps and keep = 1 among them."""
    g = np.random.default_rng(seed)
    ks = []
    for T in Ts:
        k = g.integers(1, T + 1, B)
        k[0] = T          # a session that keeps every row: nothing to replay
        k[-1] = 1         # the shortest replay
        ks.append([int(x) for x in k])
    return ks


@pytest.mark.parametrize("bf16,Ts", [(True, [8, 8, 8, 8]), (True, [8, 5, 15, 1, 3]), (False, [6, 9, 2])])
def test_deferred_rounds_equal_rollback_then_pingpong(bf16, Ts):
    L, B, H = 2, 4, 6
    w0 = synth.Workload("d", L=L, B=B, H=H, T=Ts[0], bf16=bf16, V=64, rounds=1, seed=0x9930, accept="uniform")
    state0, ring0, cw = small_case(w0)
    rounds = [rows_to_dev(r, bf16) for r in _rounds(L, B, H, Ts, bf16, 0x9931)]
    keeps = _keeps(B, Ts, 0x9932)
    a = kb.PingPong(layer_state(state0, ring0, cw))  # rollback, then ping-pong verify
    b = kb.PingPong(layer_state(state0, ring0, cw))  # deferred rounds
    for r, T in enumerate(Ts):
        out_a = torch.full((L, B, T, H, 128), float("nan"), device="cuda")
        out_b = torch.full_like(out_a, float("nan"))
        x = [rounds[r][n] for n in NAMES]
        if r > 0:
            kb.kda_rollback_pingpong(a, keeps[r - 1])
        kb.kda_verify_scan_pingpong(a, *x, out=out_a)
        if r == 0:
            kb.kda_verify_scan_pingpong(b, *x, out=out_b)
        else:
            kb.kda_verify_scan_deferred(b, *x, torch.tensor(keeps[r - 1], dtype=torch.int32, device="cuda"),
                                        out=out_b)
        torch.cuda.synchronize()
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        # this round's snapshot (the committed state) and post-round state, state and ring
        for nm, ta, tb in (("snapshot", a.states[a.last], b.states[b.last]),
                           ("post-round", a.state(), b.state()),
                           ("ring snapshot", a.rings[a.last], b.rings[b.last]),
                           ("post-round ring", a.ring(), b.ring())):
            assert bits_equal(ta, tb), f"round {r}: {nm}"
    # the last round commits with an ordinary rollback on both sides
    kb.kda_rollback_pingpong(a, keeps[-1])
    kb.kda_rollback_pingpong(b, keeps[-1])
    torch.cuda.synchronize()
    assert bits_equal(a.state(), b.state()) and bits_equal(a.ring(), b.ring())


def test_deferred_matches_the_oracle(orc):
    L, B, H, Ts = 1, 3, 2, [7, 5]
    w0 = synth.Workload("do", L=L, B=B, H=H, T=7, bf16=True, V=64, rounds=1, seed=0x9933, accept="uniform")
    state0, ring0, cw = small_case(w0)
    rounds_np = _rounds(L, B, H, Ts, True, 0x9934)
    keep0 = [7, 4, 1]
    pp = kb.PingPong(layer_state(state0, ring0, cw))
    x0 = [rows_to_dev(rounds_np[0], True)[n] for n in NAMES]
    x1 = [rows_to_dev(rounds_np[1], True)[n] for n in NAMES]
    out = torch.empty((L, B, 5, H, 128), dtype=torch.float32, device="cuda")
    kb.kda_verify_scan_pingpong(pp, *x0)
    kb.kda_verify_scan_deferred(pp, *x1, torch.tensor(keep0, dtype=torch.int32, device="cuda"), out=out)
    torch.cuda.synchronize()
    for b in range(B):
        u0 = {n: rounds_np[0][n][0, b] for n in rounds_np[0]}
        u1 = {n: rounds_np[1][n][0, b] for n in rounds_np[1]}
        a0 = (u0["q"], u0["k"], u0["v"], u0["g"], u0["beta"], cw[0])
        s_T, r_T, _ = orc.verify(*a0, ring0[0, b], state0[0, b])
        s_c, r_c = orc.rollback(keep0[b], *a0, ring0[0, b], state0[0, b], r_T, s_T)
        s1, r1, o1 = orc.verify(u1["q"], u1["k"], u1["v"], u1["g"], u1["beta"], cw[0], r_c, s_c)
        assert_close(host(out[0, b]), o1, f"outputs of session {b}")
        assert_close(host(pp.state()[0, b]), s1, f"post-round state of session {b}")
        assert_close(host(pp.states[pp.last][0, b]), s_c, f"snapshot of session {b}")
        assert np.array_equal(host(pp.ring()[0, b]), r1) and np.array_equal(host(pp.rings[pp.last][0, b]), r_c)


def test_deferred_bad_keep_leaves_the_session_and_reports():
    L, B, H, Ts = 1, 3, 4, [6, 6]
    w0 = synth.Workload("db", L=L, B=B, H=H, T=6, bf16=True, V=64, rounds=1, seed=0x9935, accept="uniform")
    state0, ring0, cw = small_case(w0)
    rounds = [rows_to_dev(r, True) for r in _rounds(L, B, H, Ts, True, 0x9936)]
    good = [6, 2, 3]
    a = kb.PingPong(layer_state(state0, ring0, cw))
    b = kb.PingPong(layer_state(state0, ring0, cw))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for pp in (a, b):
        kb.kda_verify_scan_pingpong(pp, *[rounds[0][n] for n in NAMES])
    kb.kda_rollback_pingpong(a, good)
    kb.kda_verify_scan_pingpong(a, *[rounds[1][n] for n in NAMES])
    bad = [6, 0, 3]  # session 1's keep is outside 1..6
    kb.kda_verify_scan_deferred(b, *[rounds[1][n] for n in NAMES], torch.tensor(bad, dtype=torch.int32, device="cuda"),
                                dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & kb.ST_BADKEEP
    for s in (0, 2):  # the other sessions are processed as usual
        assert bits_equal(a.state()[:, s], b.state()[:, s]) and bits_equal(a.states[a.last][:, s], b.states[b.last][:, s])


def test_deferred_plan_equals_the_functions():
    L, B, H = 2, 3, 5
    w = synth.Workload("dp", L=L, B=B, H=H, T=8, bf16=True, V=500, rounds=4, seed=0x9937, accept="uniform")
    state0, ring0, cw = small_case(w)
    from gpu_util import to_dev
    rows = [rows_to_dev(synth.all_rows(w, r), True) for r in range(w.rounds)]
    logits = [to_dev(synth.logits(w, r), True) for r in range(w.rounds)]
    drafts = [to_dev(synth.drafts_for(synth.logit_argmax(w, r), synth.accept_targets(w, r), w.V))
              for r in range(w.rounds)]
    j, bonus, keep = (torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(3))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(kb.spec_accept_scratch_bytes(B, w.T, w.V), dtype=torch.uint8, device="cuda")
    out_a = torch.empty((L, B, w.T, H, 128), dtype=torch.float32, device="cuda")
    out_b = torch.empty_like(out_a)
    a = kb.PingPong(layer_state(state0, ring0, cw))
    b = kb.PingPong(layer_state(state0, ring0, cw))
    plans = [kb.DeferredRoundPlan(b, rows[r], out_b, logits[r], drafts[r], j, bonus, keep, status, scratch)
             for r in range(w.rounds)]
    first = kb.PingPongRoundPlan(b, rows[0], out_b, logits[0], drafts[0], j, bonus, keep, status, scratch)
    # plan side: round 0 verify + accept (no rollback yet), then deferred rounds
    first.verify(b.parity)
    first.accept()
    p0 = b.parity
    first._flip(p0)
    for r in range(w.rounds):
        x = [rows[r][n] for n in NAMES]
        if r > 0:
            kb.kda_rollback_pingpong(a, [int(t) + 1 for t in synth.accept_targets(w, r - 1)])
        kb.kda_verify_scan_pingpong(a, *x, out=out_a)
        if r > 0:
            plans[r]()
        torch.cuda.synchronize()
        assert [int(t) for t in j.cpu()] == list(synth.accept_targets(w, r))
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        assert bits_equal(a.state(), b.state()) and bits_equal(a.states[a.last], b.states[b.last]), f"round {r}"
    assert int(status[0]) == 0


@pytest.mark.parametrize("wl", ["stack34", "batched32"])
def test_deferred_full_size_equals_separate(wl):
    """The full-size workloads put 13 to 15 units on every CTA, so replay and verify
    items alternate through the stages and scan-input buffers across units; every
    state, ring and output bit must equal the separate rollback + ping-pong rounds.
    Keeps vary per session and round (a full keep, keep 1, and seeded ones)."""
    from speculative_decode_verify_kda_gb300 import synth_gpu
    w = synth.WORKLOADS[wl]
    dev = torch.device("cuda", 0)
    a = kb.PingPong(kb.LayerState(synth_gpu.state(w, dev), synth_gpu.ring(w, dev), synth_gpu.conv_w(w, dev)))
    b = kb.PingPong(kb.LayerState(synth_gpu.state(w, dev), synth_gpu.ring(w, dev), synth_gpu.conv_w(w, dev)))
    R = 4
    rows = [synth_gpu.rows(w, r, dev) for r in range(R)]
    keeps = _keeps(w.B, [w.T] * R, 0x9938)
    if w.B == 1:  # one session: cycle a partial keep, a full keep and keep 1 over the rounds
        keeps = [[3], [w.T], [1], [w.T - 1]]
    out_a = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device=dev)
    out_b = torch.empty_like(out_a)
    for r in range(R):
        x = [rows[r][n] for n in NAMES]
        if r > 0:
            kb.kda_rollback_pingpong(a, keeps[r - 1])
        kb.kda_verify_scan_pingpong(a, *x, out=out_a)
        if r == 0:
            kb.kda_verify_scan_pingpong(b, *x, out=out_b)
        else:
            kb.kda_verify_scan_deferred(b, *x, torch.tensor(keeps[r - 1], dtype=torch.int32, device=dev), out=out_b)
        torch.cuda.synchronize()
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        assert bits_equal(a.state(), b.state()) and bits_equal(a.ring(), b.ring()), f"round {r}: post-round"
        assert bits_equal(a.states[a.last], b.states[b.last]) and bits_equal(a.rings[a.last], b.rings[b.last]), \
            f"round {r}: snapshot"


@pytest.mark.parametrize("bounds", [None, [(0, 2), (2, 3)]], ids=["per-layer", "ranges"])
def test_per_layer_deferred_rounds_equal_one_launch(bounds):
    """A deferred round issued one launch per layer (as a model issues it) equals the
    one-launch deferred round bit for bit."""
    from gpu_util import to_dev
    L, B, H = 3, 2, 5
    w = synth.Workload("dl", L=L, B=B, H=H, T=6, bf16=True, V=300, rounds=5, seed=0x9939, accept="uniform")
    state0, ring0, cw = small_case(w)
    rows = [rows_to_dev(synth.all_rows(w, r), True) for r in range(w.rounds)]
    logits = [to_dev(synth.logits(w, r), True) for r in range(w.rounds)]
    drafts = [to_dev(synth.drafts_for(synth.logit_argmax(w, r), synth.accept_targets(w, r), w.V))
              for r in range(w.rounds)]

    def case():
        pp = kb.PingPong(layer_state(state0, ring0, cw))
        j, bonus, keep = (torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(3))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        scratch = torch.empty(kb.spec_accept_scratch_bytes(B, w.T, w.V), dtype=torch.uint8, device="cuda")
        out = torch.empty((L, B, w.T, H, 128), dtype=torch.float32, device="cuda")
        first = kb.PingPongRoundPlan(pp, rows[0], out, logits[0], drafts[0], j, bonus, keep, status, scratch)
        par = pp.parity
        first.verify(par)
        first.accept()
        first._flip(par)
        return pp, j, keep, status, scratch, out

    pa, ja, ka, sa, xa, oa = case()
    pb, jb, kb_, sb, xb, ob = case()
    lps = kb.layer_pingpongs(pb, bounds)
    for r in range(1, w.rounds):
        kb.DeferredRoundPlan(pa, rows[r], oa, logits[r], drafts[r], ja, torch.empty_like(ja), ka, sa, xa)()
        kb.LayerDeferredRoundPlan(pb, lps, rows[r], ob, logits[r], drafts[r], jb, torch.empty_like(jb), kb_, sb, xb,
                                  bounds=bounds)()
        torch.cuda.synchronize()
        assert torch.equal(ja, jb) and [int(x) for x in ja.cpu()] == list(synth.accept_targets(w, r))
        assert bits_equal(oa, ob), f"round {r}: outputs"
        assert bits_equal(pa.state(), pb.state()) and bits_equal(pa.ring(), pb.ring()), f"round {r}"
        assert bits_equal(pa.states[pa.last], pb.states[pb.last]), f"round {r}: snapshot"
    kb.kda_rollback_pingpong(pa, ka)
    kb.kda_rollback_pingpong(pb, kb_)
    torch.cuda.synchronize()
    assert bits_equal(pa.state(), pb.state()) and int(sa[0]) == 0 and int(sb[0]) == 0


@pytest.mark.parametrize("ppf,upload", [(1, "library"), (4, "library"), (3, "torch")])
def test_staged_deferred_rounds_equal_deferred_rounds(ppf, upload):
    """Deferred rounds whose raw rows arrive while the launch runs (copied from pinned host
    memory by ranges of (layer, session) pairs on a side stream, each range's flag set
    after its copy, by kda_upload_rows_staged or by torch copies and kda_stream_write_u32)
    give the bits of deferred rounds on resident rows."""
    ensure_built()
    from gpu_util import to_dev
    L, B, H = 3, 2, 5
    w = synth.Workload("st", L=L, B=B, H=H, T=6, bf16=True, V=300, rounds=5, seed=0x5791, accept="uniform")
    state0, ring0, cw = small_case(w)
    host_rows = [synth.all_rows(w, r) for r in range(w.rounds)]
    rows = [rows_to_dev(hr, True) for hr in host_rows]
    logits = [to_dev(synth.logits(w, r), True) for r in range(w.rounds)]
    drafts = [to_dev(synth.drafts_for(synth.logit_argmax(w, r), synth.accept_targets(w, r), w.V))
              for r in range(w.rounds)]
    pairs = L * B
    bounds = [(p0, min(pairs, p0 + ppf)) for p0 in range(0, pairs, ppf)]  # flag f covers pairs f*ppf ..
    flags = torch.zeros(kb.staged_flag_count(L, B, ppf), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()

    def case():
        pp = kb.PingPong(layer_state(state0, ring0, cw))
        j, bonus, keep = (torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(3))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        scratch = torch.empty(kb.spec_accept_scratch_bytes(B, w.T, w.V), dtype=torch.uint8, device="cuda")
        out = torch.empty((L, B, w.T, H, 128), dtype=torch.float32, device="cuda")
        first = kb.PingPongRoundPlan(pp, rows[0], out, logits[0], drafts[0], j, bonus, keep, status, scratch)
        par = pp.parity
        first.verify(par)
        first.accept()
        first._flip(par)
        return pp, j, bonus, keep, status, scratch, out

    pa, ja, ba, ka, sa, xa, oa = case()
    pb, jb, bb, kb_, sb, xb, ob = case()
    for r in range(1, w.rounds):
        kb.DeferredRoundPlan(pa, rows[r], oa, logits[r], drafts[r], ja, ba, ka, sa, xa)()
        # this round's rows for pb: fresh device tensors, filled while the launch waits
        pinned = {n: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
                  for n, a in host_rows[r].items()}
        if upload == "library" and ppf == 4:
            # q, k, v, g as four equal tensors of one allocation on both sides: the library
            # then copies a range of the four as one 2D copy
            shp = tuple(pinned["q"].shape)
            hblk = torch.empty((4,) + shp, dtype=torch.int16).pin_memory()
            dblk = torch.empty((4,) + shp, dtype=torch.int16, device="cuda")
            for i, n in enumerate(("q", "k", "v", "g")):
                hblk[i].copy_(pinned[n])
                pinned[n] = hblk[i]
            staged = {n: dblk[i] for i, n in enumerate(("q", "k", "v", "g"))}
            staged["beta"] = torch.empty(tuple(pinned["beta"].shape), dtype=torch.int16, device="cuda")
        else:
            staged = {n: torch.empty(t.shape, dtype=torch.int16, device="cuda") for n, t in pinned.items()}
        views = {n: t.view(torch.bfloat16) for n, t in staged.items()}
        plan = kb.DeferredRoundPlan(pb, views, ob, logits[r], drafts[r], jb, bb, kb_, sb, xb, ready_flags=flags,
                                    pairs_per_flag=ppf)
        p = pb.last
        plan.verify(p, epoch=r)
        if upload == "library":
            kb.StagedUpload(views, {n: t.view(torch.bfloat16) for n, t in pinned.items()}, flags, ppf)(r, side)
        else:
            with torch.cuda.stream(side):
                for f, (p0, p1) in enumerate(bounds):
                    for n in staged:  # [L][B] ... as pairs
                        staged[n].flatten(0, 1)[p0:p1].copy_(pinned[n].flatten(0, 1)[p0:p1], non_blocking=True)
                    kb.kda_stream_write_u32(flags[f:f + 1], r, stream=side)
        plan.accept()
        plan._flip(p)
        torch.cuda.synchronize()
        assert int(sb[0]) == 0, f"round {r}: status {int(sb[0]):#x}"
        assert torch.equal(ja, jb) and [int(x) for x in ja.cpu()] == list(synth.accept_targets(w, r))
        assert bits_equal(oa, ob), f"round {r}: outputs"
        assert bits_equal(pa.state(), pb.state()) and bits_equal(pa.ring(), pb.ring()), f"round {r}"
        assert bits_equal(pa.states[pa.last], pb.states[pb.last]), f"round {r}: snapshot"
        pb.rows = [views[n] for n in ("q", "k", "v", "g", "beta")]  # keep this round's rows alive
    kb.kda_rollback_pingpong(pa, ka)
    kb.kda_rollback_pingpong(pb, kb_)
    torch.cuda.synchronize()
    assert bits_equal(pa.state(), pb.state()) and int(sa[0]) == 0 and int(sb[0]) == 0


def test_staged_rows_that_never_arrive_time_out():
    """A ready flag that nothing sets: the launch gives up after its bounded wait, reports
    KDA_ST_TIMEOUT, and the device stays usable."""
    ensure_built()
    L, B, H = 2, 1, 3
    w = synth.Workload("to", L=L, B=B, H=H, T=4, bf16=True, V=64, rounds=2, seed=0x7101, accept="uniform")
    state0, ring0, cw = small_case(w)
    rows = [rows_to_dev(synth.all_rows(w, r), True) for r in range(2)]
    pp = kb.PingPong(layer_state(state0, ring0, cw))
    kb.kda_verify_scan_pingpong(pp, *[rows[0][n] for n in ("q", "k", "v", "g", "beta")])
    keep = torch.full((B,), 2, dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kb.kda_verify_scan_deferred_staged(pp, *[rows[1][n] for n in ("q", "k", "v", "g", "beta")], keep, flags,
                                       L * B, 7, dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & kb.ST_TIMEOUT
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float((x * 2).sum()) == 56.0


@pytest.mark.parametrize("wl,ppf", [("stack34", 9), ("batched32", 8)])
def test_staged_full_size_equals_resident(wl, ppf):
    """The e2e arrangement at full size: each round's raw rows streamed from one pinned
    block (q, k, v, g as four equal tensors, so a range of them is one 2D copy) into one
    device block by ranges of (layer, session) pairs while the staged launch runs; every
    output, state, ring and snapshot bit equals the deferred rounds on resident rows."""
    from speculative_decode_verify_kda_gb300 import synth_gpu
    w = synth.WORKLOADS[wl]
    dev = torch.device("cuda", 0)
    a = kb.PingPong(kb.LayerState(synth_gpu.state(w, dev), synth_gpu.ring(w, dev), synth_gpu.conv_w(w, dev)))
    b = kb.PingPong(kb.LayerState(synth_gpu.state(w, dev), synth_gpu.ring(w, dev), synth_gpu.conv_w(w, dev)))
    R = 3
    rows = [synth_gpu.rows(w, r, dev) for r in range(R)]
    keeps = _keeps(w.B, [w.T] * R, 0x9940)
    if w.B == 1:
        keeps = [[3], [1], [w.T]]
    shp, bshp = tuple(rows[0]["q"].shape), tuple(rows[0]["beta"].shape)
    flags = torch.zeros(kb.staged_flag_count(w.L, w.B, ppf), dtype=torch.int32, device=dev)
    side = torch.cuda.Stream()

    def block(on_dev):  # q, k, v, g in one allocation, beta apart
        kw = {"device": dev} if on_dev else {}
        qkvg = torch.empty((4,) + shp, dtype=torch.bfloat16, **kw)
        beta = torch.empty(bshp, dtype=torch.bfloat16, **kw)
        if not on_dev:
            qkvg, beta = qkvg.pin_memory(), beta.pin_memory()
        return dict(zip(NAMES, [qkvg[0], qkvg[1], qkvg[2], qkvg[3], beta]))

    out_a = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device=dev)
    out_b = torch.empty_like(out_a)
    dev_blocks = [block(True) for _ in range(2)]
    for r in range(R):
        x = [rows[r][n] for n in NAMES]
        db = dev_blocks[r % 2]
        if r == 0:
            kb.kda_verify_scan_pingpong(a, *x, out=out_a)
            for n in NAMES:
                db[n].copy_(rows[r][n])
            kb.kda_verify_scan_pingpong(b, *[db[n] for n in NAMES], out=out_b)
        else:
            keep = torch.tensor(keeps[r - 1], dtype=torch.int32, device=dev)
            kb.kda_verify_scan_deferred(a, *x, keep, out=out_a)
            hb = block(False)
            for n in NAMES:
                hb[n].copy_(rows[r][n].cpu())
            torch.cuda.synchronize()
            kb.kda_verify_scan_deferred_staged(b, *[db[n] for n in NAMES], keep, flags, ppf, r, out=out_b)
            kb.StagedUpload(db, hb, flags, ppf)(r, side)
        torch.cuda.synchronize()
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        assert bits_equal(a.state(), b.state()) and bits_equal(a.ring(), b.ring()), f"round {r}: post-round"
        assert bits_equal(a.states[a.last], b.states[b.last]) and bits_equal(a.rings[a.last], b.rings[b.last]), \
            f"round {r}: snapshot"


def test_staged_rounds_with_f32_rows():
    """f32 raw rows through kda_upload_rows_staged (4-byte elements) and the staged launch:
    the bits of deferred rounds on resident rows."""
    ensure_built()
    L, B, H = 2, 3, 4
    w = synth.Workload("sf", L=L, B=B, H=H, T=5, bf16=False, V=64, rounds=4, seed=0x5F32, accept="uniform")
    state0, ring0, cw = small_case(w)
    host_rows = [synth.all_rows(w, r) for r in range(w.rounds)]
    rows = [rows_to_dev(hr, False) for hr in host_rows]
    keeps = _keeps(B, [w.T] * w.rounds, 0x5F33)
    ppf = 2
    flags = torch.zeros(kb.staged_flag_count(L, B, ppf), dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    pa = kb.PingPong(layer_state(state0, ring0, cw))
    pb = kb.PingPong(layer_state(state0, ring0, cw))
    out_a = torch.empty((L, B, w.T, H, 128), dtype=torch.float32, device="cuda")
    out_b = torch.empty_like(out_a)
    kb.kda_verify_scan_pingpong(pa, *[rows[0][n] for n in NAMES], out=out_a)
    kb.kda_verify_scan_pingpong(pb, *[rows[0][n] for n in NAMES], out=out_b)
    keep_alive = []
    for r in range(1, w.rounds):
        keep = torch.tensor(keeps[r - 1], dtype=torch.int32, device="cuda")
        kb.kda_verify_scan_deferred(pa, *[rows[r][n] for n in NAMES], keep, out=out_a)
        pinned = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for n, a in host_rows[r].items()}
        staged = {n: torch.empty(t.shape, dtype=torch.float32, device="cuda") for n, t in pinned.items()}
        keep_alive.append(staged)
        kb.kda_verify_scan_deferred_staged(pb, *[staged[n] for n in NAMES], keep, flags, ppf, r, out=out_b)
        kb.StagedUpload(staged, pinned, flags, ppf)(r, side)
        torch.cuda.synchronize()
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        assert bits_equal(pa.state(), pb.state()) and bits_equal(pa.ring(), pb.ring()), f"round {r}"


@pytest.mark.parametrize("bf16,with_w", [(True, False), (True, True), (False, False)])
def test_deferred_rows_read_in_place_from_host(bf16, with_w):
    """kda_verify_scan_deferred_host reads this round's raw rows in place from pinned host
    memory: outputs, snapshots, states and rings bit-identical to the same rounds from
    device rows, and the device copy it leaves equals the host rows byte for byte (the
    next round replays from it)."""
    L, B, H, Ts = 2, 4, 5, [8, 6, 15, 3]
    w0 = synth.Workload("dh", L=L, B=B, H=H, T=Ts[0], bf16=bf16, V=64, rounds=1, seed=0x9940, accept="uniform")
    state0, ring0, cw = small_case(w0)
    rounds_np = _rounds(L, B, H, Ts, bf16, 0x9941)
    keeps = _keeps(B, Ts, 0x9942)
    dt = torch.bfloat16 if bf16 else torch.float32

    def host_set(r):
        out = {}
        for n in NAMES:
            t = torch.from_numpy(np.ascontiguousarray(rounds_np[r][n]))
            out[n] = (t.view(torch.bfloat16) if bf16 else t).pin_memory()
        return out

    a = kb.PingPong(layer_state(state0, ring0, cw))
    b = kb.PingPong(layer_state(state0, ring0, cw))
    hold = []
    for r, T in enumerate(Ts):
        x = rows_to_dev(rounds_np[r], bf16)
        out_a = torch.full((L, B, T, H, 128), float("nan"), device="cuda")
        out_b = torch.full_like(out_a, float("nan"))
        wa = torch.empty((L, B, T, H, 128), dtype=torch.float32, device="cuda") if with_w else None
        wb = torch.empty_like(wa) if with_w else None
        if r == 0:
            kb.kda_verify_scan_pingpong(a, *[x[n] for n in NAMES], out=out_a, w=wa)
            kb.kda_verify_scan_pingpong(b, *[x[n] for n in NAMES], out=out_b, w=wb)
            hold.append((x, wa, wb))
            continue
        keep = torch.tensor(keeps[r - 1], dtype=torch.int32, device="cuda")
        kb.kda_verify_scan_deferred(a, *[x[n] for n in NAMES], keep, out=out_a, w=wa)
        h = host_set(r)
        dev = {n: torch.full_like(x[n], 0) for n in NAMES}
        if with_w:
            dev["w"] = wb
        kb.kda_verify_scan_deferred_host(b, h, dev, keep, out=out_b)
        torch.cuda.synchronize()
        hold.append((x, h, dev, wa, wb))
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        for n in NAMES:
            assert torch.equal(dev[n].cpu().view(torch.int16 if bf16 else torch.int32),
                               h[n].view(torch.int16 if bf16 else torch.int32)), f"round {r}: device copy of {n}"
        for nm, ta, tb in (("snapshot", a.states[a.last], b.states[b.last]),
                           ("post-round", a.state(), b.state()),
                           ("ring snapshot", a.rings[a.last], b.rings[b.last]),
                           ("post-round ring", a.ring(), b.ring())):
            assert bits_equal(ta, tb), f"round {r}: {nm}"
    kb.kda_rollback_pingpong(a, keeps[-1])
    kb.kda_rollback_pingpong(b, keeps[-1])
    torch.cuda.synchronize()
    assert bits_equal(a.state(), b.state()) and bits_equal(a.ring(), b.ring())
