"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar: accept j / bonus / vam and conv rings bit-exact; f32 outputs and states
within rel 1e-4 / abs 1e-5 of the oracle (gpu_util.RTOL/ATOL).  GPU-vs-GPU
contracts (batched T rows == T chained one-row launches; rollback == a fresh
verify of the kept rows) are bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import assert_close, bits_equal, host, layer_state, rows_to_dev, small_case, to_dev
from libs import ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth, synth_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def _unit_dict(rows, l, b):
    return {n: rows[n][l, b] for n in synth.ROW_TENSORS}


def _oracle_round(orc, w, r, l, b, state, ring, conv_w, keep):
    """One round of one unit on the oracle: verify, then rollback to keep."""
    u = synth.unit_rows(w, r, l, b)
    args = (u["q"], u["k"], u["v"], u["g"], u["beta"])
    st_T, ring_T, out = orc.verify(*args, conv_w, ring, state)
    st_k, ring_k = orc.rollback(keep, *args, conv_w, ring, state, ring_T, st_T)
    return out, st_T, ring_T, st_k, ring_k


def _run_round(st: kb.LayerState, rows: dict, logits, drafts, stash, out):
    kb.kda_verify_scan(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], out=out, stash=stash)
    j, bonus, keep = kb.spec_accept(logits, drafts)
    kb.kda_rollback(st, stash, keep)
    return j, bonus, keep


# ---------------------------------------------------------------------------
def test_tiny_every_accept_j(orc):
    """One head, f32 rows, V=32: rounds sweep j = 0..7 with state carried round to round."""
    w = synth.WORKLOADS["tiny"]
    state0, ring0, cw = small_case(w)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    out = torch.empty((1, 1, w.T, 1, 128), dtype=torch.float32, device="cuda")
    s_ref, r_ref = state0[0, 0], ring0[0, 0]
    for r in range(w.rounds):
        rows = synth.all_rows(w, r)
        lg = synth.logits(w, r)
        d = synth.drafts_for(synth.logit_argmax(w, r), synth.accept_targets(w, r), w.V)
        pre_state = st.state.clone()
        j, bonus, keep = _run_round(st, rows_to_dev(rows, False), to_dev(lg), to_dev(d), stash, out)
        torch.cuda.synchronize()
        jr, br, vam, rc = orc.accept(lg[0], d[0])
        assert rc == 0 and jr == r and int(j[0]) == jr and int(bonus[0]) == br and int(keep[0]) == jr + 1
        o, st_T, ring_T, st_k, ring_k = _oracle_round(orc, w, r, 0, 0, s_ref, r_ref, cw[0], jr + 1)
        assert bits_equal(stash.state_snap, pre_state), "fused snapshot must equal the pre-round state"
        assert_close(host(out)[0, 0], o, f"round {r} out")
        assert_close(host(st.state)[0, 0], st_k, f"round {r} state after rollback")
        assert np.array_equal(host(st.conv_ring)[0, 0], ring_k), f"round {r} ring"
        s_ref, r_ref = st_k, ring_k


def test_layer64_rounds(orc):
    """One glm5_next-shaped layer (64 heads, bf16 rows, V=32768), four rounds carried."""
    w = synth.WORKLOADS["layer64"]
    state0, ring0, cw = small_case(w)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    out = torch.empty((1, 1, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    s_ref, r_ref = state0[0, 0], ring0[0, 0]
    for r in range(4):
        rows = synth.all_rows(w, r)
        lg = synth.logits(w, r)
        jt = synth.accept_targets(w, r)
        d = synth.drafts_for(synth.logit_argmax(w, r), jt, w.V)
        j, bonus, keep = _run_round(st, rows_to_dev(rows, True), to_dev(lg, True), to_dev(d), stash, out)
        torch.cuda.synchronize()
        jr, br, _, _ = orc.accept(lg[0], d[0])
        assert (int(j[0]), int(bonus[0])) == (jr, br) and jr == jt[0]
        o, st_T, ring_T, st_k, ring_k = _oracle_round(orc, w, r, 0, 0, s_ref, r_ref, cw[0], jr + 1)
        assert_close(host(out)[0, 0], o, f"round {r} out")
        assert_close(host(st.state)[0, 0], st_k, f"round {r} state")
        assert np.array_equal(host(st.conv_ring)[0, 0], ring_k)
        s_ref, r_ref = st_k, ring_k


@pytest.mark.parametrize("name", ["tiny", "layer64"])
def test_batched_launch_equals_chained_single_rows(name):
    """T rows in one launch == T launches of one row each (state, ring, outputs bit-identical)."""
    w = synth.WORKLOADS[name]
    state0, ring0, cw = small_case(w)
    rows = rows_to_dev(synth.all_rows(w, 0), w.bf16)
    a = layer_state(state0, ring0, cw)
    out_a = torch.empty((1, 1, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    kb.kda_verify_scan(a, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], out=out_a)
    c = layer_state(state0, ring0, cw)
    out_c = torch.empty_like(out_a)
    for t in range(w.T):
        sl = {n: x[:, :, t:t + 1].contiguous() for n, x in rows.items()}
        o = torch.empty((1, 1, 1, w.H, 128), dtype=torch.float32, device="cuda")
        kb.kda_verify_scan(c, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], out=o)
        out_c[:, :, t] = o[:, :, 0]
    torch.cuda.synchronize()
    assert bits_equal(a.state, c.state)
    assert bits_equal(a.conv_ring, c.conv_ring)
    assert bits_equal(out_a, out_c)


@pytest.mark.parametrize("name", ["tiny", "batched32"])
def test_rollback_equals_verify_of_kept_rows(name):
    """Verify(T) + rollback(keep) == verify of rows 0..keep-1 from the same start, bit for bit."""
    w = synth.WORKLOADS[name]
    if name == "batched32":
        w = synth.Workload("b4", L=2, B=4, H=8, T=15, bf16=True, V=64, rounds=1, seed=77, accept="uniform")
    state0, ring0, cw = small_case(w)
    rows = rows_to_dev(synth.all_rows(w, 0), w.bf16)
    for shift in range(w.T):
        keep = [((k + shift) % w.T) + 1 for k in range(w.B)]
        a = layer_state(state0, ring0, cw)
        stash = kb.Stash(a)
        kb.kda_verify_scan(a, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], stash=stash)
        kb.kda_rollback(a, stash, keep)
        for b in range(w.B):
            ref = layer_state(state0[:, b:b + 1], ring0[:, b:b + 1], cw)
            kk = keep[b]
            sl = {n: x[:, b:b + 1, :kk].contiguous() for n, x in rows.items()}
            kb.kda_verify_scan(ref, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"])
            torch.cuda.synchronize()
            assert bits_equal(a.state[:, b], ref.state[:, 0]), (shift, b, kk)
            assert bits_equal(a.conv_ring[:, b], ref.conv_ring[:, 0]), (shift, b, kk)


def test_rollback_host_and_device_keep_agree():
    w = synth.Workload("hk", L=1, B=6, H=4, T=7, bf16=True, V=64, rounds=1, seed=78, accept="uniform")
    state0, ring0, cw = small_case(w)
    rows = rows_to_dev(synth.all_rows(w, 0), True)
    keep = [1, 7, 3, 7, 6, 2]
    res = []
    for mode in ("host", "device"):
        st = layer_state(state0, ring0, cw)
        stash = kb.Stash(st)
        kb.kda_verify_scan(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], stash=stash)
        k = keep if mode == "host" else torch.tensor(keep, dtype=torch.int32, device="cuda")
        kb.kda_rollback(st, stash, k)
        res.append((st.state.clone(), st.conv_ring.clone()))
    torch.cuda.synchronize()
    assert bits_equal(res[0][0], res[1][0]) and bits_equal(res[0][1], res[1][1])


def test_bad_device_keep_sets_status_and_leaves_state():
    w = synth.Workload("bk", L=1, B=3, H=2, T=5, bf16=False, V=64, rounds=1, seed=79, accept="uniform")
    state0, ring0, cw = small_case(w)
    rows = rows_to_dev(synth.all_rows(w, 0), False)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    kb.kda_verify_scan(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], stash=stash)
    after = st.state.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kb.kda_rollback(st, stash, torch.tensor([0, 6, 5], dtype=torch.int32, device="cuda"), dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & kb.ST_BADKEEP
    assert bits_equal(st.state, after)


@pytest.mark.parametrize("H,T", [(1, 1), (3, 15), (5, 2)])
def test_shapes_and_edges(orc, H, T):
    """Odd head counts, T = 1 (no drafts) and the T = 15 cap, f32 and bf16 rows."""
    for bf16 in (False, True):
        w = synth.Workload("e", L=2, B=2, H=H, T=T, bf16=bf16, V=40, rounds=1, seed=80 + H + T, accept="uniform")
        state0, ring0, cw = small_case(w)
        rows_np = synth.all_rows(w, 0)
        st = layer_state(state0, ring0, cw)
        stash = kb.Stash(st)
        out = torch.empty((2, 2, T, H, 128), dtype=torch.float32, device="cuda")
        rows = rows_to_dev(rows_np, bf16)
        kb.kda_verify_scan(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], out=out, stash=stash)
        torch.cuda.synchronize()
        ref = orc.verify_units(rows_np, cw, ring0, state0)
        for (l, b), (s_o, r_o, o_o) in ref.items():
            assert_close(host(out)[l, b], o_o, f"out {l},{b}")
            assert_close(host(st.state)[l, b], s_o, f"state {l},{b}")
            assert np.array_equal(host(st.conv_ring)[l, b], r_o)
        assert bits_equal(stash.state_snap, to_dev(state0)) and bits_equal(stash.ring_snap, to_dev(ring0))


def test_empty_problem_is_a_no_op():
    """L*B*H = 0: verify and rollback succeed without touching memory (torch gives NULL pointers)."""
    st = kb.LayerState(torch.zeros((0, 1, 64, 128, 128), device="cuda"), torch.zeros((0, 1, 64, 3, 3, 128), device="cuda"),
                       torch.zeros((0, 64, 3, 128, 4), device="cuda"))
    z = torch.zeros((0, 1, 8, 64, 128), dtype=torch.bfloat16, device="cuda")
    stash = kb.Stash(st)
    kb.kda_verify_scan(st, z, z, z, z, torch.zeros((0, 1, 8, 64), dtype=torch.bfloat16, device="cuda"), stash=stash)
    assert stash.T == 8
    kb.kda_rollback(st, stash, [3])
    j, bonus, keep = kb.spec_accept(torch.zeros((0, 4, 100), device="cuda"),
                                    torch.zeros((0, 3), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert j.numel() == 0


# ---------------------------------------------------------------------------
# accept
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 7, 33, 1000, 4096, 32768, 40000])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_accept_against_oracle(orc, V, dtype):
    """Ragged and small vocabularies, many ties, an all -inf row; f32 and bf16 logits."""
    rng = np.random.default_rng(V)
    B, T = 5, 6
    x = rng.integers(-4, 5, (B, T, V)).astype(np.float32)  # values -4..4: ties everywhere
    plant = rng.integers(0, V, (B, T))
    for b in range(1, B, 2):  # odd sessions get a unique row maximum, even ones keep the ties
        x[b, np.arange(T), plant[b]] = 7.0
    x[1, 2, :] = -np.inf
    xin = synth.to_bf16_bits(x) if dtype == "bf16" else x
    vam = np.stack([orc.accept(xin[b], np.zeros(T - 1, np.int32))[2] for b in range(B)])
    d = synth.drafts_for(vam, np.array([0, 5, 2, 4, 1]), max(V, 2))
    j, bonus, keep = kb.spec_accept(to_dev(xin, dtype == "bf16"), to_dev(d))
    torch.cuda.synchronize()
    for b in range(B):
        jr, br, _, rc = orc.accept(xin[b], d[b])
        assert rc == 0
        assert (int(j[b]), int(bonus[b]), int(keep[b])) == (jr, br, jr + 1), (b, V)


def test_accept_nan_rows():
    V, T = 64, 4
    x = np.zeros((3, T, V), np.float32)
    x[:, :, 5] = 1.0
    x[0, 2, 9] = np.nan   # consulted: drafts match rows 0,1 -> j reaches row 2
    x[1, 2, 9] = np.nan   # not consulted: mismatch at row 0
    d = np.array([[5, 5, 5], [4, 5, 5], [5, 5, 5]], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    j, bonus, _ = kb.spec_accept(to_dev(x), to_dev(d), dev_status=status)
    torch.cuda.synchronize()
    assert (int(j[0]), int(bonus[0])) == (2, -1)
    assert (int(j[1]), int(bonus[1])) == (0, 5)
    assert (int(j[2]), int(bonus[2])) == (3, 5)
    assert int(status[0]) & kb.ST_NAN


# ---------------------------------------------------------------------------
# full-size workloads in the bench's launch configuration (sampled units)
# ---------------------------------------------------------------------------
def _device_case(w):
    st = kb.LayerState(synth_gpu.state(w), synth_gpu.ring(w), synth_gpu.conv_w(w))
    return st


@pytest.mark.parametrize("name,rounds,units", [
    ("stack34", 12, [(0, 0), (17, 0), (33, 0)]),
    ("batched32", 2, [(0, 0), (0, 13), (0, 31)]),
])
def test_multiround_sampled_units(orc, name, rounds, units):
    w = synth.WORKLOADS[name]
    st = _device_case(w)
    stash = kb.Stash(st)
    out = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    ref = {(l, b): (synth.unit_state(w, l, b), synth.unit_ring(w, l, b), synth.layer_conv_w(w, l)) for l, b in units}
    for r in range(rounds):
        rows = synth_gpu.rows(w, r)
        lg = synth_gpu.logits(w, r)
        d, jt = synth_gpu.drafts(w, r)
        j, bonus, keep = _run_round(st, rows, lg, d, stash, out)
        torch.cuda.synchronize()
        assert [int(x) for x in j.cpu()] == jt
        for (l, b) in units:
            s, rg, cw = ref[(l, b)]
            o, st_T, ring_T, st_k, ring_k = _oracle_round(orc, w, r, l, b, s, rg, cw, jt[b] + 1)
            assert_close(host(out[l, b]), o, f"{name} r{r} unit {l},{b} out")
            assert_close(host(st.state[l, b]), st_k, f"{name} r{r} unit {l},{b} state")
            assert np.array_equal(host(st.conv_ring[l, b]), ring_k)
            ref[(l, b)] = (st_k, ring_k, cw)


def test_stress_full_size_one_round(orc):
    """64 sessions x 34 layers x 64 heads at T = 15 (~8.5 GiB of state): one round, sampled units,
    plus size-independent properties on every unit."""
    w = synth.WORKLOADS["stress64x34"]
    st = _device_case(w)
    stash = kb.Stash(st)
    out = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    rows = synth_gpu.rows(w, 0)
    lg = synth_gpu.logits(w, 0)
    d, jt = synth_gpu.drafts(w, 0)
    kb.kda_verify_scan(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], out=out, stash=stash)
    post = st.state[:, [b for b in range(w.B) if jt[b] == w.K]].clone()
    j, bonus, keep = kb.spec_accept(lg, d)
    kb.kda_rollback(st, stash, keep)
    torch.cuda.synchronize()
    assert [int(x) for x in j.cpu()] == jt
    # the snapshot is the pre-round state of every unit, bit for bit
    assert bits_equal(stash.state_snap, synth_gpu.state(w))
    # full-accept sessions keep the post-verify state untouched
    assert bits_equal(st.state[:, [b for b in range(w.B) if jt[b] == w.K]], post)
    full = [b for b in range(w.B) if jt[b] == w.K][:1]
    low = [b for b in range(w.B) if jt[b] == 0][:1]
    units = [(0, 0), (33, 63), (17, 31)] + [(5, b) for b in full + low]
    for (l, b) in units:
        s, rg, cw = synth.unit_state(w, l, b), synth.unit_ring(w, l, b), synth.layer_conv_w(w, l)
        o, _, _, st_k, ring_k = _oracle_round(orc, w, 0, l, b, s, rg, cw, jt[b] + 1)
        assert_close(host(out[l, b]), o, f"stress unit {l},{b} out")
        assert_close(host(st.state[l, b]), st_k, f"stress unit {l},{b} state")
        assert np.array_equal(host(st.conv_ring[l, b]), ring_k)


@pytest.mark.parametrize("name", ["tiny", "layer64"])
def test_state_does_not_depend_on_asking_for_outputs(name):
    """A verify that writes output rows and one that does not (the replay path) leave the
    same state and ring bits; so do rollbacks after each."""
    w = synth.WORKLOADS[name]
    state0, ring0, cw = small_case(w)
    rows = rows_to_dev(synth.all_rows(w, 0), w.bf16)
    a = layer_state(state0, ring0, cw)
    b = layer_state(state0, ring0, cw)
    sa, sb = kb.Stash(a), kb.Stash(b)
    out = torch.empty((1, 1, w.T, w.H, 128), dtype=torch.float32, device="cuda")
    kb.kda_verify_scan(a, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], out=out, stash=sa)
    kb.kda_verify_scan(b, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], stash=sb)
    torch.cuda.synchronize()
    assert bits_equal(a.state, b.state) and bits_equal(a.conv_ring, b.conv_ring)
    kb.kda_rollback(a, sa, [3])
    kb.kda_rollback(b, sb, [3])
    torch.cuda.synchronize()
    assert bits_equal(a.state, b.state) and bits_equal(a.conv_ring, b.conv_ring)
