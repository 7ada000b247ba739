"""GPU: rounds whose length differs per session (variable T inside one batched grid).

* spec_window (glm_spec.rs glm5_conf_keep; dflash.rs dspark_confidence_vt and
  dspark_slot_confidence_vt) against the oracle and the pages' unit-test fixtures;
* kda_verify_scan_var / spec_accept_var / kda_rollback_var: per session bit-identical
  to the fixed-T calls on that session's rows, and within tolerance of the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import assert_close, bits_equal, host, layer_state, rows_to_dev, small_case, to_dev
from libs import ensure_built
from oracle_pins import _golden_windows, _logit_f32

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


# ---------------------------------------------------------------------------
# spec_window
# ---------------------------------------------------------------------------
def test_window_page_fixtures_on_device():
    for kind, vals, param, flag, exp in _golden_windows():
        if kind == "conf_keep":
            scores, policy, cap, want = vals, kb.WIN_CONF_KEEP, 15, min(exp + 1, 15)
            pmin0 = flag
        else:
            scores = _logit_f32(vals)
            policy = kb.WIN_CONFIDENCE if kind == "confidence" else kb.WIN_SLOT_CONFIDENCE
            cap, want, pmin0 = flag, exp, 0
        s = torch.from_numpy(np.ascontiguousarray(scores.reshape(1, -1), np.float32)).cuda()
        got = kb.spec_window(s, policy, float(param), cap, pmin0)
        torch.cuda.synchronize()
        assert int(got[0]) == want, (kind, list(vals), float(param), flag)


def _near_threshold(values: np.ndarray, thr: np.float32) -> bool:
    """Whether any value sits within 4 ulp of the threshold (the device and host exp may
    then round to opposite sides)."""
    if values.size == 0:
        return False
    return bool(np.any(np.abs(values.astype(np.float64) - float(thr)) <= 4 * np.spacing(np.float32(thr))))


@pytest.mark.parametrize("policy", [kb.WIN_CONF_KEEP, kb.WIN_CONFIDENCE, kb.WIN_SLOT_CONFIDENCE])
def test_window_kernel_against_oracle(orc, policy):
    rng = np.random.default_rng(100 + policy)
    B, K = 513, 14
    if policy == kb.WIN_CONF_KEEP:
        scores = rng.uniform(0, 1, (B, K)).astype(np.float32)
        scores[::7, 0] = 0.05  # slot-0 misses
    else:
        scores = rng.normal(1.5, 2.0, (B, K)).astype(np.float32)
    for param in (0.0, 0.2, 0.5, 0.9):
        for cap in ((1, 8, 15) if policy == kb.WIN_CONF_KEEP else (2, 5, 15)):
            for pmin0 in (0, 1):
                got = host(kb.spec_window(to_dev(scores), policy, param, cap, pmin0))
                torch.cuda.synchronize()
                bad = 0
                for b in range(B):
                    if policy == kb.WIN_CONF_KEEP:
                        want = min(orc.conf_keep(scores[b], param, pmin0) + 1, cap)
                    elif policy == kb.WIN_CONFIDENCE:
                        want = orc.confidence_vt(scores[b], param, cap)
                    else:
                        want = orc.slot_confidence_vt(scores[b], param, cap)
                    if int(got[b]) != want:
                        sig = (np.float32(1) / (np.float32(1) + np.exp(-scores[b]).astype(np.float32)))
                        stat = np.cumprod(sig, dtype=np.float32) if policy == kb.WIN_CONFIDENCE else sig
                        assert policy != kb.WIN_CONF_KEEP and _near_threshold(stat, np.float32(param)), \
                            (b, int(got[b]), want)
                        bad += 1
                assert bad <= 2


# ---------------------------------------------------------------------------
# verify / accept / rollback with per-session rows
# ---------------------------------------------------------------------------
W = synth.Workload("var", L=2, B=6, H=4, T=9, bf16=True, V=300, rounds=2, seed=131, accept="uniform")
T_ROWS = [9, 1, 5, 2, 9, 7]


def _session_fixed(state0, ring0, cw, rows, b, n):
    """Session b alone through the fixed-T call on its first n rows."""
    ref = layer_state(state0[:, b:b + 1], ring0[:, b:b + 1], cw)
    sl = {k: x[:, b:b + 1, :n].contiguous() for k, x in rows.items()}
    out = torch.empty((W.L, 1, n, W.H, 128), dtype=torch.float32, device="cuda")
    stash = kb.Stash(ref)
    kb.kda_verify_scan(ref, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], out=out, stash=stash)
    return ref, out, stash


@pytest.mark.parametrize("mem", ["host", "device"])
def test_verify_var_equals_fixed_per_session(orc, mem):
    state0, ring0, cw = small_case(W)
    rows_np = synth.all_rows(W, 0)
    rows = rows_to_dev(rows_np, W.bf16)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    out = torch.zeros((W.L, W.B, W.T, W.H, 128), dtype=torch.float32, device="cuda")
    t = T_ROWS if mem == "host" else torch.tensor(T_ROWS, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kb.kda_verify_scan_var(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], t, out=out, stash=stash,
                           dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == 0
    assert bits_equal(stash.state_snap, to_dev(state0)) and bits_equal(stash.ring_snap, to_dev(ring0))
    for b, n in enumerate(T_ROWS):
        ref, ref_out, _ = _session_fixed(state0, ring0, cw, rows, b, n)
        torch.cuda.synchronize()
        assert bits_equal(st.state[:, b], ref.state[:, 0]), b
        assert bits_equal(st.conv_ring[:, b], ref.conv_ring[:, 0]), b
        assert bits_equal(out[:, b, :n], ref_out[:, 0]), b
        assert not out[:, b, n:].any(), "rows past a session's count are not written"
        for l in range(W.L):  # and the oracle, on the session's rows
            sl = {k: x[l, b, :n] for k, x in rows_np.items()}
            s_o, r_o, o_o = orc.verify(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], cw[l], ring0[l, b],
                                       state0[l, b])
            assert_close(host(st.state[l, b]), s_o, f"state {l},{b}")
            assert_close(host(out[l, b, :n]), o_o, f"out {l},{b}")
            assert np.array_equal(host(st.conv_ring[l, b]), r_o)


def test_accept_var_against_oracle(orc):
    rng = np.random.default_rng(7)
    B, T, V = 9, 12, 777
    x = rng.normal(0, 1, (B, T, V)).astype(np.float32)
    plant = rng.integers(0, V, (B, T))
    x[np.arange(B)[:, None], np.arange(T)[None, :], plant] = 9.0
    t_rows = np.array([12, 1, 2, 7, 12, 3, 5, 11, 6], np.int32)
    jt = np.array([rng.integers(0, t) for t in t_rows])
    d = synth.drafts_for(plant, jt, V)
    d[1] = -5  # a one-row round reads no drafts
    j, bonus, keep = kb.spec_accept_var(to_dev(x), to_dev(d), to_dev(t_rows))
    torch.cuda.synchronize()
    for b in range(B):
        n = int(t_rows[b])
        jr, br, _, rc = orc.accept(x[b, :n], d[b, :n - 1])
        assert rc == 0 and jr == jt[b]
        assert (int(j[b]), int(bonus[b]), int(keep[b])) == (jr, br, jr + 1), b


@pytest.mark.parametrize("mem", ["host", "device"])
def test_rollback_var_equals_verify_of_kept_rows(mem):
    state0, ring0, cw = small_case(W)
    rows = rows_to_dev(synth.all_rows(W, 0), W.bf16)
    for shift in range(3):
        keep = [((b + shift) % n) + 1 for b, n in enumerate(T_ROWS)]
        st = layer_state(state0, ring0, cw)
        stash = kb.Stash(st)
        kb.kda_verify_scan_var(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], T_ROWS, stash=stash)
        post = st.state.clone()
        if mem == "host":
            kb.kda_rollback_var(st, stash, T_ROWS, keep)
        else:
            kb.kda_rollback_var(st, stash, torch.tensor(T_ROWS, dtype=torch.int32, device="cuda"),
                                torch.tensor(keep, dtype=torch.int32, device="cuda"))
        for b, kk in enumerate(keep):
            ref, _, _ = _session_fixed(state0, ring0, cw, rows, b, kk)
            torch.cuda.synchronize()
            assert bits_equal(st.state[:, b], ref.state[:, 0]), (shift, b, kk)
            assert bits_equal(st.conv_ring[:, b], ref.conv_ring[:, 0]), (shift, b, kk)
            if kk == T_ROWS[b]:
                assert bits_equal(st.state[:, b], post[:, b])


def test_invalid_device_rows_leave_the_session_untouched():
    state0, ring0, cw = small_case(W)
    rows = rows_to_dev(synth.all_rows(W, 0), W.bf16)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = torch.tensor([9, 0, 5, 10, 9, 7], dtype=torch.int32, device="cuda")
    kb.kda_verify_scan_var(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], t, stash=stash,
                           dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & kb.ST_BADKEEP
    for b in (1, 3):
        assert bits_equal(st.state[:, b], to_dev(state0)[:, b]) and bits_equal(st.conv_ring[:, b], to_dev(ring0)[:, b])
    j, bonus, keep = kb.spec_accept_var(torch.zeros((W.B, W.T, 64), device="cuda"),
                                        torch.zeros((W.B, W.T - 1), dtype=torch.int32, device="cuda"), t,
                                        dev_status=status)
    torch.cuda.synchronize()
    assert [int(x) for x in keep.cpu()][1] == 0 and [int(x) for x in keep.cpu()][3] == 0


def test_device_round_window_verify_accept_rollback(orc):
    """A whole variable-length round with every decision on the device: spec_window sizes
    the rounds, then verify, accept and rollback read its counts."""
    state0, ring0, cw = small_case(W)
    rows_np = synth.all_rows(W, 0)
    rows = rows_to_dev(rows_np, W.bf16)
    rng = np.random.default_rng(11)
    conf = rng.uniform(0.3, 1.0, (W.B, W.K)).astype(np.float32)
    t = kb.spec_window(to_dev(conf), kb.WIN_CONF_KEEP, 0.5, W.T)
    t_host = [min(orc.conf_keep(conf[b], 0.5, False) + 1, W.T) for b in range(W.B)]
    lg = synth.logits(W, 0)
    plant = synth.logit_argmax(W, 0)
    jt = np.array([rng.integers(0, n) for n in t_host])
    d = synth.drafts_for(plant, jt, W.V)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    kb.kda_verify_scan_var(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], t, stash=stash)
    j, bonus, keep = kb.spec_accept_var(to_dev(lg, W.bf16), to_dev(d), t)
    kb.kda_rollback_var(st, stash, t, keep)
    torch.cuda.synchronize()
    assert [int(x) for x in t.cpu()] == t_host
    assert [int(x) for x in j.cpu()] == list(jt)
    for b in range(W.B):
        for l in range(W.L):
            n = int(jt[b]) + 1
            sl = {k: x[l, b, :n] for k, x in rows_np.items()}
            s_o, r_o, _ = orc.verify(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], cw[l], ring0[l, b], state0[l, b])
            assert_close(host(st.state[l, b]), s_o, f"state {l},{b}")
            assert np.array_equal(host(st.conv_ring[l, b]), r_o)
