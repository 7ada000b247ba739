"""GPU: replays that read the update vectors the verify stored.

A rollback (glm_spec.rs, glm5_verify_rollback: restore the pre-round snapshot and
replay rows 0..keep-1) re-runs rows whose update vector w_t = beta_t (v_t - S'^T k_t)
the verify already formed.  With kda_rows.w the verify writes w_t and the replay reads
it back, so a replayed row is only S' = d S and S = S' + k w^T.  Those are the operations
the verify applied, on the same operands, so every state, ring and output must be
bit-identical to the same rounds run without w; and a replay must really read w (a
changed w changes the replayed state).
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
    out = []
    for r, T in enumerate(Ts):
        w = synth.Workload(f"w{T}", L=L, B=B, H=H, T=T, bf16=bf16, V=64, rounds=r + 1, seed=seed + 11 * T,
                           accept="uniform")
        out.append(rows_to_dev(synth.all_rows(w, r), bf16))
    return out


def _keeps(B, Ts, seed):
    g = np.random.default_rng(seed)
    ks = []
    for T in Ts:
        k = g.integers(1, T + 1, B)
        k[0] = T   # nothing to replay
        k[-1] = 1  # the shortest replay
        ks.append([int(x) for x in k])
    return ks


def _wbuf(L, B, T, H):
    # NaN-filled: a row the verify did not write would poison the replay
    return torch.full((L, B, T, H, 128), float("nan"), dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("bf16,Ts", [(True, [8, 8, 8, 8, 8]), (True, [8, 5, 15, 1, 3, 15]), (False, [6, 9, 2, 7])])
def test_deferred_rounds_with_w_are_bit_identical(bf16, Ts):
    L, B, H = 2, 5, 6
    w0 = synth.Workload("wd", L=L, B=B, H=H, T=Ts[0], bf16=bf16, V=64, rounds=1, seed=0x7710, accept="uniform")
    state0, ring0, cw = small_case(w0)
    rounds = _rounds(L, B, H, Ts, bf16, 0x7711)
    keeps = _keeps(B, Ts, 0x7712)
    a = kb.PingPong(layer_state(state0, ring0, cw))  # without w
    b = kb.PingPong(layer_state(state0, ring0, cw))  # with the update vectors stored
    wb = [_wbuf(L, B, T, H) for T in Ts]  # a round's replay reads the previous round's
    for r, T in enumerate(Ts):
        out_a = torch.full((L, B, T, H, 128), float("nan"), device="cuda")
        out_b = torch.full_like(out_a, float("nan"))
        x = [rounds[r][n] for n in NAMES]
        wr = wb[r]
        if r == 0:
            kb.kda_verify_scan_pingpong(a, *x, out=out_a)
            kb.kda_verify_scan_pingpong(b, *x, out=out_b, w=wr)
        else:
            keep = torch.tensor(keeps[r - 1], dtype=torch.int32, device="cuda")
            kb.kda_verify_scan_deferred(a, *x, keep, out=out_a)
            kb.kda_verify_scan_deferred(b, *x, keep, out=out_b, w=wr)
        torch.cuda.synchronize()
        assert bits_equal(out_a, out_b), f"round {r}: outputs"
        for nm, ta, tb in (("snapshot", a.states[a.last], b.states[b.last]),
                           ("post-round", a.state(), b.state()),
                           ("ring snapshot", a.rings[a.last], b.rings[b.last]),
                           ("post-round ring", a.ring(), b.ring())):
            assert bits_equal(ta, tb), f"round {r}: {nm}"
    kb.kda_rollback_pingpong(a, keeps[-1])
    kb.kda_rollback_pingpong(b, keeps[-1])  # the last round's replay reads its w
    torch.cuda.synchronize()
    assert bits_equal(a.state(), b.state()) and bits_equal(a.ring(), b.ring())


@pytest.mark.parametrize("bf16,device_keep", [(True, False), (True, True), (False, True)])
def test_rollback_with_w_is_bit_identical(bf16, device_keep):
    L, B, H, T = 2, 4, 5, 11
    w0 = synth.Workload("wr", L=L, B=B, H=H, T=T, bf16=bf16, V=64, rounds=1, seed=0x7720, accept="uniform")
    state0, ring0, cw = small_case(w0)
    x = [_rounds(L, B, H, [T], bf16, 0x7721)[0][n] for n in NAMES]
    keep = [3, T, 1, 7]
    kd = torch.tensor(keep, dtype=torch.int32, device="cuda") if device_keep else keep
    res = []
    for use_w in (False, True):
        st = layer_state(state0, ring0, cw)
        stash = kb.Stash(st)
        wb = _wbuf(L, B, T, H) if use_w else None
        out = torch.full((L, B, T, H, 128), float("nan"), device="cuda")
        kb.kda_verify_scan(st, *x, out=out, stash=stash, w=wb)
        kb.kda_rollback(st, stash, kd)
        torch.cuda.synchronize()
        res.append((out, st.state.clone(), st.conv_ring.clone(), wb))
    (oa, sa, ra, _), (ob, sb, rb, wb) = res
    assert bits_equal(oa, ob) and bits_equal(sa, sb) and bits_equal(ra, rb)
    assert not torch.isnan(wb).any()  # the verify wrote every row's update vector


def test_pingpong_var_rollback_with_w_is_bit_identical():
    L, B, H, T = 1, 4, 4, 9
    w0 = synth.Workload("wv", L=L, B=B, H=H, T=T, bf16=True, V=64, rounds=1, seed=0x7730, accept="uniform")
    state0, ring0, cw = small_case(w0)
    x = [_rounds(L, B, H, [T], True, 0x7731)[0][n] for n in NAMES]
    t_rows = torch.tensor([9, 4, 6, 1], dtype=torch.int32, device="cuda")
    keep = torch.tensor([5, 2, 6, 1], dtype=torch.int32, device="cuda")
    pps = []
    for use_w in (False, True):
        pp = kb.PingPong(layer_state(state0, ring0, cw))
        kb.kda_verify_scan_pingpong(pp, *x, t_rows=t_rows, w=_wbuf(L, B, T, H) if use_w else None)
        kb.kda_rollback_pingpong(pp, keep, t_rows=t_rows)
        pps.append(pp)
    torch.cuda.synchronize()
    assert bits_equal(pps[0].state(), pps[1].state()) and bits_equal(pps[0].ring(), pps[1].ring())


def test_the_replay_reads_w():
    """A replay with a changed w leaves a different state: the stored vectors are what
    it applies (the bit-identity tests above show they are the right ones)."""
    L, B, H, T = 1, 2, 3, 6
    w0 = synth.Workload("wx", L=L, B=B, H=H, T=T, bf16=True, V=64, rounds=1, seed=0x7740, accept="uniform")
    state0, ring0, cw = small_case(w0)
    x = [_rounds(L, B, H, [T], True, 0x7741)[0][n] for n in NAMES]
    keep = [4, 2]
    st0 = layer_state(state0, ring0, cw)
    stash0 = kb.Stash(st0)
    kb.kda_verify_scan(st0, *x, stash=stash0)
    kb.kda_rollback(st0, stash0, keep)
    st = layer_state(state0, ring0, cw)
    stash = kb.Stash(st)
    wb = _wbuf(L, B, T, H)
    kb.kda_verify_scan(st, *x, stash=stash, w=wb)
    snap = stash.state_snap.clone()
    ring_snap = stash.ring_snap.clone()
    wb[:, :, 1] *= 0.5  # row 1's update vectors of both sessions (both replay row 1)
    kb.kda_rollback(st, stash, keep)
    torch.cuda.synchronize()
    assert bits_equal(stash.state_snap, snap) and bits_equal(stash.ring_snap, ring_snap)
    for b in range(B):
        assert not bits_equal(st.state[:, b], st0.state[:, b]), f"session {b} did not apply the stored w"
    assert bits_equal(st.conv_ring, st0.conv_ring)  # the ring does not depend on w


def test_w_rows_match_the_oracle_update_vectors(orc):
    """The stored w_t of every unit and row against the oracle's: its activations of the
    rows (conv, SiLU, L2 norm, gates) and the state before row t from its recurrence,
    then w_t = beta_t (v_t - (diag(exp g_t) S)^T k_t) in float64."""
    L, B, H, T = 1, 2, 3, 7
    w0 = synth.Workload("wo", L=L, B=B, H=H, T=T, bf16=False, V=64, rounds=1, seed=0x7750, accept="uniform")
    state0, ring0, cw = small_case(w0)
    rows_np = synth.all_rows(synth.Workload(f"w{T}", L=L, B=B, H=H, T=T, bf16=False, V=64, rounds=1,
                                            seed=0x7751 + 11 * T, accept="uniform"), 0)
    x = [rows_to_dev(rows_np, False)[n] for n in NAMES]
    st = layer_state(state0, ring0, cw)
    wb = _wbuf(L, B, T, H)
    kb.kda_verify_scan(st, *x, w=wb)
    torch.cuda.synchronize()
    for b in range(B):
        u = {n: rows_np[n][0, b] for n in rows_np}
        q, k, v, g, beta, _ = orc.prepare(u["q"], u["k"], u["v"], u["g"], u["beta"], cw[0], ring0[0, b])
        S = np.asarray(state0[0, b], np.float64)
        for t in range(T):
            for h in range(H):
                Sp = np.exp(g[t, h])[:, None] * S[h]
                w_ref = beta[t, h] * (v[t, h] - Sp.T @ k[t, h])
                assert_close(host(wb[0, b, t, h]), w_ref, f"w of session {b}, row {t}, head {h}",
                             rtol=1e-3, atol=1e-4)
            S, _ = orc.core(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S)
