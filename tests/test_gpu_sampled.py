"""GPU: sampled acceptance (glm_spec.rs, SAMPLED ACCEPTANCE / glm5_sampled_accept)
through the C ABI against the oracle, and the speculative-sampling identity on the
device.

The walk's decisions compare floats (u * q~ < p~, running weight > u * W) that the
device computes in f32 and the oracle in double.  Each session must match the oracle
exactly, except where the oracle itself reaches the device's answer when the session's
uniforms move by 1e-5 (a decision that close to its boundary has no unique answer at f32
precision); such near-ties are counted and bounded.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest
import torch

from gpu_util import to_dev
from libs import ensure_built
from oracle_pins import _chi2_ok

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu

FILTERS = [
    dict(temperature=1.0, top_k=0, top_p=1.0, min_p=0.0),
    dict(temperature=0.7, top_k=50, top_p=0.9, min_p=0.0),
    dict(temperature=1.3, top_k=200, top_p=0.95, min_p=0.02),
    dict(temperature=1.0, top_k=0, top_p=1.0, min_p=0.1),
    dict(temperature=0.5, top_k=1, top_p=1.0, min_p=0.0),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def _case(rng, B, T, V, orc, filt, bf16):
    """Target rows, draft rows near them (some sessions) or not, drafts drawn from q~."""
    K = T - 1
    P = rng.normal(0, 2.0, (B, T, V)).astype(np.float32)
    noise = np.where(rng.uniform(size=(B, 1, 1)) < 0.6, 0.3, 3.0).astype(np.float32)
    Q = (P[:, :K] + rng.normal(0, 1, (B, K, V)).astype(np.float32) * noise).astype(np.float32)
    if bf16:
        P, Q = synth.to_bf16_bits(P), synth.to_bf16_bits(Q)
    d = np.zeros((B, K), np.int32)
    for b in range(B):
        for r in range(K):
            qt = orc.filtered(Q[b, r], **filt)
            d[b, r] = rng.choice(V, p=qt / qt.sum())
    ua = rng.uniform(0, 1, (B, K)).astype(np.float32)
    us = rng.uniform(0, 1, B).astype(np.float32)
    return P, Q, d, ua, us


def _near_tie(orc, P, Q, d, ua, us, filt, want):
    """Whether the oracle reaches `want` with some uniform of the session moved by 1e-5."""
    for r in range(len(ua)):
        for s in (-1e-5, 1e-5):
            u2 = ua.astype(np.float64).copy()
            u2[r] = min(max(u2[r] + s, 0.0), 1.0 - 1e-12)
            if orc.sampled_accept(P, Q, d, u2, float(us), **filt) == want:
                return True
    for s in (-1e-5, 1e-5):
        if orc.sampled_accept(P, Q, d, ua, min(max(float(us) + s, 0.0), 1.0 - 1e-12), **filt) == want:
            return True
    return False


@pytest.mark.parametrize("fi", range(len(FILTERS)))
@pytest.mark.parametrize("V,bf16", [(300, False), (32768, True)])
def test_sampled_accept_against_oracle(orc, fi, V, bf16):
    filt = FILTERS[fi]
    rng = np.random.default_rng(1000 + 10 * fi + V % 7)
    B, T = (48 if V > 1000 else 96), 8
    P, Q, d, ua, us = _case(rng, B, T, V, orc, filt, bf16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    j, tok, keep = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                          dev_status=status, **filt)
    j2, tok2, _ = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                         **filt)
    torch.cuda.synchronize()
    assert torch.equal(j, j2) and torch.equal(tok, tok2), "results must be reproducible"
    assert int(status[0]) == 0
    jg, tg, kg = (x.cpu().numpy() for x in (j, tok, keep))
    near, seen_j = 0, set()
    for b in range(B):
        want = orc.sampled_accept(P[b], Q[b], d[b], ua[b], float(us[b]), **filt)
        got = (int(jg[b]), int(tg[b]))
        assert kg[b] == jg[b] + 1
        seen_j.add(want[0])
        if got != want:
            assert _near_tie(orc, P[b], Q[b], d[b], ua[b], us[b], filt, got), (b, got, want)
            near += 1
    assert near <= 2, near
    assert len(seen_j) >= 3, "the case should exercise several accept lengths"


def test_emitted_token_follows_the_target_on_device(orc):
    """The first emitted token (the accepted draft, else the residual draw) is distributed as
    the filtered target p~_0, whatever q~_0: one session per sample, chi-square."""
    rng = np.random.default_rng(77)
    V, n = 6, 20000
    for filt in (dict(temperature=1.0, top_k=0, top_p=1.0, min_p=0.0), dict(temperature=0.8, top_k=4, top_p=0.85, min_p=0.0)):
        p_row = rng.normal(0, 1.5, V).astype(np.float32)
        q_row = rng.normal(0, 1.5, V).astype(np.float32)
        pt, qt = orc.filtered(p_row, **filt), orc.filtered(q_row, **filt)
        P = np.broadcast_to(np.stack([p_row, p_row]), (n, 2, V)).copy()
        Q = np.broadcast_to(q_row, (n, 1, V)).copy()
        x0 = rng.choice(V, n, p=qt).astype(np.int32).reshape(n, 1)
        ua = rng.uniform(0, 1, (n, 1)).astype(np.float32)
        us = rng.uniform(0, 1, n).astype(np.float32)
        j, tok, _ = kb.spec_accept_sampled(to_dev(P), to_dev(Q), to_dev(x0), to_dev(ua), to_dev(us), **filt)
        torch.cuda.synchronize()
        emitted = np.where(j.cpu().numpy() == 1, x0[:, 0], tok.cpu().numpy())
        assert _chi2_ok(np.bincount(emitted, minlength=V), pt, n)


def test_top_k_one_is_greedy_accept():
    rng = np.random.default_rng(5)
    B, T, V = 64, 6, 1000
    P = rng.normal(0, 1, (B, T, V)).astype(np.float32)
    Q = rng.normal(0, 1, (B, T - 1, V)).astype(np.float32)
    d = np.where(rng.uniform(size=(B, T - 1)) < 0.8, np.argmax(P[:, :T - 1], -1), np.argmax(Q, -1)).astype(np.int32)
    ua = rng.uniform(0, 1, (B, T - 1)).astype(np.float32)
    us = rng.uniform(0, 1, B).astype(np.float32)
    js, ts, _ = kb.spec_accept_sampled(to_dev(P), to_dev(Q), to_dev(d), to_dev(ua), to_dev(us), top_k=1)
    jg, bg, _ = kb.spec_accept(to_dev(P), to_dev(d))
    torch.cuda.synchronize()
    assert torch.equal(js, jg) and torch.equal(ts, bg)


def test_nan_row_is_refused():
    B, T, V = 3, 3, 64
    P = np.zeros((B, T, V), np.float32)
    P[:, :, 7] = 5.0
    P[1, 0, 3] = np.nan
    Q = P[:, :T - 1].copy()
    Q[1, 0, 3] = 0.0
    d = np.full((B, T - 1), 7, np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    j, tok, keep = kb.spec_accept_sampled(to_dev(P), to_dev(Q), to_dev(d), to_dev(np.zeros((B, T - 1), np.float32)),
                                          to_dev(np.full(B, 0.5, np.float32)), dev_status=status)
    torch.cuda.synchronize()
    assert int(status[0]) & kb.ST_NAN
    assert int(tok[1]) == -1 and int(j[1]) == 0
    assert (int(j[0]), int(tok[0])) == (2, 7) and (int(j[2]), int(tok[2])) == (2, 7)


def test_single_row_round_is_a_bonus_draw(orc):
    """T = 1 (no drafts): the token is a draw from p~_0 with u_sample."""
    rng = np.random.default_rng(9)
    B, V = 200, 50
    P = rng.normal(0, 1, (B, 1, V)).astype(np.float32)
    us = rng.uniform(0, 1, B).astype(np.float32)
    j, tok, _ = kb.spec_accept_sampled(to_dev(P), torch.zeros((B, 0, V), device="cuda"),
                                       torch.zeros((B, 0), dtype=torch.int32, device="cuda"),
                                       torch.zeros((B, 0), device="cuda"), to_dev(us), top_k=20, top_p=0.9)
    torch.cuda.synchronize()
    bad = 0
    for b in range(B):
        want = orc.sampled_accept(P[b], np.zeros((0, V), np.float32), [], [], float(us[b]), top_k=20, top_p=0.9)
        if (int(j[b]), int(tok[b])) != want:
            assert _near_tie(orc, P[b], np.zeros((0, V), np.float32), [], np.zeros(0), us[b],
                             dict(top_k=20, top_p=0.9), (int(j[b]), int(tok[b])))
            bad += 1
    assert bad <= 2
