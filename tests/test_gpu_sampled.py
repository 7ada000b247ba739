"""GPU: sampled acceptance (glm_spec.rs, SAMPLED ACCEPTANCE / glm5_sampled_accept /
glm5_sampled_bonus) through the C ABI against the oracle, the session form on its
Philox counters, the device Philox4x32-10 against its published known answers and
against cuRAND's device generator, and the speculative-sampling identity on the device.

The device and the oracle take every decision at the same precision: the filter's
thresholds on the f32 values of e, the accept test u * q~ < p~ in double on the f32
values of p~ and q~ (as the page does), the top-p running sum and the final draw in
double.  The sampling parameters are f32 in the C ABI, so the oracle gets the same
f32 values.  Every session must match the oracle exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from gpu_util import to_dev
from libs import ensure_built
from oracle_pins import _chi2_ok, _philox_kat

from speculative_decode_verify_kda_gb300 import binding as kb
from speculative_decode_verify_kda_gb300 import synth

pytestmark = pytest.mark.gpu

FILTERS = [
    dict(temperature=1.0, top_k=0, top_p=1.0, min_p=0.0),
    dict(temperature=0.7, top_k=50, top_p=0.9, min_p=0.0),
    dict(temperature=1.3, top_k=200, top_p=0.95, min_p=0.02),
    dict(temperature=1.0, top_k=0, top_p=1.0, min_p=0.1),
    dict(temperature=0.5, top_k=1, top_p=1.0, min_p=0.0),
    dict(temperature=0.8, top_k=0, top_p=0.9, min_p=0.0),      # nucleus sampling alone
    dict(temperature=1.1, top_k=2000, top_p=0.8, min_p=0.0),   # top_k beyond the old 512 limit
]


def f32(filt):
    """The filter as the C ABI sees it: f32 temperature, top_p and min_p."""
    return {k: (float(np.float32(v)) if isinstance(v, float) else v) for k, v in filt.items()}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()
    kb.lib()


def _case(rng, B, T, V, orc, filt, bf16, ties=False):
    """Target rows, draft rows near them (some sessions) or not, drafts drawn from q~.
    ties: logits on a coarse grid, so thousands of tokens share a value."""
    K = T - 1
    P = rng.normal(0, 2.0, (B, T, V)).astype(np.float32)
    noise = np.where(rng.uniform(size=(B, 1, 1)) < 0.6, 0.3, 3.0).astype(np.float32)
    Q = (P[:, :K] + rng.normal(0, 1, (B, K, V)).astype(np.float32) * noise).astype(np.float32)
    if ties:
        P, Q = np.round(P), np.round(Q)
    if bf16:
        P, Q = synth.to_bf16_bits(P), synth.to_bf16_bits(Q)
    d = np.zeros((B, K), np.int32)
    for b in range(B):
        for r in range(K):
            qt = orc.filtered(Q[b, r], **f32(filt))
            d[b, r] = rng.choice(V, p=qt / qt.sum())
    ua = rng.uniform(0, 1, (B, K)).astype(np.float32)
    us = rng.uniform(0, 1, B).astype(np.float32)
    return P, Q, d, ua, us


@pytest.mark.parametrize("fi", range(len(FILTERS)))
@pytest.mark.parametrize("V,bf16,ties", [(300, False, False), (32768, True, False), (32768, True, True)])
def test_sampled_accept_against_oracle(orc, fi, V, bf16, ties):
    filt = FILTERS[fi]
    rng = np.random.default_rng(1000 + 10 * fi + V % 7 + ties)
    B, T = (32 if V > 1000 else 96), 8
    P, Q, d, ua, us = _case(rng, B, T, V, orc, filt, bf16, ties)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    j, tok, keep = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                          dev_status=status, **filt)
    j2, tok2, _ = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                         **filt)
    torch.cuda.synchronize()
    assert torch.equal(j, j2) and torch.equal(tok, tok2), "results must be reproducible"
    assert int(status[0]) == 0
    jg, tg, kg = (x.cpu().numpy() for x in (j, tok, keep))
    seen_j = set()
    for b in range(B):
        want = orc.sampled_accept(P[b], Q[b], d[b], ua[b], float(us[b]), **f32(filt))
        assert (int(jg[b]), int(tg[b])) == want, (b, (int(jg[b]), int(tg[b])), want)
        assert kg[b] == jg[b] + 1
        seen_j.add(want[0])
    assert len(seen_j) >= 3, "the case should exercise several accept lengths"


@pytest.mark.parametrize("fi", range(len(FILTERS)))
@pytest.mark.parametrize("V,bf16,ties", [(300, False, False), (32768, True, False), (32768, True, True)])
def test_sampled_accept_few_rows_against_oracle(orc, fi, V, bf16, ties):
    """One session of T = 8 (15 rows): each row's statistics come from a cluster of CTAs
    sharing the row (few rows leave the GPU room for them); the result must equal the
    oracle's exactly, as with one CTA a row."""
    filt = FILTERS[fi]
    seen_j = set()
    for case in range(8):
        rng = np.random.default_rng(5000 + 97 * fi + 13 * case + V % 5 + ties)
        P, Q, d, ua, us = _case(rng, 1, 8, V, orc, filt, bf16, ties)
        if case % 2:
            # the draft rows equal the target rows: every draft passes, the bonus comes
            # from the target's last row
            Q = P[:, :7].copy()
            for r in range(7):
                pt = orc.filtered(P[0, r], **f32(filt))
                d[0, r] = rng.choice(V, p=pt / pt.sum())
        j, tok, keep = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                              **filt)
        torch.cuda.synchronize()
        want = orc.sampled_accept(P[0], Q[0], d[0], ua[0], float(us[0]), **f32(filt))
        assert (int(j[0]), int(tok[0])) == want, (case, (int(j[0]), int(tok[0])), want)
        assert int(keep[0]) == int(j[0]) + 1
        seen_j.add(want[0])
    assert len(seen_j) >= 2, "the cases should exercise several accept lengths"


@pytest.mark.parametrize("B", [1, 12])
@pytest.mark.parametrize("fi", [1, 2, 5, 6])
@pytest.mark.parametrize("V,bf16", [(300, False), (32768, True)])
def test_negative_logits_against_oracle(orc, B, fi, V, bf16):
    """Every logit below zero: the top-k and top-p boundaries fall on negative values,
    whose order keys are complemented bit patterns (B = 1: a cluster of CTAs a row;
    B = 12: one CTA a row)."""
    filt = FILTERS[fi]
    rng = np.random.default_rng(7000 + 31 * fi + B + bf16)
    P, Q, d, ua, us = _case(rng, B, 5, V, orc, filt, False)
    P, Q = P - 40.0, Q - 40.0
    if bf16:
        P, Q = synth.to_bf16_bits(P), synth.to_bf16_bits(Q)
    for b in range(B):  # drafts drawn again from the shifted draft rows
        for r in range(4):
            qt = orc.filtered(Q[b, r], **f32(filt))
            d[b, r] = rng.choice(V, p=qt / qt.sum())
    j, tok, _ = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                       **filt)
    torch.cuda.synchronize()
    for b in range(B):
        want = orc.sampled_accept(P[b], Q[b], d[b], ua[b], float(us[b]), **f32(filt))
        assert (int(j[b]), int(tok[b])) == want, (b, (int(j[b]), int(tok[b])), want)


@pytest.mark.parametrize("B", [1, 12])
@pytest.mark.parametrize("fi", [1, 2, 5, 6])
@pytest.mark.parametrize("V,bf16", [(4000, False), (32768, True)])
def test_flat_logits_against_oracle(orc, B, fi, V, bf16):
    """Logits N(0, 1), as in the verify workloads: a flat distribution on which top-k
    binds far below top-p (the device then proves it from a lower bound of S and forms
    no S), and nucleus sampling alone keeps about half the vocabulary."""
    filt = FILTERS[fi]
    rng = np.random.default_rng(8100 + 17 * fi + B + bf16)
    T, K = 6, 5
    P = rng.normal(0, 1.0, (B, T, V)).astype(np.float32)
    Q = (P[:, :K] + rng.normal(0, 0.3, (B, K, V))).astype(np.float32)
    if bf16:
        P, Q = synth.to_bf16_bits(P), synth.to_bf16_bits(Q)
    d = np.zeros((B, K), np.int32)
    for b in range(B):
        for r in range(K):
            qt = orc.filtered(Q[b, r], **f32(filt))
            d[b, r] = rng.choice(V, p=qt / qt.sum())
    ua = rng.uniform(0, 1, (B, K)).astype(np.float32)
    us = rng.uniform(0, 1, B).astype(np.float32)
    j, tok, _ = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                       **filt)
    torch.cuda.synchronize()
    for b in range(B):
        want = orc.sampled_accept(P[b], Q[b], d[b], ua[b], float(us[b]), **f32(filt))
        assert (int(j[b]), int(tok[b])) == want, (b, (int(j[b]), int(tok[b])), want)


@pytest.mark.parametrize("B", [1, 12])
@pytest.mark.parametrize("V,bf16", [(1001, True), (37, False), (4099, False)])
def test_unvectorised_rows_against_oracle(orc, B, V, bf16):
    """Rows that are not whole 16-byte vectors are read one logit at a time, and a
    cluster's CTAs then split the row by logits (B = 1) rather than by vectors."""
    rng = np.random.default_rng(8300 + V + B)
    for fi in (1, 2, 5, 6):
        filt = FILTERS[fi]
        P, Q, d, ua, us = _case(rng, B, 5, V, orc, filt, bf16)
        j, tok, _ = kb.spec_accept_sampled(to_dev(P, bf16), to_dev(Q, bf16), to_dev(d), to_dev(ua), to_dev(us),
                                           **filt)
        torch.cuda.synchronize()
        for b in range(B):
            want = orc.sampled_accept(P[b], Q[b], d[b], ua[b], float(us[b]), **f32(filt))
            assert (int(j[b]), int(tok[b])) == want, (fi, b, (int(j[b]), int(tok[b])), want)


@pytest.mark.parametrize("sd", [1.0, 4.0])
def test_largest_batch_against_oracle(orc, sd):
    """64 sessions of T = 15 at V = 32768 (the largest seeded batch: 1856 rows, several
    waves of one CTA a row), flat (top-k binds, S skipped) and peaked (top-p binds) rows;
    six sessions across the batch against the oracle (its filter takes about 0.15 s a
    row here), every session's result a valid walk length and token."""
    filt = FILTERS[1]
    rng = np.random.default_rng(8400 + int(sd))
    B, T, K, V = 64, 15, 14, 32768
    P = (rng.normal(0, sd, (B, T, V))).astype(np.float32)
    Q = (P[:, :K] + rng.normal(0, 0.3 * sd, (B, K, V))).astype(np.float32)
    P, Q = synth.to_bf16_bits(P), synth.to_bf16_bits(Q)
    d = np.argmax(synth.bf16_bits_to_f32(Q), axis=-1).astype(np.int32)  # the draft rows' modes
    ua = rng.uniform(0, 1, (B, K)).astype(np.float32)
    us = rng.uniform(0, 1, B).astype(np.float32)
    j, tok, _ = kb.spec_accept_sampled(to_dev(P, True), to_dev(Q, True), to_dev(d), to_dev(ua), to_dev(us), **filt)
    torch.cuda.synchronize()
    jg, tg = j.cpu().numpy(), tok.cpu().numpy()
    assert ((jg >= 0) & (jg <= K)).all() and ((tg >= 0) & (tg < V)).all()
    for b in (0, 13, 31, 40, 52, 63):
        want = orc.sampled_accept(P[b], Q[b], d[b], ua[b], float(us[b]), **f32(filt))
        assert (int(jg[b]), int(tg[b])) == want, (b, (int(jg[b]), int(tg[b])), want)


def test_top_p_with_thousands_of_ties(orc):
    """Rows whose top-p boundary falls inside a tie group of more than 1024 tokens: the
    kept set takes the whole group, on the device as in the oracle."""
    V, B = 32768, 8
    rng = np.random.default_rng(55)
    P = np.full((B, 1, V), -4.0, np.float32)
    for b in range(B):
        P[b, 0, rng.choice(V, 1500 + 300 * b, replace=False)] = 0.0  # the tie group at the top
        P[b, 0, rng.choice(V, 20, replace=False)] = 1.0
    us = rng.uniform(0, 1, B).astype(np.float32)
    for filt in (dict(top_p=0.5), dict(top_p=0.05), dict(top_k=1200, top_p=0.9)):
        j, tok, _ = kb.spec_accept_sampled(to_dev(P), torch.zeros((B, 0, V), device="cuda"),
                                           torch.zeros((B, 0), dtype=torch.int32, device="cuda"),
                                           torch.zeros((B, 0), device="cuda"), to_dev(us), **filt)
        torch.cuda.synchronize()
        for b in range(B):
            want = orc.sampled_accept(P[b], np.zeros((0, V), np.float32), [], [], float(us[b]), **f32(filt))
            assert (int(j[b]), int(tok[b])) == want, (filt, b)


@pytest.mark.parametrize("B", [24, 3, 50])
def test_session_rounds_against_oracle(orc, B):
    """spec_accept_sampled_session over several rounds in a row: every round draws its
    uniforms from the session's counters and advances them on the device, exactly as the
    oracle's session walk does (B = 3, 24, 50: each session's walk shared by a cluster of
    8, 4 or 2 CTAs, one of which writes the counters the others have read)."""
    rng = np.random.default_rng(71 + B)
    T, V = 6, 2000
    seeds = rng.integers(0, 2**63, B, dtype=np.int64)
    ctr = np.stack([rng.integers(0, 2**31, B), rng.integers(0, 2**31, B)], 1).astype(np.int64)
    counters = torch.from_numpy(ctr.astype(np.int32)).cuda()
    sd = torch.from_numpy(seeds).cuda()
    oc = [(int(ctr[b, 0]), int(ctr[b, 1])) for b in range(B)]
    for rnd, filt in enumerate([FILTERS[1], FILTERS[5], FILTERS[2], FILTERS[0]]):
        P, Q, d, _, _ = _case(rng, B, T, V, orc, filt, False)
        j, tok, keep = kb.spec_accept_sampled_session(to_dev(P), to_dev(Q), to_dev(d), sd, counters, **filt)
        torch.cuda.synchronize()
        cg = counters.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
        for b in range(B):
            want = orc.sampled_accept_session(P[b], Q[b], d[b], int(seeds[b]) & (2**64 - 1), oc[b][0], oc[b][1],
                                              **f32(filt))
            assert (int(j[b]), int(tok[b])) == want[:2], (rnd, b)
            assert (int(cg[b, 0]), int(cg[b, 1])) == want[2:], (rnd, b)
            oc[b] = want[2:]


def test_philox_known_answers_on_device():
    kat = _philox_kat()
    ctr = torch.tensor(np.array([c for c, _, _ in kat], np.uint32).view(np.int32), device="cuda")
    key = torch.tensor(np.array([k for _, k, _ in kat], np.uint32).view(np.int32), device="cuda")
    out = kb.philox4x32_10(ctr, key).cpu().numpy().view(np.uint32)
    assert [list(map(int, o)) for o in out] == [w for _, _, w in kat]


_CURAND_SRC = r"""
#include <curand_kernel.h>
__global__ void k(const unsigned long long *seeds, uint4 *out, int n, int per)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    curandStatePhilox4_32_10_t st;
    curand_init(seeds[i], 0ull, 0ull, &st);
    for (int r = 0; r < per; ++r)
        out[i * per + r] = curand4(&st);
}
extern "C" int curand_philox(const unsigned long long *seeds, void *out, int n, int per)
{
    k<<<(n + 127) / 128, 128>>>(seeds, static_cast<uint4 *>(out), n, per);
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 1;
}
"""


def test_philox_matches_curand(orc, tmp_path):
    """The library's Philox4x32-10 against cuRAND's device generator of the same name:
    cuRAND's state seeded with s (subsequence 0, offset 0) returns, call after call, the
    generator at counters (0, 0, 0, 0), (1, 0, 0, 0), ... under key (s low, s high)."""
    src = tmp_path / "curand_philox.cu"
    src.write_text(_CURAND_SRC)
    so = tmp_path / "libcurand_philox.so"
    nvcc = os.environ.get("NVCC", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    str(src), "-o", str(so)], check=True)
    lib = ctypes.CDLL(str(so))
    lib.curand_philox.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    rng = np.random.default_rng(7)
    n, per = 64, 5
    seeds = rng.integers(0, 2**63, n, dtype=np.int64)
    seeds[0] = 0
    sd = torch.from_numpy(seeds).cuda()
    ref = torch.empty((n, per, 4), dtype=torch.int32, device="cuda")
    assert lib.curand_philox(sd.data_ptr(), ref.data_ptr(), n, per) == 0
    s64 = seeds.view(np.uint64)
    ctr = np.zeros((n, per, 4), np.uint32)
    ctr[:, :, 0] = np.arange(per, dtype=np.uint32)[None]
    key = np.stack([s64 & 0xFFFFFFFF, s64 >> 32], -1).astype(np.uint32)[:, None, :].repeat(per, 1)
    got = kb.philox4x32_10(torch.from_numpy(ctr.reshape(-1, 4).view(np.int32)).cuda(),
                           torch.from_numpy(np.ascontiguousarray(key.reshape(-1, 2)).view(np.int32)).cuda())
    torch.cuda.synchronize()
    assert torch.equal(got.view(n, per, 4), ref)
    # and the oracle's generator on a sample of the same counters
    g = got.cpu().numpy().view(np.uint32).reshape(n, per, 4)
    for i in range(0, n, 9):
        for r in range(per):
            assert list(map(int, orc.philox(ctr[i, r], key[i, r]))) == list(map(int, g[i, r]))


def test_emitted_token_follows_the_target_on_device(orc):
    """The first emitted token (the accepted draft, else the residual draw) is distributed as
    the filtered target p~_0, whatever q~_0: one session per sample, chi-square.  The
    uniforms come from the sessions' own Philox streams."""
    rng = np.random.default_rng(77)
    V, n = 6, 20000
    for filt in (dict(temperature=1.0, top_k=0, top_p=1.0, min_p=0.0),
                 dict(temperature=0.8, top_k=4, top_p=0.85, min_p=0.0),
                 dict(temperature=0.9, top_k=0, top_p=0.7, min_p=0.0)):
        p_row = rng.normal(0, 1.5, V).astype(np.float32)
        q_row = rng.normal(0, 1.5, V).astype(np.float32)
        pt, qt = orc.filtered(p_row, **f32(filt)), orc.filtered(q_row, **f32(filt))
        P = np.broadcast_to(np.stack([p_row, p_row]), (n, 2, V)).copy()
        Q = np.broadcast_to(q_row, (n, 1, V)).copy()
        x0 = rng.choice(V, n, p=qt).astype(np.int32).reshape(n, 1)
        seeds = torch.from_numpy(rng.integers(0, 2**63, n, dtype=np.int64)).cuda()
        counters = torch.zeros((n, 2), dtype=torch.int32, device="cuda")
        j, tok, _ = kb.spec_accept_sampled_session(to_dev(P), to_dev(Q), to_dev(x0), seeds, counters, **filt)
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
    filt = dict(top_k=20, top_p=0.9)
    j, tok, _ = kb.spec_accept_sampled(to_dev(P), torch.zeros((B, 0, V), device="cuda"),
                                       torch.zeros((B, 0), dtype=torch.int32, device="cuda"),
                                       torch.zeros((B, 0), device="cuda"), to_dev(us), **filt)
    torch.cuda.synchronize()
    for b in range(B):
        want = orc.sampled_accept(P[b], np.zeros((0, V), np.float32), [], [], float(us[b]), **f32(filt))
        assert (int(j[b]), int(tok[b])) == want, b
