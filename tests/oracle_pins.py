"""Pins of the CPU oracle against things other than itself.

Each ``pin_*`` takes a loaded oracle and raises AssertionError when it is wrong.
The checks are closed forms, invariants, special cases that reduce to library
routines, brute force on tiny inputs in an independent formulation (the matrix
form of the recurrence, ``np.correlate`` for the conv, sorting for the argmax),
and the values printed on the pages (``tests/golden``).  The mutation test runs
every pin against deliberately broken copies of the oracle and requires each
copy to fail at least one of them.
"""
from __future__ import annotations

import math
import os

import numpy as np
from scipy.special import expit

D = 128
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# independent helpers (numpy / scipy, no oracle code)
# ---------------------------------------------------------------------------
def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _post_inputs(rng, T, H, g_lo=-5.0):
    q = _unit(rng.standard_normal((T, H, D)))
    k = _unit(rng.standard_normal((T, H, D)))
    v = rng.standard_normal((T, H, D))
    g = rng.uniform(g_lo, 0.0, (T, H, D))
    beta = rng.uniform(0.05, 0.95, (T, H))
    S = 0.01 * rng.standard_normal((H, D, D))
    return q, k, v, g, beta, S


def matrix_form(q, k, v, g, beta, S0):
    """S_t = (I - beta k k^T) diag(exp g) S_{t-1} + beta k v^T ; o_t = S_t^T q / sqrt(128)."""
    T, H = q.shape[0], q.shape[1]
    S = S0.copy()
    out = np.empty((T, H, D))
    eye = np.eye(D)
    for t in range(T):
        for h in range(H):
            kk = k[t, h][:, None]
            A = (eye - beta[t, h] * kk @ kk.T) @ np.diag(np.exp(g[t, h]))
            S[h] = A @ S[h] + beta[t, h] * kk @ v[t, h][None, :]
            out[t, h] = S[h].T @ q[t, h] / math.sqrt(D)
    return S, out


def silu(x):
    return x * expit(x)


def _raw_inputs(rng, T, H):
    xq, xk, xv, xg = (rng.standard_normal((T, H, D)).astype(np.float32) for _ in range(4))
    xb = rng.standard_normal((T, H)).astype(np.float32)
    conv_w = rng.uniform(-0.5, 0.5, (H, 3, D, 4)).astype(np.float32)
    ring = (0.1 * rng.standard_normal((H, 3, 3, D))).astype(np.float32)
    state = (0.01 * rng.standard_normal((H, D, D))).astype(np.float32)
    return xq, xk, xv, xg, xb, conv_w, ring, state


def brute_verify(xq, xk, xv, xg, xb, conv_w, ring, state):
    """The whole verify of one unit from library routines, in float64."""
    T, H = xq.shape[0], xq.shape[1]
    raw = [xq.astype(np.float64), xk.astype(np.float64), xv.astype(np.float64)]
    y = np.empty((3, T, H, D))
    for s in range(3):
        for h in range(H):
            for c in range(D):
                seq = np.concatenate([ring[h, s, :, c].astype(np.float64), raw[s][:, h, c]])
                # correlate(seq, w, 'valid')[t] = sum_m seq[t+m] w[m]: tap 3 meets row t
                y[s, :, h, c] = silu(np.correlate(seq, conv_w[h, s, c].astype(np.float64), "valid"))
    q = y[0] / np.sqrt((y[0] ** 2).sum(-1, keepdims=True) + 1e-6)
    k = y[1] / np.sqrt((y[1] ** 2).sum(-1, keepdims=True) + 1e-6)
    g = -5.0 * expit(xg.astype(np.float64))
    beta = expit(xb.astype(np.float64))
    S, out = matrix_form(q, k, y[2], g, beta, state.astype(np.float64))
    ring_out = np.empty_like(ring)
    for s in range(3):
        seq = np.concatenate([ring[:, s].transpose(1, 0, 2), raw[s].astype(np.float32)], axis=0)
        ring_out[:, s] = seq[-3:].transpose(1, 0, 2)
    return S, out, ring_out


def _close(a, b, rtol, atol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    err = np.abs(a - b) - (atol + rtol * np.abs(b))
    assert np.all(err <= 0), f"{what}: max excess {err.max():.3e}"


# ---------------------------------------------------------------------------
# the recurrence (core entry)
# ---------------------------------------------------------------------------
def pin_core_matrix_form(orc):
    """Brute force in the matrix form, tiny inputs, several heads and rows."""
    rng = _rng(11)
    for T, H in ((1, 1), (5, 2), (8, 1)):
        q, k, v, g, beta, S0 = _post_inputs(rng, T, H)
        S, out = orc.core(q, k, v, g, beta, S0)
        Sb, outb = matrix_form(q, k, v, g, beta, S0)
        _close(S, Sb, 1e-12, 1e-14, "state vs matrix form")
        _close(out, outb, 1e-11, 1e-14, "out vs matrix form")


def pin_core_closed_form_first_write(orc):
    """From S = 0 one row gives S = beta k v^T and o = beta (q.k) v / sqrt(128)."""
    rng = _rng(12)
    q, k, v, g, beta, _ = _post_inputs(rng, 1, 3)
    S, out = orc.core(q, k, v, g, beta, np.zeros((3, D, D)))
    for h in range(3):
        _close(S[h], beta[0, h] * np.outer(k[0, h], v[0, h]), 1e-13, 1e-15, "S closed form")
        o = beta[0, h] * float(q[0, h] @ k[0, h]) * v[0, h] / math.sqrt(D)
        _close(out[0, h], o, 1e-12, 1e-15, "o closed form")


def pin_core_identity(orc):
    """beta = 0 and g = 0 leave S unchanged, bit for bit."""
    rng = _rng(13)
    q, k, v, _, _, S0 = _post_inputs(rng, 6, 2)
    S, _ = orc.core(q, k, v, np.zeros_like(q), np.zeros((6, 2)), S0)
    assert np.array_equal(S, S0), "beta=0, g=0 must leave the state unchanged"


def pin_core_orthonormal_writes(orc):
    """g = 0, beta = 1 and orthonormal keys: afterwards S^T k_t = v_t for every row t."""
    rng = _rng(14)
    T = 7
    basis, _ = np.linalg.qr(rng.standard_normal((D, D)))
    k = basis[:, :T].T.reshape(T, 1, D)
    q = _unit(rng.standard_normal((T, 1, D)))
    v = rng.standard_normal((T, 1, D))
    S0 = 0.01 * rng.standard_normal((1, D, D))
    S, _ = orc.core(q, k, v, np.zeros((T, 1, D)), np.ones((T, 1)), S0)
    for t in range(T):
        _close(S[0].T @ k[t, 0], v[t, 0], 1e-12, 1e-12, f"read back row {t}")
    # the part of S orthogonal to every written key is untouched
    P = np.eye(D) - k[:, 0].T @ k[:, 0]
    _close(P @ S[0], P @ S0[0], 1e-12, 1e-14, "orthogonal complement")


def pin_core_decay_only(orc):
    """beta = 0: S_T = diag(exp(sum_t g_t)) S_0 and o_t = S_t^T q_t / sqrt(128)."""
    rng = _rng(15)
    q, k, v, g, _, S0 = _post_inputs(rng, 5, 2)
    S, out = orc.core(q, k, v, g, np.zeros((5, 2)), S0)
    for h in range(2):
        _close(S[h], np.exp(g[:, h].sum(0))[:, None] * S0[h], 1e-13, 1e-16, "pure decay")
        St = S0[h].copy()
        for t in range(5):
            St = np.exp(g[t, h])[:, None] * St
            _close(out[t, h], St.T @ q[t, h] / math.sqrt(D), 1e-12, 1e-16, "decay-only output")


# ---------------------------------------------------------------------------
# activations (prepare entry)
# ---------------------------------------------------------------------------
def _taps(H, tap):
    w = np.zeros((H, 3, D, 4), np.float32)
    w[..., tap] = 1.0
    return w


def pin_prepare_current_tap(orc):
    """Weights [0,0,0,1]: the conv is the identity, so v = SiLU(x) and q, k are SiLU(x)/norm."""
    rng = _rng(21)
    xq, xk, xv, xg, xb, _, ring, _ = _raw_inputs(rng, 4, 2)
    q, k, v, g, b, _ = orc.prepare(xq, xk, xv, xg, xb, _taps(2, 3), ring)
    _close(v, silu(xv.astype(np.float64)), 1e-15, 1e-300, "v = SiLU(x)")
    for got, x in ((q, xq), (k, xk)):
        y = silu(x.astype(np.float64))
        n = (y ** 2).sum(-1, keepdims=True)
        _close((got ** 2).sum(-1, keepdims=True), n / (n + 1e-6), 1e-14, 0, "|x_hat|^2 = n/(n+eps)")
        _close(got * np.linalg.norm(y, axis=-1, keepdims=True), y * np.sqrt(n / (n + 1e-6)),
               1e-13, 1e-15, "x_hat parallel to SiLU(x)")


def pin_prepare_shifted_taps(orc):
    """Weights with one tap m pick x[t-3+m]: the ring supplies the rows before row 0, oldest first."""
    rng = _rng(22)
    T, H = 5, 2
    xq, xk, xv, xg, xb, _, ring, _ = _raw_inputs(rng, T, H)
    for m in range(3):
        _, _, v, _, _, _ = orc.prepare(xq, xk, xv, xg, xb, _taps(H, m), ring)
        seq = np.concatenate([ring[:, 2].transpose(1, 0, 2), xv], axis=0)  # [3+T][H][D]
        _close(v, silu(seq[m:m + T].astype(np.float64)), 1e-15, 1e-300, f"tap {m}")


def pin_prepare_vs_correlate(orc):
    """Random weights: the conv equals np.correlate over [ring, rows]."""
    rng = _rng(23)
    T, H = 6, 2
    xq, xk, xv, xg, xb, conv_w, ring, _ = _raw_inputs(rng, T, H)
    _, _, v, _, _, _ = orc.prepare(xq, xk, xv, xg, xb, conv_w, ring)
    for h in range(H):
        for c in (0, 17, 127):
            seq = np.concatenate([ring[h, 2, :, c], xv[:, h, c]]).astype(np.float64)
            a = np.correlate(seq, conv_w[h, 2, c].astype(np.float64), "valid")
            _close(v[:, h, c], silu(a), 1e-14, 1e-16, "conv vs correlate")


def pin_prepare_gates(orc):
    """g = -5 sigmoid(raw): raw 0 -> -2.5, raw -inf -> 0 (no decay), raw +inf -> -5; beta likewise."""
    T, H = 3, 2
    z = np.zeros((T, H, D), np.float32)
    xg = np.zeros((T, H, D), np.float32)
    xg[1] = -np.inf
    xg[2] = np.inf
    xb = np.array([[0.0, -np.inf], [np.inf, 0.0], [2.0, -2.0]], np.float32)
    _, _, _, g, b, _ = orc.prepare(z, z, z, xg, xb, _taps(H, 3), np.zeros((H, 3, 3, D), np.float32))
    assert np.all(g[0] == -2.5) and np.all(g[1] == 0.0) and np.all(g[2] == -5.0), "gate specials"
    _close(b, [[0.5, 0.0], [1.0, 0.5], [expit(2.0), expit(-2.0)]], 1e-15, 0, "beta = sigmoid")
    rng = _rng(24)
    xg = rng.standard_normal((T, H, D)).astype(np.float32)
    _, _, _, g, _, _ = orc.prepare(z, z, z, xg, xb, _taps(H, 3), np.zeros((H, 3, 3, D), np.float32))
    _close(g, -5.0 * expit(xg.astype(np.float64)), 1e-15, 0, "g = -5 expit")


def pin_prepare_ring_reroll(orc):
    """ring_out = the last 3 raw inputs of [ring, x_0..x_{T-1}] per stream, for T = 1, 2, 3, 7."""
    rng = _rng(25)
    H = 2
    for T in (1, 2, 3, 7):
        xq, xk, xv, xg, xb, conv_w, ring, _ = _raw_inputs(rng, T, H)
        *_, ring_out = orc.prepare(xq, xk, xv, xg, xb, conv_w, ring)
        for s, x in enumerate((xq, xk, xv)):
            seq = np.concatenate([ring[:, s].transpose(1, 0, 2), x], axis=0)
            assert np.array_equal(ring_out[:, s], seq[-3:].transpose(1, 0, 2)), f"ring T={T} s={s}"


def _golden_bf16():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_widen.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                bits, val = line.split()
                rows.append((int(bits, 16), float(val)))
    return rows


def pin_bf16_widening(orc):
    """bf16 rows widen exactly (tests/golden/bf16_widen.txt); checked through v = SiLU(x)."""
    rows = _golden_bf16()
    bits = np.array([b for b, _ in rows], np.uint16)
    vals = np.array([v for _, v in rows], np.float64)
    H = 1
    xv = np.zeros((1, H, D), np.uint16)
    xv[0, 0, : len(bits)] = bits
    z = np.zeros((1, H, D), np.uint16)
    _, _, v, _, _, _ = orc.prepare(z, z, xv, z, np.zeros((1, H), np.uint16), _taps(H, 3),
                                   np.zeros((H, 3, 3, D), np.float32))
    got = v[0, 0, : len(bits)]
    fin = np.isfinite(vals)
    assert np.array_equal(got[fin], silu(vals[fin])), "bf16 widening"
    assert np.isinf(got[~fin]).all()
    # (the sign of a zero does not survive the conv sum 0 + (-0) = +0, so -0.0 is
    # checked by value only here; the accept pins compare -0.0 with +0.0 directly)


# ---------------------------------------------------------------------------
# the whole verify, rollback
# ---------------------------------------------------------------------------
def pin_verify_brute_force(orc):
    """The full unit verify equals the library-routine brute force (conv, SiLU, norm, gates, matrix form)."""
    rng = _rng(31)
    for T, H in ((1, 1), (4, 2), (8, 1)):
        args = _raw_inputs(rng, T, H)
        st, ring_out, out = orc.verify(*args)
        Sb, outb, ringb = brute_verify(*args)
        _close(st, Sb, 2e-7, 1e-9, "verify state")
        _close(out, outb, 2e-6, 1e-9, "verify out")
        assert np.array_equal(ring_out, ringb), "verify ring"


def pin_verify_chained_rows(orc):
    """Running rows one launch at a time (f32 state between) stays within f32 rounding of one launch."""
    rng = _rng(32)
    T, H = 6, 2
    xq, xk, xv, xg, xb, conv_w, ring, state = _raw_inputs(rng, T, H)
    st_all, ring_all, out_all = orc.verify(xq, xk, xv, xg, xb, conv_w, ring, state)
    st, rg = state, ring
    for t in range(T):
        sl = slice(t, t + 1)
        st, rg, out = orc.verify(xq[sl], xk[sl], xv[sl], xg[sl], xb[sl], conv_w, rg, st)
        _close(out[0], out_all[t], 1e-5, 1e-8, f"row {t} output")
    _close(st, st_all, 1e-5, 1e-8, "chained state")
    assert np.array_equal(rg, ring_all), "chained ring"


def pin_rollback(orc):
    """keep == T keeps the resident state; keep < T equals a fresh run of rows 0..keep-1; bad keep refused."""
    import oracle
    rng = _rng(33)
    T, H = 5, 2
    xq, xk, xv, xg, xb, conv_w, ring, state = _raw_inputs(rng, T, H)
    st_T, ring_T, _ = orc.verify(xq, xk, xv, xg, xb, conv_w, ring, state)
    for keep in range(1, T + 1):
        st, rg = orc.rollback(keep, xq, xk, xv, xg, xb, conv_w, ring, state, ring_T, st_T)
        if keep == T:
            assert np.array_equal(st, st_T) and np.array_equal(rg, ring_T), "keep == T"
        else:
            sl = slice(0, keep)
            st_k, ring_k, _ = orc.verify(xq[sl], xk[sl], xv[sl], xg[sl], xb[sl], conv_w, ring, state)
            assert np.array_equal(st, st_k) and np.array_equal(rg, ring_k), f"keep={keep}"
            # and the rollback really moved the state off the post-row-T value
            assert not np.array_equal(st, st_T)
    for bad in (0, T + 1):
        try:
            orc.rollback(bad, xq, xk, xv, xg, xb, conv_w, ring, state, ring_T, st_T)
        except oracle.OracleError as e:
            assert e.rc == oracle.EINVAL
        else:
            raise AssertionError(f"keep={bad} accepted")


# ---------------------------------------------------------------------------
# greedy accept
# ---------------------------------------------------------------------------
def _planted_logits(vam, V, rng):
    x = rng.uniform(-3.0, 3.0, (len(vam), V)).astype(np.float32)
    for r, a in enumerate(vam):
        x[r, a] = 10.0
    return x


def _golden_harvest():
    out = []
    with open(os.path.join(GOLDEN, "accept_harvest_fixture.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                name, T, vam, drafts, j, bonus = line.split()
                out.append((name, int(T), [int(x) for x in vam.split(",")],
                            [int(x) for x in drafts.split(",")], int(j), int(bonus)))
    return out


def pin_accept_page_fixture(orc):
    """The harvest-alignment fixture printed on the pages: aligned -> full block, misaligned -> 0."""
    rng = _rng(41)
    for name, T, vam, drafts, j_exp, bonus_exp in _golden_harvest():
        x = _planted_logits(vam, 1024, rng)
        j, bonus, got_vam, rc = orc.accept(x, drafts)
        assert rc == 0 and list(got_vam) == vam, name
        assert (j, bonus) == (j_exp, bonus_exp), f"{name}: {(j, bonus)} != {(j_exp, bonus_exp)}"


def _first_argmax_by_sort(row):
    order = sorted(range(len(row)), key=lambda c: (-row[c], c))
    return order[0]


def _accept_brute(logits, drafts):
    vam = [_first_argmax_by_sort(list(r)) for r in logits]
    K = len(drafts)
    j = max(m for m in range(K + 1) if all(drafts[r] == vam[r] for r in range(m)))
    return j, vam[j], vam


def pin_accept_brute_force(orc):
    """Tiny vocabularies with many ties, every draft combination: j, bonus, vam as brute force gives."""
    rng = _rng(42)
    V = 3
    for trial in range(30):
        T = 1 + trial % 4
        x = rng.integers(0, 3, (T, V)).astype(np.float32)  # values in {0,1,2}: ties everywhere
        for code in range(V ** (T - 1)):
            drafts = [(code // V ** r) % V for r in range(T - 1)]
            j, bonus, vam, rc = orc.accept(x, np.array(drafts, np.int32))
            jb, bb, vb = _accept_brute(x, drafts)
            assert rc == 0 and (j, bonus) == (jb, bb) and list(vam) == vb, (x, drafts)


def pin_accept_nan(orc):
    """A NaN in a consulted row is refused (sentinel bonus); a NaN in a row past j is not consulted."""
    import oracle
    rng = _rng(43)
    vam = [5, 6, 7, 8]
    x = _planted_logits(vam, 16, rng)
    x_bad = x.copy()
    x_bad[2, 3] = np.nan
    # drafts match rows 0 and 1, so the walk reaches the NaN row 2
    j, bonus, got, rc = orc.accept(x_bad, np.array([5, 6, 7], np.int32))
    assert rc == oracle.ENAN and j == 2 and bonus == oracle.SENTINEL and got[2] == oracle.SENTINEL
    # drafts mismatch at row 0: row 2 is never consulted
    j, bonus, got, rc = orc.accept(x_bad, np.array([4, 6, 7], np.int32))
    assert rc == 0 and (j, bonus) == (0, 5)


def pin_accept_ties(orc):
    """Equal maxima: the lowest index wins, for f32 and bf16 rows and for -0.0 against +0.0."""
    x = np.array([[1.0, 3.0, 3.0, 2.0], [-0.0, 0.0, -1.0, -0.0], [-np.inf, -np.inf, -np.inf, -np.inf]],
                 np.float32)
    _, _, vam, rc = orc.accept(x, np.array([9, 9], np.int32))
    assert rc == 0 and list(vam) == [1, 0, 0], vam
    bits = (np.ascontiguousarray(x).view(np.uint32) >> 16).astype(np.uint16)
    _, _, vam, rc = orc.accept(bits, np.array([9, 9], np.int32))
    assert rc == 0 and list(vam) == [1, 0, 0], vam
    # a bf16 row whose values differ only below bf16 precision in f32 would tie; bf16 decides
    y = np.array([[0x3F80, 0x3F81, 0x3F81, 0x3F80]], np.uint16)
    _, bonus, vam, _ = orc.accept(y, np.zeros(0, np.int32))
    assert vam[0] == 1 and bonus == 1


def _golden_windows():
    rows = []
    with open(os.path.join(GOLDEN, "window_policy_fixture.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            kind, vals, param, flag, exp = line.split()
            v = [] if vals == "-" else [float(x) for x in vals.split(",")]
            rows.append((kind, np.array(v, np.float32), np.float32(param), int(flag), int(exp)))
    return rows


def _logit_f32(p):
    """ln(p / (1 - p)) in f32, the way the page's tests build raw scores."""
    p = np.asarray(p, np.float32)
    return np.log((p / (np.float32(1.0) - p)).astype(np.float32)).astype(np.float32)


def pin_window_page_fixture(orc):
    """glm5_conf_keep, dspark_confidence_vt and dspark_slot_confidence_vt on the cases
    printed in the pages' unit tests (tests/golden/window_policy_fixture.txt)."""
    for kind, vals, param, flag, exp in _golden_windows():
        if kind == "conf_keep":
            got = orc.conf_keep(vals, param, flag)
        elif kind == "confidence":
            got = orc.confidence_vt(_logit_f32(vals), param, flag)
        else:
            got = orc.slot_confidence_vt(_logit_f32(vals), param, flag)
        assert got == exp, (kind, list(vals), float(param), flag, got, exp)


def pin_window_brute_force(orc):
    """Each window is the longest prefix whose every slot passes its own test, written as
    a search over prefix lengths; survival never keeps more than the per-slot arm."""
    rng = np.random.default_rng(2024)
    for _ in range(400):
        n = int(rng.integers(0, 9))
        q = rng.uniform(0, 1, n).astype(np.float32)
        p_min = np.float32(rng.choice([0.0, 0.3, 0.5, 0.8]))
        pmin0 = int(rng.integers(0, 2))
        ok = [bool(q[j] >= p_min or (j == 0 and not pmin0)) for j in range(n)]
        want = max(m for m in range(n + 1) if all(ok[:m]))
        assert orc.conf_keep(q, p_min, pmin0) == want
        raws = rng.normal(0, 3, n).astype(np.float32)
        sig = (np.float32(1) / (np.float32(1) + np.exp(-raws).astype(np.float32))).astype(np.float32)
        tau = np.float32(rng.choice([0.05, 0.3, 0.5, 0.9]))
        cap = int(rng.integers(1, 16))
        surv = np.cumprod(sig, dtype=np.float32) if n else np.zeros(0, np.float32)
        clamp = lambda m: min(max(1 + m, 2), max(cap, 2))
        keep_s = max(m for m in range(n + 1) if all(surv[:m] >= tau))
        keep_p = max(m for m in range(n + 1) if all(sig[:m] >= tau))
        vt, vt_slot = orc.confidence_vt(raws, tau, cap), orc.slot_confidence_vt(raws, tau, cap)
        assert vt == clamp(keep_s) and vt_slot == clamp(keep_p), (raws, tau, cap)
        assert vt <= vt_slot


def pin_window_limits(orc):
    """Scores at the extremes: certain slots keep every draft up to the cap, hopeless ones
    keep none (the vt floor is anchor + 1 draft); p_min = 0 switches the break off."""
    for n in range(0, 15):
        assert orc.conf_keep(np.zeros(n), 0.0, 1) == n
        assert orc.conf_keep(np.ones(n), 1.0, 1) == n
        assert orc.confidence_vt(np.full(n, np.inf, np.float32), 0.5, 15) == max(2, n + 1)
        assert orc.confidence_vt(np.full(n, -np.inf, np.float32), 0.5, 15) == 2
        assert orc.slot_confidence_vt(np.full(n, 30.0, np.float32), 0.99, 4) == min(max(2, n + 1), 4)


def _softmax(z):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max())
    return e / e.sum()


def pin_filter_closed_forms(orc):
    """No filter is softmax(x / temperature); top_k = 1 is the argmax; top_k = V, top_p = 1 and
    min_p = 0 filter nothing; the filtered distribution sums to 1."""
    rng = np.random.default_rng(31)
    for V in (1, 2, 7, 100):
        x = rng.normal(0, 2, V).astype(np.float32)
        for tau in (0.3, 1.0, 2.5):
            ref = _softmax(x.astype(np.float64) / tau)
            assert np.allclose(orc.filtered(x, tau), ref, rtol=1e-12, atol=1e-15)
            assert np.allclose(orc.filtered(x, tau, top_k=V, top_p=1.0, min_p=0.0), ref, rtol=1e-12, atol=1e-15)
            one = orc.filtered(x, tau, top_k=1)
            assert one[int(np.argmax(x))] == 1.0 and one.sum() == 1.0
            for kw in ({"top_k": 3}, {"top_p": 0.5}, {"min_p": 0.2}, {"top_k": 5, "top_p": 0.8, "min_p": 0.05}):
                assert abs(orc.filtered(x, tau, **kw).sum() - 1.0) < 1e-12


def pin_filter_brute_force(orc):
    """Kept sets from their set definitions: top-k keeps a token when fewer than k tokens are
    strictly more likely; top-p keeps it when the tokens strictly more likely hold less than
    top_p of the mass; min-p keeps p >= min_p * max p.  Ties included."""
    rng = np.random.default_rng(32)
    for _ in range(300):
        V = int(rng.integers(1, 9))
        x = rng.integers(-3, 4, V).astype(np.float32)  # small integers: ties everywhere
        tau = float(rng.choice([0.5, 1.0, 3.0]))
        k = int(rng.integers(0, V + 2))
        tp = float(rng.choice([1.0, 0.9, 0.5, 0.2]))
        mp = float(rng.choice([0.0, 0.1, 0.5]))
        p = _softmax(x.astype(np.float64) / tau)
        keep = np.ones(V, bool)
        for v in range(V):
            larger = p > p[v]
            if 0 < k < V and larger.sum() >= k:
                keep[v] = False
            if tp < 1.0 and p[larger].sum() >= tp:
                keep[v] = False
            if mp > 0 and p[v] < mp * p.max():
                keep[v] = False
        want = np.where(keep, p, 0.0)
        want /= want.sum()
        got = orc.filtered(x, tau, top_k=k, top_p=tp, min_p=mp)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-15), (x, tau, k, tp, mp, got, want)


def pin_filter_top_p_boundary(orc):
    """top_p reached exactly by the first token's mass keeps that token alone (the running
    sum "reaches" top_p * S: >=, not >)."""
    for a in (-1.0, -0.5, -2.0):
        x = np.array([0.0, a, a], np.float32)
        e = np.exp(x.astype(np.float64))
        S = 0.0
        for v in e:  # the oracle's order of summation
            S += v
        tp = 1.0 / S
        assert tp * S == 1.0
        got = orc.filtered(x, 1.0, top_p=tp)
        assert list(got) == [1.0, 0.0, 0.0], (a, got)


def _chi2_ok(counts, probs, n):
    """Pearson chi-square of counts against probs, p-value above 1e-4 (scipy)."""
    from scipy.stats import chisquare
    m = probs > 0
    assert counts[~m].sum() == 0, "a token outside the support was emitted"
    if m.sum() == 1:  # one token carries all the mass: every draw must be it
        return bool(counts[m].sum() == n)
    exp = probs[m] * n
    return chisquare(counts[m], exp * counts[m].sum() / exp.sum()).pvalue > 1e-4


def pin_sampled_accept_is_exact(orc):
    """Speculative sampling emits its first token distributed exactly as the filtered target
    p~_0 whatever the draft distribution q~_0 (the draft token is drawn from q~_0, u ~ U(0,1)):
    Monte Carlo with a chi-square test, for several draft/target pairs and filters."""
    rng = np.random.default_rng(33)
    V, n = 6, 20000
    for case in range(4):
        p_row = rng.normal(0, 1.5, V).astype(np.float32)
        q_row = rng.normal(0, 1.5, V).astype(np.float32) if case != 3 else p_row.copy()
        filt = [{}, {"top_k": 4}, {"top_p": 0.8, "min_p": 0.05}, {"temperature": 0.7}][case]
        pt = orc.filtered(p_row, **{"temperature": 1.0, **filt})
        qt = orc.filtered(q_row, **{"temperature": 1.0, **filt})
        logits = np.stack([p_row, rng.normal(0, 1, V).astype(np.float32)])
        counts = np.zeros(V, np.int64)
        xs = rng.choice(V, n, p=qt)
        us = rng.uniform(0, 1, (n, 2))
        for i in range(n):
            j, tok = orc.sampled_accept(logits, q_row[None], [int(xs[i])], [us[i, 0]], us[i, 1],
                                        **{"temperature": 1.0, **filt})
            counts[int(xs[i]) if j == 1 else tok] += 1
        assert _chi2_ok(counts, pt, n), (case, counts, pt)
        if case == 3:  # q = p: every draft is accepted
            assert counts.sum() == n


def pin_sampled_accept_bonus_and_greedy(orc):
    """All drafts accepted: the bonus follows p~_K (chi-square).  top_k = 1 turns the walk into
    greedy acceptance: j and the token equal the greedy accept of the same rows."""
    rng = np.random.default_rng(34)
    V, T = 5, 3
    logits = rng.normal(0, 1, (T, V)).astype(np.float32)
    pK = orc.filtered(logits[T - 1])
    counts = np.zeros(V, np.int64)
    drafts = [int(np.argmax(orc.filtered(logits[r]))) for r in range(T - 1)]
    n = 20000
    us = rng.uniform(0, 1, n)
    for i in range(n):
        j, tok = orc.sampled_accept(logits, logits[:T - 1], drafts, [0.999999, 0.999999], us[i])
        assert j == T - 1
        counts[tok] += 1
    assert _chi2_ok(counts, pK, n)
    for _ in range(200):
        T = int(rng.integers(1, 6))
        V = int(rng.integers(2, 30))
        lg = rng.normal(0, 1, (T, V)).astype(np.float32)
        dl = rng.normal(0, 1, (max(T - 1, 1), V)).astype(np.float32)[:T - 1]
        d = [int(np.argmax(dl[r])) if rng.uniform() < 0.7 else int(np.argmax(lg[r])) for r in range(T - 1)]
        jg, bg, _, _ = orc.accept(lg, np.array(d, np.int32))
        js, ts = orc.sampled_accept(lg, dl, d, rng.uniform(0, 1, T - 1), float(rng.uniform()), top_k=1)
        assert (js, ts) == (jg, bg), (lg, d)
        # u = 0 still rejects a draft the filtered target excludes (p~ = 0 at it)
        js0, ts0 = orc.sampled_accept(lg, dl, d, np.zeros(T - 1), 0.0, top_k=1)
        assert (js0, ts0) == (jg, bg), (lg, d)


def _philox_kat():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                w = [int(x, 16) for x in ln.split()]
                rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def pin_philox_known_answers(orc):
    """Philox4x32-10 reproduces the generator's published known-answer vectors
    (tests/golden/philox4x32_10_kat.txt)."""
    kat = _philox_kat()
    assert len(kat) == 3
    for ctr, key, want in kat:
        assert [int(x) for x in orc.philox(ctr, key)] == want, (ctr, key)


def pin_u01_layout(orc):
    """A session uniform is output word 0 of Philox4x32-10 at counter (n, 0, 0, tag) under
    key (seed low, seed high), top 24 bits times 2^-24: exact in f32, in [0, 1), and
    uniform (chi-square over 16 bins of 20000 draws)."""
    rng = np.random.default_rng(40)
    for _ in range(50):
        seed = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        n = int(rng.integers(0, 2**32))
        tag = int(rng.choice([0xFFFFFFFE, 0xFFFFFFFF, 0]))
        w0 = int(orc.philox([n, 0, 0, tag], [seed & 0xFFFFFFFF, seed >> 32])[0])
        u = orc.u01(seed, n, tag)
        assert u == (w0 >> 8) / 16777216.0 and 0.0 <= u < 1.0 and float(np.float32(u)) == u
    us = np.array([orc.u01(99, n, 0xFFFFFFFE) for n in range(20000)])
    assert _chi2_ok(np.histogram(us, bins=16, range=(0, 1))[0], np.full(16, 1 / 16), us.size)
    assert orc.u01(99, 5, 0xFFFFFFFE) != orc.u01(99, 5, 0xFFFFFFFF)  # the two tags are two streams


def pin_sampled_session_counters(orc):
    """The session walk equals the uniform-input walk fed from its counters: accept test r
    uses u01(seed, uctr + r, 0xFFFFFFFE) and the final draw u01(seed, sctr, 0xFFFFFFFF);
    uctr advances by the tests run (j + 1 on a rejection, K when every draft is accepted),
    sctr by one.  Rounds in a row never reuse a counter."""
    rng = np.random.default_rng(41)
    V = 40
    for case in range(200):
        T = int(rng.integers(1, 8))
        K = T - 1
        lg = rng.normal(0, 1.5, (T, V)).astype(np.float32)
        dl = (lg[:K] + rng.normal(0, 1.0, (K, V)).astype(np.float32)).astype(np.float32)
        d = [int(np.argmax(dl[r])) if rng.uniform() < 0.7 else int(rng.integers(0, V)) for r in range(K)]
        seed, uctr, sctr = int(rng.integers(0, 2**62)), int(rng.integers(0, 2**32 - 20)), int(rng.integers(0, 2**32 - 2))
        filt = dict(temperature=0.8, top_k=int(rng.choice([0, 5])), top_p=float(rng.choice([1.0, 0.9])))
        j, tok, u2, s2 = orc.sampled_accept_session(lg, dl, d, seed, uctr, sctr, **filt)
        ua = [orc.u01(seed, uctr + r, 0xFFFFFFFE) for r in range(K)]
        us = orc.u01(seed, sctr, 0xFFFFFFFF)
        assert (j, tok) == orc.sampled_accept(lg, dl, d, ua, us, **filt)
        assert u2 == uctr + (j + 1 if j < K else K) and s2 == sctr + 1
        # the next round starts where this one stopped: its first test uniform is new
        if K:
            assert u2 > uctr


PINS = [
    pin_core_matrix_form,
    pin_core_closed_form_first_write,
    pin_core_identity,
    pin_core_orthonormal_writes,
    pin_core_decay_only,
    pin_prepare_current_tap,
    pin_prepare_shifted_taps,
    pin_prepare_vs_correlate,
    pin_prepare_gates,
    pin_prepare_ring_reroll,
    pin_bf16_widening,
    pin_verify_brute_force,
    pin_verify_chained_rows,
    pin_rollback,
    pin_accept_page_fixture,
    pin_accept_brute_force,
    pin_accept_nan,
    pin_accept_ties,
    pin_window_page_fixture,
    pin_window_brute_force,
    pin_window_limits,
    pin_filter_closed_forms,
    pin_filter_brute_force,
    pin_filter_top_p_boundary,
    pin_sampled_accept_is_exact,
    pin_sampled_accept_bonus_and_greedy,
    pin_philox_known_answers,
    pin_u01_layout,
    pin_sampled_session_counters,
]
