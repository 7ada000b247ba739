"""CPU oracle for the KDA speculative-verify walk (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this package.  The CUDA library never imports, links or calls
it, and it shares no code with the CUDA path.  The arithmetic lives in
``kda_oracle.c`` (plain single-threaded C, double precision, f32 storage);
this module compiles it with gcc and marshals numpy arrays through ctypes.

Every function works on one (session, layer) unit; ``verify_units`` only
slices the [L][B] leading axes of the library's layouts and loops.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

D = 128
TMAX = 15
F32, BF16 = 0, 1
OK, EINVAL, ENAN, ENOMEM = 0, 1, 2, 5
SENTINEL = -1

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kda_oracle.c")
HEADER_DIR = _HERE
BUILD_DIR = os.path.join(_HERE, "_build")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def build(out_path: str | None = None, source: str | None = None) -> str:
    """Compile the oracle into a shared library and return its path.

    ``source`` is the path of the C file to compile (the tests use this to build
    deliberately broken copies of the oracle); by default ``kda_oracle.c``.
    """
    src = source or SOURCE
    if out_path is None:
        out_path = os.path.join(BUILD_DIR, "libkda_oracle.so")
    os.makedirs(os.path.dirname(os.path.abspath(out_path)), exist_ok=True)
    tmp = f"{out_path}.{os.getpid()}.tmp"
    cmd = ["gcc", *CFLAGS, "-I", HEADER_DIR, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _raw(a):
    """Raw rows: float32 values, or uint16 arrays holding bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"raw rows must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        super().__init__(f"oracle {fn} returned {rc}")
        self.rc = rc


class Oracle:
    """ctypes view of one compiled copy of the oracle."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        vp, ci = ctypes.c_void_p, ctypes.c_int
        self.lib.kdao_prepare.argtypes = [ci, ci, ci] + [vp] * 13
        self.lib.kdao_core.argtypes = [ci, ci] + [vp] * 7
        self.lib.kdao_verify.argtypes = [ci, ci, ci] + [vp] * 11
        self.lib.kdao_rollback.argtypes = [ci, ci, ci, ci] + [vp] * 12
        self.lib.kdao_accept.argtypes = [ci, ci, ci, vp, vp, vp, vp, vp]
        cf = ctypes.c_float
        self.lib.kdao_conf_keep.argtypes = [ci, vp, cf, ci]
        self.lib.kdao_confidence_vt.argtypes = [ci, vp, cf, ci]
        self.lib.kdao_slot_confidence_vt.argtypes = [ci, vp, cf, ci]
        cd = ctypes.c_double
        self.lib.kdao_filtered.argtypes = [ci, ci, vp, cd, ci, cd, cd, vp]
        self.lib.kdao_sampled_accept.argtypes = [ci, ci, ci, vp, vp, vp, vp, cd, cd, ci, cd, cd, vp, vp]
        cu, cull = ctypes.c_uint, ctypes.c_ulonglong
        self.lib.kdao_philox4x32_10.argtypes = [vp, vp, vp]
        self.lib.kdao_philox4x32_10.restype = None
        self.lib.kdao_u01.argtypes = [cull, cu, cu]
        self.lib.kdao_u01.restype = cf
        self.lib.kdao_sampled_accept_session.argtypes = [ci, ci, ci, vp, vp, vp, cull, vp, vp, cd, ci, cd, cd, vp,
                                                         vp]
        for fn in ("kdao_prepare", "kdao_core", "kdao_verify", "kdao_rollback", "kdao_accept", "kdao_conf_keep",
                   "kdao_confidence_vt", "kdao_slot_confidence_vt", "kdao_filtered", "kdao_sampled_accept",
                   "kdao_sampled_accept_session"):
            getattr(self.lib, fn).restype = ci

    @staticmethod
    def _check(fn, rc, allowed=(OK,)):
        if rc not in allowed:
            raise OracleError(fn, rc)
        return rc

    # -- activations ----------------------------------------------------------
    def prepare(self, xq, xk, xv, xg, xb, conv_w, ring_in):
        """Conv + SiLU, L2 norm and gates of one unit.

        Returns (q_hat, k_hat, v, g, beta, ring_out): float64 [T][H][128] except
        beta [T][H]; ring_out float32 [H][3][3][128].
        """
        xq, dt = _raw(xq)
        xk, xv, xg, xb = (_raw(a)[0] for a in (xk, xv, xg, xb))
        T, H = xq.shape[0], xq.shape[1]
        conv_w, ring_in = _f32(conv_w), _f32(ring_in)
        q = np.empty((T, H, D))
        k, v, g = np.empty_like(q), np.empty_like(q), np.empty_like(q)
        b = np.empty((T, H))
        ring_out = np.empty((H, 3, 3, D), np.float32)
        rc = self.lib.kdao_prepare(H, T, dt, _p(xq), _p(xk), _p(xv), _p(xg), _p(xb), _p(conv_w),
                                   _p(ring_in), _p(q), _p(k), _p(v), _p(g), _p(b), _p(ring_out))
        self._check("kdao_prepare", rc)
        return q, k, v, g, b, ring_out

    # -- the recurrence on post-activation inputs -----------------------------
    def core(self, q_hat, k_hat, v, g, beta, S):
        """Run the gated delta rule; returns (S_after [H][128][128], out [T][H][128])."""
        q_hat, k_hat, v, g, beta = (_f64(a) for a in (q_hat, k_hat, v, g, beta))
        S = _f64(S).copy()
        T, H = q_hat.shape[0], q_hat.shape[1]
        out = np.empty((T, H, D))
        rc = self.lib.kdao_core(H, T, _p(q_hat), _p(k_hat), _p(v), _p(g), _p(beta), _p(S), _p(out))
        self._check("kdao_core", rc)
        return S, out

    # -- one verify launch for one unit ---------------------------------------
    def verify(self, xq, xk, xv, xg, xb, conv_w, ring_in, state_in):
        """Returns (state_out, ring_out, out) as float32."""
        xq, dt = _raw(xq)
        xk, xv, xg, xb = (_raw(a)[0] for a in (xk, xv, xg, xb))
        T, H = xq.shape[0], xq.shape[1]
        conv_w, ring_in, state_in = _f32(conv_w), _f32(ring_in), _f32(state_in)
        state_out = np.empty((H, D, D), np.float32)
        ring_out = np.empty((H, 3, 3, D), np.float32)
        out = np.empty((T, H, D), np.float32)
        rc = self.lib.kdao_verify(H, T, dt, _p(xq), _p(xk), _p(xv), _p(xg), _p(xb), _p(conv_w),
                                  _p(ring_in), _p(state_in), _p(ring_out), _p(state_out), _p(out))
        self._check("kdao_verify", rc)
        return state_out, ring_out, out

    def rollback(self, keep, xq, xk, xv, xg, xb, conv_w, ring_snap, state_snap, ring_cur, state_cur):
        """Accept-j rollback of one unit; returns (state, ring) as float32."""
        xq, dt = _raw(xq)
        xk, xv, xg, xb = (_raw(a)[0] for a in (xk, xv, xg, xb))
        T, H = xq.shape[0], xq.shape[1]
        arrs = [_f32(a) for a in (conv_w, ring_snap, state_snap, ring_cur, state_cur)]
        state_out = np.empty((H, D, D), np.float32)
        ring_out = np.empty((H, 3, 3, D), np.float32)
        rc = self.lib.kdao_rollback(H, T, int(keep), dt, _p(xq), _p(xk), _p(xv), _p(xg), _p(xb),
                                    *(_p(a) for a in arrs), _p(ring_out), _p(state_out))
        self._check("kdao_rollback", rc)
        return state_out, ring_out

    def accept(self, logits, drafts):
        """Greedy accept of one session.

        logits: [T][V] float32 or uint16 (bf16 bits); drafts: [T-1] ints.
        Returns (j, bonus, vam, rc) with rc OK or ENAN.
        """
        logits, dt = _raw(logits)
        T, V = logits.shape
        drafts = np.ascontiguousarray(drafts, dtype=np.int32).reshape(-1)
        assert drafts.shape == (T - 1,)
        vam = np.empty(T, np.int32)
        j, bonus = ctypes.c_int(), ctypes.c_int()
        dptr = _p(drafts) if T > 1 else None
        rc = self.lib.kdao_accept(T, V, dt, _p(logits), dptr, _p(vam), ctypes.byref(j),
                                  ctypes.byref(bonus))
        self._check("kdao_accept", rc, (OK, ENAN))
        return j.value, bonus.value, vam, rc

    # -- verify-window policies (f32 decisions) --------------------------------
    def conf_keep(self, q, p_min, pmin0):
        """Drafts kept by the p-min break over the slot confidences q (glm5_conf_keep)."""
        q = _f32(q).reshape(-1)
        return int(self.lib.kdao_conf_keep(q.size, _p(q) if q.size else None, float(p_min), int(bool(pmin0))))

    def confidence_vt(self, raws, tau, vt_cap):
        """Verify rows from cumulative survival of sigmoid(raws) (dspark_confidence_vt)."""
        r = _f32(raws).reshape(-1)
        return int(self.lib.kdao_confidence_vt(r.size, _p(r) if r.size else None, float(tau), int(vt_cap)))

    def slot_confidence_vt(self, raws, tau, vt_cap):
        """Verify rows from per-slot sigmoid(raws) (dspark_slot_confidence_vt)."""
        r = _f32(raws).reshape(-1)
        return int(self.lib.kdao_slot_confidence_vt(r.size, _p(r) if r.size else None, float(tau), int(vt_cap)))

    # -- sampled acceptance ----------------------------------------------------
    def filtered(self, row, temperature=1.0, top_k=0, top_p=1.0, min_p=0.0):
        """Filtered distribution of one logits row (float32 or bf16 bits) as float64 [V]."""
        row, dt = _raw(row)
        V = row.shape[-1]
        p = np.empty(V)
        rc = self.lib.kdao_filtered(V, dt, _p(row), float(temperature), int(top_k), float(top_p), float(min_p),
                                    _p(p))
        self._check("kdao_filtered", rc)
        return p

    def sampled_accept(self, logits, draft_logits, drafts, u_accept, u_sample, temperature=1.0, top_k=0,
                       top_p=1.0, min_p=0.0):
        """Sampled accept walk of one session; returns (j, token)."""
        logits, dt = _raw(logits)
        T, V = logits.shape
        K = T - 1
        draft_logits = _raw(draft_logits)[0] if K else np.zeros((1, V), logits.dtype)
        drafts = np.ascontiguousarray(drafts, dtype=np.int32).reshape(-1)
        u_accept = _f64(u_accept).reshape(-1)
        assert drafts.shape == (K,) and u_accept.shape == (K,)
        j, tok = ctypes.c_int(), ctypes.c_int()
        rc = self.lib.kdao_sampled_accept(T, V, dt, _p(logits), _p(draft_logits), _p(drafts) if K else None,
                                          _p(u_accept) if K else None, float(u_sample), float(temperature),
                                          int(top_k), float(top_p), float(min_p), ctypes.byref(j), ctypes.byref(tok))
        self._check("kdao_sampled_accept", rc)
        return j.value, tok.value

    def philox(self, ctr, key):
        """Philox4x32-10 of one 4-word counter under a 2-word key; returns 4 uint32."""
        c = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(4)
        k = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
        o = np.empty(4, np.uint32)
        self.lib.kdao_philox4x32_10(_p(c), _p(k), _p(o))
        return o

    def u01(self, seed, counter, tag):
        """The uniform of a session's stream at (counter, tag)."""
        return float(self.lib.kdao_u01(int(seed) & (2**64 - 1), int(counter) & 0xFFFFFFFF, int(tag) & 0xFFFFFFFF))

    def sampled_accept_session(self, logits, draft_logits, drafts, seed, uctr, sctr, temperature=1.0, top_k=0,
                               top_p=1.0, min_p=0.0):
        """Sampled accept walk of one session drawing from its Philox counters; returns
        (j, token, uctr after, sctr after)."""
        logits, dt = _raw(logits)
        T, V = logits.shape
        K = T - 1
        draft_logits = _raw(draft_logits)[0] if K else np.zeros((1, V), logits.dtype)
        drafts = np.ascontiguousarray(drafts, dtype=np.int32).reshape(-1)
        assert drafts.shape == (K,)
        j, tok = ctypes.c_int(), ctypes.c_int()
        uc, sc = ctypes.c_uint(int(uctr) & 0xFFFFFFFF), ctypes.c_uint(int(sctr) & 0xFFFFFFFF)
        rc = self.lib.kdao_sampled_accept_session(T, V, dt, _p(logits), _p(draft_logits), _p(drafts) if K else None,
                                                  int(seed) & (2**64 - 1), ctypes.byref(uc), ctypes.byref(sc),
                                                  float(temperature), int(top_k), float(top_p), float(min_p),
                                                  ctypes.byref(j), ctypes.byref(tok))
        self._check("kdao_sampled_accept_session", rc)
        return j.value, tok.value, uc.value, sc.value

    # -- [L][B] helper ---------------------------------------------------------
    def verify_units(self, rows, conv_w, ring, state, units=None):
        """Run ``verify`` on every (l, b) unit (or the listed ones).

        rows: dict q,k,v,g,beta with [L][B][T][H](128); conv_w [L][H][3][128][4];
        ring [L][B][H][3][3][128]; state [L][B][H][128][128].
        Returns dict {(l, b): (state_out, ring_out, out)}.
        """
        L, B = state.shape[0], state.shape[1]
        units = units if units is not None else [(l, b) for l in range(L) for b in range(B)]
        return {
            (l, b): self.verify(rows["q"][l, b], rows["k"][l, b], rows["v"][l, b],
                                rows["g"][l, b], rows["beta"][l, b], conv_w[l], ring[l, b],
                                state[l, b])
            for (l, b) in units
        }


_cache: dict[str, Oracle] = {}
_lock = threading.Lock()


def load(path: str | None = None) -> Oracle:
    """Return the oracle, compiling it first if its library is missing or stale."""
    with _lock:
        if path is None:
            path = os.path.join(BUILD_DIR, "libkda_oracle.so")
            srcs = [SOURCE, os.path.join(_HERE, "kda_oracle.h")]
            if not os.path.exists(path) or os.path.getmtime(path) < max(map(os.path.getmtime, srcs)):
                build(path)
        if path not in _cache:
            _cache[path] = Oracle(path)
        return _cache[path]
