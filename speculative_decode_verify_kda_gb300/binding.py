"""Thin ctypes binding of the C ABI in include/kda_spec.h.

Argument marshalling only: torch tensors are checked for device, dtype, shape and
contiguity, their data pointers and the current CUDA stream go to the library,
and every step of the path runs in the library's kernels.  There is no fallback:
if the compiled library is missing, loading it raises.

Names follow the C ABI: ``kda_verify_scan``, ``kda_rollback``, ``spec_accept``.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libkda_spec.so")

D = 128
TMAX = 15
HOST_KEEP_MAX = 2048
OK, EINVAL, ENAN, ECUDA, ETIMEOUT = 0, 1, 2, 3, 4
ST_NAN, ST_BADKEEP, ST_TIMEOUT = 0x1, 0x2, 0x4
TAG_ACCEPT, TAG_DRAW = 0xFFFFFFFE, 0xFFFFFFFF  # counter word 3 of a session's accept tests / draws
F32, BF16 = 0, 1
MEM_HOST, MEM_DEVICE = 0, 1

# every symbol the header declares (checked by the CPU test of the library load)
EXPORTS = ("kda_verify_scan", "kda_rollback", "kda_verify_scan_var", "kda_rollback_var", "kda_verify_scan_pingpong",
           "kda_verify_scan_deferred", "kda_verify_scan_deferred_staged", "kda_stream_write_u32",
           "kda_upload_rows_staged", "kda_round_host", "kda_verify_scan_deferred_host",
           "kda_verify_scan_cols",
           "kda_rollback_cols", "spec_accept_var",
           "spec_window", "spec_accept_sampled", "spec_accept_sampled_session", "kda_philox4x32_10",
           "spec_accept_sampled_scratch_bytes", "spec_accept_scratch_bytes", "spec_accept", "spec_accept_noalloc", "kda_error_string",
           "kda_last_error", "kda_abi_version")
ABI_VERSION = 9
WIN_CONF_KEEP, WIN_CONFIDENCE, WIN_SLOT_CONFIDENCE = 0, 1, 2


class KdaDims(ctypes.Structure):
    _fields_ = [("L", ctypes.c_int), ("B", ctypes.c_int), ("H", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("dtype", ctypes.c_int)]


class KdaLayerState(ctypes.Structure):
    _fields_ = [("state", ctypes.c_void_p), ("conv_ring", ctypes.c_void_p), ("conv_w", ctypes.c_void_p)]


class KdaRows(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("w", ctypes.c_void_p)]


class KdaStashC(ctypes.Structure):
    _fields_ = [("state_snap", ctypes.c_void_p), ("ring_snap", ctypes.c_void_p),
                ("rows", KdaRows), ("T", ctypes.c_int)]


class KdaSampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int), ("top_p", ctypes.c_float),
                ("min_p", ctypes.c_float)]


class KdaError(RuntimeError):
    def __init__(self, fn: str, rc: int, msg: str):
        super().__init__(f"{fn} failed ({rc}): {msg}")
        self.rc = rc


_lib = None


def lib(path: str | None = None):
    """Load the compiled library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library {p} is missing: run __graft_entry__.build() "
                           "(or python -m speculative_decode_verify_kda_gb300.build) first")
    L = ctypes.CDLL(p)
    vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.kda_verify_scan.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                  ctypes.POINTER(KdaRows), ci, vp, ctypes.POINTER(KdaStashC), vp]
    L.kda_verify_scan.restype = ci
    L.kda_rollback.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                               ctypes.POINTER(KdaStashC), vp, ci, vp, vp]
    L.kda_rollback.restype = ci
    L.kda_verify_scan_var.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                      ctypes.POINTER(KdaRows), ci, vp, ci, vp, ctypes.POINTER(KdaStashC), vp, vp]
    L.kda_verify_scan_var.restype = ci
    L.kda_rollback_var.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                   ctypes.POINTER(KdaStashC), vp, vp, ci, vp, vp]
    L.kda_rollback_var.restype = ci
    L.kda_verify_scan_pingpong.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                           ctypes.POINTER(KdaRows), ci, vp, ci, vp, ctypes.POINTER(KdaStashC), vp,
                                           vp]
    L.kda_verify_scan_pingpong.restype = ci
    L.kda_verify_scan_deferred.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                           ctypes.POINTER(KdaStashC), vp, ctypes.POINTER(KdaRows), ci, vp, vp, vp]
    L.kda_verify_scan_deferred.restype = ci
    L.kda_verify_scan_deferred_staged.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                                  ctypes.POINTER(KdaStashC), vp, ctypes.POINTER(KdaRows), ci, vp, vp,
                                                  ci, ctypes.c_uint, vp, vp]
    L.kda_verify_scan_deferred_staged.restype = ci
    L.kda_stream_write_u32.argtypes = [vp, ctypes.c_uint, vp]
    L.kda_stream_write_u32.restype = ci
    L.kda_upload_rows_staged.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaRows), ctypes.POINTER(KdaRows),
                                         ci, vp, ci, ctypes.c_uint, vp]
    L.kda_upload_rows_staged.restype = ci
    L.kda_round_host.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState), ctypes.POINTER(KdaStashC),
                                 ci, ctypes.POINTER(KdaRows), ctypes.POINTER(KdaRows), vp, vp, ci, ci, vp, vp, vp,
                                 vp, vp, vp, ci, ctypes.c_uint, vp, vp, vp, ci, ci]
    L.kda_round_host.restype = ci
    L.kda_verify_scan_deferred_host.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                                ctypes.POINTER(KdaStashC), vp, ctypes.POINTER(KdaRows),
                                                ctypes.POINTER(KdaRows), ci, vp, vp, vp]
    L.kda_verify_scan_deferred_host.restype = ci
    L.kda_verify_scan_cols.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState),
                                       ctypes.POINTER(KdaRows), ci, vp, vp, vp, vp]
    L.kda_verify_scan_cols.restype = ci
    L.kda_rollback_cols.argtypes = [ctypes.POINTER(KdaDims), ctypes.POINTER(KdaLayerState), vp, vp, ci, vp, ci, vp,
                                    vp]
    L.kda_rollback_cols.restype = ci
    L.spec_accept_var.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_accept_var.restype = ci
    L.spec_window.argtypes = [vp, ci, ci, ci, ctypes.c_float, ci, ci, vp, vp]
    L.spec_window.restype = ci
    L.spec_accept_sampled.argtypes = [vp, vp, ci, ci, ci, ci, vp, vp, vp, ctypes.POINTER(KdaSampling), vp, vp, vp,
                                      vp, vp, sz, vp]
    L.spec_accept_sampled_session.argtypes = [vp, vp, ci, ci, ci, ci, vp, vp, vp, ctypes.POINTER(KdaSampling), vp,
                                              vp, vp, vp, vp, sz, vp]
    L.spec_accept_sampled_session.restype = ci
    L.kda_philox4x32_10.argtypes = [vp, vp, vp, ci, vp]
    L.kda_philox4x32_10.restype = ci
    L.spec_accept_sampled_scratch_bytes.argtypes = [ci, ci]
    L.spec_accept_sampled_scratch_bytes.restype = sz
    L.spec_accept_sampled.restype = ci
    L.spec_accept_scratch_bytes.argtypes = [ci, ci, ci]
    L.spec_accept_scratch_bytes.restype = sz
    L.spec_accept.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, vp, vp, vp, sz, vp]
    L.spec_accept.restype = ci
    L.kda_error_string.argtypes = [ci]
    L.kda_error_string.restype = ctypes.c_char_p
    L.kda_last_error.argtypes = []
    L.kda_last_error.restype = ctypes.c_char_p
    L.kda_abi_version.argtypes = []
    L.kda_abi_version.restype = ci
    if path is None:
        _lib = L
    return L


def _check(fn: str, rc: int):
    if rc != OK:
        raise KdaError(fn, rc, lib().kda_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _row_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"raw rows must be float32 or bfloat16, got {t.dtype}")


class LayerState:
    """Resident state of L layers x B sessions x H heads (device tensors).

    state [L][B][H][128][128] f32, conv_ring [L][B][H][3][3][128] f32,
    conv_w [L][H][3][128][4] f32.
    """

    def __init__(self, state: torch.Tensor, conv_ring: torch.Tensor, conv_w: torch.Tensor):
        L, B, H = state.shape[:3]
        self.L, self.B, self.H = int(L), int(B), int(H)
        self.state = _dev(state, "state", torch.float32, (L, B, H, D, D))
        self.conv_ring = _dev(conv_ring, "conv_ring", torch.float32, (L, B, H, 3, 3, D))
        self.conv_w = _dev(conv_w, "conv_w", torch.float32, (L, H, 3, D, 4))

    def c(self) -> KdaLayerState:
        return KdaLayerState(self.state.data_ptr(), self.conv_ring.data_ptr(), self.conv_w.data_ptr())

    def dims(self, dtype: int) -> KdaDims:
        return KdaDims(self.L, self.B, self.H, D, D, dtype)

    def layer(self, l: int) -> "LayerState":
        """Layer l alone (L = 1), as views of these tensors (layer-major, so contiguous)."""
        return LayerState(self.state[l:l + 1], self.conv_ring[l:l + 1], self.conv_w[l:l + 1])


class Stash:
    """Rollback material of one verify round: snapshots (owned here) + the raw rows.

    The raw-row tensors are referenced, not copied, and stay alive with the stash.
    """

    def __init__(self, st: LayerState | None = None, state_snap: torch.Tensor | None = None,
                 ring_snap: torch.Tensor | None = None):
        self.state_snap = torch.empty_like(st.state) if state_snap is None else state_snap
        self.ring_snap = torch.empty_like(st.conv_ring) if ring_snap is None else ring_snap
        self.c = KdaStashC(self.state_snap.data_ptr(), self.ring_snap.data_ptr(), KdaRows(), 0)
        self.rows = None
        self.dtype = None

    def layer(self, l: int) -> "Stash":
        """A stash for layer l alone whose snapshots are views of these snapshots."""
        return Stash(state_snap=self.state_snap[l:l + 1], ring_snap=self.ring_snap[l:l + 1])

    @property
    def T(self) -> int:
        return int(self.c.T)


def _rows(st: LayerState, q, k, v, g, beta, T: int | None = None, w: torch.Tensor | None = None):
    """The kda_rows of one round; w (optional): f32 [L][B][T][H][128], the update vectors
    the verify writes and a replay of these rows reads."""
    dt = q.dtype
    if T is None:
        T = int(q.shape[2])
    shp = (st.L, st.B, T, st.H, D)
    tensors = [_dev(q, "q", dt, shp), _dev(k, "k", dt, shp), _dev(v, "v", dt, shp),
               _dev(g, "g", dt, shp), _dev(beta, "beta", dt, shp[:4])]
    wp = None
    if w is not None:
        tensors.append(_dev(w, "w", torch.float32, shp))
        wp = w.data_ptr()
    return KdaRows(*(x.data_ptr() for x in tensors[:5]), wp), tensors, _row_dtype(q), T


def kda_verify_scan(st: LayerState, q, k, v, g, beta, out: torch.Tensor | None = None,
                    stash: Stash | None = None, stream=None, w: torch.Tensor | None = None) -> Stash | None:
    """One verify round of T = q.shape[2] rows for every (layer, session, head).

    q, k, v, g: [L][B][T][H][128], beta [L][B][T][H] (float32 or bfloat16, raw rows);
    out: None or f32 [L][B][T][H][128].  state and conv_ring advance in place.
    With a stash, its snapshots receive the pre-round state and ring.  w: None or f32
    [L][B][T][H][128], receives the rows' update vectors, which the rollback then reads.
    """
    rows, tensors, dt, T = _rows(st, q, k, v, g, beta, w=w)
    if out is not None:
        _dev(out, "out", torch.float32, (st.L, st.B, T, st.H, D))
    dims, cst = st.dims(dt), st.c()
    rc = lib().kda_verify_scan(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(rows), T,
                               _ptr(out), ctypes.byref(stash.c) if stash is not None else None,
                               ctypes.c_void_p(_stream(stream)))
    _check("kda_verify_scan", rc)
    if stash is not None:
        stash.rows, stash.dtype = tensors, dt
    return stash


def kda_rollback(st: LayerState, stash: Stash, keep, dev_status: torch.Tensor | None = None,
                 stream=None) -> None:
    """Accept-j rollback.  keep: host sequence of B ints, or a device int32 tensor [B]."""
    if stash.rows is None:
        raise ValueError("stash holds no verify round")
    dims, cst = st.dims(stash.dtype), st.c()
    if isinstance(keep, torch.Tensor) and keep.is_cuda:
        _dev(keep, "keep", torch.int32, (st.B,))
        kp, mem = ctypes.c_void_p(keep.data_ptr()), MEM_DEVICE
        hold = keep
    else:
        hold = (ctypes.c_int * max(st.B, 1))(*[int(x) for x in keep])
        if len(list(keep)) != st.B:
            raise ValueError(f"keep must have {st.B} entries")
        kp, mem = ctypes.cast(hold, ctypes.c_void_p), MEM_HOST
    if dev_status is not None:
        _dev(dev_status, "dev_status", torch.int32)
    rc = lib().kda_rollback(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(stash.c), kp, mem,
                            _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
    del hold
    _check("kda_rollback", rc)


def _int_array(x, B: int, name: str):
    """A host int array (ctypes) or a device int32 tensor [B] -> (pointer, mem kind, holder)."""
    if isinstance(x, torch.Tensor) and x.is_cuda:
        _dev(x, name, torch.int32, (B,))
        return ctypes.c_void_p(x.data_ptr()), MEM_DEVICE, x
    vals = [int(v) for v in x]
    if len(vals) != B:
        raise ValueError(f"{name} must have {B} entries")
    hold = (ctypes.c_int * max(B, 1))(*vals)
    return ctypes.cast(hold, ctypes.c_void_p), MEM_HOST, hold


def kda_verify_scan_var(st: LayerState, q, k, v, g, beta, t_rows, out: torch.Tensor | None = None,
                        stash: Stash | None = None, dev_status: torch.Tensor | None = None, stream=None,
                        w: torch.Tensor | None = None):
    """Verify round where session b runs t_rows[b] of the T = q.shape[2] rows.

    t_rows: host sequence of B ints or a device int32 tensor [B]; the other arguments
    as for kda_verify_scan.
    """
    rows, tensors, dt, T = _rows(st, q, k, v, g, beta, w=w)
    if out is not None:
        _dev(out, "out", torch.float32, (st.L, st.B, T, st.H, D))
    tp, mem, hold = _int_array(t_rows, st.B, "t_rows")
    dims, cst = st.dims(dt), st.c()
    rc = lib().kda_verify_scan_var(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(rows), T, tp, mem, _ptr(out),
                                   ctypes.byref(stash.c) if stash is not None else None, _ptr(dev_status),
                                   ctypes.c_void_p(_stream(stream)))
    del hold
    _check("kda_verify_scan_var", rc)
    if stash is not None:
        stash.rows, stash.dtype = tensors, dt
    return stash


def kda_rollback_var(st: LayerState, stash: Stash, t_rows, keep, dev_status: torch.Tensor | None = None,
                     stream=None) -> None:
    """Rollback of a kda_verify_scan_var round: t_rows and keep both host or both device."""
    if stash.rows is None:
        raise ValueError("stash holds no verify round")
    tp, m1, h1 = _int_array(t_rows, st.B, "t_rows")
    kp, m2, h2 = _int_array(keep, st.B, "keep")
    if m1 != m2:
        raise ValueError("t_rows and keep must both be host arrays or both device tensors")
    dims, cst = st.dims(stash.dtype), st.c()
    rc = lib().kda_rollback_var(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(stash.c), tp, kp, m1,
                                _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
    del h1, h2
    _check("kda_rollback_var", rc)


class PingPong:
    """The state and conv ring of L x B x H units in two buffers whose roles swap
    every round (kda_verify_scan_pingpong): a round reads the committed buffer, which
    it leaves untouched as the round's snapshot, and writes the other one.

    ``state()`` / ``ring()`` are the committed tensors.  A round is ``verify`` then,
    where some session keeps fewer than all rows, ``rollback`` (both address the
    buffers of the last verify); ``verify`` flips which buffer is committed.
    """

    def __init__(self, st: LayerState, spare_state: torch.Tensor | None = None,
                 spare_ring: torch.Tensor | None = None):
        self.L, self.B, self.H = st.L, st.B, st.H
        spare_state = torch.empty_like(st.state) if spare_state is None else spare_state
        spare_ring = torch.empty_like(st.conv_ring) if spare_ring is None else spare_ring
        _dev(spare_state, "spare_state", torch.float32, tuple(st.state.shape))
        _dev(spare_ring, "spare_ring", torch.float32, tuple(st.conv_ring.shape))
        self.conv_w = st.conv_w
        self.states = (st.state, spare_state)
        self.rings = (st.conv_ring, spare_ring)
        # a round of parity p reads buffer p (its stash) and writes buffer 1 - p
        self.cst = [KdaLayerState(self.states[1 - p].data_ptr(), self.rings[1 - p].data_ptr(),
                                  st.conv_w.data_ptr()) for p in (0, 1)]
        self.cstash = [KdaStashC(self.states[p].data_ptr(), self.rings[p].data_ptr(), KdaRows(), 0) for p in (0, 1)]
        self.parity = 0  # the committed state is in buffer `parity`
        self.last = None  # parity of the last verify
        self.rows, self.dtype = None, None

    def state(self) -> torch.Tensor:
        return self.states[self.parity]

    def ring(self) -> torch.Tensor:
        return self.rings[self.parity]

    def dims(self, dtype: int) -> KdaDims:
        return KdaDims(self.L, self.B, self.H, D, D, dtype)


def kda_verify_scan_pingpong(pp: PingPong, q, k, v, g, beta, out: torch.Tensor | None = None, t_rows=None,
                             dev_status: torch.Tensor | None = None, stream=None,
                             w: torch.Tensor | None = None) -> PingPong:
    """One verify round from the committed buffer of ``pp`` into the other one.

    Arguments as for kda_verify_scan (t_rows: None, or per-session rows as for
    kda_verify_scan_var).  Afterwards the other buffer is committed.
    """
    shape_ref = LayerState(pp.states[0], pp.rings[0], pp.conv_w)
    rows, tensors, dt, T = _rows(shape_ref, q, k, v, g, beta, w=w)
    if out is not None:
        _dev(out, "out", torch.float32, (pp.L, pp.B, T, pp.H, D))
    tp, mem, hold = (None, MEM_HOST, None) if t_rows is None else _int_array(t_rows, pp.B, "t_rows")
    p = pp.parity
    dims = pp.dims(dt)
    rc = lib().kda_verify_scan_pingpong(ctypes.byref(dims), ctypes.byref(pp.cst[p]), ctypes.byref(rows), T, tp, mem,
                                        _ptr(out), ctypes.byref(pp.cstash[p]), _ptr(dev_status),
                                        ctypes.c_void_p(_stream(stream)))
    del hold
    _check("kda_verify_scan_pingpong", rc)
    pp.rows, pp.dtype, pp.last, pp.parity = tensors, dt, p, 1 - p
    return pp


def kda_verify_scan_deferred(pp: PingPong, q, k, v, g, beta, prev_keep: torch.Tensor, out: torch.Tensor | None = None,
                             dev_status: torch.Tensor | None = None, stream=None,
                             w: torch.Tensor | None = None) -> PingPong:
    """A ping-pong round that first commits the previous one: each session with
    prev_keep[b] < the previous T is replayed from the previous pre-round buffer (the
    rollback), then this round's rows run from the committed state.  prev_keep: device
    int32 [B] (the previous round's keep).  Afterwards, as after kda_verify_scan_pingpong,
    the round's snapshot is kept and the post-round buffer is the one to commit next.
    w: None or f32 [L][B][T][H][128], this round's update vectors; the replay reads
    the previous round's (when that round had them), so two w buffers alternate.
    """
    if pp.last is None:
        raise ValueError("a deferred round follows a ping-pong round (no previous round to commit)")
    shape_ref = LayerState(pp.states[0], pp.rings[0], pp.conv_w)
    rows, tensors, dt, T = _rows(shape_ref, q, k, v, g, beta, w=w)
    if dt != pp.dtype:
        raise TypeError("the raw rows must have the previous round's element type")
    if out is not None:
        _dev(out, "out", torch.float32, (pp.L, pp.B, T, pp.H, D))
    _dev(prev_keep, "prev_keep", torch.int32, (pp.B,))
    p = pp.last
    prev = pp.cstash[p]
    cst = KdaLayerState(pp.states[1 - p].data_ptr(), pp.rings[1 - p].data_ptr(), pp.conv_w.data_ptr())
    cstash = KdaStashC(pp.states[p].data_ptr(), pp.rings[p].data_ptr(), prev.rows, prev.T)
    dims = pp.dims(dt)
    rc = lib().kda_verify_scan_deferred(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(cstash), _ptr(prev_keep),
                                        ctypes.byref(rows), T, _ptr(out), _ptr(dev_status),
                                        ctypes.c_void_p(_stream(stream)))
    _check("kda_verify_scan_deferred", rc)
    # this round's snapshot is in buffer 1 - p, its post-round state in buffer p
    pp.cstash[1 - p].rows, pp.cstash[1 - p].T = rows, T
    pp.rows, pp.dtype, pp.last, pp.parity = tensors, dt, 1 - p, p
    return pp


def kda_verify_scan_deferred_staged(pp: PingPong, q, k, v, g, beta, prev_keep: torch.Tensor,
                                    ready_flags: torch.Tensor, pairs_per_flag: int, epoch: int,
                                    out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                                    stream=None, w: torch.Tensor | None = None) -> PingPong:
    """kda_verify_scan_deferred whose raw rows of (layer, session) pair lb = l B + b may
    be read once ready_flags[lb // pairs_per_flag] has reached epoch (see
    kda_upload_rows_staged, kda_stream_write_u32).  ready_flags: device int32 flags
    (compared as unsigned)."""
    if pp.last is None:
        raise ValueError("a deferred round follows a ping-pong round (no previous round to commit)")
    _dev(ready_flags, "ready_flags", torch.int32, (staged_flag_count(pp.L, pp.B, pairs_per_flag),))
    shape_ref = LayerState(pp.states[0], pp.rings[0], pp.conv_w)
    rows, tensors, dt, T = _rows(shape_ref, q, k, v, g, beta, w=w)
    if dt != pp.dtype:
        raise TypeError("the raw rows must have the previous round's element type")
    if out is not None:
        _dev(out, "out", torch.float32, (pp.L, pp.B, T, pp.H, D))
    _dev(prev_keep, "prev_keep", torch.int32, (pp.B,))
    p = pp.last
    prev = pp.cstash[p]
    cst = KdaLayerState(pp.states[1 - p].data_ptr(), pp.rings[1 - p].data_ptr(), pp.conv_w.data_ptr())
    cstash = KdaStashC(pp.states[p].data_ptr(), pp.rings[p].data_ptr(), prev.rows, prev.T)
    dims = pp.dims(dt)
    rc = lib().kda_verify_scan_deferred_staged(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(cstash),
                                               _ptr(prev_keep), ctypes.byref(rows), T, _ptr(out), _ptr(ready_flags),
                                               int(pairs_per_flag), ctypes.c_uint(epoch & 0xffffffff),
                                               _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
    _check("kda_verify_scan_deferred_staged", rc)
    pp.cstash[1 - p].rows, pp.cstash[1 - p].T = rows, T
    pp.rows, pp.dtype, pp.last, pp.parity = tensors, dt, 1 - p, p
    return pp


def kda_verify_scan_deferred_host(pp: PingPong, host: dict, dev: dict, prev_keep: torch.Tensor,
                                  out: torch.Tensor | None = None, dev_status: torch.Tensor | None = None,
                                  stream=None) -> PingPong:
    """kda_verify_scan_deferred whose raw rows are read in place from pinned host memory:
    host holds CPU tensors q, k, v, g, beta (pinned); dev device tensors of the same
    shapes (and optionally w) that receive their copy, which the stash records."""
    if pp.last is None:
        raise ValueError("a deferred round follows a ping-pong round (no previous round to commit)")
    shape_ref = LayerState(pp.states[0], pp.rings[0], pp.conv_w)
    rows, tensors, dt, T = _rows(shape_ref, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], w=dev.get("w"))
    names = ("q", "k", "v", "g", "beta")
    for n in names:
        h = host[n]
        if h.is_cuda or not h.is_contiguous() or h.dtype != dev[n].dtype or tuple(h.shape) != tuple(dev[n].shape):
            raise ValueError(f"host {n} must be a contiguous CPU tensor of the device tensor's shape and type")
    hrows = KdaRows(*(host[n].data_ptr() for n in names))
    if dt != pp.dtype:
        raise TypeError("the raw rows must have the previous round's element type")
    if out is not None:
        _dev(out, "out", torch.float32, (pp.L, pp.B, T, pp.H, D))
    _dev(prev_keep, "prev_keep", torch.int32, (pp.B,))
    p = pp.last
    prev = pp.cstash[p]
    cst = KdaLayerState(pp.states[1 - p].data_ptr(), pp.rings[1 - p].data_ptr(), pp.conv_w.data_ptr())
    cstash = KdaStashC(pp.states[p].data_ptr(), pp.rings[p].data_ptr(), prev.rows, prev.T)
    dims = pp.dims(dt)
    rc = lib().kda_verify_scan_deferred_host(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(cstash),
                                             _ptr(prev_keep), ctypes.byref(hrows), ctypes.byref(rows), T, _ptr(out),
                                             _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
    _check("kda_verify_scan_deferred_host", rc)
    pp.cstash[1 - p].rows, pp.cstash[1 - p].T = rows, T
    pp.rows, pp.dtype, pp.last, pp.parity = tensors, dt, 1 - p, p
    return pp


def staged_flag_count(L: int, B: int, pairs_per_flag: int) -> int:
    """Flags of a staged round: one a range of pairs_per_flag (layer, session) pairs."""
    if int(pairs_per_flag) < 1:
        raise ValueError("pairs_per_flag must be >= 1")
    return -(-(int(L) * int(B)) // int(pairs_per_flag))


def kda_stream_write_u32(flag: torch.Tensor, value: int, stream=None) -> None:
    """flag[0] = value in the order of ``stream``, written by the stream itself (a stream
    memory operation): the ready flags of kda_verify_scan_deferred_staged.  flag: a
    device int32 tensor (its first element is written)."""
    if not isinstance(flag, torch.Tensor) or not flag.is_cuda or flag.dtype != torch.int32 or flag.numel() < 1:
        raise TypeError("flag must be a device int32 tensor")
    _check("kda_stream_write_u32", lib().kda_stream_write_u32(_ptr(flag), ctypes.c_uint(value & 0xffffffff),
                                                              ctypes.c_void_p(_stream(stream))))


class StagedUpload:
    """kda_upload_rows_staged for one pair of raw-row sets: ``host`` (pinned CPU tensors)
    into ``dev`` (device tensors of the same shapes and element type), by ranges of
    pairs_per_flag (layer, session) pairs, each range's flag in ``ready_flags`` set to the
    call's epoch after its copies.  ``__call__(epoch, stream)`` issues the copies on
    ``stream``."""

    def __init__(self, dev: dict, host: dict, ready_flags: torch.Tensor, pairs_per_flag: int):
        names = ("q", "k", "v", "g", "beta")
        L_, B, T, H = (int(x) for x in dev["q"].shape[:4])
        for n in names:
            if tuple(host[n].shape) != tuple(dev[n].shape) or host[n].dtype != dev[n].dtype:
                raise ValueError(f"host and device {n} must have the same shape and element type")
            if not dev[n].is_cuda or host[n].is_cuda or not host[n].is_contiguous() or not dev[n].is_contiguous():
                raise ValueError(f"{n}: dev must be a contiguous device tensor and host a contiguous CPU tensor")
        dt = BF16 if dev["q"].dtype == torch.bfloat16 else F32
        _dev(ready_flags, "ready_flags", torch.int32, (staged_flag_count(L_, B, pairs_per_flag),))
        self.dims = KdaDims(L_, B, H, D, D, dt)
        self.dst = KdaRows(*(dev[n].data_ptr() for n in names))
        self.src = KdaRows(*(host[n].data_ptr() for n in names))
        self.T, self.flags, self.ppf = T, ready_flags, int(pairs_per_flag)
        self._keep = (dev, host)

    def __call__(self, epoch: int, stream=None):
        _check("kda_upload_rows_staged", lib().kda_upload_rows_staged(
            ctypes.byref(self.dims), ctypes.byref(self.dst), ctypes.byref(self.src), self.T, _ptr(self.flags),
            self.ppf, ctypes.c_uint(epoch & 0xffffffff), ctypes.c_void_p(_stream(stream))))


def kda_rollback_pingpong(pp: PingPong, keep, t_rows=None, dev_status: torch.Tensor | None = None,
                          stream=None) -> None:
    """kda_rollback (or kda_rollback_var with t_rows) of the last ping-pong round: the
    sessions that keep fewer than all rows are replayed from the round's pre-round
    buffer into the committed one."""
    if pp.last is None:
        raise ValueError("no ping-pong verify round to roll back")
    p = pp.last
    dims = pp.dims(pp.dtype)
    kp, m2, h2 = _int_array(keep, pp.B, "keep")
    if t_rows is None:
        rc = lib().kda_rollback(ctypes.byref(dims), ctypes.byref(pp.cst[p]), ctypes.byref(pp.cstash[p]), kp, m2,
                                _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
        fn, h1 = "kda_rollback", None
    else:
        tp, m1, h1 = _int_array(t_rows, pp.B, "t_rows")
        if m1 != m2:
            raise ValueError("t_rows and keep must both be host arrays or both device tensors")
        rc = lib().kda_rollback_var(ctypes.byref(dims), ctypes.byref(pp.cst[p]), ctypes.byref(pp.cstash[p]), tp, kp,
                                    m1, _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
        fn = "kda_rollback_var"
    del h1, h2
    _check(fn, rc)


class ColStash:
    """The state and conv ring after every row of one round (column-stash rollback)."""

    def __init__(self, st: LayerState, T: int):
        dev = st.state.device
        self.T = int(T)
        self.state_cols = torch.empty((st.L, st.B, st.H, self.T, D, D), dtype=torch.float32, device=dev)
        self.ring_cols = torch.empty((st.L, st.B, st.H, self.T, 3, 3, D), dtype=torch.float32, device=dev)


def kda_verify_scan_cols(st: LayerState, q, k, v, g, beta, cols: ColStash, out: torch.Tensor | None = None,
                         stream=None) -> ColStash:
    """Verify round that also stashes the state and ring after every row."""
    rows, tensors, dt, T = _rows(st, q, k, v, g, beta)
    if T != cols.T:
        raise ValueError(f"the column stash holds {cols.T} rows, the round has {T}")
    if out is not None:
        _dev(out, "out", torch.float32, (st.L, st.B, T, st.H, D))
    dims, cst = st.dims(dt), st.c()
    rc = lib().kda_verify_scan_cols(ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(rows), T, _ptr(out),
                                    _ptr(cols.state_cols), _ptr(cols.ring_cols), ctypes.c_void_p(_stream(stream)))
    _check("kda_verify_scan_cols", rc)
    cols.dtype = dt
    return cols


def kda_rollback_cols(st: LayerState, cols: ColStash, keep, dev_status: torch.Tensor | None = None,
                      stream=None) -> None:
    """Commit keep[b] rows of a column-stash round by copying the kept column."""
    kp, mem, hold = _int_array(keep, st.B, "keep")
    dims, cst = st.dims(getattr(cols, "dtype", BF16)), st.c()
    rc = lib().kda_rollback_cols(ctypes.byref(dims), ctypes.byref(cst), _ptr(cols.state_cols), _ptr(cols.ring_cols),
                                 cols.T, kp, mem, _ptr(dev_status), ctypes.c_void_p(_stream(stream)))
    del hold
    _check("kda_rollback_cols", rc)


def spec_accept_var(logits: torch.Tensor, drafts: torch.Tensor, t_rows: torch.Tensor, j_out=None, bonus_out=None,
                    keep_out=None, dev_status=None, scratch: torch.Tensor | None = None, stream=None):
    """Greedy accept when session b's round has t_rows[b] (device int32 [B]) of the T rows."""
    _dev(logits, "logits")
    B, T, V = (int(x) for x in logits.shape)
    _dev(drafts, "drafts", torch.int32, (B, T - 1))
    _dev(t_rows, "t_rows", torch.int32, (B,))
    dev = logits.device
    j_out = torch.empty(B, dtype=torch.int32, device=dev) if j_out is None else j_out
    bonus_out = torch.empty(B, dtype=torch.int32, device=dev) if bonus_out is None else bonus_out
    keep_out = torch.empty(B, dtype=torch.int32, device=dev) if keep_out is None else keep_out
    nb = 0 if scratch is None else scratch.numel() * scratch.element_size()  # not used by the library
    rc = lib().spec_accept_var(_ptr(logits), _row_dtype(logits), B, T, V, _ptr(t_rows), _ptr(drafts), _ptr(j_out),
                               _ptr(bonus_out), _ptr(keep_out), _ptr(dev_status), _ptr(scratch), nb,
                               ctypes.c_void_p(_stream(stream)))
    _check("spec_accept_var", rc)
    return j_out, bonus_out, keep_out


def spec_window(scores: torch.Tensor, policy: int, param: float, t_cap: int, pmin0: bool = False,
                t_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per-session verify rows from slot scores (device f32 [B][K]); returns int32 [B]."""
    _dev(scores, "scores", torch.float32)
    B, K = (int(x) for x in scores.shape)
    t_out = torch.empty(B, dtype=torch.int32, device=scores.device) if t_out is None else t_out
    _dev(t_out, "t_out", torch.int32, (B,))
    rc = lib().spec_window(_ptr(scores), B, K, int(policy), float(param), int(bool(pmin0)), int(t_cap), _ptr(t_out),
                           ctypes.c_void_p(_stream(stream)))
    _check("spec_window", rc)
    return t_out


def spec_accept_sampled(logits: torch.Tensor, draft_logits: torch.Tensor, drafts: torch.Tensor,
                        u_accept: torch.Tensor, u_sample: torch.Tensor, temperature: float = 1.0, top_k: int = 0,
                        top_p: float = 1.0, min_p: float = 0.0, j_out=None, token_out=None, keep_out=None,
                        dev_status=None, scratch: torch.Tensor | None = None, stream=None):
    """Sampled acceptance: logits [B][T][V], draft_logits [B][T-1][V] (same dtype), drafts
    int32 [B][T-1], u_accept f32 [B][T-1], u_sample f32 [B].  Returns (j, token, keep)."""
    _dev(logits, "logits")
    B, T, V = (int(x) for x in logits.shape)
    _dev(draft_logits, "draft_logits", logits.dtype, (B, T - 1, V))
    _dev(drafts, "drafts", torch.int32, (B, T - 1))
    _dev(u_accept, "u_accept", torch.float32, (B, T - 1))
    _dev(u_sample, "u_sample", torch.float32, (B,))
    dev = logits.device
    j_out = torch.empty(B, dtype=torch.int32, device=dev) if j_out is None else j_out
    token_out = torch.empty(B, dtype=torch.int32, device=dev) if token_out is None else token_out
    keep_out = torch.empty(B, dtype=torch.int32, device=dev) if keep_out is None else keep_out
    sp = KdaSampling(float(temperature), int(top_k), float(top_p), float(min_p))
    need = int(lib().spec_accept_sampled_scratch_bytes(B, T))
    if scratch is None:
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib().spec_accept_sampled(_ptr(logits), _ptr(draft_logits), _row_dtype(logits), B, T, V, _ptr(drafts),
                                   _ptr(u_accept), _ptr(u_sample), ctypes.byref(sp), _ptr(j_out), _ptr(token_out),
                                   _ptr(keep_out), _ptr(dev_status), _ptr(scratch),
                                   scratch.numel() * scratch.element_size(), ctypes.c_void_p(_stream(stream)))
    _check("spec_accept_sampled", rc)
    return j_out, token_out, keep_out


def spec_accept_sampled_session(logits: torch.Tensor, draft_logits: torch.Tensor, drafts: torch.Tensor,
                                seeds: torch.Tensor, counters: torch.Tensor, temperature: float = 1.0, top_k: int = 0,
                                top_p: float = 1.0, min_p: float = 0.0, j_out=None, token_out=None, keep_out=None,
                                dev_status=None, scratch: torch.Tensor | None = None, stream=None):
    """Sampled acceptance drawing from each session's Philox stream: seeds int64 [B] (the
    64-bit key, two's complement), counters int32 [B][2] (uctr, sctr; advanced in place on
    the device).  Other arguments as spec_accept_sampled.  Returns (j, token, keep)."""
    _dev(logits, "logits")
    B, T, V = (int(x) for x in logits.shape)
    _dev(draft_logits, "draft_logits", logits.dtype, (B, T - 1, V))
    _dev(drafts, "drafts", torch.int32, (B, T - 1))
    _dev(seeds, "seeds", torch.int64, (B,))
    _dev(counters, "counters", torch.int32, (B, 2))
    dev = logits.device
    j_out = torch.empty(B, dtype=torch.int32, device=dev) if j_out is None else j_out
    token_out = torch.empty(B, dtype=torch.int32, device=dev) if token_out is None else token_out
    keep_out = torch.empty(B, dtype=torch.int32, device=dev) if keep_out is None else keep_out
    sp = KdaSampling(float(temperature), int(top_k), float(top_p), float(min_p))
    need = int(lib().spec_accept_sampled_scratch_bytes(B, T))
    if scratch is None:
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    rc = lib().spec_accept_sampled_session(_ptr(logits), _ptr(draft_logits), _row_dtype(logits), B, T, V,
                                           _ptr(drafts), _ptr(seeds), _ptr(counters), ctypes.byref(sp), _ptr(j_out),
                                           _ptr(token_out), _ptr(keep_out), _ptr(dev_status), _ptr(scratch),
                                           scratch.numel() * scratch.element_size(), ctypes.c_void_p(_stream(stream)))
    _check("spec_accept_sampled_session", rc)
    return j_out, token_out, keep_out


def philox4x32_10(ctr: torch.Tensor, key: torch.Tensor, stream=None) -> torch.Tensor:
    """The library's Philox4x32-10 on the device: ctr int32 [n][4] and key int32 [n][2] (the
    uint32 bit patterns); returns int32 [n][4]."""
    n = int(ctr.shape[0])
    _dev(ctr, "ctr", torch.int32, (n, 4))
    _dev(key, "key", torch.int32, (n, 2))
    out = torch.empty((n, 4), dtype=torch.int32, device=ctr.device)
    rc = lib().kda_philox4x32_10(_ptr(ctr), _ptr(key), _ptr(out), n, ctypes.c_void_p(_stream(stream)))
    _check("kda_philox4x32_10", rc)
    return out


def spec_accept_scratch_bytes(B: int, T: int, V: int) -> int:
    return int(lib().spec_accept_scratch_bytes(B, T, V))


def spec_accept(logits: torch.Tensor, drafts: torch.Tensor, j_out=None, bonus_out=None, keep_out=None,
                dev_status=None, scratch: torch.Tensor | None = None, stream=None):
    """Greedy accept for B sessions: logits [B][T][V] (f32/bf16), drafts int32 [B][T-1].

    Returns (j_out, bonus_out, keep_out) device int32 tensors [B] (allocated here
    by torch when not given).
    """
    _dev(logits, "logits")
    B, T, V = (int(x) for x in logits.shape)
    _dev(drafts, "drafts", torch.int32, (B, T - 1))
    dev = logits.device
    j_out = torch.empty(B, dtype=torch.int32, device=dev) if j_out is None else j_out
    bonus_out = torch.empty(B, dtype=torch.int32, device=dev) if bonus_out is None else bonus_out
    keep_out = torch.empty(B, dtype=torch.int32, device=dev) if keep_out is None else keep_out
    nb = 0 if scratch is None else scratch.numel() * scratch.element_size()  # not used by the library
    rc = lib().spec_accept(_ptr(logits), _row_dtype(logits), B, T, V, _ptr(drafts), _ptr(j_out),
                           _ptr(bonus_out), _ptr(keep_out), _ptr(dev_status), _ptr(scratch), nb,
                           ctypes.c_void_p(_stream(stream)))
    _check("spec_accept", rc)
    return j_out, bonus_out, keep_out


class RoundPlan:
    """Pre-marshalled arguments of one verify round, for calling it many times.

    Holds the ctypes argument tuples of kda_verify_scan, spec_accept and
    kda_rollback (device keep from spec_accept's keep_out) for fixed tensors, so
    each call is one foreign call with no per-call marshalling.  The tensors are
    referenced and must keep their storage while the plan is used.  ``rows`` holds
    q, k, v, g, beta and optionally w (the update vectors; see _rows), in which case
    the verify writes them and the replay reads them.
    """

    def __init__(self, st: LayerState, rows: dict, out, stash: Stash, logits, drafts, j_out, bonus_out,
                 keep_out, dev_status, scratch, stream=None):
        L = lib()
        self._keep = (st, rows, out, stash, logits, drafts, j_out, bonus_out, keep_out, dev_status, scratch)
        crows, tensors, dt, T = _rows(st, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], w=rows.get("w"))
        B, Tl, V = (int(x) for x in logits.shape)
        if Tl != T or B != st.B:
            raise ValueError("logits must be [B][T][V] of the round")
        _dev(drafts, "drafts", torch.int32, (B, T - 1))
        for name, t in (("j_out", j_out), ("bonus_out", bonus_out), ("keep_out", keep_out)):
            _dev(t, name, torch.int32, (B,))
        if out is not None:
            _dev(out, "out", torch.float32, (st.L, st.B, T, st.H, D))
        self.dims, self.cst, self.crows = st.dims(dt), st.c(), crows
        s = ctypes.c_void_p(_stream(stream))
        self._verify = (ctypes.byref(self.dims), ctypes.byref(self.cst), ctypes.byref(self.crows), T,
                        _ptr(out), ctypes.byref(stash.c), s)
        nbytes = scratch.numel() * scratch.element_size()
        self._accept = (_ptr(logits), _row_dtype(logits), B, T, V, _ptr(drafts), _ptr(j_out), _ptr(bonus_out),
                        _ptr(keep_out), _ptr(dev_status), _ptr(scratch), nbytes, s)
        self._rollback = (ctypes.byref(self.dims), ctypes.byref(self.cst), ctypes.byref(stash.c),
                          _ptr(keep_out), MEM_DEVICE, _ptr(dev_status), s)
        self._stash, self._tensors, self._dt = stash, tensors, dt
        self._L = L
        self.stream = stream if isinstance(stream, torch.cuda.Stream) else None
        self.graph = None

    def verify(self):
        rc = self._L.kda_verify_scan(*self._verify)
        if rc:
            _check("kda_verify_scan", rc)
        self._stash.rows, self._stash.dtype = self._tensors, self._dt

    def accept(self):
        rc = self._L.spec_accept(*self._accept)
        if rc:
            _check("spec_accept", rc)

    def rollback(self):
        rc = self._L.kda_rollback(*self._rollback)
        if rc:
            _check("kda_rollback", rc)

    def __call__(self):
        self.verify()
        self.accept()
        self.rollback()

    def capture(self):
        """Capture one round (verify, accept, rollback) into a CUDA graph on the plan's
        side stream (a torch.cuda.Stream other than the default one).  Run the round
        eagerly once before, so every one-time setup call has happened."""
        if self.stream is None:
            raise ValueError("capture needs a plan built on a side torch.cuda.Stream")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self()
        return self.graph

    def replay(self):
        self.graph.replay()


class PingPongRoundPlan:
    """RoundPlan for ping-pong rounds: kda_verify_scan_pingpong, spec_accept and
    kda_rollback (device keep) with their arguments marshalled once for each parity
    of the shared PingPong buffers.  Each call runs the round at the buffers' current
    parity and flips it.  ``capture()`` records one CUDA graph per parity; ``replay()``
    replays the one of the current parity and flips it.
    """

    def __init__(self, pp: PingPong, rows: dict, out, logits, drafts, j_out, bonus_out, keep_out, dev_status,
                 scratch, stream=None):
        self._keep = (pp, rows, out, logits, drafts, j_out, bonus_out, keep_out, dev_status, scratch)
        self.pp = pp
        shape_ref = LayerState(pp.states[0], pp.rings[0], pp.conv_w)
        crows, tensors, dt, T = _rows(shape_ref, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"],
                                      w=rows.get("w"))
        B, Tl, V = (int(x) for x in logits.shape)
        if Tl != T or B != pp.B:
            raise ValueError("logits must be [B][T][V] of the round")
        _dev(drafts, "drafts", torch.int32, (B, T - 1))
        for name, t in (("j_out", j_out), ("bonus_out", bonus_out), ("keep_out", keep_out)):
            _dev(t, name, torch.int32, (B,))
        if out is not None:
            _dev(out, "out", torch.float32, (pp.L, pp.B, T, pp.H, D))
        self.dims, self.crows = pp.dims(dt), crows
        # per-parity copies of the structs: the library records the rows in the stash
        self.cst = [KdaLayerState(c.state, c.conv_ring, c.conv_w) for c in pp.cst]
        self.cstash = [KdaStashC(c.state_snap, c.ring_snap, KdaRows(), 0) for c in pp.cstash]
        s = ctypes.c_void_p(_stream(stream))
        self._verify = [(ctypes.byref(self.dims), ctypes.byref(self.cst[p]), ctypes.byref(self.crows), T, None,
                         MEM_HOST, _ptr(out), ctypes.byref(self.cstash[p]), _ptr(dev_status), s) for p in (0, 1)]
        nbytes = scratch.numel() * scratch.element_size()
        self._accept = (_ptr(logits), _row_dtype(logits), B, T, V, _ptr(drafts), _ptr(j_out), _ptr(bonus_out),
                        _ptr(keep_out), _ptr(dev_status), _ptr(scratch), nbytes, s)
        self._rollback = [(ctypes.byref(self.dims), ctypes.byref(self.cst[p]), ctypes.byref(self.cstash[p]),
                           _ptr(keep_out), MEM_DEVICE, _ptr(dev_status), s) for p in (0, 1)]
        self._tensors, self._dt = tensors, dt
        self._L = lib()
        self.stream = stream if isinstance(stream, torch.cuda.Stream) else None
        self.graphs = None

    def verify(self, p: int):
        rc = self._L.kda_verify_scan_pingpong(*self._verify[p])
        if rc:
            _check("kda_verify_scan_pingpong", rc)

    def accept(self):
        rc = self._L.spec_accept(*self._accept)
        if rc:
            _check("spec_accept", rc)

    def rollback(self, p: int):
        rc = self._L.kda_rollback(*self._rollback[p])
        if rc:
            _check("kda_rollback", rc)

    def _flip(self, p: int):
        pp = self.pp
        pp.rows, pp.dtype, pp.last, pp.parity = self._tensors, self._dt, p, 1 - p
        pp.cstash[p].rows, pp.cstash[p].T = self.crows, self.cstash[p].T

    def __call__(self):
        p = self.pp.parity
        self.verify(p)
        self.accept()
        self.rollback(p)
        self._flip(p)

    def capture(self):
        """Capture the round at each parity into a CUDA graph on the plan's side stream.
        Run the round eagerly at both parities before, so every one-time setup call has
        happened."""
        if self.stream is None:
            raise ValueError("capture needs a plan built on a side torch.cuda.Stream")
        self.graphs = []
        for p in (0, 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.verify(p)
                self.accept()
                self.rollback(p)
            self.graphs.append(g)
        return self.graphs

    def replay(self):
        p = self.pp.parity
        self.graphs[p].replay()
        self._flip(p)


class DeferredRoundPlan:
    """A round whose rollback is deferred into the next round's verify: one call runs
    kda_verify_scan_deferred (committing the previous round with the device keep_out
    that the previous round's spec_accept left) and then spec_accept of this round.
    The previous round must be a ping-pong round (or a deferred one) of the same
    PingPong buffers whose keep is in keep_out.  Arguments as for PingPongRoundPlan.
    """

    def __init__(self, pp: PingPong, rows: dict, out, logits, drafts, j_out, bonus_out, keep_out, dev_status,
                 scratch, stream=None, ready_flags=None, pairs_per_flag: int = 1):
        self._keep = (pp, rows, out, logits, drafts, j_out, bonus_out, keep_out, dev_status, scratch, ready_flags)
        self.pp = pp
        shape_ref = LayerState(pp.states[0], pp.rings[0], pp.conv_w)
        crows, tensors, dt, T = _rows(shape_ref, rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"],
                                      w=rows.get("w"))
        B, Tl, V = (int(x) for x in logits.shape)
        if Tl != T or B != pp.B:
            raise ValueError("logits must be [B][T][V] of the round")
        _dev(drafts, "drafts", torch.int32, (B, T - 1))
        for name, t in (("j_out", j_out), ("bonus_out", bonus_out), ("keep_out", keep_out)):
            _dev(t, name, torch.int32, (B,))
        if out is not None:
            _dev(out, "out", torch.float32, (pp.L, pp.B, T, pp.H, D))
        self.dims, self.crows, self.T = pp.dims(dt), crows, T
        w = pp.conv_w.data_ptr()
        # for the previous round's snapshot in buffer p: st is buffer 1 - p, the stash buffer p
        self.cst = [KdaLayerState(pp.states[1 - p].data_ptr(), pp.rings[1 - p].data_ptr(), w) for p in (0, 1)]
        self.cstash = [KdaStashC(pp.states[p].data_ptr(), pp.rings[p].data_ptr(), KdaRows(), 0) for p in (0, 1)]
        s = ctypes.c_void_p(_stream(stream))
        self._verify = [(ctypes.byref(self.dims), ctypes.byref(self.cst[p]), ctypes.byref(self.cstash[p]),
                         _ptr(keep_out), ctypes.byref(self.crows), T, _ptr(out), _ptr(dev_status), s) for p in (0, 1)]
        # staged raw rows (kda_verify_scan_deferred_staged): the epoch is given per call
        self._staged = None
        if ready_flags is not None:
            _dev(ready_flags, "ready_flags", torch.int32, (staged_flag_count(pp.L, pp.B, pairs_per_flag),))
            self._staged = [(ctypes.byref(self.dims), ctypes.byref(self.cst[p]), ctypes.byref(self.cstash[p]),
                             _ptr(keep_out), ctypes.byref(self.crows), T, _ptr(out), _ptr(ready_flags),
                             int(pairs_per_flag)) for p in (0, 1)]
            self._staged_tail = (_ptr(dev_status), s)
        nbytes = scratch.numel() * scratch.element_size()
        self._accept = (_ptr(logits), _row_dtype(logits), B, T, V, _ptr(drafts), _ptr(j_out), _ptr(bonus_out),
                        _ptr(keep_out), _ptr(dev_status), _ptr(scratch), nbytes, s)
        self._tensors, self._dt = tensors, dt
        self._L = lib()

    def verify(self, p: int, epoch: int | None = None):
        """The deferred verify launch; with staged rows (ready_flags given) ``epoch`` is
        the flag value that marks this call's rows as in place."""
        pp = self.pp
        prev = pp.cstash[p]
        # the library swaps the pointers in the structs it is given: restore them
        c, st = self.cst[p], self.cstash[p]
        c.state, c.conv_ring = pp.states[1 - p].data_ptr(), pp.rings[1 - p].data_ptr()
        st.state_snap, st.ring_snap = pp.states[p].data_ptr(), pp.rings[p].data_ptr()
        st.rows, st.T = prev.rows, prev.T
        if self._staged is not None:
            if epoch is None:
                raise ValueError("a plan with staged rows needs the call's epoch")
            rc = self._L.kda_verify_scan_deferred_staged(*self._staged[p], ctypes.c_uint(epoch & 0xffffffff),
                                                         *self._staged_tail)
            if rc:
                _check("kda_verify_scan_deferred_staged", rc)
            return
        rc = self._L.kda_verify_scan_deferred(*self._verify[p])
        if rc:
            _check("kda_verify_scan_deferred", rc)

    def accept(self):
        rc = self._L.spec_accept(*self._accept)
        if rc:
            _check("spec_accept", rc)

    def _flip(self, p: int):
        pp = self.pp
        pp.cstash[1 - p].rows, pp.cstash[1 - p].T = self.crows, self.T
        pp.rows, pp.dtype, pp.last, pp.parity = self._tensors, self._dt, 1 - p, p

    def __call__(self):
        p = self.pp.last
        if p is None:
            raise ValueError("a deferred round follows a ping-pong round")
        self.verify(p)
        self.accept()
        self._flip(p)


class LayerDeferredRoundPlan:
    """A deferred round issued the way a model issues it: one kda_verify_scan_deferred
    per layer (each over that layer's views of the PingPong buffers and raw rows, in
    layer order), then one spec_accept.  Each layer commits its own part of the
    previous round.  ``layers`` are the PingPong views of ``pp`` made by
    ``layer_pingpongs(pp, bounds)`` and shared by every plan of the sequence (one view a
    layer by default; ``bounds`` groups consecutive layers into one launch); the
    results are bit-identical to DeferredRoundPlan over all layers.
    """

    def __init__(self, pp: PingPong, layers: list, rows: dict, out, logits, drafts, j_out, bonus_out, keep_out,
                 dev_status, scratch, stream=None, bounds=None):
        bounds = layer_bounds(pp.L, bounds)
        if len(bounds) != len(layers):
            raise ValueError("one PingPong view per layer range")
        self.pp, self.layers = pp, layers
        self.full = DeferredRoundPlan(pp, rows, out, logits, drafts, j_out, bonus_out, keep_out, dev_status, scratch,
                                      stream)
        self.plans = []
        for (l0, l1), lp in zip(bounds, layers):
            rl = {n: t[l0:l1] for n, t in rows.items()}
            self.plans.append(DeferredRoundPlan(lp, rl, None if out is None else out[l0:l1], logits, drafts, j_out,
                                                bonus_out, keep_out, dev_status, scratch, stream))

    def __call__(self):
        p = self.pp.last
        if p is None:
            raise ValueError("a deferred round follows a ping-pong round")
        for lp, plan in zip(self.layers, self.plans):
            plan.verify(p)
            plan._flip(p)
        self.full.accept()
        self.full._flip(p)


def layer_bounds(L: int, bounds=None) -> list:
    """[(l0, l1), ...]: consecutive layer ranges covering 0..L-1, one a layer by default;
    an int n splits the layers into n ranges of near-equal length."""
    if bounds is None:
        return [(l, l + 1) for l in range(L)]
    if isinstance(bounds, int):
        n = max(1, min(bounds, L))
        edges = [L * i // n for i in range(n + 1)]
        return [(edges[i], edges[i + 1]) for i in range(n)]
    bounds = [(int(a), int(b)) for a, b in bounds]
    if not bounds or bounds[0][0] != 0 or bounds[-1][1] != L or any(
            b0[1] != b1[0] for b0, b1 in zip(bounds, bounds[1:])) or any(a >= b for a, b in bounds):
        raise ValueError("layer ranges must be consecutive, non-empty and cover 0..L-1")
    return bounds


def layer_pingpongs(pp: PingPong, bounds=None) -> list:
    """PingPong views of pp's buffers over consecutive layer ranges (``layer_bounds``:
    one view a layer by default; layer-major, so each is contiguous), with pp's parity
    and last round.  For LayerDeferredRoundPlan and per-range deferred rounds; the last
    round must be recorded in pp by a ping-pong or deferred round over all layers."""
    out = []
    for l0, l1 in layer_bounds(pp.L, bounds):
        st = LayerState(pp.states[0][l0:l1], pp.rings[0][l0:l1], pp.conv_w[l0:l1])
        lp = PingPong(st, spare_state=pp.states[1][l0:l1], spare_ring=pp.rings[1][l0:l1])
        lp.parity, lp.last, lp.dtype = pp.parity, pp.last, pp.dtype
        if pp.last is not None:
            full = pp.cstash[pp.last]
            rows = {n: t[l0:l1] for n, t in zip(("q", "k", "v", "g", "beta", "w"), pp.rows)} if pp.rows else None
            if rows is not None:
                names = ("q", "k", "v", "g", "beta", "w") if "w" in rows else ("q", "k", "v", "g", "beta")
                lp.rows = [rows[n] for n in names]
                lp.cstash[pp.last].rows = KdaRows(*(rows[n].data_ptr() for n in names))
                lp.cstash[pp.last].T = full.T
        out.append(lp)
    return out


class LayerRoundPlan:
    """One verify round issued the way a model issues it: one kda_verify_scan per layer
    (each over that layer's views, in layer order), then spec_accept, then one
    kda_rollback over all layers from the snapshots the per-layer calls wrote.

    Same arguments as RoundPlan; the results are bit-identical to it.  A plan built on
    a side stream (a torch.cuda.Stream other than the default one) can capture its round
    into a CUDA graph with ``capture()`` and replay it with ``replay()``: the library
    allocates nothing and never synchronises, so the captured launches are the eager ones.
    """

    def __init__(self, st: LayerState, rows: dict, out, stash: Stash, logits, drafts, j_out, bonus_out,
                 keep_out, dev_status, scratch, stream=None):
        self.full = RoundPlan(st, rows, out, stash, logits, drafts, j_out, bonus_out, keep_out, dev_status,
                              scratch, stream)
        self.layers = []
        self._views = []
        for l in range(st.L):
            stl, stashl = st.layer(l), stash.layer(l)
            rl = {n: t[l:l + 1] for n, t in rows.items()}
            outl = None if out is None else out[l:l + 1]
            crows, tensors, dt, T = _rows(stl, rl["q"], rl["k"], rl["v"], rl["g"], rl["beta"], w=rl.get("w"))
            dims, cst = stl.dims(dt), stl.c()
            self._views.append((stl, stashl, rl, outl, crows, dims, cst, tensors))
            self.layers.append((ctypes.byref(dims), ctypes.byref(cst), ctypes.byref(crows), T, _ptr(outl),
                                ctypes.byref(stashl.c), ctypes.c_void_p(_stream(stream))))
        self.stream = stream if isinstance(stream, torch.cuda.Stream) else None
        self.graph = None

    def verify(self):
        L = self.full._L
        for args in self.layers:
            rc = L.kda_verify_scan(*args)
            if rc:
                _check("kda_verify_scan", rc)
        # the all-layer stash now describes this round: its snapshots were written by
        # the per-layer calls, its rows are the round's full raw-row tensors
        f = self.full
        f._stash.c.rows, f._stash.c.T = f.crows, self.layers[0][3]
        f._stash.rows, f._stash.dtype = f._tensors, f._dt

    def accept(self):
        self.full.accept()

    def rollback(self):
        self.full.rollback()

    def __call__(self):
        self.verify()
        self.accept()
        self.rollback()

    def capture(self):
        """Capture one round (all launches) into a CUDA graph on the plan's side stream.
        Run the round eagerly once before, so every one-time setup call has happened."""
        if self.stream is None:
            raise ValueError("capture needs a plan built on a side torch.cuda.Stream")
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self()
        return self.graph

    def replay(self):
        self.graph.replay()


class HostRounds:
    """A chain of speculative rounds driven from host memory, one kda_round_host call a
    round: the round's raw rows, logits and drafts go up from pinned host tensors, the
    verify folds in the previous round's accept, the accept runs and j and the bonus
    come back.

    st: the committed state and ring (and conv weights); spare_state / spare_ring: the
    second buffer pair (allocated here when None).  dev_sets: two dicts of device
    tensors, each with q, k, v, g, beta (optionally w), logits [B][T][V] and drafts
    int32 [B][T-1]; the rounds alternate between them.  The per-round host inputs are
    dicts of pinned CPU tensors with the same keys (w excepted).  pairs_per_flag: the
    (layer, session) pairs of a staged range (default: four ranges).  in_place: after the
    first round the verify reads the raw rows in place from the host tensors (they must
    be addressable by the device) and leaves their copy in the device set.  ``commit()`` applies
    the last round's accept; ``state()`` / ``ring()`` are then the committed tensors.
    """

    def __init__(self, st: LayerState, dev_sets: list, out=None, ready_flags=None, pairs_per_flag: int | None = None,
                 dev_status=None, stream=None, copy_stream=None, spare_state=None, spare_ring=None,
                 in_place: bool = False):
        if len(dev_sets) != 2:
            raise ValueError("two device input sets alternate")
        self.L, self.B, self.H = st.L, st.B, st.H
        spare_state = torch.empty_like(st.state) if spare_state is None else spare_state
        spare_ring = torch.empty_like(st.conv_ring) if spare_ring is None else spare_ring
        _dev(spare_state, "spare_state", torch.float32, tuple(st.state.shape))
        _dev(spare_ring, "spare_ring", torch.float32, tuple(st.conv_ring.shape))
        self._bufs = {st.state.data_ptr(): st.state, spare_state.data_ptr(): spare_state,
                      st.conv_ring.data_ptr(): st.conv_ring, spare_ring.data_ptr(): spare_ring}
        # the first round reads the committed pair from the stash's buffers
        self.cst = KdaLayerState(spare_state.data_ptr(), spare_ring.data_ptr(), st.conv_w.data_ptr())
        self.cstash = KdaStashC(st.state.data_ptr(), st.conv_ring.data_ptr(), KdaRows(), 0)
        q0 = dev_sets[0]["q"]
        self.T = int(q0.shape[2])
        self.dt = _row_dtype(q0)
        self.dims = KdaDims(self.L, self.B, self.H, D, D, self.dt)
        self.sets, self.crows = [], []
        for ds in dev_sets:
            crows, tensors, _, T = _rows(st, ds["q"], ds["k"], ds["v"], ds["g"], ds["beta"], w=ds.get("w"))
            lg, dr = ds["logits"], ds["drafts"]
            _dev(lg, "logits")
            if lg.dim() != 3 or int(lg.shape[0]) != self.B or int(lg.shape[1]) != self.T:
                raise ValueError("logits must be [B][T][V] of the round")
            _dev(dr, "drafts", torch.int32, (self.B, self.T - 1))
            self.sets.append((crows, tensors, lg, dr))
        self.V = int(dev_sets[0]["logits"].shape[2])
        self.ldt = _row_dtype(dev_sets[0]["logits"])
        self.jbk = torch.zeros((3, self.B), dtype=torch.int32, device=q0.device)
        self.host_jb = torch.zeros((2, self.B), dtype=torch.int32).pin_memory()
        if out is not None:
            _dev(out, "out", torch.float32, (self.L, self.B, self.T, self.H, D))
        pairs = self.L * self.B
        if pairs_per_flag is None:  # four ranges (measured best of 1, 2, 4, 8 on stack34 and batched32)
            pairs_per_flag = max(1, -(-pairs // 4))
        if ready_flags is None:
            ready_flags = torch.zeros(staged_flag_count(self.L, self.B, pairs_per_flag), dtype=torch.int32,
                                   device=q0.device)
        _dev(ready_flags, "ready_flags", torch.int32, (staged_flag_count(self.L, self.B, pairs_per_flag),))
        self.out, self.flags, self.ppf, self.status = out, ready_flags, int(pairs_per_flag), dev_status
        self.stream = stream
        self.copy_stream = copy_stream if copy_stream is not None else torch.cuda.Stream(q0.device)
        self._hold = (st, spare_state, spare_ring, dev_sets, ready_flags, dev_status, out, pairs)
        self._host = {}
        self.epoch = 0
        self.rounds = 0
        self.in_place = bool(in_place)
        self._L = lib()

    def _host_rows(self, hs: dict):
        key = id(hs)
        if key not in self._host:
            names = ("q", "k", "v", "g", "beta")
            for n in names + ("logits", "drafts"):
                if hs[n].is_cuda or not hs[n].is_contiguous():
                    raise ValueError(f"host input {n} must be a contiguous CPU tensor (pinned)")
            self._host[key] = (KdaRows(*(hs[n].data_ptr() for n in names)), hs)
        return self._host[key][0]

    def __call__(self, hs: dict, wait: bool = True):
        """One round from the host inputs hs; returns (j, bonus) as host int32 tensors
        [B] (views of one pinned buffer, overwritten by the next round) when wait."""
        crows, _, lg, dr = self.sets[self.rounds % 2]
        hrows = self._host_rows(hs)
        self.epoch = (self.epoch + 1) & 0xffffffff
        rc = self._L.kda_round_host(ctypes.byref(self.dims), ctypes.byref(self.cst), ctypes.byref(self.cstash),
                                    self.T, ctypes.byref(hrows), ctypes.byref(crows), hs["logits"].data_ptr(),
                                    lg.data_ptr(), self.ldt, self.V, hs["drafts"].data_ptr(), dr.data_ptr(),
                                    self.jbk.data_ptr(), self.host_jb.data_ptr(), _ptr(self.out),
                                    self.flags.data_ptr(), self.ppf, ctypes.c_uint(self.epoch), _ptr(self.status),
                                    ctypes.c_void_p(_stream(self.stream)),
                                    ctypes.c_void_p(_stream(self.copy_stream)), 1 if self.in_place else 0,
                                    1 if wait else 0)
        if rc:
            _check("kda_round_host", rc)
        self.rounds += 1
        return (self.host_jb[0], self.host_jb[1]) if wait else None

    def commit(self):
        """Apply the last round's accept (kda_rollback with the device keep)."""
        if self.rounds == 0:
            return
        rc = self._L.kda_rollback(ctypes.byref(self.dims), ctypes.byref(self.cst), ctypes.byref(self.cstash),
                                  ctypes.c_void_p(self.jbk[2].data_ptr()), MEM_DEVICE, _ptr(self.status),
                                  ctypes.c_void_p(_stream(self.stream)))
        _check("kda_rollback", rc)

    def state(self):
        return self._bufs[self.cst.state]

    def ring(self):
        return self._bufs[self.cst.conv_ring]
