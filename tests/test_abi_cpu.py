"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
include/kda_spec.h declares, and rejects invalid calls on the host (KDA_EINVAL)
before anything touches a device.  No call here reaches a launch."""
import ctypes
import os
import re

import pytest

from libs import ROOT, ensure_built

from speculative_decode_verify_kda_gb300 import binding as kb

HEADER = os.path.join(ROOT, "include", "kda_spec.h")


@pytest.fixture(scope="module")
def L():
    ensure_built()
    return kb.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^(?:int|size_t|const char \*)\s*(\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == set(kb.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n
    assert L.kda_abi_version() == kb.ABI_VERSION
    assert L.kda_error_string(kb.EINVAL) == b"invalid argument"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation first


def _state(H=64, B=1, L_=1, dtype=kb.BF16, dk=128):
    return (kb.KdaDims(L_, B, H, dk, 128, dtype), kb.KdaLayerState(FAKE, FAKE, FAKE),
            kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE))


@pytest.mark.parametrize("case", ["T0", "T16", "dk64", "dtype", "null_state", "null_rows", "misaligned",
                                  "w_misaligned", "snap_alias", "snap_null", "negB"])
def test_verify_rejects_on_host(L, case):
    dims, st, rows = _state()
    T, stash = 8, None
    if case == "T0":
        T = 0
    elif case == "T16":
        T = 16
    elif case == "dk64":
        dims.dk = 64
    elif case == "dtype":
        dims.dtype = 7
    elif case == "null_state":
        st.state = None
    elif case == "null_rows":
        rows.v = None
    elif case == "misaligned":
        rows.q = FAKE + 2
    elif case == "w_misaligned":  # the update vectors are read as 16-byte vectors
        rows.w = FAKE + 4
    elif case == "snap_alias":
        stash = kb.KdaStashC(FAKE, FAKE + 0x100, kb.KdaRows(), 0)
    elif case == "snap_null":
        stash = kb.KdaStashC(None, FAKE, kb.KdaRows(), 0)
    elif case == "negB":
        dims.B = -1
    rc = L.kda_verify_scan(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), T, None,
                           ctypes.byref(stash) if stash is not None else None, None)
    assert rc == kb.EINVAL
    assert L.kda_last_error()  # a reason is recorded


@pytest.mark.parametrize("keep", [[0], [9], [-1]])
def test_rollback_rejects_bad_host_keep(L, keep):
    dims, st, rows = _state()
    stash = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, rows, 8)
    arr = (ctypes.c_int * 1)(*keep)
    rc = L.kda_rollback(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(stash),
                        ctypes.cast(arr, ctypes.c_void_p), kb.MEM_HOST, None, None)
    assert rc == kb.EINVAL
    assert b"outside 1..8" in L.kda_last_error()


def test_rollback_full_accept_host_keep_is_a_no_op(L):
    # keep == T for every session: nothing to restore, nothing launched, OK
    dims, st, rows = _state(B=3)
    stash = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, rows, 8)
    arr = (ctypes.c_int * 3)(8, 8, 8)
    assert L.kda_rollback(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(stash),
                          ctypes.cast(arr, ctypes.c_void_p), kb.MEM_HOST, None, None) == kb.OK


def test_rollback_rejects_missing_round_and_bad_mode(L):
    dims, st, rows = _state()
    arr = (ctypes.c_int * 1)(1)
    empty = kb.KdaStashC(FAKE, FAKE, rows, 0)
    assert L.kda_rollback(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(empty),
                          ctypes.cast(arr, ctypes.c_void_p), kb.MEM_HOST, None, None) == kb.EINVAL
    stash = kb.KdaStashC(FAKE, FAKE, rows, 4)
    assert L.kda_rollback(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(stash),
                          ctypes.cast(arr, ctypes.c_void_p), 5, None, None) == kb.EINVAL
    big = kb.KdaDims(1, kb.HOST_KEEP_MAX + 1, 64, 128, 128, kb.BF16)
    arr2 = (ctypes.c_int * (kb.HOST_KEEP_MAX + 1))(*([1] * (kb.HOST_KEEP_MAX + 1)))
    assert L.kda_rollback(ctypes.byref(big), ctypes.byref(st), ctypes.byref(stash),
                          ctypes.cast(arr2, ctypes.c_void_p), kb.MEM_HOST, None, None) == kb.EINVAL


def test_accept_rejects_on_host(L):
    need = L.spec_accept_scratch_bytes(2, 8, 32768)
    assert need == 2 * 8 * 8 * 16
    args = dict(logits=FAKE, dt=kb.BF16, B=2, T=8, V=32768, drafts=FAKE)

    def call(**kw):
        a = {**args, **kw}
        return L.spec_accept(a["logits"], a["dt"], a["B"], a["T"], a["V"], a["drafts"], None, None, None,
                             None, kw.get("scratch", FAKE), kw.get("nbytes", need), None)
    assert call(T=16) == kb.EINVAL
    assert call(T=0) == kb.EINVAL
    assert call(V=0) == kb.EINVAL
    assert call(dt=3) == kb.EINVAL
    assert call(logits=FAKE + 4) == kb.EINVAL
    assert call(drafts=None) == kb.EINVAL
    assert call(B=0) == kb.OK  # nothing to do


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        kb.lib(str(tmp_path / "libkda_spec.so"))


def test_var_entry_points_reject_on_host(L):
    dims, st, rows = _state(B=3)
    t = (ctypes.c_int * 3)(8, 9, 1)   # 9 > T
    assert L.kda_verify_scan_var(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), 8,
                                 ctypes.cast(t, ctypes.c_void_p), kb.MEM_HOST, None, None, None, None) == kb.EINVAL
    assert b"outside 1..8" in L.kda_last_error()
    assert L.kda_verify_scan_var(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), 8, None, kb.MEM_HOST,
                                 None, None, None, None) == kb.EINVAL
    t_ok = (ctypes.c_int * 3)(8, 5, 1)
    assert L.kda_verify_scan_var(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), 8,
                                 ctypes.cast(t_ok, ctypes.c_void_p), 7, None, None, None, None) == kb.EINVAL
    stash = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, rows, 8)
    keep = (ctypes.c_int * 3)(8, 6, 1)   # keep 6 > t_rows 5
    assert L.kda_rollback_var(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(stash),
                              ctypes.cast(t_ok, ctypes.c_void_p), ctypes.cast(keep, ctypes.c_void_p), kb.MEM_HOST,
                              None, None) == kb.EINVAL
    assert b"outside 1..5" in L.kda_last_error()
    # every session keeps all of its own rows: nothing launched
    full = (ctypes.c_int * 3)(8, 5, 1)
    assert L.kda_rollback_var(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(stash),
                              ctypes.cast(t_ok, ctypes.c_void_p), ctypes.cast(full, ctypes.c_void_p), kb.MEM_HOST,
                              None, None) == kb.OK


def test_window_and_accept_var_reject_on_host(L):
    assert L.spec_window(FAKE, 4, 7, 3, 0.5, 0, 8, FAKE, None) == kb.EINVAL           # unknown policy
    assert L.spec_window(FAKE, 4, 7, kb.WIN_CONFIDENCE, 0.5, 0, 1, FAKE, None) == kb.EINVAL  # cap below 2
    assert L.spec_window(FAKE, 4, 7, kb.WIN_CONF_KEEP, 0.5, 0, 16, FAKE, None) == kb.EINVAL  # cap above 15
    assert L.spec_window(FAKE, 4, 7, kb.WIN_CONF_KEEP, float("nan"), 0, 8, FAKE, None) == kb.EINVAL
    assert L.spec_window(None, 0, 7, kb.WIN_CONF_KEEP, 0.5, 0, 8, None, None) == kb.OK   # nothing to do
    need = L.spec_accept_scratch_bytes(2, 8, 1000)
    assert L.spec_accept_var(FAKE, kb.BF16, 2, 8, 1000, None, FAKE, None, None, None, None, FAKE, need,
                             None) == kb.EINVAL
    assert L.spec_accept_var(FAKE, kb.BF16, 2, 8, 1000, FAKE + 2, FAKE, None, None, None, None, FAKE, need,
                             None) == kb.EINVAL


@pytest.mark.parametrize("sp", [(0.0, 0, 1.0, 0.0), (1.0, -1, 1.0, 0.0), (1.0, 10, 0.0, 0.0), (1.0, 10, 1.5, 0.0),
                                (1.0, 0, 1.0, 1.0), (float("inf"), 0, 1.0, 0.0), (float("nan"), 0, 1.0, 0.0),
                                (1.0, 0, float("nan"), 0.0), (1.0, 0, 1.0, -0.1)])
def test_sampled_accept_rejects_bad_parameters(L, sp):
    s = kb.KdaSampling(*sp)
    rc = L.spec_accept_sampled(FAKE, FAKE, kb.BF16, 2, 8, 1000, FAKE, FAKE, FAKE, ctypes.byref(s), FAKE, FAKE, None,
                               None, FAKE, 1 << 20, None)
    assert rc == kb.EINVAL and L.kda_last_error()


def test_sampled_accept_rejects_bad_shapes_and_pointers(L):
    s = kb.KdaSampling(1.0, 50, 0.9, 0.0)
    call = lambda **k: L.spec_accept_sampled(k.get("lg", FAKE), FAKE, k.get("dt", kb.BF16), k.get("B", 2),
                                             k.get("T", 8), k.get("V", 1000), FAKE, FAKE, k.get("us", FAKE),
                                             ctypes.byref(s), FAKE, FAKE, None, None, k.get("scr", FAKE),
                                             k.get("nb", 1 << 20), None)
    assert call(T=0) == kb.EINVAL and call(T=16) == kb.EINVAL and call(V=0) == kb.EINVAL
    # the fixed-point sums of V weights of at most 1 (units of 2^-46) must fit 64 bits
    assert call(V=2**18) == kb.EINVAL and call(V=2**18 - 1, B=0) == kb.OK
    assert call(dt=9) == kb.EINVAL and call(us=None) == kb.EINVAL and call(lg=FAKE + 1) == kb.EINVAL
    assert call(scr=None) == kb.EINVAL and call(scr=FAKE + 8) == kb.EINVAL
    assert L.spec_accept_sampled_scratch_bytes(2, 8) == 2 * 15 * 32
    assert call(nb=2 * 15 * 32 - 1) == kb.EINVAL
    assert call(B=0) == kb.OK
    assert L.spec_accept_sampled(FAKE, FAKE, kb.BF16, 2, 8, 1000, FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None,
                                 FAKE, 1 << 20, None) == kb.EINVAL


def test_sampled_filters_need_no_top_k():
    """top_p alone and any top_k >= 1 are valid filters (checked on the host before launch: with
    B = 0 nothing is launched and the call succeeds)."""
    L = kb.lib()
    for sp in ((1.0, 0, 0.9, 0.0), (1.0, 100000, 1.0, 0.0), (0.7, 0, 0.5, 0.05)):
        s = kb.KdaSampling(*sp)
        assert L.spec_accept_sampled(FAKE, FAKE, kb.BF16, 0, 8, 1000, FAKE, FAKE, FAKE, ctypes.byref(s), FAKE, FAKE,
                                     None, None, FAKE, 1 << 20, None) == kb.OK


def test_sampled_session_rejects_on_host(L):
    s = kb.KdaSampling(1.0, 50, 0.9, 0.0)
    call = lambda **k: L.spec_accept_sampled_session(FAKE, FAKE, kb.BF16, k.get("B", 2), 8, 1000, FAKE,
                                                     k.get("seeds", FAKE), k.get("ctr", FAKE), ctypes.byref(s), FAKE,
                                                     FAKE, None, None, FAKE, 1 << 20, None)
    assert call(seeds=None) == kb.EINVAL and call(ctr=None) == kb.EINVAL
    assert call(seeds=FAKE + 4) == kb.EINVAL and call(ctr=FAKE + 4) == kb.EINVAL
    assert call(B=0) == kb.OK


def test_philox_rejects_on_host(L):
    assert L.kda_philox4x32_10(FAKE, FAKE, FAKE, -1, None) == kb.EINVAL
    assert L.kda_philox4x32_10(None, FAKE, FAKE, 4, None) == kb.EINVAL
    assert L.kda_philox4x32_10(FAKE + 8, FAKE, FAKE, 4, None) == kb.EINVAL
    assert L.kda_philox4x32_10(FAKE, FAKE + 4, FAKE, 4, None) == kb.EINVAL
    assert L.kda_philox4x32_10(None, None, None, 0, None) == kb.OK


def test_cols_entry_points_reject_on_host(L):
    dims, st, rows = _state(B=2)
    assert L.kda_verify_scan_cols(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), 8, None, None, FAKE,
                                  None) == kb.EINVAL
    assert L.kda_verify_scan_cols(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), 8, None, FAKE + 4, FAKE,
                                  None) == kb.EINVAL
    assert L.kda_verify_scan_cols(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), 16, None, FAKE, FAKE,
                                  None) == kb.EINVAL
    keep = (ctypes.c_int * 2)(3, 9)
    assert L.kda_rollback_cols(ctypes.byref(dims), ctypes.byref(st), FAKE, FAKE, 8, ctypes.cast(keep, ctypes.c_void_p),
                               kb.MEM_HOST, None, None) == kb.EINVAL
    full = (ctypes.c_int * 2)(8, 8)
    assert L.kda_rollback_cols(ctypes.byref(dims), ctypes.byref(st), FAKE, FAKE, 8, ctypes.cast(full, ctypes.c_void_p),
                               kb.MEM_HOST, None, None) == kb.OK


def test_pingpong_rejects_on_host(L):
    dims, st, rows = _state(B=2)

    def call(stash, T=8, t=None, mem=kb.MEM_HOST):
        return L.kda_verify_scan_pingpong(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(rows), T,
                                          ctypes.cast(t, ctypes.c_void_p) if t is not None else None, mem, None,
                                          ctypes.byref(stash) if stash is not None else None, None, None)
    good = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(), 0)
    assert call(None) == kb.EINVAL  # the stash holds the pre-round state: required
    assert b"pre-round" in L.kda_last_error()
    assert call(kb.KdaStashC(FAKE, FAKE + 0x2000, kb.KdaRows(), 0)) == kb.EINVAL  # state buffers alias
    assert call(kb.KdaStashC(None, FAKE + 0x2000, kb.KdaRows(), 0)) == kb.EINVAL
    assert call(good, T=16) == kb.EINVAL
    bad_t = (ctypes.c_int * 2)(8, 0)
    assert call(good, t=bad_t) == kb.EINVAL
    assert call(good, t=(ctypes.c_int * 2)(8, 8), mem=9) == kb.EINVAL
    empty = kb.KdaDims(0, 2, 64, 128, 128, kb.BF16)
    assert L.kda_verify_scan_pingpong(ctypes.byref(empty), ctypes.byref(st), ctypes.byref(rows), 8, None,
                                      kb.MEM_HOST, None, ctypes.byref(good), None, None) == kb.OK


def test_deferred_rejects_on_host(L):
    dims, st, rows = _state(B=2)

    def call(stash, keep=FAKE + 0x3000, T=8):
        return L.kda_verify_scan_deferred(ctypes.byref(dims), ctypes.byref(st),
                                          ctypes.byref(stash) if stash is not None else None, keep,
                                          ctypes.byref(rows), T, None, None, None)
    prev = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE), 8)
    assert call(None) == kb.EINVAL
    assert call(kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE), 0)) == kb.EINVAL
    assert b"ping-pong" in L.kda_last_error()
    assert call(prev, keep=None) == kb.EINVAL
    assert call(prev, keep=FAKE + 2) == kb.EINVAL
    assert call(prev, T=16) == kb.EINVAL
    assert call(kb.KdaStashC(FAKE, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE), 8)) == kb.EINVAL
    assert call(kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(), 8)) == kb.EINVAL  # no previous rows
    # the update vectors: this round's must not overwrite the previous round's, which
    # the replay reads, and both are 16-byte aligned
    rows.w = FAKE + 0x4000
    assert call(kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 0x4000),
                             8)) == kb.EINVAL
    assert b"previous round" in L.kda_last_error()
    assert call(kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 0x4008),
                             8)) == kb.EINVAL
    rows.w = FAKE + 0x4004
    assert call(prev) == kb.EINVAL
    rows.w = None
    # an empty problem only exchanges the buffers and records the round
    empty = kb.KdaDims(0, 2, 64, 128, 128, kb.BF16)
    st2 = kb.KdaLayerState(FAKE, FAKE + 0x100, FAKE + 0x200)
    s2 = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(), 8)
    assert L.kda_verify_scan_deferred(ctypes.byref(empty), ctypes.byref(st2), ctypes.byref(s2), None,
                                      ctypes.byref(rows), 5, None, None, None) == kb.OK
    assert st2.state == FAKE + 0x1000 and s2.state_snap == FAKE and s2.T == 5


def test_layer_bounds_cover_the_layers_in_order():
    assert kb.layer_bounds(3) == [(0, 1), (1, 2), (2, 3)]
    assert kb.layer_bounds(34, 4) == [(0, 8), (8, 17), (17, 25), (25, 34)]
    assert kb.layer_bounds(2, 5) == [(0, 1), (1, 2)]  # at most one range a layer
    assert kb.layer_bounds(5, [(0, 2), (2, 5)]) == [(0, 2), (2, 5)]
    for bad in ([(0, 2), (3, 5)], [(1, 5)], [(0, 4)], [(0, 0), (0, 5)], []):
        with pytest.raises(ValueError):
            kb.layer_bounds(5, bad)


def test_staged_deferred_and_flag_writer_reject_on_host(L):
    dims, st, rows = _state(B=2)
    prev = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE), 8)

    def call(ready=FAKE + 0x4000, lpf=1, keep=FAKE + 0x3000):
        return L.kda_verify_scan_deferred_staged(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(prev), keep,
                                                 ctypes.byref(rows), 8, None, ready, lpf, 1, None, None)
    assert call(ready=None) == kb.EINVAL and b"ready_flags" in L.kda_last_error()
    assert call(ready=FAKE + 0x4002) == kb.EINVAL
    assert call(lpf=0) == kb.EINVAL and b"pairs_per_flag" in L.kda_last_error()
    assert call(keep=None) == kb.EINVAL  # the deferred round's own checks still apply
    assert L.kda_stream_write_u32(None, 1, None) == kb.EINVAL
    assert L.kda_stream_write_u32(FAKE + 2, 1, None) == kb.EINVAL

    def upload(dst=rows, src=rows, T=8, ready=FAKE + 0x4000, lpf=1, d=dims):
        return L.kda_upload_rows_staged(ctypes.byref(d), ctypes.byref(dst) if dst is not None else None,
                                        ctypes.byref(src) if src is not None else None, T, ready, lpf, 1, None)
    assert upload(dst=None) == kb.EINVAL and upload(src=None) == kb.EINVAL
    assert upload(T=0) == kb.EINVAL and upload(T=16) == kb.EINVAL
    assert upload(ready=None) == kb.EINVAL and upload(ready=FAKE + 1) == kb.EINVAL and upload(lpf=0) == kb.EINVAL
    assert upload(src=kb.KdaRows(FAKE, FAKE, None, FAKE, FAKE)) == kb.EINVAL
    assert upload(d=kb.KdaDims(0, 2, 64, 128, 128, kb.BF16)) == kb.OK  # nothing to copy
    assert kb.staged_flag_count(34, 1, 9) == 4 and kb.staged_flag_count(1, 32, 8) == 4
    assert kb.staged_flag_count(3, 2, 4) == 2 and kb.staged_flag_count(3, 2, 1) == 6
    with pytest.raises(ValueError):
        kb.staged_flag_count(3, 2, 0)


def test_round_host_rejects_on_host(L):
    dims, st, rows = _state(B=2)
    hrows = kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE)

    def call(stash, T=8, V=1000, ldt=kb.BF16, jbk=FAKE + 0x5000, s1=None, s2=None, hl=FAKE):
        return L.kda_round_host(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(stash) if stash else None, T,
                                ctypes.byref(hrows), ctypes.byref(rows), hl, FAKE, ldt, V, FAKE, FAKE, jbk,
                                FAKE + 0x6000, None, FAKE + 0x7000, 1, 1, None, s1, s2, 0, 0)
    prev = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE), 8)
    assert call(None) == kb.EINVAL
    assert call(prev, T=0) == kb.EINVAL and call(prev, T=16) == kb.EINVAL
    assert call(prev, V=0) == kb.EINVAL and call(prev, ldt=5) == kb.EINVAL
    assert call(prev, jbk=FAKE + 0x5002) == kb.EINVAL
    assert call(prev, hl=None) == kb.EINVAL
    # after the first round the copies need a stream of their own: the verify waits for them
    assert call(prev, s1=None, s2=None) == kb.EINVAL
    assert b"copy_stream" in L.kda_last_error()


def test_deferred_host_rejects_on_host(L):
    dims, st, rows = _state(B=2)
    prev = kb.KdaStashC(FAKE + 0x1000, FAKE + 0x2000, kb.KdaRows(FAKE, FAKE, FAKE, FAKE, FAKE), 8)
    assert L.kda_verify_scan_deferred_host(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(prev), FAKE + 0x3000,
                                           None, ctypes.byref(rows), 8, None, None, None) == kb.EINVAL
    bad = kb.KdaRows(FAKE, FAKE, FAKE, FAKE + 2, FAKE)  # misaligned before any device query
    assert L.kda_verify_scan_deferred_host(ctypes.byref(dims), ctypes.byref(st), ctypes.byref(prev), FAKE + 0x3000,
                                           ctypes.byref(bad), ctypes.byref(rows), 8, None, None, None) == kb.EINVAL
