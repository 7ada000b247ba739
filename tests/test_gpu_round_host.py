"""GPU: kda_round_host, one speculative round from host memory in one call (glm_spec.rs,
glm5_spec_round: verify, accept and rollback a round, the host reading j before the
next round's drafts), against the same rounds issued entry point by entry point:
a ping-pong verify and spec_accept for the first round, then kda_verify_scan_deferred
(folding in the previous accept) and spec_accept, and a final kda_rollback.  Outputs,
j, bonus, states and rings must agree bit for bit; j must equal the accept count the
inputs were built for (the drafts follow the planted row maxima up to that count)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import bits_equal, layer_state, small_case
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


def _host_round(w, r):
    """Pinned host tensors of round r: raw rows, logits, drafts; and the target j."""
    rows = synth.all_rows(w, r)
    dt = torch.bfloat16 if w.bf16 else torch.float32
    h = {}
    for n in NAMES:
        t = torch.from_numpy(np.ascontiguousarray(rows[n]))
        h[n] = (t.view(torch.bfloat16) if w.bf16 else t).pin_memory()
    lg = torch.from_numpy(np.ascontiguousarray(synth.logits(w, r)))
    h["logits"] = (lg.view(torch.bfloat16) if w.bf16 else lg).to(dt).pin_memory()
    j = synth.accept_targets(w, r)
    h["drafts"] = torch.from_numpy(synth.drafts_for(synth.logit_argmax(w, r), j, w.V)).pin_memory()
    return h, [int(x) for x in j]


def _dev_set(w, with_w):
    dt = torch.bfloat16 if w.bf16 else torch.float32
    shp = (w.L, w.B, w.T, w.H, 128)
    d = {n: torch.empty(shp, dtype=dt, device="cuda") for n in ("q", "k", "v", "g")}
    d["beta"] = torch.empty(shp[:4], dtype=dt, device="cuda")
    d["logits"] = torch.empty((w.B, w.T, w.V), dtype=dt, device="cuda")
    d["drafts"] = torch.empty((w.B, w.T - 1), dtype=torch.int32, device="cuda")
    if with_w:
        d["w"] = torch.empty(shp, dtype=torch.float32, device="cuda")
    return d


@pytest.mark.parametrize("bf16,ppf,with_w,in_place", [(True, 2, False, False), (True, 1, True, False),
                                                      (False, 4, False, False), (True, 2, False, True),
                                                      (True, 1, True, True), (False, 1, False, True)])
def test_host_rounds_equal_the_entry_points(bf16, ppf, with_w, in_place):
    w = synth.Workload("rh", L=2, B=3, H=4, T=8, bf16=bf16, V=96, rounds=6, seed=0x5150, accept="uniform")
    state0, ring0, cw = small_case(w)
    R = 5
    host = [_host_round(w, r) for r in range(R)]
    # the rounds issued one entry point at a time, from the same inputs
    ref = kb.PingPong(layer_state(state0, ring0, cw))
    jb = torch.empty((3, w.B), dtype=torch.int32, device="cuda")
    outs, js = [], []
    for r in range(R):
        h, _ = host[r]
        x = [h[n].cuda() for n in NAMES]
        out = torch.full((w.L, w.B, w.T, w.H, 128), float("nan"), device="cuda")
        if r == 0:
            kb.kda_verify_scan_pingpong(ref, *x, out=out)
        else:
            kb.kda_verify_scan_deferred(ref, *x, jb[2].clone(), out=out)
        kb.spec_accept(h["logits"].cuda(), h["drafts"].cuda(), jb[0], jb[1], jb[2])
        torch.cuda.synchronize()
        outs.append(out)
        js.append(jb[:2].cpu().clone())
    kb.kda_rollback_pingpong(ref, jb[2])
    # the same rounds through kda_round_host
    st = layer_state(state0, ring0, cw)
    out = torch.full((w.L, w.B, w.T, w.H, 128), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hr = kb.HostRounds(st, [_dev_set(w, with_w), _dev_set(w, with_w)], out=out, pairs_per_flag=ppf,
                       dev_status=status, in_place=in_place)
    for r in range(R):
        h, jt = host[r]
        j, bonus = hr(h)
        assert [int(v) for v in j] == jt, f"round {r}: j is not the count the drafts were built for"
        assert torch.equal(torch.stack([j, bonus]), js[r]), f"round {r}: j / bonus"
        assert bits_equal(out, outs[r]), f"round {r}: outputs"
    hr.commit()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bits_equal(hr.state(), ref.state()) and bits_equal(hr.ring(), ref.ring())


def test_host_rounds_reject_one_stream_after_the_first_round():
    w = synth.Workload("rs", L=1, B=2, H=2, T=4, bf16=True, V=64, rounds=2, seed=0x5151, accept="uniform")
    state0, ring0, cw = small_case(w)
    s = torch.cuda.current_stream()
    hr = kb.HostRounds(layer_state(state0, ring0, cw), [_dev_set(w, False), _dev_set(w, False)], stream=s,
                       copy_stream=s)
    h0, _ = _host_round(w, 0)
    hr(h0)  # the first round runs on one stream
    h1, _ = _host_round(w, 1)
    with pytest.raises(kb.KdaError):
        hr(h1)
