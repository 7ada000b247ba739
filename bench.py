"""Benchmark: KDA speculative-verify rounds on one GB300 (or N replicas).

A step is one verify round of the whole hot path on resident inputs:
  kda_verify_scan_deferred  (one launch: the previous round's accept-j rollback, i.e.
                    the replay of its rows 0..keep-1 from its snapshot where keep < T,
                    then this round's conv + activations + gated delta rule over T
                    rows; ping-pong state buffers, no snapshot copy)  ->  spec_accept
                    (device argmax per row, first mismatch, keep = j+1, applied by the
                    next round's launch).
Beside it: the same rounds with the rollback as its own launch ("separate_rollback":
kda_verify_scan_pingpong, spec_accept, kda_rollback) and the in-place round
("in_place": kda_verify_scan copying the snapshot as it reads the state).
Default workload: the 34-layer KDA stack of one session, 64 heads x 128x128 f32
state per layer, K = 7 drafts (T = 8), 64 seeded rounds cycled, accept j drawn
per round.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "KDA verify rows/s (T=K+1, 64 heads) and achieved HBM GB/s vs 8 TB/s roofline"
UNIT = "verify rows/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes read + written by one deferred-round launch of kda_scan_kernel, from one
# ncu capture per workload (dram__bytes_read.sum + dram__bytes_write.sum), with the
# kernel's own byte count (deferred_bytes with the update vectors stored and read back,
# the default) of the captured launch, so the figure can be scaled to a run's mean
# launch.  TRAFFIC_SOURCE is the hash of kda_scan.cu (code
# only: comments and blank space removed) the captures were taken on; with any other
# source the traffic is reported as null.
TRAFFIC_SOURCE = "4210bf2b757b85d42b500a53fa83fda9836cbd789d37a1bbbe01722c582abe9f"
TRAFFIC_BYTES = {"stack34": (205_133_056 + 266_830_080, 516_995_840),
                 "batched32": (213_674_496 + 258_313_984, 512_188_800),
                 "stress64x34": (13_887_103_232 + 18_720_913_664, 31_932_887_040)}
SCAN_SOURCE = os.path.join(ROOT, "speculative_decode_verify_kda_gb300", "csrc", "kda_scan.cu")


def code_hash(path: str) -> str:
    """sha256 of a C/C++/CUDA source with its comments and white space removed."""
    import hashlib
    import re
    with open(path) as f:
        src = f.read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":  # string or char literal, copied whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    code = re.sub(r"\s+", "", "".join(out))
    return hashlib.sha256(code.encode()).hexdigest()


WORKLOAD_TEXT = {
    "stack34": "34 KDA layers x 64 heads x 128x128 f32 state (136 MiB/round), K=7 (T=8), 1 session, "
               "64 seeded rounds cycled, accept j ~ U{0..7}, logits [8][32768] bf16",
    "stress64x34": "64 sessions x 34 layers x 64 heads x 128x128 f32 state, K=14 (T=15), skewed accept, "
                   "16 rounds cycled",
    "batched32": "32 sessions x 1 layer x 64 heads, K=14 (T=15), 16 rounds cycled",
    "layer64": "one 64-head KDA layer, K=7 (T=8), 1 session",
    "tiny": "1 layer, 1 head, K=7, f32 rows, V=32",
}


# ---------------------------------------------------------------------------
# byte accounting (algorithmic bytes: every tensor element moved once)
# ---------------------------------------------------------------------------
def verify_bytes(w, snapshot_copy: bool = False, stored_w: bool = False) -> int:
    """One verify launch.  Ping-pong (the default): S read + S write, ring read + write.
    snapshot_copy: the in-place verify that also writes the snapshot of S and ring.
    stored_w: the verify also writes each row's update vector (f32, 512 B a head)."""
    es = 2 if w.bf16 else 4
    D = 128
    n = 3 if snapshot_copy else 2
    per_head = n * D * D * 4 + n * 9 * D * 4
    rows = w.T * w.H * (4 * D + 1) * es
    out = w.T * w.H * D * 4
    wv = w.T * w.H * D * 4 if stored_w else 0
    return w.L * w.B * (w.H * per_head + rows + out + wv) + w.L * w.H * 3 * D * 4 * 4


def deferred_bytes(w, prev_keeps, stored_w: bool = False) -> int:
    """One kda_verify_scan_deferred launch: per session that rolls back (keep < T) the
    state is read, written as the snapshot and written again, the ring likewise, and
    the replayed rows are read besides this round's; a session that kept every row
    reads and writes its state and ring once.  stored_w: the launch also writes this
    round's update vectors and reads the replayed rows' (f32, 512 B a head and row)."""
    es = 2 if w.bf16 else 4
    D = 128
    row = w.H * (4 * D + 1) * es
    wrow = w.H * D * 4 if stored_w else 0
    n = 0
    for k in prev_keeps:
        pending = k < w.T
        m = 3 if pending else 2
        kr = k if pending else 0
        n += w.L * (w.H * m * (D * D * 4 + 9 * D * 4) + kr * (row + wrow) + w.T * (row + wrow) +
                    w.T * w.H * D * 4)
    return n + w.L * w.H * 3 * D * 4 * 4


def algorithmic_bytes(w, prev_keeps) -> int:
    """The bytes the round's steps must move, each tensor once: this round's verify at
    the ping-pong minimum (per session and layer the state read and written, 2 x 4 MiB
    at 64 heads; T raw rows of 65,664 B; T output rows of 32 KiB; the conv ring read
    and written, 2 x 288 KiB) plus the layer's conv weights (384 KiB), and the
    previous accept's rollback of every session that kept fewer than T rows (the
    snapshot read and the state written, the ring snapshot read and the ring written,
    and the kept raw rows).  This is what the roofline fraction divides by: a launch
    that folds the rollback into the verify moves fewer bytes than this."""
    es = 2 if w.bf16 else 4
    D = 128
    row = w.H * (4 * D + 1) * es
    state = w.H * D * D * 4
    ring = w.H * 9 * D * 4
    verify = 2 * state + 2 * ring + w.T * row + w.T * w.H * D * 4
    n = w.L * w.B * verify + w.L * w.H * 3 * D * 4 * 4
    for k in prev_keeps:
        if k < w.T:
            n += w.L * (2 * state + 2 * ring + k * row)
    return n


def rollback_bytes(w, keeps) -> int:
    es = 2 if w.bf16 else 4
    D = 128
    n = 0
    for k in keeps:
        if k < w.T:
            n += w.L * (w.H * (2 * D * D * 4 + 2 * 9 * D * 4) + k * w.H * (4 * D + 1) * es)
    if n:
        n += w.L * w.H * 3 * D * 4 * 4
    return n


def verify_bytes_var(w, t_rows, stored_w: bool = False) -> int:
    """verify_bytes (in place, snapshot copied) with session b running t_rows[b] rows."""
    es = 2 if w.bf16 else 4
    D = 128
    per_head = 3 * D * D * 4 + 3 * 9 * D * 4
    n = 0
    for t in t_rows:
        n += w.L * (w.H * per_head + t * w.H * (4 * D + 1) * es + t * w.H * D * 4 * (2 if stored_w else 1))
    return n + w.L * w.H * 3 * D * 4 * 4


def accept_bytes(w) -> int:
    return w.B * w.T * w.V * (2 if w.bf16 else 4) + w.B * (w.T - 1) * 4 + 3 * w.B * 4


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# replicas on several GPUs: every rank runs the whole workload (weak scaling, no
# collective on the data path); a time is the slowest rank's, the throughput counts
# every rank's rows
# ---------------------------------------------------------------------------
def slowest(ms: float, world: int, device=None) -> float:
    """The largest of every rank's ms (identity with one rank)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class nvtx_range:
    """An NVTX range around a bench section, so a profiler can pick a section's launches
    (ncu --nvtx --nvtx-include "<name>/")."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        import torch
        torch.cuda.nvtx.range_push(self.name)
        return self

    def __exit__(self, *exc):
        import torch
        torch.cuda.nvtx.range_pop()
        return False


def job_rows_per_s(world: int, B: int, T: int, ms: float) -> float:
    """Verify rows per second of the whole job: world replicas of B sessions x T rows per step."""
    return world * B * T / (ms * 1e-3)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi every 20 ms from before the first warm-up step to after the last timed
    section; the summary keeps the samples taken while the GPU was busy (utilization
    at least 50 %)."""
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap", "utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, pw, reasons, total = [], [], [], set(), 0
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                clk, cmax, util = float(parts[0]), float(parts[1]), float(parts[7])
            except ValueError:
                continue
            total += 1
            if util < 50:
                continue
            sm.append(clk)
            mx.append(cmax)
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "samples_total": total}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_total": total, "power_w_max": max(pw) if pw else None,
                "window": "from before the first warm-up step to after the last timed section, "
                          "samples at >= 50 % GPU utilization"}


# ---------------------------------------------------------------------------
# CPU oracle baseline (the reference arm and the cpu_baseline key)
# ---------------------------------------------------------------------------
class OracleArm:
    """The CPU oracle, as it stands, on one (layer, session) unit of the workload.

    Inputs for a few rounds are drawn once (untimed); each call runs accept +
    verify + rollback of one round on a slice of the unit's heads (heads are
    independent) and returns the oracle's own time.  State carries across rounds.
    """

    def __init__(self, w, n_rounds: int = 4):
        import oracle
        from speculative_decode_verify_kda_gb300 import synth
        self.orc = oracle.load()
        self.w = w
        l, b = 0, 0
        self.state = synth.unit_state(w, l, b)
        self.ring = synth.unit_ring(w, l, b)
        self.cw = synth.layer_conv_w(w, l)
        self.rounds = []
        for r in range(min(n_rounds, w.rounds)):
            d = synth.drafts_for(synth.logit_argmax(w, r, [b]), synth.accept_targets(w, r)[b:b + 1], w.V)[0]
            self.rounds.append((synth.unit_rows(w, r, l, b), synth.logits(w, r, sessions=[b])[0], d))
        self.r = 0
        self.h0 = 0

    def step(self, n_heads: int):
        """One round of accept + verify + rollback on the next n_heads heads."""
        rows, lg, d = self.rounds[self.r % len(self.rounds)]
        hs = slice(self.h0, min(self.w.H, self.h0 + n_heads))
        args = tuple(np.ascontiguousarray(rows[n][:, hs]) for n in ("q", "k", "v", "g", "beta"))
        s, rg, cw = (np.ascontiguousarray(a[hs]) for a in (self.state, self.ring, self.cw))
        t0 = time.perf_counter()
        j, _, _, _ = self.orc.accept(lg, d)
        t1 = time.perf_counter()
        st_T, ring_T, _ = self.orc.verify(*args, cw, rg, s)
        st_k, ring_k = self.orc.rollback(j + 1, *args, cw, rg, s, ring_T, st_T)
        t2 = time.perf_counter()
        self.state[hs], self.ring[hs] = st_k, ring_k
        done = hs.stop - hs.start
        self.h0 = hs.stop
        if self.h0 >= self.w.H:
            self.h0 = 0
            self.r += 1
        return t2 - t1, t1 - t0, done

    def rows_per_s(self, scan_s_per_head: float, accept_s: float) -> float:
        w = self.w
        round_s = scan_s_per_head * w.H * w.L * w.B + accept_s * w.B
        return w.B * w.T / round_s


def oracle_baseline(w, budget_s: float):
    """cpu_baseline: whole unit-rounds of the oracle for about budget_s seconds."""
    arm = OracleArm(w)
    t_scan = t_acc = 0.0
    heads = rounds = 0
    while t_scan + t_acc < budget_s or rounds == 0:
        ts, ta, n = arm.step(w.H)
        t_scan, t_acc, heads, rounds = t_scan + ts, t_acc + ta, heads + n, rounds + 1
    val = arm.rows_per_s(t_scan / heads, t_acc / rounds)
    desc = (f"{rounds} rounds of one (layer, session) unit of {w.name} ({w.H} heads, T={w.T}: accept + "
            f"verify + rollback), {t_scan + t_acc:.1f} s of single-threaded oracle time, extrapolated "
            f"linearly to {w.L} layers x {w.B} sessions per round")
    return {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc}


def oracle_baseline_threads(w, budget_s: float, threads: int):
    """A second CPU figure: the same oracle, unchanged, on independent (layer, session)
    units in `threads` host threads at once (the C calls release the interpreter lock),
    for about budget_s seconds of wall time."""
    from concurrent.futures import ThreadPoolExecutor
    arms = [OracleArm(w) for _ in range(threads)]

    def work(arm):
        heads = rounds = 0
        t_end = time.perf_counter() + budget_s
        while time.perf_counter() < t_end or rounds == 0:
            _, _, n = arm.step(w.H)
            heads, rounds = heads + n, rounds + 1
        return heads, rounds

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        done = list(ex.map(work, arms))
    wall = time.perf_counter() - t0
    heads = sum(d[0] for d in done)
    rounds = sum(d[1] for d in done)
    # a round of the workload is L*B unit-rounds of H heads; here every unit-round also ran
    # its accept, so the figure errs low
    round_s = wall / heads * (w.H * w.L * w.B)
    desc = (f"{rounds} unit-rounds of {w.name} ({w.H} heads, T={w.T}: accept + verify + rollback) in {threads} "
            f"threads over {wall:.1f} s of wall time, extrapolated linearly to {w.L} layers x {w.B} sessions")
    return {"value": w.B * w.T / round_s, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_e2e(args, w, R, pp, rows, logits, drafts, out, status, scratch, stream, dev, world, nc, use_w=False,
            in_place=True):
    """The deferred round end to end from pinned host buffers through the public API:
    one kda_round_host call a round (binding.HostRounds).

    A round's inputs sit in one pinned host block (logits, drafts, then each raw-row
    tensor whole).  in_place: the deferred round launch reads the raw rows in place from
    the host block over the host link while it runs (leaving their device copy for the
    next round's replay), the logits and drafts go up on a copy stream meanwhile.  Else
    the call copies the raw rows by nc consecutive ranges of (layer, session) pairs on a
    copy stream, each range followed by a stream write of its ready flag, and the launch
    scans each range once its flag is set (nc == 1: the whole block before the scan).
    Then the accept, whose j and bonus land in pinned host memory.  The call returns once
    the host has j (a round's inputs follow from the previous accept).  Leaves pp
    committed."""
    import time

    import torch
    from speculative_decode_verify_kda_gb300 import binding as kb

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    names = ("q", "k", "v", "g", "beta")
    parts = [("logits", logits[0]), ("drafts", drafts[0])] + [(n, rows[0][n]) for n in names]
    offs, off = {}, 0
    for n, t in parts:
        offs[n] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    block_bytes = off
    HR = min(R, 4 if block_bytes < (1 << 30) else 2)  # pinned host rounds cycled
    pairs = w.L * w.B  # (layer, session) pairs, the unit of a staged range
    ppf = -(-pairs // max(1, min(nc, pairs)))  # pairs a flag covers
    nranges = -(-pairs // ppf)

    def views(buf):
        out_ = {}
        for n, t in parts:
            nb = t.numel() * t.element_size()
            out_[n] = buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        return out_

    host_views = []
    for r in range(HR):
        hb = torch.empty(block_bytes, dtype=torch.uint8).pin_memory()
        hv = views(hb)
        src = dict(rows[r], logits=logits[r], drafts=drafts[r])
        for n, _ in parts:
            hv[n].copy_(src[n].cpu())
        host_views.append(hv)
    # two device blocks: a deferred round reads the previous round's raw rows (and the
    # update vectors, two buffers, stay on the device)
    dev_sets = []
    for _ in range(2):
        v = views(torch.empty(block_bytes, dtype=torch.uint8, device=dev))
        if use_w:
            v["w"] = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device=dev)
        dev_sets.append(v)
    h2d = sum(t.numel() * t.element_size() for _, t in parts)
    d2h = 2 * w.B * 4  # j and the bonus
    Ke = max(1, min(args.e2e_steps, args.steps))
    copy_stream = torch.cuda.Stream(dev)
    p = pp.parity
    hr = kb.HostRounds(kb.LayerState(pp.states[p], pp.rings[p], pp.conv_w), dev_sets, out=out,
                       pairs_per_flag=ppf, dev_status=status, stream=stream, copy_stream=copy_stream,
                       spare_state=pp.states[1 - p], spare_ring=pp.rings[1 - p], in_place=in_place)
    # the chain opens with a ping-pong round, then deferred rounds
    for i in range(4):
        hr(host_views[i % HR])
    barrier()
    t0 = time.perf_counter()
    with nvtx_range("e2e_in_place" if in_place else "e2e_staged"):
        for i in range(4, 4 + Ke):
            hr(host_views[i % HR])
    barrier()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / Ke
    e2e_ms = slowest(e2e_ms, world, dev)
    hr.commit()
    torch.cuda.synchronize(dev)
    if int(status.item()):
        raise RuntimeError(f"device status {int(status.item()):#x} after the e2e steps")
    # the committed state is in one of pp's two buffers
    pp.parity = 0 if hr.state().data_ptr() == pp.states[0].data_ptr() else 1
    pp.last = None
    res = {"value": job_rows_per_s(world, w.B, w.T, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms, "steps": Ke,
           "call": "kda_round_host (one call a round)",
           "raw_rows": ("read in place from the pinned host block by the verify launch over the host link"
                        if in_place else f"copied in {nranges} range(s) of (layer, session) pairs")}
    if not in_place and nranges > 1:
        res["staged_ranges"] = nranges
        res["pairs_per_range"] = ppf
    return res


def run_sampled(args, w, logits, K, j_out, keep_out, status, stream, dev, barrier, accept_ms):
    """The sampled acceptance of one workload's first round: the rejection walk with
    filtered target and draft rows (the draft rows equal the target rows, so every draft
    is accepted: the longest walk), from caller uniforms and from the sessions' Philox
    streams."""
    import torch

    from speculative_decode_verify_kda_gb300 import binding as kb
    filt = dict(temperature=0.7, top_k=50, top_p=0.9, min_p=0.0)
    lg0 = logits[0]
    dl = lg0[:, :w.K].contiguous()
    dr = torch.argmax(lg0[:, :w.K].float(), dim=-1).to(torch.int32).contiguous()
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    ua = torch.rand((w.B, w.K), generator=g, device=dev)
    us = torch.rand((w.B,), generator=g, device=dev)
    tok = torch.empty_like(j_out)
    Ks = max(1, min(args.sampled_steps, K))
    for _ in range(3):
        kb.spec_accept_sampled(lg0, dl, dr, ua, us, j_out=j_out, token_out=tok, keep_out=keep_out,
                               dev_status=status, stream=stream, **filt)
    barrier()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with nvtx_range("sampled"):
        a_.record(stream)
        for _ in range(Ks):
            kb.spec_accept_sampled(lg0, dl, dr, ua, us, j_out=j_out, token_out=tok, keep_out=keep_out,
                                   dev_status=status, stream=stream, **filt)
        b_.record(stream)
    barrier()
    if int(status.item()) or int(j_out.min().item()) != w.K:
        raise RuntimeError("sampled accept: unexpected status or walk length")
    s_ms = a_.elapsed_time(b_) / Ks
    # the same walk drawing from the sessions' Philox streams (counters advanced on the device)
    seeds = torch.arange(w.B, dtype=torch.int64, device=dev) + w.seed
    counters = torch.zeros((w.B, 2), dtype=torch.int32, device=dev)
    for _ in range(3):
        kb.spec_accept_sampled_session(lg0, dl, dr, seeds, counters, j_out=j_out, token_out=tok, keep_out=keep_out,
                                       dev_status=status, stream=stream, **filt)
    barrier()
    with nvtx_range("sampled_session"):
        a_.record(stream)
        for _ in range(Ks):
            kb.spec_accept_sampled_session(lg0, dl, dr, seeds, counters, j_out=j_out, token_out=tok,
                                           keep_out=keep_out, dev_status=status, stream=stream, **filt)
        b_.record(stream)
    barrier()
    if int(status.item()) or int(j_out.min().item()) != w.K:
        raise RuntimeError("sampled accept (session): unexpected status or walk length")
    ss_ms = a_.elapsed_time(b_) / Ks
    nbytes = w.B * (2 * w.K + 1) * w.V * lg0.element_size()
    return {"filter": filt, "walk": "every draft accepted (draft rows = target rows)",
            "ms": s_ms, "session_ms": ss_ms, "greedy_accept_ms": accept_ms,
            "logit_rows_per_call": w.B * (2 * w.K + 1),
            "logits_gbs": nbytes / (s_ms * 1e-3) / 1e9}


def run_gpu(args, rank, world, local_rank, wname, full=True):
    """One workload on this rank's GPU.  full: every section; else the timed deferred
    rounds and the e2e rounds only."""
    import torch
    from speculative_decode_verify_kda_gb300 import binding as kb
    from speculative_decode_verify_kda_gb300 import synth, synth_gpu

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synth.WORKLOADS[wname]
    R = min(w.rounds, args.rounds) if args.rounds else w.rounds
    # stored update vectors, for the deferred rounds only (a deferred round's replay
    # reads the previous round's, so consecutive rounds need different w buffers and
    # the cycle of rounds is even); the rounds with a separate rollback run without them
    # (with them a separate verify measured ~3 % slower and the rollback ~8 %)
    use_w = args.replay_w == "on" and R >= 2
    if use_w and R % 2:
        R -= 1

    st = kb.LayerState(synth_gpu.state(w, dev), synth_gpu.ring(w, dev), synth_gpu.conv_w(w, dev))
    stash = kb.Stash(st)
    rows = [synth_gpu.rows(w, r, dev) for r in range(R)]
    plain = rows  # q, k, v, g, beta
    if use_w:
        wbufs = [torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device=dev) for _ in range(2)]
        rows = [dict(rows[r], w=wbufs[r % 2]) for r in range(R)]
    logits = [synth_gpu.logits(w, r, dev) for r in range(R)]
    drafts, jt = zip(*[synth_gpu.drafts(w, r, dev, lg=logits[r]) for r in range(R)])
    out = torch.empty((w.L, w.B, w.T, w.H, 128), dtype=torch.float32, device=dev)
    j_out = torch.empty(w.B, dtype=torch.int32, device=dev)
    bonus_out = torch.empty_like(j_out)
    keep_out = torch.empty_like(j_out)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scratch = torch.empty(max(kb.spec_accept_scratch_bytes(w.B, w.T, w.V), 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # the timed round: ping-pong state buffers (the resident state and the stash's
    # snapshot buffers swap roles every round; the verify reads one and writes the other)
    pp = kb.PingPong(st, spare_state=stash.state_snap, spare_ring=stash.ring_snap)
    pplans = [kb.PingPongRoundPlan(pp, plain[r], out, logits[r], drafts[r], j_out, bonus_out, keep_out, status,
                                   scratch, stream) for r in range(R)]
    # the in-place round (snapshot copied by the verify), reported beside it
    plans = [kb.RoundPlan(st, plain[r], out, stash, logits[r], drafts[r], j_out, bonus_out, keep_out, status,
                          scratch, stream) for r in range(R)]

    def step(r, ev=None, plans_=None):
        p = (plans_ or pplans)[r]
        if ev is None:
            p()
            return
        if plans_ is None:
            par = pp.parity
            ev[0].record(stream)
            p.verify(par)
            ev[1].record(stream)
            p.accept()
            ev[2].record(stream)
            p.rollback(par)
            ev[3].record(stream)
            p._flip(par)
            return
        ev[0].record(stream)
        p.verify()
        ev[1].record(stream)
        p.accept()
        ev[2].record(stream)
        p.rollback()
        ev[3].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # the timed round: kda_verify_scan_deferred (the previous round's rollback and this
    # round's verify in one launch) then spec_accept, whose keep the next round applies
    dplans = [kb.DeferredRoundPlan(pp, rows[r], out, logits[r], drafts[r], j_out, bonus_out, keep_out, status,
                                   scratch, stream) for r in range(R)]

    def dstep(r, ev=None):
        p = dplans[r]
        par = pp.last
        if ev is not None:
            ev[0].record(stream)
        p.verify(par)
        if ev is not None:
            ev[1].record(stream)
        p.accept()
        if ev is not None:
            ev[2].record(stream)
        p._flip(par)

    # the first round opens the chain: a ping-pong verify and its accept (its rollback
    # runs inside the next round's launch)
    par0 = pp.parity
    pplans[0].verify(par0)
    pplans[0].accept()
    pplans[0]._flip(par0)
    for i in range(1, args.warmup + 1):
        dstep(i % R)
    barrier()
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    # the timed steps: only the two events around them, so that each launch follows the
    # previous one as a programmatic dependent (an event between two launches would
    # serialise them); then the same number of steps again with events around each
    # launch, for the per-kernel times
    t_wall = time.perf_counter()
    with nvtx_range("deferred"):
        e0.record(stream)
        for i in range(K):
            dstep((args.warmup + 1 + i) % R)
        e1.record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    total_ms = e0.elapsed_time(e1)
    with nvtx_range("deferred_events"):
        for i in range(K):
            dstep((args.warmup + 1 + K + i) % R, evs[i])
    barrier()
    round_ms = [e[0].elapsed_time(e[1]) for e in evs]
    accept_ms = [e[1].elapsed_time(e[2]) for e in evs]
    st_word = int(status.item())
    if st_word:
        raise RuntimeError(f"device status {st_word:#x} after the timed steps")
    ms_step = total_ms / K
    ms_step = slowest(ms_step, world, dev)
    # commit the last round, so the committed state is in the ping-pong buffers
    kb.kda_rollback_pingpong(pp, keep_out, dev_status=status, stream=stream)

    # the kept rows each round of the second pass replays: the previous round's accept
    prev_keeps = [[j + 1 for j in jt[(args.warmup + K + i) % R]] for i in range(K)]
    round_bytes = [deferred_bytes(w, k, stored_w=use_w) for k in prev_keeps]
    algo_bytes = [algorithmic_bytes(w, k) for k in prev_keeps]
    step_bytes = [rb + accept_bytes(w) for rb in round_bytes]
    round_avg_ms = sum(round_ms) / K
    peak, peak_kind = measured_peak()
    achieved = sum(algo_bytes) / (sum(round_ms) * 1e-3) / 1e9
    achieved_kernel = sum(round_bytes) / (sum(round_ms) * 1e-3) / 1e9
    res = {
        "rows_per_s": job_rows_per_s(world, w.B, w.T, ms_step),
        "ms_per_step": ms_step,
        "round_kernel_ms": round_avg_ms,
        "accept_ms": sum(accept_ms) / K,
        "wall_s": t_wall,
        "round_bytes_mean": sum(round_bytes) / K,
        "algo_bytes_mean": sum(algo_bytes) / K,
        "step_bytes_mean": sum(step_bytes) / K,
        "step_gbs": sum(deferred_bytes(w, [j + 1 for j in jt[(args.warmup + i) % R]], stored_w=use_w) +
                        accept_bytes(w) for i in range(K)) / (total_ms * 1e-3) / 1e9,
        "achieved": achieved,
        "achieved_kernel": achieved_kernel,
        "peak": peak,
        "peak_kind": peak_kind,
        "launches_per_step": 2,  # kda_scan_kernel (deferred round) and accept_cluster_kernel
        "replay_w": use_w,
    }
    if not full:
        if not args.no_e2e:
            res["e2e"] = run_e2e(args, w, R, pp, rows, logits, drafts, out, status, scratch, stream, dev, world,
                                 args.e2e_chunks, use_w, in_place=args.e2e_rows == "in_place")
        if not args.no_sampled:
            res["sampled_accept"] = run_sampled(args, w, logits, K, j_out, keep_out, status, stream, dev, barrier,
                                                res["accept_ms"])
        return res

    # the same rounds with the rollback as its own launch: ping-pong verify, accept,
    # rollback
    Kp = max(1, min(K, 1000))
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Kp)]
    for i in range(3):
        step(i % R)
    barrier()
    pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with nvtx_range("separate"):  # the step time without events between the launches
        pa.record(stream)
        for i in range(Kp):
            step((3 + i) % R)
        pb.record(stream)
        for i in range(Kp):  # the per-kernel times
            step((3 + Kp + i) % R, evp[i])
    barrier()
    if int(status.item()):
        raise RuntimeError(f"device status {int(status.item()):#x} after the ping-pong steps")
    s_ms = slowest(pa.elapsed_time(pb) / Kp, world, dev)
    s_verify = sum(e[0].elapsed_time(e[1]) for e in evp) / Kp
    vb = verify_bytes(w)
    separate = {"steps": Kp, "ms_per_step": s_ms, "rows_per_s": job_rows_per_s(world, w.B, w.T, s_ms),
                "verify_ms": s_verify, "accept_ms": sum(e[1].elapsed_time(e[2]) for e in evp) / Kp,
                "rollback_ms": sum(e[2].elapsed_time(e[3]) for e in evp) / Kp, "verify_bytes": vb,
                "verify_gbs": vb / (s_verify * 1e-3) / 1e9, "verify_frac_of_peak": vb / (s_verify * 1e-3) / 1e9 / peak,
                "launches_per_step": 4}

    # the in-place round: kda_verify_scan writes the snapshot copy as it reads the state
    Ki = max(1, min(K, 1000))
    evi = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Ki)]
    for i in range(3):
        step(i % R, plans_=plans)
    barrier()
    ia, ib = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with nvtx_range("in_place"):  # the step time without events between the launches
        ia.record(stream)
        for i in range(Ki):
            step(i % R, plans_=plans)
        ib.record(stream)
        for i in range(Ki):  # the per-kernel times
            step((Ki + i) % R, evi[i], plans_=plans)
    barrier()
    if int(status.item()):
        raise RuntimeError(f"device status {int(status.item()):#x} after the in-place steps")
    i_ms = slowest(ia.elapsed_time(ib) / Ki, world, dev)
    i_verify = sum(e[0].elapsed_time(e[1]) for e in evi) / Ki
    vb_in = verify_bytes(w, snapshot_copy=True)
    in_place = {"steps": Ki, "ms_per_step": i_ms, "rows_per_s": job_rows_per_s(world, w.B, w.T, i_ms),
                "verify_ms": i_verify, "accept_ms": sum(e[1].elapsed_time(e[2]) for e in evi) / Ki,
                "rollback_ms": sum(e[2].elapsed_time(e[3]) for e in evi) / Ki, "verify_bytes": vb_in,
                "verify_gbs": vb_in / (i_verify * 1e-3) / 1e9,
                "verify_frac_of_peak": vb_in / (i_verify * 1e-3) / 1e9 / peak}
    # the committed state is back in the ping-pong buffers' hands from here on: the
    # in-place rounds above advanced st.state, which is one of them
    pp.parity = 0

    res["separate_rollback"] = separate
    res["in_place"] = in_place

    # the same rounds replayed from CUDA graphs (one graph per resident round): the
    # launch gaps between the round's kernels shrink
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        gp = [kb.PingPongRoundPlan(pp, plain[r], out, logits[r], drafts[r], j_out, bonus_out, keep_out, status,
                                   scratch, side) for r in range(R)]
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for g in gp:
                g()  # both parities of every plan run once eagerly before capture
                g()
        stream.wait_stream(side)
        barrier()
        for g in gp:
            g.capture()
        for i in range(args.warmup):
            gp[i % R].replay()
        barrier()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        for i in range(K):
            gp[(args.warmup + i) % R].replay()
        gb.record(stream)
        barrier()
        g_ms = ga.elapsed_time(gb) / K
        if int(status.item()):
            raise RuntimeError(f"device status {int(status.item()):#x} after the graph steps")
        g_ms = slowest(g_ms, world, dev)
        res["graph"] = {"ms_per_step": g_ms, "rows_per_s": job_rows_per_s(world, w.B, w.T, g_ms), "steps": K,
                        "round": "ping-pong verify, accept, rollback (separate launches), one graph per round"}

    # e2e: host buffers through the public API, copies inside the timed region (run_e2e):
    # the raw rows stream in by range of (layer, session) pairs while the one launch
    # scans the ranges already in place; the one-copy round (the whole block, then the
    # launch) is reported beside it.
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, w, R, pp, rows, logits, drafts, out, status, scratch, stream, dev, world,
                             args.e2e_chunks, use_w, in_place=args.e2e_rows == "in_place")
        # the copy-based rounds beside it: the rows staged by range, and in one copy
        for key, nc_, ip in (("staged_copy", args.e2e_chunks, False), ("one_copy", 1, False)):
            if args.e2e_rows == "in_place" or key == "one_copy":
                alt = run_e2e(args, w, R, pp, rows, logits, drafts, out, status, scratch, stream, dev, world, nc_,
                              use_w, in_place=ip)
                res["e2e"][key] = {"value": alt["value"], "ms_per_step": alt["ms_per_step"]}

    # per-layer issue: one kda_verify_scan per layer (as a model issues them), then accept
    # and one all-layer rollback; eagerly, and replayed from CUDA graphs (one per round)
    if w.L > 1 and not args.no_per_layer:
        Kp = max(1, min(args.per_layer_steps, K))
        RP = min(R, 8)
        lplans = [kb.LayerRoundPlan(st, plain[r], out, stash, logits[r], drafts[r], j_out, bonus_out, keep_out,
                                    status, scratch, stream) for r in range(RP)]
        side = torch.cuda.Stream(dev)
        gplans = [kb.LayerRoundPlan(st, plain[r], out, stash, logits[r], drafts[r], j_out, bonus_out, keep_out,
                                    status, scratch, side) for r in range(RP)]

        def timed(fn):
            for i in range(4):  # even: a deferred round's update vectors alternate with the round's parity
                fn(i % RP)
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(Kp):
                fn(i % RP)
            b.record(stream)
            barrier()
            return a.elapsed_time(b) / Kp

        eager_ms = timed(lambda r: lplans[r]())
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for g in gplans:
                g()  # one eager round on the capture stream: every one-time setup call has run
        stream.wait_stream(side)
        barrier()
        for g in gplans:
            g.capture()
        graph_ms = timed(lambda r: gplans[r].replay())
        if int(status.item()):
            raise RuntimeError(f"device status {int(status.item()):#x} after the per-layer steps")
        eager_ms, graph_ms = slowest(eager_ms, world, dev), slowest(graph_ms, world, dev)
        # deferred rounds issued one launch per layer, then the accept (the round's
        # rollbacks run inside the layer launches)
        pp.parity = 0  # the in-place rounds above left the committed state in st.state
        par = pp.parity
        pplans[0].verify(par)
        pplans[0].accept()
        pplans[0]._flip(par)
        lps = kb.layer_pingpongs(pp)
        dl_plans = [kb.LayerDeferredRoundPlan(pp, lps, rows[r], out, logits[r], drafts[r], j_out, bonus_out,
                                              keep_out, status, scratch, stream) for r in range(RP)]
        deferred_ms = timed(lambda r: dl_plans[(r + 1) % RP]())
        kb.kda_rollback_pingpong(pp, keep_out, dev_status=status, stream=stream)
        if int(status.item()):
            raise RuntimeError(f"device status {int(status.item()):#x} after the per-layer deferred steps")
        deferred_ms = slowest(deferred_ms, world, dev)
        res["per_layer"] = {"launches_per_step": w.L + 3, "steps": Kp, "eager_ms_per_step": eager_ms,
                            "graph_ms_per_step": graph_ms,
                            "graph_rows_per_s": job_rows_per_s(world, w.B, w.T, graph_ms),
                            "deferred": {"launches_per_step": w.L + 1, "eager_ms_per_step": deferred_ms,
                                         "rows_per_s": job_rows_per_s(world, w.B, w.T, deferred_ms)}}
    # column-stash rollback (the alternative to snapshot + replay): the verify also
    # writes the state and ring after every row, the rollback copies the kept column
    col_bytes = w.L * w.B * w.H * w.T * (128 * 128 + 9 * 128) * 4
    if not args.no_cols and col_bytes <= 16e9:
        cols = kb.ColStash(st, w.T)
        Kc = max(1, min(args.cols_steps, K))
        evc = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(Kc + 3)]

        def col_step(i, ev):
            r = i % R
            rr = plain[r]
            ev[0].record(stream)
            kb.kda_verify_scan_cols(st, rr["q"], rr["k"], rr["v"], rr["g"], rr["beta"], cols, out=out, stream=stream)
            ev[1].record(stream)
            plans[r].accept()
            ev[2].record(stream)
            kb.kda_rollback_cols(st, cols, keep_out, dev_status=status, stream=stream)
            ev[3].record(stream)

        for i in range(3):
            col_step(i, evc[Kc + i])
        barrier()
        with nvtx_range("col_stash"):
            for i in range(Kc):
                col_step(i, evc[i])
        barrier()
        if int(status.item()):
            raise RuntimeError(f"device status {int(status.item()):#x} after the column-stash steps")
        cv = sum(e[0].elapsed_time(e[1]) for e in evc[:Kc]) / Kc
        cr = sum(e[2].elapsed_time(e[3]) for e in evc[:Kc]) / Kc
        cs = sum(e[0].elapsed_time(e[3]) for e in evc[:Kc]) / Kc
        es = 2 if w.bf16 else 4
        per_head = (2 + w.T) * 128 * 128 * 4 + (2 + w.T) * 9 * 128 * 4
        cvb = w.L * w.B * (w.H * per_head + w.T * w.H * (4 * 128 + 1) * es + w.T * w.H * 128 * 4) + \
            w.L * w.H * 3 * 128 * 4 * 4
        keeps = [[j + 1 for j in jt[i % R]] for i in range(Kc)]
        crb = sum(w.L * w.H * sum(1 for k in ks if k < w.T) * 2 * (128 * 128 + 9 * 128) * 4 for ks in keeps) / Kc
        res["col_stash"] = {"stash_bytes": col_bytes, "steps": Kc, "verify_ms": cv, "rollback_ms": cr,
                            "round_ms": cs, "verify_bytes": cvb, "rollback_bytes_mean": crb,
                            "verify_gbs": cvb / (cv * 1e-3) / 1e9,
                            "snapshot_replay": {"verify_ms": res["separate_rollback"]["verify_ms"],
                                                "rollback_ms": res["separate_rollback"]["rollback_ms"],
                                                "round_ms": res["separate_rollback"]["ms_per_step"],
                                                "stash_bytes": w.L * w.B * w.H * (128 * 128 + 9 * 128) * 4}}

    # sampled acceptance (run_sampled)
    if not args.no_sampled:
        res["sampled_accept"] = run_sampled(args, w, logits, K, j_out, keep_out, status, stream, dev, barrier,
                                            res["accept_ms"])

    # variable T per session: the window of each session's round from seeded drafter
    # confidences (glm5_conf_keep, p_min 0.5), then verify / accept / rollback with
    # per-session row counts, all decided on the device
    if w.B > 1 and not args.no_var_t:
        g = np.random.default_rng(w.seed + 17)
        conf = torch.from_numpy(g.uniform(0.3, 1.0, (w.B, w.K)).astype(np.float32)).to(dev)
        t_dev = kb.spec_window(conf, kb.WIN_CONF_KEEP, 0.5, w.T)
        t_host = [int(x) for x in t_dev.cpu()]
        Kv = max(1, min(args.var_t_steps, K))

        def var_step(r, ev):
            rr = plain[r]
            ev[0].record(stream)
            kb.kda_verify_scan_var(st, rr["q"], rr["k"], rr["v"], rr["g"], rr["beta"], t_dev, out=out, stash=stash,
                                   dev_status=status, stream=stream)
            ev[1].record(stream)
            kb.spec_accept_var(logits[r], drafts[r], t_dev, j_out, bonus_out, keep_out, status, scratch, stream)
            kb.kda_rollback_var(st, stash, t_dev, keep_out, status, stream)
            ev[2].record(stream)

        evv = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Kv + 3)]
        for i in range(3):
            var_step(i % R, evv[Kv + i])
        barrier()
        with nvtx_range("var_t"):
            for i in range(Kv):
                var_step(i % R, evv[i])
        barrier()
        if int(status.item()):
            raise RuntimeError(f"device status {int(status.item()):#x} after the variable-T steps")
        v_ms = sum(e[0].elapsed_time(e[1]) for e in evv[:Kv]) / Kv
        s_ms = sum(e[0].elapsed_time(e[2]) for e in evv[:Kv]) / Kv
        vb_var = verify_bytes_var(w, t_host)
        res["var_t"] = {"window": "glm5_conf_keep, p_min 0.5, slot confidences ~ U(0.3, 1) (seeded)",
                        "rows_mean": sum(t_host) / len(t_host), "rows_min": min(t_host), "rows_max": max(t_host),
                        "steps": Kv, "verify_ms": v_ms, "round_gpu_ms": s_ms,
                        "rows_per_s": world * sum(t_host) / (slowest(s_ms, world, dev) * 1e-3),
                        "verify_gbs": vb_var / (v_ms * 1e-3) / 1e9,
                        "verify_frac_of_peak": vb_var / (v_ms * 1e-3) / 1e9 / peak}
    return res


def host_cpu() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def workload_config(wname, args, step_bytes=None):
    from speculative_decode_verify_kda_gb300 import synth
    w = synth.WORKLOADS[wname]
    if step_bytes:
        l2 = (f"no flush: each step moves {step_bytes / 1e9:.2f} GB (the launch's own bytes and the accept's "
              f"logits), {step_bytes / 129e6:.1f}x the 129 MB L2")
    else:
        l2 = "no flush: every step moves more bytes than the 129 MB L2"
    return {"workload": wname, "description": WORKLOAD_TEXT[wname], "L": w.L, "B": w.B, "H": w.H, "T": w.T,
            "V": w.V, "rows_dtype": "bf16" if w.bf16 else "f32", "state_dtype": "f32", "l2": l2,
            "update_vectors": ("stored by each verify, read back by the replay" if args.replay_w == "on"
                               else "formed again by the replay"),
            "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single GPU"}


def roofline_of(wname, res, clocks) -> dict:
    """The roofline object of the deferred-round launch: achieved = algorithmic bytes per
    launch over its mean time; the kernel's own bytes and the DRAM traffic of an ncu
    capture (while the kernel source is the captured one) beside it."""
    peak = res["peak"]
    traffic = frac_dram = None
    same = code_hash(SCAN_SOURCE) == TRAFFIC_SOURCE
    captured_form = res.get("replay_w", True)  # the captures ran the launch that stores update vectors
    if wname in TRAFFIC_BYTES and same and captured_form:
        dram, own = TRAFFIC_BYTES[wname]
        traffic = dram * res["round_bytes_mean"] / own
        frac_dram = traffic / (res["round_kernel_ms"] * 1e-3) / 1e9 / peak
    if wname not in TRAFFIC_BYTES:
        tsrc = "no ncu capture of this workload's launch"
    elif same and not captured_form:
        tsrc = "null: the ncu captures ran the launch that stores the update vectors (--replay-w on)"
    elif same:
        tsrc = ("ncu capture of one launch (dram__bytes_read.sum + dram__bytes_write.sum) on this kernel "
                "source, scaled to the run's mean kernel bytes per launch")
    else:
        tsrc = "null: kda_scan.cu differs from the source the ncu capture was taken on"
    out = {"bound": "hbm", "kernel": "kda_scan_kernel (deferred round: rollback + verify)",
           "achieved": res["achieved"], "peak": peak, "unit": "GB/s", "frac": res["achieved"] / peak,
           "basis": "algorithmic bytes per launch: this round's verify at the ping-pong minimum and the "
                    "previous accept's rollback, each tensor once; over the launch's mean CUDA-event time",
           "target": "frac >= 0.70 on the 64-head, 34-layer workloads",
           "frac_of_nominal_8tbs": res["achieved"] / NOMINAL_HBM_GBS,
           "peak_source": f"{res['peak_kind']} (MEASURED_PEAKS.json hbm_gbs)",
           "bytes_per_launch": res["algo_bytes_mean"],
           "kernel_bytes_per_launch": res["round_bytes_mean"],
           "frac_kernel_bytes": res["achieved_kernel"] / peak,
           "traffic": traffic, "frac_dram": frac_dram, "traffic_source": tsrc,
           "launch_ms": res["round_kernel_ms"]}
    if clocks and clocks.get("sm_mhz"):
        out["launch_kcycles_at_median_clock"] = res["round_kernel_ms"] * clocks["sm_mhz"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stack34", choices=sorted(WORKLOAD_TEXT),
                    help="the headline workload (every section)")
    ap.add_argument("--workloads", default="batched32,stress64x34",
                    help="further workloads timed in the same run (deferred rounds and e2e), reported under "
                         "'workloads'; empty for none")
    ap.add_argument("--rounds", type=int, default=0, help="distinct input rounds kept resident (0: all)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--replay-w", choices=["on", "off"], default="on",
                    help="verifies store each row's update vector and replays read it back")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--e2e-rows", choices=["in_place", "staged"], default="in_place",
                    help="e2e raw rows: read in place from pinned host memory by the verify launch, or copied "
                         "to the device by range first")
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="ranges of (layer, session) pairs the e2e round's raw rows are copied in (the one "
                         "launch waits for each range's ready flag); 1: one copy, then the launch")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--no-per-layer", action="store_true", help="skip the per-layer (and CUDA graph) rounds")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the rounds")
    ap.add_argument("--per-layer-steps", type=int, default=200)
    ap.add_argument("--no-var-t", action="store_true", help="skip the variable-T rounds")
    ap.add_argument("--no-sampled", action="store_true", help="skip the sampled-accept timing")
    ap.add_argument("--no-cols", action="store_true", help="skip the column-stash rounds")
    ap.add_argument("--cols-steps", type=int, default=200)
    ap.add_argument("--sampled-steps", type=int, default=200)
    ap.add_argument("--var-t-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from speculative_decode_verify_kda_gb300 import synth
    w = synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        config = workload_config(args.workload, args)
        arm = OracleArm(w)
        ts, ta, n = arm.step(w.H)  # calibration: one whole unit-round
        per_head = ts / n
        budget = min(0.5, 90.0 / (args.steps + args.warmup))
        hps = int(max(1, min(w.H, budget // max(per_head, 1e-9))))
        t_scan = t_acc = 0.0
        heads = rounds = 0
        t_steps = 0.0
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            ts, ta, n = arm.step(hps)
            dt = time.perf_counter() - t0
            if i >= args.warmup:
                t_scan += ts
                t_steps += dt
                heads += n
                t_acc += ta * n / w.H  # one accept per round, spread over the round's heads
        val = arm.rows_per_s(t_scan / heads, t_acc / heads * w.H)
        sample = (f"each step: accept + verify + rollback of {hps} heads of one (layer, session) unit of "
                  f"{args.workload} (single-threaded oracle); value extrapolated linearly to {w.H} heads x "
                  f"{w.L} layers x {w.B} sessions per round")
        cores = 1
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_steps * 1e3 / args.steps,
                "step": f"{hps} heads of one (layer, session) unit: accept + verify + rollback",
                "extrapolated_ms_per_round": w.B * w.T / val * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded counter-based draws)", "config": config,
                "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                                 "cpu_model": host_cpu(), "host_cores": os.cpu_count()},
                "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import gc

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    subs = [x for x in args.workloads.split(",") if x and x != args.workload]
    for x in subs:
        if x not in WORKLOAD_TEXT:
            ap.error(f"unknown workload {x}")
    with ClockSampler(local_rank) as clk:
        res = run_gpu(args, rank, world, local_rank, args.workload, full=True)
        subres = {}
        for wn in subs:
            gc.collect()
            torch.cuda.empty_cache()
            subres[wn] = run_gpu(args, rank, world, local_rank, wn, full=False)
    clocks = clk.summary()
    cpu = cpu_threads = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = oracle_baseline(w, args.cpu_budget)
        cpu_threads = oracle_baseline_threads(w, args.cpu_budget, os.cpu_count() or 1)
        model = host_cpu()
        for c in (cpu, cpu_threads):
            c["cpu_model"] = model
            c["host_cores"] = os.cpu_count()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return
    workloads = {}
    for wn, r in subres.items():
        workloads[wn] = {"config": workload_config(wn, args, r["step_bytes_mean"]), "value": r["rows_per_s"],
                         "unit": UNIT, "steps": args.steps, "ms_per_step": r["ms_per_step"],
                         "round_kernel_ms": r["round_kernel_ms"], "accept_ms": r["accept_ms"],
                         "roofline": roofline_of(wn, r, clocks), "e2e": r.get("e2e"),
                         "sampled_accept": r.get("sampled_accept"),
                         "gpu_launches": r["launches_per_step"] * args.steps}
    line = {
        "metric": METRIC, "value": res["rows_per_s"], "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded counter-based draws; bf16 raw rows)",
        "config": workload_config(args.workload, args, res["step_bytes_mean"]),
        "roofline": roofline_of(args.workload, res, clocks),
        "round_kernel_ms": res["round_kernel_ms"], "accept_ms": res["accept_ms"],
        "step_achieved_gbs": res["step_gbs"],
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "cpu_baseline_threads": cpu_threads,
        "e2e": res.get("e2e"),
        "workloads": workloads,
        "separate_rollback": res.get("separate_rollback"),
        "in_place": res.get("in_place"),
        "graph": res.get("graph"),
        "per_layer": res.get("per_layer"),
        "var_t": res.get("var_t"),
        "sampled_accept": res.get("sampled_accept"),
        "col_stash": res.get("col_stash"),
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
