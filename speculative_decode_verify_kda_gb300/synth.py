"""Seeded synthetic inputs for the KDA verify walk.

This module is the one piece that both the CUDA path's callers (tests, bench)
and the CPU oracle's callers share.  It holds none of the method's arithmetic:
it only draws numbers and lays them out.

Generator (counter based, so any slice of any tensor can be drawn on its own,
on the CPU here or on the GPU by ``csrc/synth_fill.cu``, bit for bit the same):

* ``out(c)`` is output number ``c`` of a SplitMix64 stream whose state starts at
  the tensor key: ``mix(key + (c + 1) * GAMMA)`` with SplitMix64's published
  golden-ratio increment and finaliser (Steele, Lea and Flood, 2014).
* A normal-like draw for element ``n`` sums twelve 16-bit uniforms taken from
  ``out(3n)``, ``out(3n+1)``, ``out(3n+2)`` (Irwin-Hall with 12 terms: mean 0,
  variance exactly 1, support [-6, 6]); the sum minus its mean, times 2^-16, is
  exact in f32.  A sigma other than 1 is applied by one f32 multiply.
* A symmetric uniform draw for element ``n`` takes the top 24 bits of ``out(n)``:
  ``(u - 2^23) * 2^-24`` in [-0.5, 0.5), exact in f32, then one f32 multiply.
* bf16 values are the f32 draws rounded to nearest-even on the top 16 bits.

Workloads (the five shapes the library is measured and checked on) are described
by ``Workload``; layouts are the library's: raw rows [L][B][T][H][128] (beta
[L][B][T][H]), state [L][B][H][128][128], conv ring [L][B][H][3][3][128], conv
weights [L][H][3][128][4], logits [B][T][V].
"""
from __future__ import annotations

import dataclasses

import numpy as np

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
KEY_MUL = 0xD1B54A32D192ED03

D = 128
TAPS = 4

# stable tensor ids: keys must never change, stored fixtures depend on them
TENSOR_IDS = {
    "state": 1, "ring": 2, "conv_w": 3,
    "q": 4, "k": 5, "v": 6, "g": 7, "beta": 8,
    "logits": 9, "plant": 10, "accept": 11,  # "plant": no longer drawn, its id stays reserved
}
ROW_TENSORS = ("q", "k", "v", "g", "beta")


def _mix_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def tensor_key(seed: int, name: str, round_idx: int = 0) -> int:
    """64-bit stream key of one tensor (of one verify round)."""
    k = _mix_int(seed + TENSOR_IDS[name] * KEY_MUL)
    return _mix_int(k + (round_idx + 1) * GAMMA)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def stream(key: int, counters: np.ndarray) -> np.ndarray:
    """``out(c)`` for each counter ``c`` (uint64 array)."""
    c = counters.astype(np.uint64) + np.uint64(1)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + c * np.uint64(GAMMA))


def normal(key: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """Elements ``start .. start+count-1`` of a normal-like f32 tensor."""
    n = np.arange(start, start + count, dtype=np.uint64)
    total = np.zeros(count, dtype=np.int64)
    for m in range(3):
        r = stream(key, n * np.uint64(3) + np.uint64(m))
        for f in range(4):
            total += ((r >> np.uint64(16 * f)) & np.uint64(0xFFFF)).astype(np.int64)
    z = (total - 393210).astype(np.float32) * np.float32(2.0 ** -16)
    if sigma != 1.0:
        z = z * np.float32(sigma)
    return z


def uniform_sym(key: int, start: int, count: int, half_width: float = 0.5) -> np.ndarray:
    """Elements of a U(-half_width, half_width) f32 tensor."""
    n = np.arange(start, start + count, dtype=np.uint64)
    u = (stream(key, n) >> np.uint64(40)).astype(np.int64)
    x = (u - (1 << 23)).astype(np.float32) * np.float32(2.0 ** -24)
    if half_width != 0.5:
        x = x * np.float32(2.0 * half_width)
    return x


def integers(key: int, start: int, count: int, bound: int) -> np.ndarray:
    """Integers in [0, bound) (modulo reduction of ``out(n)``; the bias is immaterial)."""
    n = np.arange(start, start + count, dtype=np.uint64)
    return (stream(key, n) % np.uint64(bound)).astype(np.int64)


def unit_floats(key: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of ``out(n)``."""
    n = np.arange(start, start + count, dtype=np.uint64)
    return (stream(key, n) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """f32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    L: int
    B: int
    H: int
    T: int
    bf16: bool
    V: int
    rounds: int
    seed: int
    accept: str  # "uniform" j ~ U{0..K}; "skewed" P(j=K)=0.3 else U{0..K-1}; "sweep" j = round mod (K+1)
    state_sigma: float = 0.01
    ring_sigma: float = 0.1
    conv_half_width: float = 0.5

    @property
    def K(self) -> int:
        return self.T - 1

    def per_row(self, name: str) -> int:
        return self.H * (D if name != "beta" else 1)

    def per_unit(self, name: str) -> int:
        return self.T * self.per_row(name)


WORKLOADS = {
    # one head, f32 rows, V=32 logits, every accept j swept
    "tiny": Workload("tiny", L=1, B=1, H=1, T=8, bf16=False, V=32, rounds=8,
                     seed=0x5EED0001, accept="sweep"),
    # one glm5_next-shaped KDA layer
    "layer64": Workload("layer64", L=1, B=1, H=64, T=8, bf16=True, V=32768, rounds=1000,
                        seed=0x5EED0002, accept="uniform"),
    # the 34-layer KDA stack of one session, 64 consecutive rounds
    "stack34": Workload("stack34", L=34, B=1, H=64, T=8, bf16=True, V=32768, rounds=64,
                        seed=0x5EED0003, accept="uniform"),
    # 32 independent sessions of one layer at the T=15 cap
    "batched32": Workload("batched32", L=1, B=32, H=64, T=15, bf16=True, V=32768, rounds=16,
                          seed=0x5EED0004, accept="uniform"),
    # 64 sessions x 34 layers at T=15, skewed accept, 16 rounds
    "stress64x34": Workload("stress64x34", L=34, B=64, H=64, T=15, bf16=True, V=32768,
                            rounds=16, seed=0x5EED0005, accept="skewed"),
}


def unit_rows(w: Workload, round_idx: int, l: int, b: int, T: int | None = None) -> dict:
    """Raw rows q, k, v, g, beta of one (layer, session) unit of one round.

    Shapes [T][H][128] (beta [T][H]); f32, or uint16 bf16 bits when ``w.bf16``.
    A smaller ``T`` draws only the first rows (a prefix of the full draw).
    """
    T = w.T if T is None else T
    out = {}
    for name in ROW_TENSORS:
        start = (l * w.B + b) * w.per_unit(name)
        x = normal(tensor_key(w.seed, name, round_idx), start, T * w.per_row(name))
        x = x.reshape((T, w.H, D) if name != "beta" else (T, w.H))
        out[name] = to_bf16_bits(x) if w.bf16 else x
    return out


def all_rows(w: Workload, round_idx: int) -> dict:
    """Raw rows of every unit: [L][B][T][H](128) each."""
    out = {}
    for name in ROW_TENSORS:
        x = normal(tensor_key(w.seed, name, round_idx), 0, w.L * w.B * w.per_unit(name))
        x = x.reshape((w.L, w.B, w.T, w.H) + ((D,) if name != "beta" else ()))
        out[name] = to_bf16_bits(x) if w.bf16 else x
    return out


def unit_state(w: Workload, l: int, b: int) -> np.ndarray:
    n = w.H * D * D
    return normal(tensor_key(w.seed, "state"), (l * w.B + b) * n, n, w.state_sigma).reshape(w.H, D, D)


def unit_ring(w: Workload, l: int, b: int) -> np.ndarray:
    n = w.H * 3 * 3 * D
    return normal(tensor_key(w.seed, "ring"), (l * w.B + b) * n, n, w.ring_sigma).reshape(w.H, 3, 3, D)


def layer_conv_w(w: Workload, l: int) -> np.ndarray:
    n = w.H * 3 * D * TAPS
    return uniform_sym(tensor_key(w.seed, "conv_w"), l * n, n, w.conv_half_width).reshape(w.H, 3, D, TAPS)


def all_state(w: Workload) -> np.ndarray:
    n = w.L * w.B * w.H * D * D
    return normal(tensor_key(w.seed, "state"), 0, n, w.state_sigma).reshape(w.L, w.B, w.H, D, D)


def all_ring(w: Workload) -> np.ndarray:
    n = w.L * w.B * w.H * 9 * D
    return normal(tensor_key(w.seed, "ring"), 0, n, w.ring_sigma).reshape(w.L, w.B, w.H, 3, 3, D)


def all_conv_w(w: Workload) -> np.ndarray:
    n = w.L * w.H * 3 * D * TAPS
    return uniform_sym(tensor_key(w.seed, "conv_w"), 0, n, w.conv_half_width).reshape(w.L, w.H, 3, D, TAPS)


# ---------------------------------------------------------------------------
# Accept-side inputs: normal logits and drafts that follow the row argmax up to j
# ---------------------------------------------------------------------------
def accept_targets(w: Workload, round_idx: int) -> np.ndarray:
    """Target accepted-draft count j per session for one round."""
    K = w.K
    if w.accept == "sweep":
        return np.full(w.B, round_idx % (K + 1), dtype=np.int64)
    key = tensor_key(w.seed, "accept", round_idx)
    if w.accept == "uniform":
        return integers(key, 0, w.B, K + 1)
    if w.accept == "skewed":
        u = unit_floats(key, 0, 2 * w.B).reshape(w.B, 2)
        j = np.minimum((u[:, 1] * K).astype(np.int64), K - 1)
        return np.where(u[:, 0] < 0.3, K, j)
    raise ValueError(w.accept)


def drafts_for(vam: np.ndarray, j: np.ndarray, V: int) -> np.ndarray:
    """Drafts [B][T-1]: the row argmax (vam [B][T]) before position j, a different id from
    j on, so that greedy acceptance accepts exactly j drafts."""
    B, T = vam.shape
    r = np.arange(T - 1)[None, :]
    hit = vam[:, : T - 1]
    miss = (hit + 1) % V
    return np.where(r < np.asarray(j)[:, None], hit, miss).astype(np.int32)


def logits(w: Workload, round_idx: int, sessions=None) -> np.ndarray:
    """Logits [B][T][V]: normal draws (mean 0, variance 1), rounded to bf16 for bf16
    workloads, so that at V = 32768 a row's maximum can tie."""
    sessions = range(w.B) if sessions is None else sessions
    key = tensor_key(w.seed, "logits", round_idx)
    rows = []
    for b in sessions:
        x = normal(key, b * w.T * w.V, w.T * w.V).reshape(w.T, w.V)
        rows.append(to_bf16_bits(x) if w.bf16 else x)
    return np.stack(rows)


def logit_argmax(w: Workload, round_idx: int, sessions=None) -> np.ndarray:
    """The argmax of each logits row, [B][T], the lowest index winning ties (bf16 rows
    compared after exact widening): the token a draft must equal to be accepted."""
    sessions = range(w.B) if sessions is None else sessions
    out = []
    for b in sessions:
        x = logits(w, round_idx, [b])[0]
        out.append((bf16_bits_to_f32(x) if w.bf16 else x).argmax(-1))
    return np.stack(out).astype(np.int64)
