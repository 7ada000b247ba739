"""Host-side checks of bench.py's accounting (no GPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decode_verify_kda_gb300 import synth  # noqa: E402


def test_traffic_constants_belong_to_this_kernel_source():
    """The DRAM traffic bench.py reports comes from an ncu capture of kda_scan_kernel; a
    change to the kernel's code (comments aside) needs a new capture and new constants."""
    assert bench.code_hash(bench.SCAN_SOURCE) == bench.TRAFFIC_SOURCE


def test_code_hash_ignores_comments_and_space(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text('int f(int x) { return x + 1; }  // one\n/* block */ const char *s = "a // b";\n')
    b.write_text('// other words\nint f(int x)\n{\n    return x + 1;\n}\nconst char *s = "a // b";\n')
    c.write_text('int f(int x) { return x + 2; }\nconst char *s = "a // b";\n')
    assert bench.code_hash(str(a)) == bench.code_hash(str(b))
    assert bench.code_hash(str(a)) != bench.code_hash(str(c))


def test_algorithmic_bytes_by_hand():
    """Per (session, layer) at 64 heads with bf16 rows: the verify moves the state twice
    (8 MiB), T raw rows of 64 x (4 x 128 + 1) x 2 B, T output rows of 32 KiB and the
    ring twice (576 KiB); the layer's conv weights are 384 KiB; a rollback to keep rows
    moves the state and ring twice again and reads keep raw rows."""
    w = synth.WORKLOADS["stack34"]
    row = 64 * (4 * 128 + 1) * 2
    assert row == 65664
    verify = 8 * 2**20 + 8 * row + 8 * 32768 + 576 * 1024 + 384 * 1024
    rollback = 8 * 2**20 + 576 * 1024 + 4 * row
    assert bench.algorithmic_bytes(w, [4]) == 34 * (verify + rollback)
    assert bench.algorithmic_bytes(w, [8]) == 34 * verify  # a full accept rolls nothing back
    wb = synth.WORKLOADS["batched32"]
    v15 = 8 * 2**20 + 15 * row + 15 * 32768 + 576 * 1024
    keeps = [1, 15, 7] + [15] * 29
    expect = 32 * v15 + 384 * 1024 + sum(8 * 2**20 + 576 * 1024 + k * row for k in keeps if k < 15)
    assert bench.algorithmic_bytes(wb, keeps) == expect


def test_fused_launch_moves_fewer_bytes_than_the_steps():
    """The deferred launch folds the rollback into the verify: its own bytes never
    exceed the algorithmic bytes of the two steps, beyond the update vectors it stores
    and reads back when it keeps them (f32, 512 B a head and row)."""
    for name in ("stack34", "batched32", "stress64x34"):
        w = synth.WORKLOADS[name]
        for keeps in ([1] * w.B, [w.T] * w.B, [max(1, w.T // 2)] * w.B):
            algo = bench.algorithmic_bytes(w, keeps)
            assert bench.deferred_bytes(w, keeps) <= algo
            wv = w.L * w.H * 512 * sum(w.T + (k if k < w.T else 0) for k in keeps)
            assert bench.deferred_bytes(w, keeps, stored_w=True) == bench.deferred_bytes(w, keeps) + wv
