"""The device fill of the seeded inputs equals the CPU draw bit for bit."""
import numpy as np
import pytest
import torch

from gpu_util import host
from libs import ensure_built

from speculative_decode_verify_kda_gb300 import synth, synth_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def test_device_fill_equals_cpu_draw():
    w = synth.Workload("s", L=2, B=3, H=4, T=5, bf16=True, V=300, rounds=2, seed=123, accept="uniform")
    rows_c = synth.all_rows(w, 1)
    rows_g = synth_gpu.rows(w, 1)
    for n in synth.ROW_TENSORS:
        assert np.array_equal(host(rows_g[n]), rows_c[n]), n
    assert np.array_equal(host(synth_gpu.state(w)), synth.all_state(w))
    assert np.array_equal(host(synth_gpu.ring(w)), synth.all_ring(w))
    assert np.array_equal(host(synth_gpu.conv_w(w)), synth.all_conv_w(w))
    assert np.array_equal(host(synth_gpu.logits(w, 1)), synth.logits(w, 1))
    wf = synth.WORKLOADS["tiny"]
    assert np.array_equal(host(synth_gpu.rows(wf, 3)["k"]), synth.all_rows(wf, 3)["k"])
    assert np.array_equal(host(synth_gpu.logits(wf, 3)), synth.logits(wf, 3))


def test_device_fill_at_large_offsets():
    key = synth.tensor_key(5, "q", 9)
    t = torch.empty(100_000, dtype=torch.bfloat16, device="cuda")
    synth_gpu.fill_normal(t, key, start=3_000_000_000)
    assert np.array_equal(host(t), synth.to_bf16_bits(synth.normal(key, 3_000_000_000, 100_000)))
