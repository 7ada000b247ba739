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


def test_device_drafts_equal_cpu_drafts_with_ties():
    """The bench's drafts (row argmax of the device logits, the lowest index among equal
    maxima) equal the CPU's at V = 32768 in bf16, where row maxima tie now and then."""
    w = synth.Workload("dr", L=1, B=4, H=1, T=15, bf16=True, V=32768, rounds=3, seed=0x79, accept="uniform")
    ties = 0
    for r in range(3):
        d_gpu, j = synth_gpu.drafts(w, r)
        vam = synth.logit_argmax(w, r)
        assert np.array_equal(host(d_gpu), synth.drafts_for(vam, synth.accept_targets(w, r), w.V))
        assert j == [int(x) for x in synth.accept_targets(w, r)]
        x = synth.bf16_bits_to_f32(synth.logits(w, r))
        ties += int(((x == x.max(-1, keepdims=True)).sum(-1) > 1).sum())
    assert ties > 0
