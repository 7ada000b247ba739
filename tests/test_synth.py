"""The seeded input generator: determinism, slicing, distributions, bf16 rounding."""
import numpy as np
import torch

from speculative_decode_verify_kda_gb300 import synth


def test_splitmix_reference_value():
    # SplitMix64 seeded with 0: its first output is 0xE220A8397B1DCDAF (Vigna's reference code)
    assert int(synth.stream(0, np.array([0], np.uint64))[0]) == 0xE220A8397B1DCDAF


def test_slices_equal_full_draw():
    key = synth.tensor_key(7, "q", 3)
    full = synth.normal(key, 0, 5000)
    assert np.array_equal(full[1234:1234 + 777], synth.normal(key, 1234, 777))
    w = synth.WORKLOADS["batched32"]
    w = synth.Workload("t", L=2, B=3, H=2, T=4, bf16=True, V=64, rounds=2, seed=9, accept="uniform")
    rows = synth.all_rows(w, 1)
    u = synth.unit_rows(w, 1, 1, 2)
    for n in synth.ROW_TENSORS:
        assert np.array_equal(rows[n][1, 2], u[n])
    assert np.array_equal(synth.all_state(w)[1, 2], synth.unit_state(w, 1, 2))
    assert np.array_equal(synth.all_ring(w)[0, 1], synth.unit_ring(w, 0, 1))
    assert np.array_equal(synth.all_conv_w(w)[1], synth.layer_conv_w(w, 1))
    # a shorter T draws a prefix of the rows
    u2 = synth.unit_rows(w, 1, 1, 2, T=2)
    assert np.array_equal(u2["g"], u["g"][:2])


def test_normal_moments_and_support():
    x = synth.normal(synth.tensor_key(1, "v"), 0, 400_000).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.01
    assert x.min() >= -6.0 and x.max() <= 6.0
    s = synth.normal(synth.tensor_key(1, "state"), 0, 100_000, 0.01)
    assert abs(s.std() - 0.01) < 2e-4
    u = synth.uniform_sym(synth.tensor_key(1, "conv_w"), 0, 100_000)
    assert u.min() >= -0.5 and u.max() < 0.5 and abs(u.mean()) < 0.01


def test_bf16_rounding_matches_torch():
    x = synth.normal(synth.tensor_key(2, "q"), 0, 50_000) * np.float32(3.7)
    ours = synth.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_bits_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_accept_targets_and_drafts():
    w = synth.WORKLOADS["stress64x34"]
    js = np.concatenate([synth.accept_targets(w, r) for r in range(16)])
    assert js.min() >= 0 and js.max() <= w.K
    assert 0.2 < np.mean(js == w.K) < 0.4
    # the drafts follow the row argmax up to j, then differ from it
    wl = synth.Workload("d", L=1, B=6, H=1, T=15, bf16=True, V=4096, rounds=1, seed=0x77, accept="uniform")
    vam = synth.logit_argmax(wl, 0)
    j = synth.accept_targets(wl, 0)
    d = synth.drafts_for(vam, j, wl.V)
    for b in range(wl.B):
        for r in range(wl.K):
            assert (d[b, r] == vam[b, r]) == (r < j[b])


def test_logits_are_normal_and_argmax_takes_the_first_tie():
    """Logits are the normal draws (mean 0, variance 1), bf16-rounded for bf16 workloads;
    the argmax is the lowest index among equal maxima (brute force per row)."""
    w = synth.Workload("l", L=1, B=2, H=1, T=8, bf16=True, V=32768, rounds=4, seed=0x78, accept="uniform")
    ties = 0
    for r in range(4):
        x = synth.bf16_bits_to_f32(synth.logits(w, r))
        assert abs(float(x.mean())) < 0.01 and abs(float(x.var()) - 1.0) < 0.02
        vam = synth.logit_argmax(w, r)
        for b in range(w.B):
            for t in range(w.T):
                hits = np.flatnonzero(x[b, t] == x[b, t].max())
                assert vam[b, t] == hits[0]
                ties += len(hits) > 1
    assert ties > 0  # at V = 32768 in bf16 a row maximum ties now and then
