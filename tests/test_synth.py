"""The seeded generator: SplitMix64 vectors, bf16 rounding, moments, determinism."""
import numpy as np
import torch

import synth
from synth import generator as g


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 started from state 0 (state advances by the golden increment)
    golden = 0x9E3779B97F4A7C15
    states = np.array([0, golden, (2 * golden) & ((1 << 64) - 1)], dtype=np.uint64)
    out = [int(x) for x in g.splitmix64(states)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0, 1e-30, 3e38],
                                 dtype=np.float32)])
    ours = g.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # ties go to even
    assert g.bf16_bits_to_f64(g.f32_to_bf16_bits(np.float32(1 + 2 ** -8))) == 1.0
    assert g.bf16_bits_to_f64(g.f32_to_bf16_bits(np.float32(1 + 3 * 2 ** -8))) == 1 + 2 ** -6


def test_irwin_hall_moments_and_range():
    key = g.counter_key(1, g.TAG_K, np.arange(4000), 0, 0)
    x = g.normal_fp32(key, 256).astype(np.float64).ravel()
    assert abs(x.mean()) < 0.005 and abs(x.var() - 1.0) < 0.01
    assert np.abs(x).max() <= 6.0
    # exact multiples of 2^-12
    assert np.all(x * 4096 == np.round(x * 4096))
    # fourth moment of Irwin-Hall(12) shifted: 3 - 1.2/12 = 2.9
    assert abs((x ** 4).mean() - 2.9) < 0.05


def test_determinism_and_independence():
    a = synth.token_tensor(5, synth.TAG_Q, 3, 2, [10, 11], 4, 8, 0.25)
    b = synth.token_tensor(5, synth.TAG_Q, 3, 2, [10, 11], 4, 8, 0.25)
    c = synth.token_tensor(5, synth.TAG_K, 3, 2, [10, 11], 4, 8, 0.25)
    d = synth.token_tensor(5, synth.TAG_Q, 4, 2, [10, 11], 4, 8, 0.25)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    assert a.shape == (2, 4, 8) and a.dtype == np.uint16


def test_scale_is_an_fp32_multiply():
    key = g.counter_key(9, g.TAG_V, 0, 0, np.arange(10))
    x = g.normal_fp32(key, 64)
    s = np.float32(1 / np.sqrt(128))
    bits = g.normal_bf16_bits(key, 64, float(s))
    assert np.array_equal(bits, g.f32_to_bf16_bits(x * s))


def test_workload_recipes():
    w = synth.workload("mixed")
    assert sorted(set(w.windows().tolist())) == [188, 250, 375]
    assert w.start_offsets().max() < 2_000_000
    # every stream steps exactly once per clock period
    counts = np.zeros(w.n_streams, dtype=int)
    for t in range(12):
        counts[w.active_at_tick(t)] += 1
    assert np.array_equal(counts, 12 * 40 // w.stream_clocks())
    assert synth.workload("qwen").input_scale == float(np.float32(1 / np.sqrt(128)))
    assert synth.workload("tiny").input_scale == 1.0
