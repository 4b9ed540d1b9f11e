"""The seeded input generator (no GPU)."""
import numpy as np

import synth


def test_splitmix64_reference_words():
    # SplitMix64 seeded with 0: published first outputs of the reference
    # generator (Steele, Lea, Flood 2014; Vigna's splitmix64.c).
    out = np.empty(3, dtype=np.uint64)
    synth._get().synth_words(0, 0, 3, out.ctypes.data)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_and_deterministic():
    a = synth.words(5, 1, 2, 0, 100)
    b = synth.words(5, 1, 2, 40, 10)
    assert np.array_equal(a[40:50], b)
    assert not np.array_equal(synth.words(5, 1, 3, 0, 10), a[:10])
    x1 = synth.normal_bf16((64, 32), 9, synth.T_A, 1)
    x2 = synth.normal_bf16((64, 32), 9, synth.T_A, 1)
    assert np.array_equal(x1, x2)


def test_distributions():
    K = 2048
    x = synth.bf16_bits_to_f32(synth.normal_bf16((256, 1024), 1, synth.T_A, 0, 0.0, 1.0 / np.sqrt(K)))
    assert abs(x.mean()) < 2e-4 and abs(x.std() * np.sqrt(K) - 1) < 1e-2
    u = synth.bf16_bits_to_f32(synth.uniform_bf16((100000,), 1, synth.T_B))
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 1e-2
    g = synth.normal_f32((7168,), 1, synth.T_GAMMA, 0, 1.0, 0.1)
    assert abs(g.mean() - 1) < 5e-3 and abs(g.std() - 0.1) < 5e-3


def test_negzero_injection():
    parts, res, gamma = synth.ar_inputs(8, 64, 7168, synth.config_seed(4))
    frac = np.mean([np.mean(p == synth.BF16_NEG_ZERO) for p in parts])
    assert 0.009 < frac < 0.011
    assert res.shape == (64, 7168) and gamma.dtype == np.float32
