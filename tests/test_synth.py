"""The seeded generator shared by the oracle and the GPU side (host half)."""

import numpy as np

import synth


def test_splitmix64_reference_sequence():
    # SplitMix64 started from state 0 (Vigna's splitmix64.c): the published first outputs
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]
    got = [synth.mix64_int((synth.GOLDEN * i) & synth.MASK64) for i in range(1, 5)]
    assert got == expect
    # the counter form with key 0 is the same sequence
    z = np.arange(4, dtype=np.uint64) + np.uint64(1)
    z *= np.uint64(synth.GOLDEN)
    assert [int(v) for v in synth._mix64(z)] == expect


def test_array_and_scalar_mix_agree():
    idx = np.array([0, 1, 2, 1 << 35, (1 << 40) + 7], dtype=np.uint64)
    key = synth.stream_key(7, 11)
    arr = synth.bits(7, 11, idx)
    ref = [synth.mix64_int((key + (int(i) + 1) * synth.GOLDEN) & synth.MASK64) for i in idx]
    assert [int(a) for a in arr] == ref


def test_normal_draws_moments_bounds_and_no_negative_zero():
    b = synth.normal_bf16_bits(0, 3, 1 << 20, 1.0)
    x = synth.bf16_bits_to_f32(b).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert np.abs(x).max() <= 3.47
    assert not np.any(b == 0x8000)
    w = synth.bf16_bits_to_f32(synth.normal_bf16_bits(0, 4, 1 << 18, 0.02)).astype(np.float64)
    assert abs(w.std() - 0.02) < 2e-4


def test_chunking_and_offsets_do_not_change_values():
    a = synth.normal_bf16_bits(0, 9, 1000, 0.02, chunk=64)
    b = synth.normal_bf16_bits(0, 9, 1000, 0.02)
    c = synth.normal_bf16_bits(0, 9, 500, 0.02, start=500)
    assert np.array_equal(a, b) and np.array_equal(a[500:], c)


def test_token_ids_range_and_uniformity():
    ids = synth.token_ids(3, 0, 200000, 1024)
    assert ids.min() >= 0 and ids.max() < 1024
    counts = np.bincount(ids, minlength=1024)
    assert counts.min() > 100 and counts.max() < 300
    big = synth.token_ids(3, 0, 100000, 151936)
    assert big.max() < 151936


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-5], dtype=np.float32)
    b = synth._f32_to_bf16_bits(x)
    back = synth.bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins; 1 + 3*2^-8 rounds up to 1 + 2^-6
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0 + 2 ** -6)
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-5) / 3.0e-5 < 2 ** -8


def test_norm_weights_default_to_one():
    s = synth.TINY
    assert np.all(synth.layer_weight_bits(s, 0, synth.W_IN_NORM) == 0x3F80)
    p = synth.bf16_bits_to_f32(synth.layer_weight_bits(s, 0, synth.W_IN_NORM, perturbed_norms=True))
    assert abs(float(p.mean()) - 1.0) < 0.03 and 0.05 < float(p.std()) < 0.15
