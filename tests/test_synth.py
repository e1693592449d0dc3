"""The synthetic input recipe (CPU): each configuration's length rule, the rounding of values to
bf16, and the rotary tables' angles."""

import math

import numpy as np

import synth


def lens_of(name):
    return synth.config_lens(name, np.random.default_rng(synth.CONFIG_NAMES.index(name)))


def test_length_rules():
    assert lens_of("tiny").tolist() == [37, 64, 150]
    g = lens_of("global")
    assert g.size == 64 and g.min() >= 32 and g.max() <= 512
    loc = lens_of("local")
    assert loc.size == 16 and loc.min() >= 1024 and loc.max() <= 8192
    lg = lens_of("long")
    assert lg.sum() == 131072 and lg.min() >= 1 and lg.max() <= 8192
    sh = lens_of("short")
    assert sh.sum() == 65536 and sh.min() >= 1 and sh.max() <= 16
    # lengths are drawn until the total reaches T and only the last one is cut
    assert np.all(lg[:-1] >= 1) and np.all(sh[:-1] >= 1)


def test_lengths_are_the_seeded_draws():
    # the same seed gives the same batch; another seed another one
    a = synth.config_lens("global", np.random.default_rng(1))
    b = synth.config_lens("global", np.random.default_rng(1))
    c = synth.config_lens("global", np.random.default_rng(2))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_cu_from_lens():
    cu = synth.cu_from_lens(np.asarray([3, 0, 5], dtype=np.int64))
    assert cu.tolist() == [0, 3, 3, 8]


def test_bf16_rounding_is_nearest_even():
    one = 0x3F80
    x = np.asarray([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9, -2.5, 0.0], dtype=np.float32)
    bits = synth.to_storage(x, "bf16")
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even significand (1);
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: ties go to 1 + 2^-6
    assert bits.tolist() == [one, one, one + 2, one, 0xC020, 0x0000]
    back = synth.to_f64(bits, "bf16")
    assert back.tolist() == [1.0, 1.0, 1.0 + 2.0 ** -6, 1.0, -2.5, 0.0]


def test_rope_table_angles():
    c, s = synth.rope_tables(8, 10000.0)
    assert c.shape == (8, 32) and s.shape == (8, 32)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    ang = 3 / 10000.0 ** (2 * 5 / 64)
    assert math.isclose(c[3, 5], math.cos(ang), rel_tol=0, abs_tol=1e-15)
    assert math.isclose(s[3, 5], math.sin(ang), rel_tol=0, abs_tol=1e-15)
