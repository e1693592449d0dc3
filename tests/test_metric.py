"""The counts behind the reported metric (CPU): useful work is 256 flop per visible (query, key)
pair per head, counted here by brute force; algorithmic bytes are the sizes of the arrays the
path reads and writes once."""

import numpy as np

import synth


def brute_pairs(lens, window):
    total = 0
    for L in lens:
        for i in range(L):
            for j in range(L):
                if window == 0 or abs(i - j) <= window:
                    total += 1
    return total


def test_visible_pairs_brute_force():
    rng = np.random.default_rng(11)
    for _ in range(40):
        lens = [int(x) for x in rng.integers(0, 40, size=rng.integers(1, 6))]
        for window in (0, 1, 2, 5, 38, 39, 100):
            assert synth.visible_pairs(lens, window) == brute_pairs(lens, window), (lens, window)


def test_visible_pairs_edge_cases():
    assert synth.visible_pairs([], 0) == 0
    assert synth.visible_pairs([0, 0], 3) == 0
    assert synth.visible_pairs([1], 0) == 1
    assert synth.visible_pairs([5], 4) == 25  # a window of L - 1 lets every pair through
    assert synth.visible_pairs([5], 1) == 5 + 2 * 4  # the diagonal and the two next to it


def test_algorithmic_bytes_are_the_array_sizes():
    for name in ("tiny", "global", "short"):
        wl = synth.make_config(name)
        e = synth.elem_size(wl.dtype)
        qkv = np.asarray(wl.qkv)
        cos = np.asarray(wl.cos)
        want = (qkv.size * e                     # qkv read once
                + wl.T * wl.H * 64 * e            # out written once
                + 4 * wl.H * wl.T                 # lse (fp32) written once
                + 2 * cos.size * e                # cos and sin tables read
                + 4 * (wl.S + 1))                 # cu read
        assert synth.algorithmic_bytes(wl) == want, name
