"""The tile-autotuning cache's key (CPU): the pages' attend_tuned key, restated here from its
definition -- heads, the window as w + 1 (0 for every key), the token count and the longest
sequence rounded up to powers of two -- and the kernel each call runs without tuning."""

import random

import pytest

import rope_cu_tile_gb300 as pk


@pytest.fixture(scope="module")
def lib():
    from rope_cu_tile_gb300 import build

    build.build()
    return pk.load()


def next_pow2(n: int) -> int:
    return 1 if n <= 1 else 1 << (n - 1).bit_length()


@pytest.mark.parametrize("seed", range(4))
def test_key_is_the_pages_key(lib, seed):
    rng = random.Random(seed)
    names = {pk.PK_F32: "f32", pk.PK_BF16: "bf16", pk.PK_F16: "f16"}
    for _ in range(50):
        dt = rng.choice(list(names))
        H = rng.randint(1, 64)
        w = rng.choice([0, 0, 1, 4, 16, 17, 64, rng.randint(0, 5000)])
        T = rng.choice([1, 2, 3, 1000, 16931, 65536, 131072, rng.randint(1, 1 << 24)])
        longest = rng.randint(0, T)
        want = (f"dtype={names[dt]},heads={H},window={w + 1 if w else 0},tokens={next_pow2(T)},"
                f"longest={next_pow2(longest)}")
        assert pk.pk_tune_key(dt, H, w, T, longest) == want


def test_key_rejects_bad_arguments(lib):
    import ctypes

    buf = ctypes.create_string_buffer(8)
    assert lib.pk_tune_key(1, 12, 0, 1000, 10, buf, 8) == 1   # does not fit
    buf = ctypes.create_string_buffer(128)
    assert lib.pk_tune_key(1, 0, 0, 1000, 10, buf, 128) == 1  # H < 1
    assert lib.pk_tune_key(1, 1, -1, 1000, 10, buf, 128) == 1  # window < 0


def test_untuned_dispatch(lib):
    for dt in (pk.PK_F32, pk.PK_BF16, pk.PK_F16):
        for w in range(1, 17):
            assert pk.pk_forward_kernel(dt, w) == 0            # band: narrow windows, fp32 arithmetic
        for w in (0, 17, 64, 1000):
            assert pk.pk_forward_kernel(dt, w) == (1 if dt == pk.PK_F32 else 2)
    assert [pk.pk_kernel_name(k) for k in range(5)][:4] == [
        "pk_attend_band_kernel", "pk_attend_f32_kernel", "pk_attend_tc_kernel", "pk_attend_q4_kernel"]
    assert pk.pk_kernel_name(5) == "pk_attend_split_kernel"
    assert pk.pk_kernel_name(99) == ""
