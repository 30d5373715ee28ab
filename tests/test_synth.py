"""The seeded generator shared by both sides (synth/): determinism, rounding, recipe."""
import numpy as np
import pytest

import synth


def test_f16_rounding_matches_numpy():
    # numpy's float64 -> float16 cast is a correctly rounded library routine (RNE).
    rng = np.random.default_rng(0)
    xs = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 11.5, 20000))
    specials = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0**-24, 2.0**-25,
                         3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11])
    L = synth.lib()
    for x in np.concatenate([xs, specials, -specials]):
        want = np.array(x).astype(np.float16).view(np.uint16)
        assert L.synth_f16_from_double(float(x)) == want, x


def test_splitmix64_reference_values():
    """The finaliser reproduces SplitMix64's published first outputs for seed 0, and every
    draw of the C generator is that finaliser applied to key + (i+1)*gamma (synth.h)."""
    gamma, tagmul, m64 = 0x9E3779B97F4A7C15, 0xD1B54A32D192ED03, 2**64 - 1

    def mix(z):
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m64
        return z ^ (z >> 31)

    assert [mix((i + 1) * gamma & m64) for i in range(3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                                               0x06C45D188009454F]
    for seed, tag in [(0, 0), (1, 5), (12345, 7)]:
        key = mix(seed ^ ((tagmul * (tag + 1)) & m64))
        for i in (0, 1, 1000):
            assert synth.lib().synth_draw_u64(seed, tag, i) == mix((key + (i + 1) * gamma) & m64)


def test_normal_moments_and_determinism():
    a = synth.normal(3, 11, (200000,)).astype(np.float64)
    b = synth.normal(3, 11, (200000,)).astype(np.float64)
    c = synth.normal(4, 11, (200000,)).astype(np.float64)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    # fourth moment of a Gaussian is 3
    assert abs((a**4).mean() - 3.0) < 0.06


def test_uniform_pixels_range_and_prefix():
    p2 = synth.pixels(1, 2).astype(np.float64)
    p1 = synth.pixels(1, 1).astype(np.float64)
    assert p2.shape == (2, 729, 588)
    assert np.array_equal(p2[:1], p1)
    assert p2.min() >= -1.0 and p2.max() <= 1.0
    assert abs(p2.mean()) < 0.01 and abs(p2.var() - 1.0 / 3.0) < 0.01


def test_recipe_so400m():
    d = synth.so400m(27)
    infos = synth.tensor_infos(d)
    assert len(infos) == 3 + 12 * 27 + 15
    by = {(t.name.decode(), t.layer): t for t in infos}
    assert (by[("qkv_w", 0)].rows, by[("qkv_w", 0)].cols) == (1152, 3456)
    assert by[("qkv_w", 5)].std == pytest.approx(np.sqrt(2 / 2304))
    assert by[("fc1_w", 26)].std == pytest.approx(np.sqrt(2 / (1152 + 4304)))
    assert by[("patch_w", -1)].std == pytest.approx(np.sqrt(2 / (588 + 1152)))
    assert by[("pos", -1)].std == pytest.approx(1 / np.sqrt(1152))
    assert by[("map_kv_w", -1)].cols == 2304
    assert by[("ln1_g", 3)].kind == 1 and by[("ln1_g", 3)].mean == 1.0
    n_params = sum(t.rows * t.cols for t in infos)
    assert 420e6 < n_params < 432e6  # So400m/14 image tower with MAP head


def test_transposed_fill_matches_logical_order():
    d = synth.vit_small(2)
    import ctypes
    for tid in (0, 5, 11, 3 + 24 + 13):
        w = synth.tensor(9, d, tid)
        K, N = w.shape
        kpad = (K + 63) // 64 * 64
        out = np.full((N, kpad), np.float16(7), dtype=np.float16)
        rc = synth.lib().synth_fill_tensor_f16_t(9, ctypes.byref(d), tid, out.ctypes.data, kpad)
        assert rc == 0
        assert np.array_equal(out[:, :K], w.T)
        assert np.all(out[:, K:] == 0)
