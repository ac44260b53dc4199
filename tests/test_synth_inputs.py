"""The seeded input generators (no GPU): the arbitrary encodings that stand
in for a compressed history hold the documented bit patterns, and every
generator is a pure function of its seed and counters."""
import numpy as np

from synth import synth as SY
from synth import workloads as WL


def test_random_encoding_fields():
    H, cap, D, S, G, C = 3, 200, 128, 2, 64, 16
    codes, meta, ids, cent = SY.random_encoding(11, SY.K_TENSOR, H, cap, D, S, G, C)
    assert codes.shape == (S, H, cap, D * 2 // 32) and codes.dtype == np.uint32
    assert meta.shape == (S, H, cap, D // G) and meta.dtype == np.uint32
    assert ids.shape == (H, cap) and ids.dtype == np.uint8 and int(ids.max()) < C
    assert cent.shape == (H, C, D) and cent.dtype == np.uint16
    scale = (meta & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    zero = (meta >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    assert scale.min() >= 2.0 ** -6 and scale.max() < 2.0 ** -5
    assert np.abs(zero).min() >= 2.0 ** -4 and np.abs(zero).max() < 2.0 ** -3
    assert (zero < 0).any() and (zero > 0).any()
    # 4-bit rows are twice as wide; no clusters means no ids or centroids
    c4, m4, i4, x4 = SY.random_encoding(11, SY.V_TENSOR, H, cap, D, 1, 32, 0, bits=4)
    assert c4.shape == (1, H, cap, D * 4 // 32) and m4.shape == (1, H, cap, D // 32)
    assert i4 is None and x4 is None


def test_generators_are_deterministic_and_keyed():
    a = SY.random_encoding(5, SY.K_TENSOR, 2, 64, 64, 2, 32, 8)
    b = SY.random_encoding(5, SY.K_TENSOR, 2, 64, 64, 2, 32, 8)
    c = SY.random_encoding(5, SY.V_TENSOR, 2, 64, 64, 2, 32, 8)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a[0], c[0])
    wl = WL.TINY
    q1 = SY.mixture_unit(wl, 0, SY.Q_TENSOR, 1, 0, 50)
    np.testing.assert_array_equal(q1, SY.mixture_unit(wl, 0, SY.Q_TENSOR, 1, 0, 50))
    assert not np.array_equal(q1, SY.mixture_unit(wl, 0, SY.K_TENSOR, 1, 0, 50))
    # a token's row does not depend on the range it is drawn in
    np.testing.assert_array_equal(q1[20:], SY.mixture_unit(wl, 0, SY.Q_TENSOR, 1, 20, 50))
