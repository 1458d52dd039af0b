"""Pins for the oracle's binary16 conversions (numpy's float16 is the library
routine for round-to-nearest; directed rounding is checked by its defining
bracketing property)."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _sample_f32_patterns():
    rng = np.random.default_rng(1)
    stride = np.arange(0, 2**32, 65537, dtype=np.uint64).astype(np.uint32)
    rand = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # neighbourhoods of every binary16 value (exact, halfway points, one ulp32 around)
    h = np.arange(0, 0x7C00, 7, dtype=np.uint16)
    hv = h.view(np.float16).astype(np.float32)
    nxt = (h + 1).view(np.float16).astype(np.float32)
    mid = ((hv.astype(np.float64) + nxt.astype(np.float64)) / 2).astype(np.float32)
    pats = [stride, rand, hv.view(np.uint32), mid.view(np.uint32), (mid.view(np.uint32) + 1),
            (mid.view(np.uint32) - 1)]
    allp = np.concatenate(pats).astype(np.uint32)
    allp = np.concatenate([allp, allp | np.uint32(0x80000000)])
    x = allp.view(np.float32)
    return x[~np.isnan(x)]


def test_f16_to_f32_exhaustive():
    h = np.arange(2**16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_round_nearest_matches_numpy():
    x = _sample_f32_patterns()
    got = oracle.f32_to_f16_bits(x, oracle.ROUND_NEAREST)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("mode", [oracle.ROUND_DOWN, oracle.ROUND_UP])
def test_directed_rounding_brackets(mode):
    x = _sample_f32_patterns()
    x = x[np.isfinite(x) & (np.abs(x) <= 65504.0)]
    h = oracle.f32_to_f16_bits(x, mode)
    v = h.view(np.float16)
    vf = v.astype(np.float64)
    xd = x.astype(np.float64)
    if mode == oracle.ROUND_DOWN:
        assert np.all(vf <= xd)
        # the next binary16 above the result is above x: the result is the largest value <= x
        up = np.nextafter(v, np.float16(np.inf)).astype(np.float64)
        assert np.all(up > xd)
    else:
        assert np.all(vf >= xd)
        dn = np.nextafter(v, np.float16(-np.inf)).astype(np.float64)
        assert np.all(dn < xd)
    # exactly representable inputs are unchanged
    exact = x.astype(np.float16).astype(np.float32) == x
    assert np.array_equal(h[exact], x[exact].astype(np.float16).view(np.uint16))


def test_directed_overflow_and_zero():
    vals = np.array([70000.0, -70000.0, 0.0, -0.0, 1e-30, -1e-30], np.float32)
    dn = oracle.f32_to_f16_bits(vals, oracle.ROUND_DOWN).view(np.float16)
    up = oracle.f32_to_f16_bits(vals, oracle.ROUND_UP).view(np.float16)
    assert dn[0] == np.float16(65504) and np.isinf(dn[1]) and dn[1] < 0
    assert np.isinf(up[0]) and up[0] > 0 and up[1] == np.float16(-65504)
    # tiny positive rounds down to +0 and up to the smallest subnormal (2^-24); mirrored for negatives
    assert dn[4] == 0 and up[4] == np.float16(2.0**-24)
    assert dn[5] == np.float16(-(2.0**-24)) and up[5] == 0
    assert oracle.f32_to_f16_bits(np.float32(-0.0), oracle.ROUND_DOWN) == 0x8000
