"""Pins of the oracle's IEEE binary16 conversions against numpy's float16,
an independent implementation: every one of the 65,536 codes widened, and
the narrowing checked on all codes, every midpoint between neighbours (the
ties), the overflow threshold, the subnormal range and a wide random sample
of binary32 bit patterns."""
import numpy as np
import pytest


def _np_half_to_float(codes):
    return codes.view(np.float16).astype(np.float32)


def _np_float_to_half(x):
    with np.errstate(over="ignore", invalid="ignore"):
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def _same_halves(a, b):
    """Equal codes, except that any two NaNs count as equal."""
    a = np.asarray(a, np.uint16)
    b = np.asarray(b, np.uint16)
    nan_a = ((a & 0x7C00) == 0x7C00) & ((a & 0x3FF) != 0)
    nan_b = ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)
    return bool(np.all(nan_a == nan_b) and np.all((a == b) | nan_a))


def test_widen_all_codes(oracle_mod):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.half_to_float(codes)
    ref = _np_half_to_float(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_narrow_round_trip_all_codes(oracle_mod):
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = _np_half_to_float(codes)
    assert _same_halves(oracle_mod.float_to_half(f), codes)


def test_narrow_ties_and_midpoints(oracle_mod):
    # every pair of neighbouring finite positive halves, and their midpoint
    # (12 significant bits: exact in binary32) plus one binary32 ulp each side
    pos = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    lo = _np_half_to_float(pos[:-1]).astype(np.float64)
    hi = _np_half_to_float(pos[1:]).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)
    cases = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)),
                            np.nextafter(mid, np.float32(0))])
    cases = np.concatenate([cases, -cases])
    assert _same_halves(oracle_mod.float_to_half(cases), _np_float_to_half(cases))


def test_narrow_overflow_subnormal_and_specials(oracle_mod):
    cases = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e30, np.inf, -np.inf,
                      np.nan, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26,
                      2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 6.0e-8, 1e-45, -1e-45,
                      np.finfo(np.float32).tiny, 3.4e38], np.float32)
    assert _same_halves(oracle_mod.float_to_half(cases), _np_float_to_half(cases))
    # the largest finite half and the first value that rounds to infinity
    assert oracle_mod.float_to_half(np.array([65519.996], np.float32))[0] == 0x7BFF
    assert oracle_mod.float_to_half(np.array([65520.0], np.float32))[0] == 0x7C00


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_narrow_random_bit_patterns(oracle_mod, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    assert _same_halves(oracle_mod.float_to_half(x), _np_float_to_half(x))


def test_narrow_in_range_sample(oracle_mod):
    # values where the step's weights live (|w| ~ 1e-6 .. 1), dense sample
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(1 << 20) * np.exp(rng.uniform(-14, 1, 1 << 20))).astype(np.float32)
    assert _same_halves(oracle_mod.float_to_half(x), _np_float_to_half(x))
