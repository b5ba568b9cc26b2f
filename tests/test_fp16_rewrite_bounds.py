"""The arithmetic facts behind the tensor-core tiles' rewrite of bf16 V as fp16,
checked on every one of the 65536 bf16 bit patterns (CPU only).

The tile kernel rewrites a staged bf16 V range as fp16 so that P can be one
fp16 value per key; a range holding a magnitude of 65536 or more (bf16 bits
0x4780 and above once the sign is cleared, inf and NaN included) is put back
to bf16 and takes the bf16 hi + lo pair instead. The design relies on:

- every finite bf16 value below 65536 in magnitude rounds to a finite fp16
  value, and 65536 is the first that does not (the threshold is exact);
- that rounding is exact from 2^-17 up (and at zero), and off by at most
  2^-25 below;
- converting the fp16 value back to bf16 (round to nearest even) returns the
  original bits wherever the first conversion was exact.

numpy's float16 cast is IEEE binary16 round-to-nearest-even, the rounding the
kernel's `cvt.rn.f16x2.f32` performs.
"""

import numpy as np

from paged_kv_cache_55_gb300 import workloads as W

ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
MAG = ALL & np.uint16(0x7FFF)
VAL = W.bf16_bits_to_f32(ALL)
FINITE = np.isfinite(VAL)
THRESHOLD = 0x4780  # bf16 bits of 65536


def test_threshold_is_65536():
    assert W.bf16_bits_to_f32(np.array([THRESHOLD], np.uint16))[0] == 65536.0
    # the largest bf16 value below it is 65280, below fp16's largest finite 65504
    assert W.bf16_bits_to_f32(np.array([THRESHOLD - 1], np.uint16))[0] == 65280.0
    assert np.finfo(np.float16).max == 65504.0


def test_below_threshold_fits_fp16_and_above_does_not():
    with np.errstate(over="ignore"):
        h = VAL.astype(np.float16)
    below = FINITE & (MAG < THRESHOLD)
    at_or_above = FINITE & (MAG >= THRESHOLD)
    assert np.isfinite(h[below]).all()
    assert np.isinf(h[at_or_above]).all()
    # inf and NaN patterns are flagged by the same comparison (they sit above 0x4780)
    assert (MAG[~FINITE] >= THRESHOLD).all()


def test_exact_from_two_to_the_minus_17_and_bounded_below():
    below = FINITE & (MAG < THRESHOLD)
    v = VAL[below].astype(np.float64)
    h = VAL[below].astype(np.float16).astype(np.float64)
    err = np.abs(h - v)
    big = (np.abs(v) >= 2.0 ** -17) | (v == 0.0)
    assert (err[big] == 0.0).all()
    assert err[~big].max() <= 2.0 ** -25
    # the bound is reached (the claim is not loose by a power of two)
    assert err[~big].max() == 2.0 ** -25
    # and 2^-17 is where exactness starts: some value just below it is not exact
    assert (err[(np.abs(v) < 2.0 ** -17)] > 0).any()


def test_round_trip_back_to_bf16_restores_exact_values():
    below = FINITE & (MAG < THRESHOLD)
    bits = ALL[below]
    v = VAL[below]
    h = v.astype(np.float16).astype(np.float32)
    back = W.f32_to_bf16_bits(h)
    exact = (np.abs(v.astype(np.float64)) >= 2.0 ** -17) | (v == 0.0)
    # +0 and -0 keep their sign through both conversions
    assert np.array_equal(back[exact], bits[exact])
    # the others come back within 2^-25 of the original value
    diff = np.abs(W.bf16_bits_to_f32(back[~exact]).astype(np.float64) - v[~exact].astype(np.float64))
    assert diff.max() <= 2.0 ** -25
