"""The arithmetic fact the folded-scale GEMM rests on, checked exhaustively on the host.

For every finite fp16 scale d and every integer code q in [-128, 127] (the weight codes of Q4_0,
Q8_0 and the IQ4_NL table, and the Q8_0 activation codes), the product v = d * q splits exactly
into two fp16 numbers: hi = fp16(v) (round to nearest even) and lo = v - hi, where lo itself is an
fp16 number, so hi + lo == v with nothing lost.  That holds wherever hi is finite; the kernel keeps
|v| below 2^15 by a per-row power of two, and a power of two times d stays exact while it is a
normal fp16 number.  Also checked: the dropped term a_lo * w_lo of the three-product sum is below
2^-22 |a w|.
"""
import numpy as np


def _all_finite_fp16():
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    d = bits.view(np.float16)
    return d[np.isfinite(d)]


def _split(v64):
    hi = v64.astype(np.float16)
    lo64 = v64 - hi.astype(np.float64)        # exact in float64 (both are multiples of 2^-24)
    lo = lo64.astype(np.float16)
    return hi, lo, lo64


def test_every_scale_times_every_code_splits_exactly():
    d = _all_finite_fp16().astype(np.float64)
    with np.errstate(invalid="ignore", over="ignore"):     # hi = inf beyond fp16's range; masked below
        for q in range(-128, 128):
            v = d * q                              # exact in float64: 11 + 8 significant bits
            hi, lo, lo64 = _split(v)
            ok = np.isfinite(hi.astype(np.float64))
            # where hi is finite, lo is an exact fp16 number and hi + lo == v
            assert np.array_equal(lo.astype(np.float64)[ok], lo64[ok]), f"q={q}: lo not representable"
            assert np.array_equal((hi.astype(np.float64) + lo.astype(np.float64))[ok], v[ok]), f"q={q}"
            # hi overflows only beyond fp16's range, i.e. never while |v| < 2^15
            assert ok[np.abs(v) < 2.0 ** 15].all()


def test_power_of_two_scaling_keeps_normal_scales_exact():
    d = _all_finite_fp16().astype(np.float64)
    d = d[np.abs(d) >= 2.0 ** -14]            # normal fp16 scales
    for t in (1, 3, 7, 9):
        s = d * 2.0 ** -t
        normal = np.abs(s) >= 2.0 ** -14
        assert np.array_equal(s.astype(np.float16).astype(np.float64)[normal], s[normal])


def test_dropped_lo_times_lo_term_is_below_2_pow_minus_22():
    rng = np.random.default_rng(7)
    d = _all_finite_fp16().astype(np.float64)
    d = d[(np.abs(d) >= 2.0 ** -14) & (np.abs(d) < 256)]
    da, dw = rng.choice(d, 200000), rng.choice(d, 200000)
    qa, qw = rng.integers(-127, 128, 200000), rng.integers(-128, 128, 200000)
    a, w = da * qa, dw * qw
    ha, la, _ = _split(a)
    hw, lw, _ = _split(w)
    prod = np.abs(a * w)
    dropped = np.abs(la.astype(np.float64) * lw.astype(np.float64))
    nz = prod > 0
    assert (dropped[nz] <= 2.0 ** -22 * prod[nz]).all()
    # and the three kept products recover a*w up to exactly that term
    kept = (ha.astype(np.float64) * hw.astype(np.float64) + ha.astype(np.float64) * lw.astype(np.float64)
            + la.astype(np.float64) * hw.astype(np.float64))
    assert np.allclose(kept + la.astype(np.float64) * lw.astype(np.float64), a * w, rtol=0, atol=0)
