"""The activation kernel's fast int4 rounding, restated on the CPU in float32.

For a block whose maximum is finite and nonzero and whose reciprocal scale is
finite, every scaled value y has |y| <= 7 (times 1 + a few ulp).  The kernel then
takes y + 1.5 * 2^23 (float32, round to nearest even): the sum lies in
[2^23, 2^24), where float32 spacing is 1, so it equals 1.5 * 2^23 plus y rounded
to the nearest integer (ties to even), and its low 4 bits are that integer's
two's complement nibble.  It checks that no value sits exactly halfway between
two integers (|y - nearest| < 0.5, NaN failing the check) and otherwise falls
back to the general rounding.  These tests check that whenever the check passes,
the nibble equals round-half-away-from-zero with the clamp to -8..7.  They cover
every float32 on a fine grid of [-7.5, 7.5], values next to each half-integer,
and the halves themselves, which must fail the check.
"""
import numpy as np

MAGIC = np.float32(12582912.0)  # 1.5 * 2^23


def fast_nibbles(y):
    y = np.asarray(y, dtype=np.float32)
    t = (y + MAGIC).astype(np.float32)
    r = (t - MAGIC).astype(np.float32)
    dd = (y - r).astype(np.float32)
    ok = np.abs(dd) < np.float32(0.5)  # NaN compares False
    nib = t.view(np.uint32) & np.uint32(0xF)
    return nib.astype(np.uint32), ok


def reference_nibbles(y):
    y = np.asarray(y, dtype=np.float64)
    r = np.sign(y) * np.floor(np.abs(y) + 0.5)  # round half away from zero (exact in float64)
    r = np.clip(r, -8, 7).astype(np.int64)
    return (r & 0xF).astype(np.uint32)


def _check(y):
    nib, ok = fast_nibbles(y)
    ref = reference_nibbles(y)
    assert np.array_equal(nib[ok], ref[ok])
    return ok


def test_grid_of_values():
    y = np.linspace(-7.5, 7.5, 2_000_001, dtype=np.float64).astype(np.float32)
    _check(y)


def test_neighbours_of_halves_and_integers():
    ys = []
    for k in range(-8, 8):
        for base in (k + 0.5, float(k)):
            up = down = np.float32(base)
            for _ in range(5):
                up = np.nextafter(up, np.float32(np.inf))
                down = np.nextafter(down, np.float32(-np.inf))
                ys += [up, down]
    # the value just below one half and other small magnitudes
    ys += [np.float32(0.5) - np.float32(2.0**-25), np.float32(2.0**-30), np.float32(-(2.0**-30)), np.float32(0.0),
           np.float32(-0.0), np.float32(7.0000005), np.float32(-7.0000005)]
    y = np.array(ys, dtype=np.float32)
    y = y[np.abs(y) < 7.5]  # the fast path's domain (see test_scaled_values_stay_below_seven_and_a_half)
    ok = _check(y)
    assert ok.all(), "no value off a half-integer may need the general path"


def test_scaled_values_stay_below_seven_and_a_half():
    # the block maximum a scaled by the kernel's reciprocal scale: d = fl(a / 7), inv
    # = fl(1 / d), a * inv; whenever inv is finite this stays below 7.5, so every
    # value of the block rounds into -7..7 and the clamp never acts
    rng = np.random.default_rng(3)
    a = np.concatenate([
        (rng.random(200_000) * 2.0 ** rng.integers(-126, 127, 200_000)).astype(np.float32),
        np.float32(2.0**-149) * np.arange(1, 200_000, dtype=np.float32),  # subnormal maxima
        np.array([np.finfo(np.float32).max, np.finfo(np.float32).tiny, 7.0, 1.0], dtype=np.float32),
    ])
    a = a[a > 0]
    with np.errstate(over="ignore", divide="ignore"):
        d = (a / np.float32(7.0)).astype(np.float32)
        inv = (np.float32(1.0) / d).astype(np.float32)
        y = (a * inv).astype(np.float32)
    fin = np.isfinite(inv) & (d > 0)
    assert fin.sum() > 150_000
    assert np.all(np.abs(y[fin]) < 7.5)


def test_halves_take_the_general_path():
    halves = np.array([k + 0.5 for k in range(-8, 7)], dtype=np.float32)
    _, ok = fast_nibbles(halves)
    assert not ok.any()


def test_nan_takes_the_general_path():
    _, ok = fast_nibbles(np.array([np.nan], dtype=np.float32))
    assert not ok.any()
