"""Host check of the arithmetic behind spec_accept's two forms of a tile (CPU only).

The kernel weighs a probability v by F(v) = floor(2^40 v) on the 2^-40 grid: in
its general form from the float's bits with 64-bit integer shifts (exact for every
float, with v >= 1 counting as 1 and anything not positive as 0), and, for a tile
whose values all convert below 2^30, as a saturating float-to-uint32 conversion of
the fp32 product v * 2^40.  These tests emulate both forms bit for bit in numpy
over every sign / exponent combination (the whole significand range at the
exponents where the forms meet) and check that the short form is exact wherever
the kernel takes it, and that no value of 2^-10 or more can take it."""
import numpy as np


def _wide_form(bits):
    """floor(2^40 v) from the float bits: (significand << 40) >> (150 - E), the shift
    clamped to 0 past 64; v >= 1 or +inf gives 2^40; zero, subnormals, negatives and
    NaN give 0."""
    bits = bits.astype(np.uint64)
    E = (bits >> np.uint64(23)) & np.uint64(0x1FF)  # with the sign bit
    x = ((bits & np.uint64(0x7FFFFF)) | np.uint64(0x800000)) << np.uint64(40)
    sh = 150 - E.astype(np.int64)
    w = np.where((sh >= 64) | (sh < 0), np.uint64(0), x >> np.clip(sh, 0, 63).astype(np.uint64))
    normal_below_one = (E >= 1) & (E <= 126)
    one = (E >= 127) & (E <= 255) & ~((E == 255) & ((bits & np.uint64(0x7FFFFF)) != 0))
    return np.where(normal_below_one, w, np.where(one, np.uint64(1 << 40), np.uint64(0)))


def _short_form(bits):
    """The fp32 product v * 2^40 converted to uint32 by truncation, saturating (NaN -> 0,
    negative -> 0, 2^32 and above -> 2^32 - 1)."""
    v = bits.astype(np.uint32).view(np.float32)
    with np.errstate(all="ignore"):
        x = (v * np.float32(2.0 ** 40)).astype(np.float64)
        r = np.where(np.isnan(x), 0.0, np.clip(np.trunc(x), 0.0, 2.0 ** 32 - 1))
    return r.astype(np.uint64)


def _floats(E, rng, dense):
    mant = np.arange(0, 1 << 23, dtype=np.uint64) if dense else rng.integers(0, 1 << 23, 4096, dtype=np.uint64)
    return (np.uint64(E) << np.uint64(23)) | mant


def test_short_form_is_exact_wherever_taken():
    rng = np.random.default_rng(3)
    dense = {0, 1, 116, 117, 118, 119, 126, 127, 255, 256, 383, 511}
    taken = 0
    for E in range(512):
        bits = _floats(E, rng, E in dense)
        wide, short = _wide_form(bits), _short_form(bits)
        fast = short < (1 << 30)
        assert np.array_equal(wide[fast], short[fast]), E
        assert not np.any(fast & (wide >= (1 << 30))), E
        taken += int(fast.sum())
    assert taken > 0


def test_forms_meet_at_two_to_minus_ten():
    # the largest float below 2^-10 takes the short form, 2^-10 itself does not
    below = np.array([np.float32(2.0 ** -10)], np.float32)
    below = np.nextafter(below, np.float32(0)).view(np.uint32)
    at = np.array([np.float32(2.0 ** -10)], np.float32).view(np.uint32)
    assert _short_form(below)[0] < (1 << 30) and _short_form(below)[0] == _wide_form(below)[0]
    assert _short_form(at)[0] == (1 << 30) == _wide_form(at)[0]


def test_wide_form_closed_values():
    f = lambda v: int(_wide_form(np.array([np.float32(v)], np.float32).view(np.uint32))[0])
    assert f(2.0 ** -40) == 1 and f(3 * 2.0 ** -40) == 3 and f(2.0 ** -41) == 0
    assert f(0.5) == 1 << 39 and f(1.0) == 1 << 40 and f(7.0) == 1 << 40 and f(np.inf) == 1 << 40
    assert f(-0.25) == 0 and f(np.nan) == 0 and f(-0.0) == 0 and f(2.0 ** -140) == 0
