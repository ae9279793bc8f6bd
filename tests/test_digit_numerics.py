"""The tensor-core path's activation operand, restated and bounded on the CPU.

The block-scaled FP4 MMA takes FP4 on both sides, so the tensor-core kernel
feeds each activation row as the sum of four NVFP4 "digit" rows: after one
power-of-two prescale of the row (largest magnitude into (1344, 2688]), digit j
holds 4^j times the residual left by digits 0..j-1, per 16-element block an
E4M3 scale rounded up and E2M1 round-to-nearest-even.  This module writes that
decomposition out from its definition (numpy, float64, no code shared with the
kernel) and pins the error bound the design relies on: after four digits every
element is within (9/8 / 6)^4 of its block's largest magnitude, i.e. about
1.24e-3, well inside the step's 2e-3 tolerance on max |y|.  It also restates
how h's per-slice digits are moved to one reference exponent per pair, and
bounds what that move costs.
"""
import numpy as np
import pytest

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_values():
    """All non-negative finite E4M3 values (codes 0x00..0x7E), ascending."""
    out = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(out)


E4M3 = e4m3_values()


def e4m3_ceil(a):
    """Smallest E4M3 value >= a (a >= 0), saturating at 448."""
    i = np.searchsorted(E4M3, a, side="left")
    return E4M3[np.minimum(i, len(E4M3) - 1)]


def e2m1_rne(v):
    """Round to the E2M1 grid, ties to the even code, saturating at 6."""
    s = np.sign(v)
    a = np.minimum(np.abs(v), 6.0)
    i = np.searchsorted(E2M1, a)  # first grid point >= a
    i = np.clip(i, 1, len(E2M1) - 1)
    lo, hi = E2M1[i - 1], E2M1[i]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((i % 2) == 0))
    return s * np.where(pick_hi, hi, lo)


def prescale_exponent(amax):
    """e with amax * 2^e in (1344, 2688]."""
    e = int(np.floor(np.log2(2688.0 / amax)))
    while amax * 2.0 ** e > 2688.0:
        e -= 1
    while amax * 2.0 ** (e + 1) <= 2688.0:
        e += 1
    return e


def digits(row, ndig=4):
    """(prescale exponent, list of digit rows as values) of one activation row."""
    e = prescale_exponent(np.max(np.abs(row)))
    r = row * 2.0 ** e
    out = []
    for j in range(ndig):
        f = 4.0 ** j
        blocks = (r * f).reshape(-1, 16)
        s = e4m3_ceil(np.max(np.abs(blocks), axis=1) / 6.0)[:, None]
        q = np.where(s > 0, e2m1_rne(np.divide(blocks, s, out=np.zeros_like(blocks), where=s > 0)), 0.0) * s
        out.append(q.reshape(-1) / f)
        r = r - q.reshape(-1) / f
    return e, out


@pytest.mark.parametrize("seed", range(6))
def test_four_digits_stay_within_the_bound(seed):
    rng = np.random.default_rng(seed)
    row = rng.standard_normal(4096) * rng.choice([1e-3, 1.0, 37.0])
    row[rng.integers(0, 4096, 8)] *= 50.0  # a few outliers, as activations have
    e, ds = digits(row)
    recon = sum(ds) * 2.0 ** -e
    blocks = np.abs(row.reshape(-1, 16)).max(axis=1).repeat(16)
    bound = (9.0 / 8.0 / 6.0) ** 4
    err = np.abs(recon - row)
    assert np.all(err <= bound * blocks * (1 + 1e-12))
    # far inside the bound on average
    assert np.mean(err / np.maximum(blocks, 1e-300)) < bound / 4


def test_each_digit_shrinks_the_residual_by_the_stated_factor():
    rng = np.random.default_rng(7)
    row = rng.standard_normal(4096)
    e, ds = digits(row, ndig=4)
    r = row * 2.0 ** e
    amax = np.abs(r.reshape(-1, 16)).max(axis=1)
    for j in range(4):
        r = r - ds[j]
        left = np.abs(r.reshape(-1, 16)).max(axis=1)
        assert np.all(left <= amax * (9.0 / 8.0 / 6.0) ** (j + 1) * (1 + 1e-12))


def test_digit_codes_never_saturate_and_zero_stays_zero():
    rng = np.random.default_rng(3)
    row = rng.standard_normal(512)
    row[:16] = 0.0  # an all-zero block: every digit and scale is zero
    e, ds = digits(row)
    assert all(np.all(d[:16] == 0.0) for d in ds)
    # scales are rounded up, so no element of any digit exceeds 6 x its scale
    r = row * 2.0 ** e
    for j in range(4):
        f = 4.0 ** j
        b = (r * f).reshape(-1, 16)
        s = e4m3_ceil(np.abs(b).max(axis=1) / 6.0)
        assert np.all(np.abs(b).max(axis=1) <= 6.0 * s + 1e-12)
        r = r - ds[j]


def test_e2m1_ties_go_to_the_even_code():
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 7.0])
    assert e2m1_rne(v).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -0.0, -4.0, 6.0]


def test_blocks_far_below_the_row_max_lose_relative_not_absolute_precision():
    """Blocks far below the row's largest magnitude reach subnormal E4M3
    scales (the prescale is shared by the row).  Relative to their own block
    their error grows past the bound (a block 2^26 down is mostly lost), but
    every element's error stays below 2^-24 of the row's largest magnitude, so
    such blocks carry no weight in a dot product."""
    rng = np.random.default_rng(11)
    row = rng.standard_normal(4096)
    shifts = [14, 17, 20, 26, 40]
    for k, sh in enumerate(shifts):
        row[16 * (k + 1):16 * (k + 2)] = rng.standard_normal(16) * 2.0 ** -sh
    e, ds = digits(row)
    err = np.abs(sum(ds) * 2.0 ** -e - row)
    rmax = np.abs(row).max()
    bound = (9.0 / 8.0 / 6.0) ** 4
    assert err.max() <= bound * rmax
    for k in range(len(shifts)):
        b = slice(16 * (k + 1), 16 * (k + 2))
        assert err[b].max() <= 2.0 ** -24 * rmax
    far = slice(16 * 4, 16 * 5)                 # the block 2^26 below
    assert err[far].max() > bound * np.abs(row[far]).max()


def e4m3_rne(a):
    """Nearest E4M3 value to a >= 0 (ties to the even code), saturating at 448."""
    i = np.clip(np.searchsorted(E4M3, a), 1, len(E4M3) - 1)
    lo, hi = E4M3[i - 1], E4M3[i]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & (i % 2 == 0))
    return np.where(a >= 448.0, 448.0, np.where(up, hi, lo))


def slice_digits(sl):
    """Prescale exponent, E2M1 values [16-blocks, 16] and E4M3 scales [16-blocks]
    of the four digit rows of one slice, from the decomposition's definition."""
    e = prescale_exponent(np.max(np.abs(sl)))
    r = sl * 2.0 ** e
    vals, scales = [], []
    for j in range(4):
        f = 4.0 ** j
        b = (r * f).reshape(-1, 16)
        s = e4m3_ceil(np.max(np.abs(b), axis=1) / 6.0)
        v = np.where(s[:, None] > 0, e2m1_rne(np.divide(b, s[:, None], out=np.zeros_like(b), where=s[:, None] > 0)), 0.0)
        vals.append(v)
        scales.append(s)
        r = r - (v * s[:, None]).reshape(-1) / f
    return e, vals, scales


@pytest.mark.parametrize("seed", range(12))
def test_h_slices_rebased_to_the_pair_reference(seed):
    """Each 128-row slice of a pair's h is decomposed with its own
    prescale, then every digit's block scales are moved to the pair's reference
    exponent (its largest slice) by an E4M3 round-to-nearest-even of
    scale x 2^-d.  The move is exact while a scale stays normal; below that a
    scale changes by at most half a subnormal step (2^-10), so with E2M1 values
    <= 6 and digit weights 4^-j the element error grows by at most
    6 * 2^-10 * 85/64 in reference units, under 2^-17 of the pair's largest |h|
    (which sits above 1344 there)."""
    rng = np.random.default_rng(100 + seed)
    I = 1024
    h = rng.standard_normal(I) * np.exp(rng.uniform(-3, 3))
    h *= np.where(rng.random(I) < 0.02, 30.0, 1.0)
    shifts = rng.integers(0, 30, I // 128)
    shifts[rng.integers(I // 128)] = 0
    for i in range(I // 128):
        h[128 * i:128 * (i + 1)] *= 2.0 ** -float(shifts[i])
    per = [slice_digits(h[128 * i:128 * (i + 1)]) for i in range(I // 128)]
    eref = min(p[0] for p in per)
    rec = np.zeros(I)
    for i, (e, vals, scales) in enumerate(per):
        d = e - eref
        out = np.zeros(128)
        for j in range(4):
            moved = e4m3_rne(scales[j] * 2.0 ** -d)
            if np.all((scales[j] == 0) | (scales[j] * 2.0 ** -d >= 2.0 ** -6)):
                assert np.array_equal(moved, scales[j] * 2.0 ** -d)     # normal: an exact shift
            out += (vals[j] * moved[:, None]).reshape(-1) / 4.0 ** j
        rec[128 * i:128 * (i + 1)] = out * 2.0 ** -eref
    err = np.abs(rec - h)
    blk = np.abs(h).reshape(-1, 16).max(axis=1).repeat(16)
    bound = (9.0 / 8.0 / 6.0) ** 4
    assert np.all(err <= bound * blk + 2.0 ** -17 * np.abs(h).max())
