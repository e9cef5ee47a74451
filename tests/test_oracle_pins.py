"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle (oracle/oracle.c) against a library routine, an
independent algorithm, a closed form or an exact invariant, chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, swapped
operands, a byte-order or signedness slip) fails at least one of them.

Definitions pinned:
* u8 sums SumI / SumISq / SumIT -- The CUDA Handbook ch. 15, section 15.5
  "Instruction-Level Parallelism and DP4A" (unsigned pixels; the page warns
  that pixels above 127 and byte order are where slips hide, so every input
  here has bright pixels and asymmetric templates).
* the normalized coefficient over those sums (the chapter's subject,
  "Normalized Correlation").
* f32 full cross-correlation, every overlap -- "Efficient GPU-accelerated
  Parallel Cross-correlation" artifact README, kernel overview.
"""
import itertools

import numpy as np
import pytest
import scipy.signal
from numpy.lib.stride_tricks import sliding_window_view

import oracle

RNG = np.random.default_rng(20261202)


def rand_u8(h, w, lo=0, hi=256, rng=RNG):
    return rng.integers(lo, hi, size=(h, w), dtype=np.uint8)


# --------------------------------------------------------------------------
# u8 sums
# --------------------------------------------------------------------------

U8_SHAPES = [  # (h, w, ht, wt)
    (5, 7, 2, 4), (6, 9, 3, 4), (1, 4, 1, 4), (4, 4, 4, 4), (9, 13, 5, 8),
    (17, 33, 7, 12), (20, 21, 1, 16), (12, 40, 12, 4), (8, 10, 3, 3),
    (11, 6, 2, 5),
]


@pytest.mark.parametrize("h,w,ht,wt", U8_SHAPES)
def test_u8_sums_match_library_valid_correlation(h, w, ht, wt):
    """SumIT = scipy correlate2d(I, T, 'valid'); SumI, SumISq = the same with
    an all-ones template on I and I^2 (exact in int64)."""
    image, tmpl = rand_u8(h, w), rand_u8(ht, wt)
    sums, _, _ = oracle.ncc_u8(image, tmpl)
    I = image.astype(np.int64)
    T = tmpl.astype(np.int64)
    ones = np.ones_like(T)
    np.testing.assert_array_equal(
        sums[2], scipy.signal.correlate2d(I, T, mode="valid"))
    np.testing.assert_array_equal(
        sums[0], scipy.signal.correlate2d(I, ones, mode="valid"))
    np.testing.assert_array_equal(
        sums[1], scipy.signal.correlate2d(I * I, ones, mode="valid"))


@pytest.mark.parametrize("h,w,ht,wt", U8_SHAPES)
def test_u8_box_sums_match_summed_area_table(h, w, ht, wt):
    """SumI and SumISq from an integral image (a different algorithm)."""
    image = rand_u8(h, w)
    sums, _, _ = oracle.ncc_u8(image, rand_u8(ht, wt))
    for plane, vals in ((0, image.astype(np.int64)),
                        (1, image.astype(np.int64) ** 2)):
        S = np.zeros((h + 1, w + 1), np.int64)
        S[1:, 1:] = vals.cumsum(0).cumsum(1)
        box = S[ht:, wt:] - S[:-ht, wt:] - S[ht:, :-wt] + S[:-ht, :-wt]
        np.testing.assert_array_equal(sums[plane], box)


def test_u8_sums_exhaustive_tiny_bruteforce():
    """Every tiny shape up to 6x6, brute force by sliding windows + einsum."""
    rng = np.random.default_rng(7)
    for h, w in itertools.product(range(1, 7), repeat=2):
        for ht, wt in itertools.product(range(1, h + 1), range(1, w + 1)):
            image = rand_u8(h, w, 100, 256, rng)   # always some bytes > 127
            tmpl = rand_u8(ht, wt, 0, 256, rng)
            sums, _, _ = oracle.ncc_u8(image, tmpl)
            win = sliding_window_view(image.astype(np.int64), (ht, wt))
            np.testing.assert_array_equal(sums[0], win.sum(axis=(2, 3)))
            np.testing.assert_array_equal(sums[1], (win * win).sum(axis=(2, 3)))
            np.testing.assert_array_equal(
                sums[2], np.einsum("yxji,ji->yx", win, tmpl.astype(np.int64)))


def test_u8_sums_byte_order_single_hot_byte():
    """A template with one hot byte at each position in turn: SumIT must pick
    exactly the image pixel under that byte (a lane swap would pick its
    neighbour)."""
    image = rand_u8(9, 16, 128, 256)
    for j, i in itertools.product(range(2), range(8)):
        tmpl = np.zeros((2, 8), np.uint8)
        tmpl[j, i] = 1
        sums, _, _ = oracle.ncc_u8(image, tmpl)
        np.testing.assert_array_equal(
            sums[2], image[j:j + 8, i:i + 9].astype(np.uint32))


def test_u8_all_ones_template_and_patch_identities():
    image = rand_u8(21, 30)
    sums, _, _ = oracle.ncc_u8(image, np.ones((5, 8), np.uint8))
    np.testing.assert_array_equal(sums[2], sums[0])       # SumIT == SumI
    x, y = 11, 7
    sums, _, _ = oracle.ncc_u8(image, image[y:y + 5, x:x + 8])
    assert sums[2, y, x] == sums[1, y, x]                 # SumIT == SumISq


def test_u8_closed_form_constant_and_ramp():
    """Constant image c: SumI = N c, SumISq = N c^2, SumIT = c SumT.
    Ramp image p(x, y) = x + 10 y: SumI has the closed form
    N (x + (wt-1)/2) + 10 N (y + (ht-1)/2)."""
    c, ht, wt = 201, 3, 4
    image = np.full((8, 12), c, np.uint8)
    tmpl = rand_u8(ht, wt)
    n = ht * wt
    sums, c64, _ = oracle.ncc_u8(image, tmpl)
    assert (sums[0] == n * c).all() and (sums[1] == n * c * c).all()
    assert (sums[2] == c * int(tmpl.astype(np.int64).sum())).all()
    assert (c64 == 0.0).all()                              # flat window -> 0
    yy, xx = np.mgrid[0:20, 0:24]
    ramp = (xx + 10 * yy).astype(np.uint8)                 # max 23 + 190 = 213
    sums, _, _ = oracle.ncc_u8(ramp, tmpl)
    oy, ox = np.mgrid[0:20 - ht + 1, 0:24 - wt + 1]
    expect = n * ox + n * (wt - 1) // 2 + 10 * (n * oy + n * (ht - 1) // 2)
    # n*(wt-1)/2 is an integer here (n=12, wt-1=3 -> 18; ht-1=2 -> 12)
    np.testing.assert_array_equal(sums[0], expect)


def test_template_sums():
    t = rand_u8(7, 12)
    st, sq = oracle.template_sums(t)
    assert st == int(t.astype(np.int64).sum())
    assert sq == int((t.astype(np.int64) ** 2).sum())


# --------------------------------------------------------------------------
# u8 coefficient
# --------------------------------------------------------------------------

@pytest.mark.parametrize("h,w,ht,wt", U8_SHAPES[:6] + [(30, 40, 8, 8)])
def test_u8_coef_matches_pearson_corrcoef(h, w, ht, wt):
    """The normalized coefficient is Pearson's r between the window and the
    template: check against numpy.corrcoef in float64."""
    if ht * wt < 2:
        pytest.skip("needs two pixels")
    image, tmpl = rand_u8(h, w), rand_u8(ht, wt)
    _, c64, c32 = oracle.ncc_u8(image, tmpl)
    win = sliding_window_view(image.astype(np.float64), (ht, wt))
    t = tmpl.astype(np.float64).ravel()
    for y, x in itertools.product(range(c64.shape[0]), range(c64.shape[1])):
        r = np.corrcoef(win[y, x].ravel(), t)[0, 1]
        assert abs(c64[y, x] - r) < 1e-12
        assert abs(float(c32[y, x]) - r) < 1e-7


def test_u8_coef_exactly_one_at_patch():
    for (h, w, ht, wt) in [(40, 50, 16, 16), (64, 64, 32, 32), (30, 90, 8, 64)]:
        image = rand_u8(h, w)
        x, y = int(RNG.integers(0, w - wt + 1)), int(RNG.integers(0, h - ht + 1))
        _, c64, c32 = oracle.ncc_u8(image, image[y:y + ht, x:x + wt])
        assert c64[y, x] == 1.0 and c32[y, x] == 1.0
        assert np.abs(c64).max() <= 1.0 + 1e-12


def test_u8_coef_sign_flip_and_affine():
    """coef(I, 255-T) = -coef(I, T) exactly (numerator negates, template
    variance unchanged); coef(I, a T + b) = coef(I, T) for a > 0."""
    image, tmpl = rand_u8(25, 33), rand_u8(6, 8)
    _, c, _ = oracle.ncc_u8(image, tmpl)
    _, cf, _ = oracle.ncc_u8(image, (255 - tmpl).astype(np.uint8))
    np.testing.assert_array_equal(cf, -c)
    small = rand_u8(6, 8, 0, 50)
    _, c1, _ = oracle.ncc_u8(image, small)
    _, c2, _ = oracle.ncc_u8(image, (3 * small + 17).astype(np.uint8))
    np.testing.assert_allclose(c2, c1, rtol=0, atol=1e-14)


def test_u8_coef_flat_template_is_zero():
    image = rand_u8(10, 12)
    _, c64, c32 = oracle.ncc_u8(image, np.full((3, 4), 77, np.uint8))
    assert (c64 == 0).all() and (c32 == 0).all()


def test_u8_sampled_matches_full():
    image, tmpl = rand_u8(37, 45), rand_u8(9, 12)
    sums, c64, _ = oracle.ncc_u8(image, tmpl)
    ys = RNG.integers(0, 37 - 9 + 1, 50)
    xs = RNG.integers(0, 45 - 12 + 1, 50)
    s2, c2 = oracle.ncc_u8_at(image, tmpl, xs, ys)
    np.testing.assert_array_equal(s2, sums[:, ys, xs])
    np.testing.assert_array_equal(c2, c64[ys, xs])


def test_u8_threads_do_not_change_result():
    image, tmpl = rand_u8(50, 61), rand_u8(7, 8)
    a = oracle.ncc_u8(image, tmpl, 1)
    b = oracle.ncc_u8(image, tmpl, 4)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_u8_argument_errors():
    with pytest.raises(oracle.oracle.OracleError):
        oracle.ncc_u8(rand_u8(4, 4), rand_u8(5, 4))       # template taller
    with pytest.raises(oracle.oracle.OracleError):
        oracle.ncc_u8(rand_u8(300, 300), rand_u8(258, 258))  # > 66051 px


@pytest.mark.parametrize("wt,ht", [(369, 179), (9, 7339)])
def test_u8_sums_at_the_template_size_limit(wt, ht):
    """Closed form at the 32-bit limit: N = 66051 pixels of 255 over a
    window of 255s give SumI = 255 N, SumISq = SumIT = 65025 N =
    4 294 966 275, the largest value below 2^32 any template can reach.
    One pixel more (66052 * 65025 >= 2^32) is refused."""
    assert wt * ht == 66051
    image = np.full((ht + 1, wt + 2), 255, np.uint8)
    s, c64, _ = oracle.ncc_u8(image, np.full((ht, wt), 255, np.uint8))
    assert (s[0] == 255 * 66051).all()
    assert (s[1] == 65025 * 66051).all() and (s[2] == 65025 * 66051).all()
    assert (c64 == 0).all()                      # flat template
    with pytest.raises(oracle.oracle.OracleError):
        oracle.ncc_u8(np.full((5, 16513), 255, np.uint8), np.full((4, 16513), 255, np.uint8))


# --------------------------------------------------------------------------
# f32 full cross-correlation
# --------------------------------------------------------------------------

F32_SHAPES = [(1, 1), (1, 3), (2, 2), (3, 5), (7, 4), (6, 11), (16, 16),
              (13, 9)]


def rand_f32(*shape, rng=RNG):
    return rng.uniform(-1, 1, size=shape).astype(np.float32)


@pytest.mark.parametrize("H,W", F32_SHAPES)
def test_xcorr_matches_scipy_full(H, W):
    """Library routine: scipy correlate2d(L, R, 'full') in float64; index
    (H-1, W-1) is the zero shift.  Also Sum|L R| = correlate2d(|L|, |R|)."""
    L, R = rand_f32(H, W), rand_f32(H, W)
    out, ab = oracle.xcorr_f32(L, R)
    Ld, Rd = L.astype(np.float64), R.astype(np.float64)
    ref = scipy.signal.correlate2d(Ld, Rd, mode="full")
    np.testing.assert_allclose(out[0, 0], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(
        ab[0, 0], scipy.signal.correlate2d(np.abs(Ld), np.abs(Rd), "full"),
        rtol=1e-12, atol=1e-12)


def test_xcorr_matches_fft():
    """Independent algorithm: zero-padded FFT correlation."""
    H, W = 24, 17
    L, R = rand_f32(H, W), rand_f32(H, W)
    out, ab = oracle.xcorr_f32(L, R)
    sh = (2 * H - 1, 2 * W - 1)
    F = np.fft.rfft2(L.astype(np.float64), sh) * np.fft.rfft2(
        R[::-1, ::-1].astype(np.float64), sh)
    ref = np.fft.irfft2(F, sh)
    assert np.all(np.abs(out[0, 0] - ref) <= 1e-9 * np.maximum(ab[0, 0], 1e-30))


def test_xcorr_delta_identities():
    """R = delta at (a, b): out[dy, dx] = L[a+dy, b+dx].
    L = delta at (a, b): out[dy, dx] = R[a-dy, b-dx]."""
    H, W, a, b = 6, 9, 2, 5
    L = rand_f32(H, W)
    D = np.zeros((H, W), np.float32)
    D[a, b] = 1
    out, _ = oracle.xcorr_f32(L, D)
    out2, _ = oracle.xcorr_f32(D, L)
    for dy, dx in itertools.product(range(-H + 1, H), range(-W + 1, W)):
        y, x = a + dy, b + dx
        e = L[y, x] if (0 <= y < H and 0 <= x < W) else 0.0
        assert out[0, 0, dy + H - 1, dx + W - 1] == e
        y, x = a - dy, b - dx
        e = L[y, x] if (0 <= y < H and 0 <= x < W) else 0.0
        assert out2[0, 0, dy + H - 1, dx + W - 1] == e


def test_xcorr_sum_flip_and_centre():
    """Sum over all shifts = sum(L) sum(R); xcorr(L, R) is xcorr(R, L) turned
    by 180 degrees; the centre of xcorr(L, L) is sum(L^2)."""
    H, W = 11, 8
    L, R = rand_f32(H, W), rand_f32(H, W)
    o, _ = oracle.xcorr_f32(L, R)
    o2, _ = oracle.xcorr_f32(R, L)
    s = float(L.astype(np.float64).sum()) * float(R.astype(np.float64).sum())
    assert abs(o.sum() - s) < 1e-10
    np.testing.assert_allclose(o[0, 0], o2[0, 0][::-1, ::-1], rtol=0, atol=1e-13)
    oo, _ = oracle.xcorr_f32(L, L)
    assert abs(oo[0, 0, H - 1, W - 1] - (L.astype(np.float64) ** 2).sum()) < 1e-12


def test_xcorr_batches_are_pairwise():
    """Pair index li*nr + ri; one-to-many and n-to-m equal one-to-one calls."""
    H, W = 5, 7
    Ls, Rs = rand_f32(3, H, W), rand_f32(4, H, W)
    out, ab = oracle.xcorr_f32(Ls, Rs)
    assert out.shape == (3, 4, 2 * H - 1, 2 * W - 1)
    for li, ri in itertools.product(range(3), range(4)):
        ref = scipy.signal.correlate2d(Ls[li].astype(np.float64),
                                       Rs[ri].astype(np.float64), "full")
        np.testing.assert_allclose(out[li, ri], ref, rtol=1e-12, atol=1e-12)


def test_xcorr_sampled_matches_full_and_threads():
    H, W = 9, 6
    Ls, Rs = rand_f32(2, H, W), rand_f32(3, H, W)
    out, ab = oracle.xcorr_f32(Ls, Rs, nthreads=4)
    out1, _ = oracle.xcorr_f32(Ls, Rs, nthreads=1)
    np.testing.assert_array_equal(out, out1)
    k = 40
    ls, rs = RNG.integers(0, 2, k), RNG.integers(0, 3, k)
    oys, oxs = RNG.integers(0, 2 * H - 1, k), RNG.integers(0, 2 * W - 1, k)
    v, a = oracle.xcorr_f32_at(Ls, Rs, ls, rs, oys, oxs)
    np.testing.assert_array_equal(v, out[ls, rs, oys, oxs])
    np.testing.assert_array_equal(a, ab[ls, rs, oys, oxs])
