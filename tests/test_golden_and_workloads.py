"""Oracle regression against the stored fixtures, and the seeded generators."""
import glob
import os

import numpy as np
import pytest
import scipy.signal

import oracle
from normalized_cross_correlation_u8_gb300 import workloads as wl
from tests.golden.make_golden import read_fixture

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "ncc_u8_*.txt"))))
def test_oracle_reproduces_ncc_fixture(path):
    fx = read_fixture(path)
    image, tmpl = fx["image"].astype(np.uint8), fx["tmpl"].astype(np.uint8)
    sums, c64, _ = oracle.ncc_u8(image, tmpl)
    np.testing.assert_array_equal(sums, fx["sums"])
    np.testing.assert_allclose(c64, fx["coef"], rtol=0, atol=1e-15)
    # and the fixture itself agrees with the library form of SumIT
    ref = scipy.signal.correlate2d(image.astype(np.int64), tmpl.astype(np.int64), "valid")
    np.testing.assert_array_equal(fx["sums"][2], ref)


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(GOLDEN, "xcorr_f32_*.txt"))))
def test_oracle_reproduces_xcorr_fixture(path):
    fx = read_fixture(path)
    left, right = fx["left"].astype(np.float32), fx["right"].astype(np.float32)
    out, ab = oracle.xcorr_f32(left, right)
    np.testing.assert_allclose(out, fx["out"], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(ab, fx["abs"], rtol=1e-15, atol=1e-15)


def test_workloads_are_deterministic_and_shaped():
    a, b = wl.ncc_256(), wl.ncc_256()
    np.testing.assert_array_equal(a.image, b.image)
    assert a.image.shape == (256, 256) and a.tmpl.shape == (16, 16)
    assert a.offsets == 241 * 241
    x, y = a.offset
    np.testing.assert_array_equal(a.tmpl, a.image[y:y + 16, x:x + 16])
    s = wl.ncc_1080p()
    assert s.image.shape == (1080, 1920) and s.tmpl.shape == (32, 32)
    assert 0.29 <= (s.image > 127).mean() <= 0.31
    assert s.offsets == 1889 * 1049
    x, y = s.offset
    d = s.tmpl.astype(int) - s.image[y:y + 32, x:x + 32].astype(int)
    assert np.abs(d).max() <= 8
    for f, shp_l, shp_r in ((wl.xcorr_one_to_one, (1, 256, 256), (1, 256, 256)),
                            (wl.xcorr_one_to_many, (1, 64, 64), (128, 64, 64)),
                            (wl.xcorr_n_to_m, (32, 16, 16), (64, 16, 16))):
        w = f()
        assert w.left.shape == shp_l and w.right.shape == shp_r
        assert w.left.dtype == np.float32
    assert wl.xcorr_one_to_one().flops == 2 * 256 ** 4
