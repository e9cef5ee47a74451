"""GPU parity of corr_ncc_u8 against the CPU oracle.

Bar (The CUDA Handbook ch. 15, section 15.5 sums; normalized coefficient):
SumI, SumISq, SumIT bit-exact; coefficient within 1e-5 absolute of the
oracle's double-precision value from the exact sums.  Inputs always contain
pixels above 127 and asymmetric templates (where signed-dp4a and byte-order
slips show).  All calls go through the C ABI via the ctypes binding.
"""
import glob
import os

import numpy as np
import pytest
import torch

import normalized_cross_correlation_u8_gb300 as corr
import oracle
from normalized_cross_correlation_u8_gb300 import workloads as wl
from tests.golden.make_golden import read_fixture

pytestmark = pytest.mark.gpu
COEF_TOL = 1e-5
NT = max(1, os.cpu_count() or 1)
RNG = np.random.default_rng(424242)


def run_gpu(image, tmpl, sums=True, coef=True, method=None):
    dev = torch.device("cuda", 0)
    s, c = corr.ncc_u8(torch.from_numpy(image).to(dev), torch.from_numpy(tmpl).to(dev),
                       sums=sums, coef=coef, method=method)
    torch.cuda.synchronize()
    s = s.cpu().numpy().view(np.uint32) if s is not None else None
    c = c.cpu().numpy() if c is not None else None
    return s, c


def assert_parity(image, tmpl, s, c, ref=None):
    if ref is None:
        ref = oracle.ncc_u8(image, tmpl, nthreads=NT)
    rs, rc64, _ = ref
    if s is not None:
        assert s.shape == rs.shape
        bad = np.argwhere(s != rs)
        assert bad.size == 0, f"{len(bad)} sum mismatches, first {bad[:5].tolist()}"
    if c is not None:
        assert c.shape == rc64.shape
        err = np.abs(c.astype(np.float64) - rc64)
        assert err.max() <= COEF_TOL, f"coef max err {err.max()} at {np.unravel_index(err.argmax(), err.shape)}"


def rand_u8(h, w, lo=0, hi=256):
    return RNG.integers(lo, hi, size=(h, w), dtype=np.uint8)


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(
    os.path.dirname(__file__), "golden", "ncc_u8_*.txt"))))
def test_fixture(path):
    fx = read_fixture(path)
    image, tmpl = fx["image"].astype(np.uint8), fx["tmpl"].astype(np.uint8)
    s, c = run_gpu(image, tmpl)
    np.testing.assert_array_equal(s, fx["sums"])
    assert np.abs(c - fx["coef"]).max() <= COEF_TOL


# fast path (wt up to 128; rows staged with 16- or 8-byte
# loads when w is a multiple of 16 or 8, else byte loads) and general path
# shapes; ragged tails in both directions (ow not a multiple of 128, oh odd)
SHAPES = [
    (40, 64, 16, 16), (97, 296, 16, 16), (77, 520, 32, 32), (130, 264, 64, 64),
    (33, 1000, 32, 7), (50, 600, 64, 3), (21, 256, 16, 21),
    (45, 300, 4, 3), (39, 100, 12, 5), (61, 333, 20, 9), (70, 515, 36, 11),
    (16, 16, 16, 16), (9, 4, 4, 1), (5, 260, 128, 5), (300, 20, 8, 200),
    (1, 1024, 64, 1), (200, 8, 8, 64),
    # fast path, every template width of 1 .. 15 words
    (45, 304, 4, 3), (41, 136, 8, 9), (39, 104, 12, 5), (61, 336, 20, 9),
    (50, 400, 24, 13), (66, 272, 28, 30), (70, 520, 36, 11), (80, 264, 40, 17),
    (90, 512, 44, 19), (100, 384, 48, 48), (75, 200, 52, 21), (120, 640, 56, 56),
    (64, 328, 60, 23),
    # fast path, templates of 17 .. 32 words (68 .. 128 wide), all three
    # staging units
    (40, 264, 68, 9), (36, 336, 96, 7), (30, 300, 124, 5), (140, 512, 128, 128),
    (50, 208, 112, 21),
    # template widths that are not a multiple of 4 (partial last word):
    # fast path with each staging unit, and the general path (wt > 128)
    (20, 64, 1, 5), (21, 136, 2, 3), (30, 64, 3, 30), (40, 304, 15, 15),
    (33, 200, 31, 17), (35, 301, 17, 9), (70, 520, 63, 41), (60, 264, 127, 7),
    (9, 300, 129, 3), (12, 270, 201, 5),
]


@pytest.mark.parametrize("method", ["box", "dp4a"])
@pytest.mark.parametrize("h,w,wt,ht", SHAPES)
def test_random_shapes(h, w, wt, ht, method):
    image, tmpl = rand_u8(h, w), rand_u8(ht, wt)
    tmpl[0, :] = 255
    tmpl[-1, -1] = 0
    s, c = run_gpu(image, tmpl, method=method)
    assert_parity(image, tmpl, s, c)


def test_methods_agree_bit_for_bit():
    """Box passes + SumIT kernel and the three-dp4a kernel: the same sums
    and the same coefficient bits (the epilogue is shared)."""
    image, tmpl = rand_u8(300, 700), rand_u8(23, 45)
    sb, cb = run_gpu(image, tmpl, method="box")
    sd, cd = run_gpu(image, tmpl, method="dp4a")
    np.testing.assert_array_equal(sb, sd)
    np.testing.assert_array_equal(cb.view(np.uint32), cd.view(np.uint32))
    assert_parity(image, tmpl, sb, cb)


@pytest.mark.parametrize("h,w,wt,ht", [(2048, 2048, 32, 32), (2000, 2064, 13, 7),
                                        (1100, 1936, 64, 20)])
def test_large_image_both_forms(h, w, wt, ht):
    """Images large enough that the box form uses 2 output rows per
    half-warp for narrow templates too: both forms bit-identical, and a band
    of rows at each edge and sampled interior offsets against the oracle."""
    image, tmpl = rand_u8(h, w), rand_u8(ht, wt)
    sb, cb = run_gpu(image, tmpl, method="box")
    sd, cd = run_gpu(image, tmpl, method="dp4a")
    np.testing.assert_array_equal(sb, sd)
    np.testing.assert_array_equal(cb.view(np.uint32), cd.view(np.uint32))
    oh, ow = cb.shape
    for y0, y1 in ((0, 9), (oh - 9, oh)):
        rb, rcb, _ = oracle.ncc_u8(image[y0:y1 + ht - 1], tmpl, nthreads=NT)
        np.testing.assert_array_equal(sb[:, y0:y1, :], rb)
        assert np.abs(cb[y0:y1, :] - rcb).max() <= COEF_TOL
    ys, xs = RNG.integers(0, oh, 300), RNG.integers(0, ow, 300)
    rs, rc = oracle.ncc_u8_at(image, tmpl, xs, ys)
    np.testing.assert_array_equal(sb[:, ys, xs], rs)
    assert np.abs(cb[ys, xs] - rc).max() <= COEF_TOL


def test_method_setting_is_per_thread_and_restored():
    assert corr.ncc_get_method() == "box"
    corr.ncc_set_method("dp4a")
    try:
        image, tmpl = rand_u8(40, 100), rand_u8(5, 7)
        s, c = run_gpu(image, tmpl, method="box")      # per-call override
        assert corr.ncc_get_method() == "dp4a"
        assert_parity(image, tmpl, s, c)
    finally:
        corr.ncc_set_method("box")
    with pytest.raises(ValueError):
        corr.ncc_set_method("fft")


def test_byte_order_single_hot_byte():
    """Hot byte at each position of a 2-row, 16-wide template in turn."""
    image = rand_u8(40, 264, 128, 256)
    for j in range(2):
        for i in range(16):
            tmpl = np.zeros((2, 16), np.uint8)
            tmpl[j, i] = 200
            s, c = run_gpu(image, tmpl)
            assert_parity(image, tmpl, s, c)


def test_unaligned_image_pointer_and_width():
    """Image viewed at a 1-byte offset (general path) and w % 8 != 0."""
    base = rand_u8(1, 64 * 301 + 1).ravel()
    dev = torch.device("cuda", 0)
    tb = torch.from_numpy(base).to(dev)
    img_t = tb[1:].view(64, 301)
    tmpl = rand_u8(8, 32)
    s, c = corr.ncc_u8(img_t, torch.from_numpy(tmpl).to(dev))
    torch.cuda.synchronize()
    assert_parity(base[1:].reshape(64, 301), tmpl, s.cpu().numpy().view(np.uint32), c.cpu().numpy())


def test_single_offset_and_thin_shapes():
    for (h, w, wt, ht) in [(16, 16, 16, 16), (7, 8, 8, 7), (1, 4, 4, 1), (3, 4, 4, 1), (1, 9, 4, 1)]:
        image, tmpl = rand_u8(h, w), rand_u8(ht, wt)
        s, c = run_gpu(image, tmpl)
        assert_parity(image, tmpl, s, c)


@pytest.mark.parametrize("h,w,wt,ht", [(260, 264, 256, 258), (440, 300, 128, 430)])
def test_largest_template(h, w, wt, ht):
    """wt*ht close to 66051: SumISq near the uint32 limit, on the general
    path (256 x 258) and on the fast path (128 x 430, a tile that fits the
    shared memory of both forms) with both methods (the box sums' slides
    wrap modulo 2^32 and must still land on the exact sums)."""
    image, tmpl = rand_u8(h, w, 200, 256), rand_u8(ht, wt, 200, 256)
    for method in ("box", "dp4a"):
        s, c = run_gpu(image, tmpl, method=method)
        assert_parity(image, tmpl, s, c)
        assert s[1].max() > 2 ** 31   # the top bit of SumISq is in use


def test_flat_window_and_flat_template_give_zero():
    image = rand_u8(40, 300)
    image[10:30, 100:200] = 77
    tmpl = rand_u8(8, 16)
    s, c = run_gpu(image, tmpl)
    assert_parity(image, tmpl, s, c)
    assert (c[10:23, 100:185] == 0).all()
    s, c = run_gpu(image, np.full((8, 16), 9, np.uint8))
    assert (c == 0).all()
    assert_parity(image, np.full((8, 16), 9, np.uint8), s, c)


@pytest.mark.parametrize("method", ["box", "dp4a"])
def test_sums_only_and_coef_only(method):
    """Coefficient only: the box method keeps SumI / SumISq in scratch."""
    image, tmpl = rand_u8(70, 270), rand_u8(16, 16)
    ref = oracle.ncc_u8(image, tmpl, nthreads=NT)
    s, _ = run_gpu(image, tmpl, sums=True, coef=False, method=method)
    assert_parity(image, tmpl, s, None, ref)
    _, c = run_gpu(image, tmpl, sums=False, coef=True, method=method)
    assert_parity(image, tmpl, None, c, ref)


def test_guard_bands_untouched():
    """Outputs written into the middle of larger buffers: the canaries on
    both sides must survive."""
    image, tmpl = rand_u8(57, 333), rand_u8(9, 20)
    oh, ow = 57 - 9 + 1, 333 - 20 + 1
    dev = torch.device("cuda", 0)
    pad = 4096
    sb = torch.full((3 * oh * ow + 2 * pad,), -559038737, dtype=torch.int32, device=dev)
    cb = torch.full((oh * ow + 2 * pad,), 12345.0, dtype=torch.float32, device=dev)
    s = sb[pad:pad + 3 * oh * ow].view(3, oh, ow)
    c = cb[pad:pad + oh * ow].view(oh, ow)
    corr.ncc_u8_into(torch.from_numpy(image).to(dev), torch.from_numpy(tmpl).to(dev), s, c)
    torch.cuda.synchronize()
    assert (sb[:pad] == -559038737).all() and (sb[-pad:] == -559038737).all()
    assert (cb[:pad] == 12345.0).all() and (cb[-pad:] == 12345.0).all()
    assert_parity(image, tmpl, s.cpu().numpy().view(np.uint32), c.cpu().numpy())


def test_argument_errors_raise():
    dev = torch.device("cuda", 0)
    img = torch.zeros(300, 300, dtype=torch.uint8, device=dev)
    with pytest.raises(corr.CorrError) as e:   # 258 x 257 > 66051 template pixels
        corr.ncc_u8(img, torch.zeros(258, 257, dtype=torch.uint8, device=dev))
    assert e.value.code == -2
    tall = torch.zeros(16520, 8, dtype=torch.uint8, device=dev)
    with pytest.raises(corr.CorrError) as e:   # 4 x 16513 = 66052 pixels: SumISq may wrap
        corr.ncc_u8(tall, torch.zeros(16513, 4, dtype=torch.uint8, device=dev))
    assert e.value.code == -2


@pytest.mark.parametrize("h,w,wt,ht", [(200, 400, 369, 179), (7400, 40, 9, 7339),
                                       (440, 300, 128, 430)])
def test_all_255_at_the_size_limit(h, w, wt, ht):
    """All-255 image and template: SumISq and SumIT reach 65025 N, at the
    32-bit limit N = 66051 on the general kernel (369 x 179, and the narrow
    9 x 7339), and at the largest template the fast kernel takes (128 x 430),
    with both methods."""
    image = np.full((h, w), 255, np.uint8)
    tmpl = np.full((ht, wt), 255, np.uint8)
    ref = oracle.ncc_u8(image, tmpl, nthreads=NT)
    for method in ("box", "dp4a"):
        s, c = run_gpu(image, tmpl, method=method)
        assert_parity(image, tmpl, s, c, ref)
        assert (s[1] == 65025 * wt * ht).all() and (s[2] == 65025 * wt * ht).all()


@pytest.mark.parametrize("h,w,wt,ht", [(15000, 8, 3, 14600), (16100, 24, 4, 16000)])
def test_tall_narrow_template_general_kernel(h, w, wt, ht):
    """Templates a few pixels wide and thousands tall: the general kernel
    packs each row into its own word count (one word here)."""
    image, tmpl = rand_u8(h, w), rand_u8(ht, wt)
    for method in ("box", "dp4a"):
        s, c = run_gpu(image, tmpl, method=method)
        assert_parity(image, tmpl, s, c)


@pytest.mark.parametrize("method", ["box", "dp4a"])
@pytest.mark.parametrize("off,pitch,h,w,wt,ht", [
    (0, 512, 70, 300, 32, 32),      # 16-byte aligned rows: vector staging
    (8, 520, 45, 264, 20, 9),       # 8-byte aligned rows
    (3, 401, 60, 333, 17, 11),      # odd pitch: byte staging
    (5, 300, 40, 290, 160, 5),      # general kernel (wt > 128)
])
def test_pitched_image(method, off, pitch, h, w, wt, ht):
    """An image whose rows are `pitch` bytes apart (a crop of a larger
    buffer, passed through corr_ncc_u8_pitched): the same results as the
    dense copy."""
    dev = torch.device("cuda", 0)
    big = rand_u8(h + 2, pitch + 16)
    flat = torch.from_numpy(big.ravel().copy()).to(dev)
    view = flat[off:off + (h - 1) * pitch + w].as_strided((h, w), (pitch, 1))
    image = np.lib.stride_tricks.as_strided(big.ravel()[off:], (h, w), (pitch, 1)).copy()
    tmpl = rand_u8(ht, wt)
    s, c = corr.ncc_u8(view, torch.from_numpy(tmpl).to(dev), method=method)
    torch.cuda.synchronize()
    assert_parity(image, tmpl, s.cpu().numpy().view(np.uint32), c.cpu().numpy())


def test_buffer_kinds_through_the_abi():
    """Pageable host memory is refused before any launch; page-locked host
    outputs are written through their device alias and match."""
    import ctypes
    image, tmpl = rand_u8(40, 160), rand_u8(6, 10)
    dev = torch.device("cuda", 0)
    img, tm = torch.from_numpy(image).to(dev), torch.from_numpy(tmpl).to(dev)
    oh, ow = 40 - 6 + 1, 160 - 10 + 1
    lib = corr.load()
    lib.corr_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    vp = ctypes.c_void_p
    pageable = np.zeros((oh, ow), np.float32)
    rc = lib.corr_ncc_u8(vp(img.data_ptr()), 160, 40, vp(tm.data_ptr()), 10, 6, None,
                         vp(pageable.ctypes.data))
    assert rc == -1
    hs = torch.zeros((3, oh, ow), dtype=torch.int32).pin_memory()
    hc = torch.zeros((oh, ow), dtype=torch.float32).pin_memory()
    rc = lib.corr_ncc_u8(vp(img.data_ptr()), 160, 40, vp(tm.data_ptr()), 10, 6,
                         vp(hs.data_ptr()), vp(hc.data_ptr()))
    assert rc == 0
    torch.cuda.synchronize()
    assert_parity(image, tmpl, hs.numpy().view(np.uint32), hc.numpy())


def test_host_tensors_round_trip():
    image, tmpl = rand_u8(50, 200), rand_u8(8, 12)
    s, c = corr.ncc_u8(torch.from_numpy(image).pin_memory(), torch.from_numpy(tmpl))
    assert not s.is_cuda and not c.is_cuda
    assert_parity(image, tmpl, s.numpy().view(np.uint32), c.numpy())


def test_nondefault_stream():
    image, tmpl = rand_u8(90, 400), rand_u8(32, 32)
    dev = torch.device("cuda", 0)
    st = torch.cuda.Stream(dev)
    ti, tt = torch.from_numpy(image).to(dev), torch.from_numpy(tmpl).to(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        s, c = corr.ncc_u8(ti, tt)
    st.synchronize()
    assert_parity(image, tmpl, s.cpu().numpy().view(np.uint32), c.cpu().numpy())


# ---- the named workloads ------------------------------------------------

def test_workload_256_full():
    w = wl.ncc_256()
    s, c = run_gpu(w.image, w.tmpl)
    assert_parity(w.image, w.tmpl, s, c)
    x, y = w.offset
    assert c[y, x] == pytest.approx(1.0, abs=1e-6)


def test_workload_1080p_full():
    w = wl.ncc_1080p()
    s, c = run_gpu(w.image, w.tmpl)
    assert_parity(w.image, w.tmpl, s, c)
    x, y = w.offset
    assert np.unravel_index(np.argmax(c), c.shape) == (y, x)   # soft: expected peak


def test_workload_4k_sampled():
    """Full 4033x4033 launch, compared on sampled offsets (rows at both
    edges, the template's own offset, random interior points)."""
    w = wl.ncc_4k()
    s, c = run_gpu(w.image, w.tmpl)
    oh, ow = c.shape
    x0, y0 = w.offset
    ys = np.concatenate([RNG.integers(0, oh, 400), [0, 0, oh - 1, oh - 1, y0]])
    xs = np.concatenate([RNG.integers(0, ow, 400), [0, ow - 1, 0, ow - 1, x0]])
    rs, rc = oracle.ncc_u8_at(w.image, w.tmpl, xs, ys)
    np.testing.assert_array_equal(s[:, ys, xs], rs)
    assert np.abs(c[ys, xs] - rc).max() <= COEF_TOL
    assert c[y0, x0] == pytest.approx(1.0, abs=1e-6)
    assert np.abs(c).max() <= 1.0 + 1e-6
    # a full band of rows at the bottom edge, all columns
    band = w.image[oh - 3:, :]
    rb, rcb, _ = oracle.ncc_u8(band, w.tmpl, nthreads=NT)
    np.testing.assert_array_equal(s[:, oh - 3:, :], rb)
    assert np.abs(c[oh - 3:, :] - rcb).max() <= COEF_TOL
