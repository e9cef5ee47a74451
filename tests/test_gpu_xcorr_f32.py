"""GPU parity of corr_xcorr_f32 against the CPU oracle (fp64).

Bar ("Efficient GPU-accelerated Parallel Cross-correlation" artifact README:
all overlaps, one-to-one / one-to-many / n-to-m): every output element within
1e-5 * sum|L*R| over its own overlap of the oracle's double-precision value.
All calls go through the C ABI via the ctypes binding.
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
REL_TOL = 1e-5
NT = max(1, os.cpu_count() or 1)
RNG = np.random.default_rng(515151)


def run_gpu(left, right):
    dev = torch.device("cuda", 0)
    out = corr.xcorr_f32(torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev))
    torch.cuda.synchronize()
    return out.cpu().numpy()


def assert_parity(got, ref, ab):
    assert got.shape == ref.shape
    err = np.abs(got.astype(np.float64) - ref)
    bound = REL_TOL * ab + 1e-30
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} elements out of tolerance; worst ratio "
                           f"{(err / bound).max():.3g} at {np.unravel_index((err / bound).argmax(), err.shape)}")


def check(left, right):
    got = run_gpu(left, right)
    ref, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    assert_parity(got, ref, ab)
    return got


def rand(n, H, W, dist="uniform"):
    if dist == "uniform":
        return RNG.uniform(-1, 1, size=(n, H, W)).astype(np.float32)
    return RNG.standard_normal(size=(n, H, W)).astype(np.float32)


@pytest.mark.parametrize("path", sorted(glob.glob(os.path.join(
    os.path.dirname(__file__), "golden", "xcorr_f32_*.txt"))))
def test_fixture(path):
    fx = read_fixture(path)
    got = run_gpu(fx["left"].astype(np.float32), fx["right"].astype(np.float32))
    assert_parity(got, fx["out"], fx["abs"])


@pytest.mark.parametrize("nl,nr,H,W", [
    (1, 1, 1, 1), (1, 1, 1, 3), (1, 1, 3, 1), (1, 1, 2, 2), (1, 1, 3, 5),
    (1, 1, 16, 16), (1, 1, 17, 33), (1, 1, 40, 9), (1, 1, 100, 130),
    (1, 5, 31, 29), (1, 37, 64, 64), (3, 4, 7, 11), (5, 9, 16, 16),
    # small matrices in batches: block shapes 16 x 32, 8 x 64 and 64 x 8
    (16, 40, 10, 10), (8, 64, 12, 12), (70, 5, 6, 7),
    # small batches, pairs of shifts per lane: W = 1, 2, 3 and odd / even W
    (20, 10, 4, 1), (10, 10, 3, 2), (12, 8, 5, 3), (64, 1, 1, 16), (9, 9, 16, 16),
    (40, 33, 13, 15),
    (2, 3, 50, 8), (33, 3, 5, 5), (1, 1, 1, 300), (1, 1, 300, 1),
    # rights in lanes: ragged right block, W % 4 != 0, short H, several lefts
    (2, 40, 20, 12), (1, 33, 30, 10), (3, 64, 9, 40), (1, 96, 33, 8),
    # row kernel: two row bands, a ragged last chunk, W % 4 != 0
    (1, 2, 130, 257), (2, 1, 200, 64),
    # row kernel, whole rows in 16-row chunks (too wide for 32): one and two
    # bands, two pairs
    (1, 1, 40, 520), (1, 1, 140, 420), (2, 1, 26, 450),
    # row kernel, windows of three x segments (rows too wide to stage whole),
    # also with W % 4 != 0 (element-wise staging)
    (1, 1, 24, 800), (1, 1, 30, 799),
    # row kernel with fewer rows than lanes (rows split along x over lanes)
    (1, 1, 5, 400), (2, 2, 3, 700), (1, 6, 4, 520), (1, 1, 16, 1000),
])
def test_shapes(nl, nr, H, W, monkeypatch):
    """The scalar kernels (the tensor-core kernels, tested on their own in
    test_gpu_xcorr_tc.py, switched off so that every block shape above still
    reaches the kernel it was written for), then the library's own choice."""
    left, right = rand(nl, H, W), rand(nr, H, W, "normal")
    monkeypatch.setenv("CORR_XCORR_TC", "0")
    monkeypatch.setenv("CORR_XCORR_TCL", "0")
    check(left, right)
    monkeypatch.delenv("CORR_XCORR_TC")
    monkeypatch.delenv("CORR_XCORR_TCL")
    check(left, right)


def test_delta_reproduces_shifted_matrix():
    H, W = 23, 37
    left = rand(1, H, W)
    d = np.zeros((1, H, W), np.float32)
    d[0, 5, 9] = 1
    got = run_gpu(left, d)[0, 0]
    for dy in range(-H + 1, H):
        for dx in range(-W + 1, W):
            y, x = 5 + dy, 9 + dx
            e = left[0, y, x] if (0 <= y < H and 0 <= x < W) else 0.0
            assert got[dy + H - 1, dx + W - 1] == e


def test_sum_identity():
    left, right = rand(2, 20, 30), rand(3, 20, 30)
    got = run_gpu(left, right).astype(np.float64)
    for li in range(2):
        for ri in range(3):
            s = left[li].astype(np.float64).sum() * right[ri].astype(np.float64).sum()
            assert abs(got[li, ri].sum() - s) <= 1e-4 * (np.abs(left[li]).sum() * np.abs(right[ri]).sum())


def test_guard_bands_untouched():
    left, right = rand(2, 13, 21), rand(3, 13, 21)
    n = 2 * 3 * 25 * 41
    pad = 2048
    dev = torch.device("cuda", 0)
    buf = torch.full((n + 2 * pad,), 777.0, dtype=torch.float32, device=dev)
    out = buf[pad:pad + n].view(2, 3, 25, 41)
    corr.xcorr_f32_into(torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev), out)
    torch.cuda.synchronize()
    assert (buf[:pad] == 777.0).all() and (buf[-pad:] == 777.0).all()
    ref, ab = oracle.xcorr_f32(left, right)
    assert_parity(out.cpu().numpy(), ref, ab)


def test_host_tensors_round_trip():
    left, right = rand(1, 30, 30), rand(2, 30, 30)
    got = corr.xcorr_f32(torch.from_numpy(left).pin_memory(), torch.from_numpy(right).pin_memory())
    assert not got.is_cuda
    ref, ab = oracle.xcorr_f32(left, right)
    assert_parity(got.numpy(), ref, ab)


# ---- the named workloads ------------------------------------------------

def test_workload_one_to_one_full():
    w = wl.xcorr_one_to_one()
    check(w.left, w.right)


def test_workload_one_to_many_full():
    w = wl.xcorr_one_to_many()
    check(w.left, w.right)


def test_workload_n_to_m_full():
    w = wl.xcorr_n_to_m()
    check(w.left, w.right)


def test_scratch_is_not_kept_between_calls():
    """A banded shape (one 256x256 pair: two row bands) takes pool scratch
    for its partial sums; once the device is synchronised the library holds
    no device memory."""
    dev = torch.device("cuda", 0)
    L = torch.from_numpy(rand(1, 256, 256)).to(dev)
    R = torch.from_numpy(rand(1, 256, 256)).to(dev)
    out = torch.empty((1, 1, 511, 511), dtype=torch.float32, device=dev)
    for _ in range(3):
        corr.xcorr_f32_into(L, R, out)          # queued back to back: one block reused
    torch.cuda.synchronize()
    assert corr.scratch_reserved(dev) == 0


@pytest.mark.parametrize("nl,nr,H,W", [(1, 2, 130, 257), (1, 1, 24, 800), (2, 2, 3, 700)])
def test_rows_kernels_item_loop(nl, nr, H, W, monkeypatch):
    """The rows kernels' work-item loop (taken by grids larger than 2^30
    CTAs) on ordinary shapes: the library caps the grid at
    CORR_XCORR_MAX_GRID, so each CTA loops over several items."""
    monkeypatch.setenv("CORR_XCORR_MAX_GRID", "37")
    check(rand(nl, H, W), rand(nr, H, W, "normal"))


@pytest.mark.parametrize("nl,nr,H,W", [(1, 1, 1, 1), (1, 1, 1, 4096), (2, 3, 2, 700),
                                       (1, 2, 5, 33), (3, 2, 7, 31), (1, 1, 40, 64),
                                       (2, 2, 16, 16)])
def test_warp_per_overlap_kernel(nl, nr, H, W, monkeypatch):
    """The warp-per-overlap kernel (CORR_XCORR_WARP=1 routes every shape to
    it): overlaps wider and narrower than a warp, single rows and columns."""
    monkeypatch.setenv("CORR_XCORR_WARP", "1")
    check(rand(nl, H, W), rand(nr, H, W, "normal"))
