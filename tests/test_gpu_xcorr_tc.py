"""GPU parity of the tensor-core form of corr_xcorr_f32 (small matrices,
H, W <= 16) against the CPU oracle (fp64).

The kernel recasts the artifact README's n-to-m batch ("Efficient
GPU-accelerated Parallel Cross-correlation", kernel overview: multi-matrix
reuse) as a dense contraction on the tensor cores with split TF32 operands
(hi*hi + hi*lo + lo*hi).  Bar: every output element within 1e-5 * sum|L*R|
over its own overlap of the oracle's double-precision value, as for the
scalar kernels.  CORR_XCORR_TC=1 routes every supported shape to it; each
case also checks that no bounded wait in the kernel gave up.
"""
import os

import numpy as np
import pytest
import torch

import normalized_cross_correlation_u8_gb300 as corr
import oracle
from normalized_cross_correlation_u8_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
REL_TOL = 1e-5
NT = max(1, os.cpu_count() or 1)
RNG = np.random.default_rng(717171)


@pytest.fixture
def tc_on(monkeypatch):
    monkeypatch.setenv("CORR_XCORR_TC", "1")


def run_check(left, right, offset=0):
    """Inputs placed `offset` floats into their device buffers (offset 1:
    rows not 16-byte aligned, so the kernel's scalar staging runs)."""
    dev = torch.device("cuda", 0)
    nl, H, W = left.shape
    nr = right.shape[0]
    Lb = torch.zeros(left.size + offset, dtype=torch.float32, device=dev)
    Rb = torch.zeros(right.size + offset, dtype=torch.float32, device=dev)
    Lb[offset:] = torch.from_numpy(left.ravel())
    Rb[offset:] = torch.from_numpy(right.ravel())
    L = Lb[offset:].view(nl, H, W)
    R = Rb[offset:].view(nr, H, W)
    out = torch.full((nl, nr, 2 * H - 1, 2 * W - 1), float("nan"), dtype=torch.float32,
                     device=dev)
    corr.xcorr_f32_into(L, R, out)
    corr.device_status()                 # raises if a bounded wait gave up
    got = out.cpu().numpy().astype(np.float64)
    ref, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    bound = REL_TOL * ab + 1e-30
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), (f"{(err > bound).sum()} elements out of tolerance; "
                                  f"worst ratio {(err / bound)[worst]:.3g} at {worst}")
    return got, ref, ab


def rand(n, H, W):
    return RNG.uniform(-1, 1, size=(n, H, W)).astype(np.float32)


# tiles: 4 lefts x (2 shifts dy x 64 rights | 4 x 32 | 8 x 16); partial
# tiles in every direction; W <= 8 takes one 8-deep K step per row
SHAPES = [
    (4, 16, 2, 2), (1, 1, 1, 1), (3, 5, 3, 5), (5, 7, 16, 16), (4, 16, 16, 16),
    (8, 20, 9, 13), (6, 33, 11, 7), (9, 64, 16, 16), (7, 100, 12, 16), (2, 70, 1, 16),
    (3, 40, 16, 1), (13, 17, 8, 8), (32, 64, 16, 16),
]


@pytest.mark.parametrize("nl,nr,H,W", SHAPES)
def test_tc_matches_oracle(tc_on, nl, nr, H, W):
    run_check(rand(nl, H, W), rand(nr, H, W))


@pytest.mark.parametrize("nl,nr,H,W", [(5, 9, 16, 16), (4, 24, 10, 12), (3, 3, 15, 15)])
def test_tc_unaligned_rows(tc_on, nl, nr, H, W):
    run_check(rand(nl, H, W), rand(nr, H, W), offset=1)


def test_tc_n_to_m_workload_full(tc_on):
    """The 32 x 64 batch of 16x16 matrices, every output."""
    w = wl.xcorr_n_to_m()
    run_check(w.left, w.right)


def test_tc_error_well_inside_the_bar(tc_on):
    """The split products leave about 3 * 2^-22 of |l*r| each, and the
    tensor cores accumulate in FP32; on random inputs the worst element
    (measured on GB300: 1.2e-6 of sum|l*r|) stays well below the 1e-5 bar,
    while a dropped hi*lo or lo*hi term would leave errors near 2^-11."""
    got, ref, ab = run_check(rand(16, 16, 16), rand(64, 16, 16))
    assert (np.abs(got - ref) / (ab + 1e-30)).max() < 4e-6


def test_tc_delta_reproduces_shifted_matrix(tc_on):
    """R = delta at (a, b): out[dy][dx] = L[a + dy][b + dx], exactly (one
    nonzero product per output, split operands hi + lo recombine it)."""
    H, W, a, b = 16, 16, 5, 9
    left = rand(4, H, W)
    right = np.zeros((16, H, W), np.float32)
    right[:, a, b] = 1.0
    got, _, _ = run_check(left, right)
    for dy in range(-(H - 1), H):
        for dx in range(-(W - 1), W):
            y, x = a + dy, b + dx
            want = left[:, y, x] if 0 <= y < H and 0 <= x < W else 0.0
            np.testing.assert_allclose(got[:, 0, dy + H - 1, dx + W - 1], want,
                                       rtol=3e-7, atol=0)


# ---- larger matrices: one left's 128 shifts dx x (shift dy, right) slots,
# K cut into 32 x 32 units whose partial sums a second kernel adds --------

@pytest.fixture
def tcl_on(monkeypatch):
    monkeypatch.setenv("CORR_XCORR_TCL", "1")
    monkeypatch.setenv("CORR_XCORR_TC", "0")
    monkeypatch.setenv("CORR_XCORR_WARP", "0")


@pytest.mark.parametrize("nl,nr,H,W", [
    (1, 1, 40, 70), (2, 3, 33, 100), (1, 5, 130, 20), (1, 2, 17, 17), (3, 1, 1, 300),
    (1, 4, 64, 64), (1, 6, 5, 129), (2, 9, 48, 33), (1, 1, 200, 1)])
def test_tcl_matches_oracle(tcl_on, nl, nr, H, W):
    assert corr.xcorr_f32_kernel(nl, nr, H, W) == "tensor_large"
    run_check(rand(nl, H, W), rand(nr, H, W))


def test_tcl_unaligned_rows(tcl_on):
    run_check(rand(1, 50, 60), rand(7, 50, 60), offset=1)


def test_tcl_one_to_one_workload_full(tcl_on):
    """The 256x256 pair, every output (1024 units of K over 16 tiles)."""
    w = wl.xcorr_one_to_one()
    run_check(w.left, w.right)


def test_tcl_one_to_many_workload_full(tcl_on):
    """One 64x64 left against 128 rights, every output."""
    w = wl.xcorr_one_to_many()
    run_check(w.left, w.right)


def test_bounded_wait_gives_up_and_reports(tc_on, monkeypatch):
    """Failure path without a fault: CORR_XCORR_TC_STALL=1 leaves out the
    kernel's last completion signal, so every wait on it runs out after
    about a second; corr_device_status reports CORR_ETIMEOUT, the outputs
    are left as they were, and the next call on the same context works."""
    dev = torch.device("cuda", 0)
    left, right = rand(4, 16, 16), rand(16, 16, 16)
    L, R = torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev)
    out = torch.full((4, 16, 31, 31), 5.0, dtype=torch.float32, device=dev)
    monkeypatch.setenv("CORR_XCORR_TC_STALL", "1")
    corr.xcorr_f32_into(L, R, out)
    with pytest.raises(corr.CorrError) as e:
        corr.device_status()
    assert e.value.code == -4                  # CORR_ETIMEOUT
    assert (out == 5.0).all()
    monkeypatch.delenv("CORR_XCORR_TC_STALL")
    run_check(left, right)                     # context still usable, status clear


@pytest.mark.parametrize("seed", range(6))
def test_tc_random_shapes(tc_on, seed):
    """Random batch shapes within the small-matrix kernel's range."""
    rng = np.random.default_rng(900 + seed)
    nl, nr = int(rng.integers(1, 40)), int(rng.integers(1, 70))
    H, W = int(rng.integers(1, 17)), int(rng.integers(1, 17))
    run_check(rand(nl, H, W), rand(nr, H, W))


@pytest.mark.parametrize("seed", range(6))
def test_tcl_random_shapes(tcl_on, seed):
    """Random shapes for the larger-matrix kernel: one or a few lefts,
    1-20 rights, sides 1-90 (tiles cut in every direction, K units that
    straddle the matrix edges)."""
    rng = np.random.default_rng(950 + seed)
    nl, nr = int(rng.integers(1, 3)), int(rng.integers(1, 21))
    H, W = int(rng.integers(1, 91)), int(rng.integers(1, 91))
    run_check(rand(nl, H, W), rand(nr, H, W))


def test_tc_large_batch_of_small_matrices(tc_on):
    """A batch of 160 x 96 pairs of 12x12 (many tiles, partial right tiles)."""
    run_check(rand(160, 12, 12), rand(96, 12, 12))


@pytest.mark.parametrize("mode,shape", [("tc", (5, 7, 13, 11)), ("tcl", (1, 6, 45, 70))])
def test_tensor_core_kernels_write_nothing_outside_the_output(monkeypatch, mode, shape):
    """Outputs written into the middle of a larger buffer: canaries on both
    sides survive (the epilogues store whole lines of runs: their edges
    must stop at the output's)."""
    monkeypatch.setenv("CORR_XCORR_TC" if mode == "tc" else "CORR_XCORR_TCL", "1")
    nl, nr, H, W = shape
    left, right = rand(nl, H, W), rand(nr, H, W)
    dev = torch.device("cuda", 0)
    n = nl * nr * (2 * H - 1) * (2 * W - 1)
    pad = 4099                                  # odd: the output starts mid-line
    buf = torch.full((n + 2 * pad,), 777.0, dtype=torch.float32, device=dev)
    out = buf[pad:pad + n].view(nl, nr, 2 * H - 1, 2 * W - 1)
    corr.xcorr_f32_into(torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev), out)
    corr.device_status()
    assert (buf[:pad] == 777.0).all() and (buf[-pad:] == 777.0).all()
    ref, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    assert (np.abs(out.cpu().numpy().astype(np.float64) - ref) <= REL_TOL * ab + 1e-30).all()
