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


def test_tcl_bounded_wait_gives_up_and_reports(tcl_on, monkeypatch):
    """The larger-matrix kernel's failure path without a fault:
    CORR_XCORR_TCL_STALL=1 leaves out the issuers' last completion signal,
    so their waits on it run out after about a second; corr_device_status
    reports CORR_ETIMEOUT, and the next call on the same context works."""
    dev = torch.device("cuda", 0)
    left, right = rand(1, 64, 64), rand(2, 64, 64)
    L, R = torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev)
    out = torch.empty((1, 2, 127, 127), dtype=torch.float32, device=dev)
    monkeypatch.setenv("CORR_XCORR_TCL_STALL", "1")
    corr.xcorr_f32_into(L, R, out)
    with pytest.raises(corr.CorrError) as e:
        corr.device_status()
    assert e.value.code == -4                  # CORR_ETIMEOUT
    monkeypatch.delenv("CORR_XCORR_TCL_STALL")
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


# Non-negative inputs: every product adds in the same direction, so the
# tensor cores' truncating FP32 accumulation drifts with the number of
# accumulates in a chain; the kernels keep chains to at most 96 and must
# stay well inside the bar.

def rand_pos(n, H, W):
    return RNG.uniform(0, 1, size=(n, H, W)).astype(np.float32)


@pytest.mark.parametrize("mode,shape", [
    ("tc", (32, 64, 16, 16)), ("tcl", (1, 1, 256, 256)), ("tcl", (1, 128, 64, 64)),
    ("tcl", (2, 3, 100, 130))])
def test_nonnegative_inputs_well_inside_the_bar(monkeypatch, mode, shape):
    monkeypatch.setenv("CORR_XCORR_TC", "1" if mode == "tc" else "0")
    monkeypatch.setenv("CORR_XCORR_TCL", "1" if mode == "tcl" else "0")
    nl, nr, H, W = shape
    got, ref, ab = run_check(rand_pos(nl, H, W), rand_pos(nr, H, W))
    assert (np.abs(got - ref) / (ab + 1e-30)).max() < 5e-6


# Items of several row units (partial tiles shrink by that factor) --------

@pytest.mark.parametrize("group,shape", [
    (2, (1, 1, 200, 130)), (3, (2, 3, 100, 70)), (4, (1, 5, 150, 40)),
    (64, (1, 2, 170, 90)), (5, (1, 1, 129, 257))])
def test_tcl_row_unit_groups(tcl_on, monkeypatch, group, shape):
    """Groups forced small (CORR_XCORR_TCL_GROUP) so that the oracle checks
    every output: a ragged last group, groups that start above a tile's
    first row, every row unit in one group; signed and non-negative."""
    monkeypatch.setenv("CORR_XCORR_TCL_GROUP", str(group))
    nl, nr, H, W = shape
    run_check(rand(nl, H, W), rand(nr, H, W))
    run_check(rand_pos(nl, H, W), rand_pos(nr, H, W))


@pytest.mark.parametrize("seed", range(4))
def test_tcl_random_larger_shapes_in_groups(tcl_on, monkeypatch, seed):
    """Random shapes with sides 90-160 (up to 5 row units, partial units at
    both ends), 1-2 lefts, 1-5 rights, a random forced group size, on
    non-negative inputs: every output against the oracle."""
    rng = np.random.default_rng(970 + seed)
    nl, nr = int(rng.integers(1, 3)), int(rng.integers(1, 6))
    H, W = int(rng.integers(90, 161)), int(rng.integers(90, 161))
    monkeypatch.setenv("CORR_XCORR_TCL_GROUP", str(int(rng.choice([1, 2, 3, 5]))))
    run_check(rand_pos(nl, H, W), rand_pos(nr, H, W))


def line_sums(v, w):
    """s[o] = sum_i v[i + o - (n - 1)] w[i] (n = len(v) = len(w)), in fp64:
    the sum of the full cross-correlation of two matrices over one output
    row (v, w their row sums) or column (their column sums)."""
    return np.convolve(v.astype(np.float64), w.astype(np.float64)[::-1])


def check_line_sums(left, right, got):
    """Row and column sums of a pair's output against line_sums of the
    matrices' row and column sums, within the parity bar summed over the
    line (inputs non-negative, so sum |L*R| is the sum itself).  A partial
    tile or a row unit left out moves some line sum by well over the bar."""
    L, R = left[0].astype(np.float64), right[0].astype(np.float64)
    g = got[0, 0]
    rows = line_sums(L.sum(1), R.sum(1))
    cols = line_sums(L.sum(0), R.sum(0))
    for have, want in ((g.sum(1), rows), (g.sum(0), cols)):
        bad = np.abs(have - want) > REL_TOL * want + 1e-9
        assert not bad.any(), f"{bad.sum()} line sums out of tolerance, first at {np.argmax(bad)}"


def test_line_sums_match_the_oracle():
    left = RNG.uniform(0, 1, size=(1, 21, 34)).astype(np.float32)
    right = RNG.uniform(0, 1, size=(1, 21, 34)).astype(np.float32)
    ref, _ = oracle.xcorr_f32(left, right)
    check_line_sums(left, right, ref)


@pytest.mark.parametrize("n", [512, 1024])
def test_tcl_large_pair(n):
    """Default choice for one n x n pair (row-unit groups of 8 and 32): at
    sampled outputs (every tile's corner rows and columns, plus random
    ones) against the oracle, and every output row and column through its
    sum."""
    for v in ("CORR_XCORR_TCL", "CORR_XCORR_TC", "CORR_XCORR_WARP", "CORR_XCORR_TCL_GROUP"):
        assert v not in os.environ
    assert corr.xcorr_f32_kernel(1, 1, n, n) == "tensor_large"
    rng = np.random.default_rng(4242 + n)
    left = rng.uniform(0, 1, size=(1, n, n)).astype(np.float32)
    right = rng.uniform(0, 1, size=(1, n, n)).astype(np.float32)
    dev = torch.device("cuda", 0)
    out = torch.full((1, 1, 2 * n - 1, 2 * n - 1), float("nan"), dtype=torch.float32,
                     device=dev)
    corr.xcorr_f32_into(torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev), out)
    corr.device_status()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    edges = sorted({e for t in range(0, 2 * n - 1, 128) for e in (t, t + 127) if e < 2 * n - 1}
                   | {2 * n - 2})
    oy, ox = np.meshgrid(edges, edges, indexing="ij")
    oy = np.concatenate([oy.ravel(), rng.integers(0, 2 * n - 1, 1500)])
    ox = np.concatenate([ox.ravel(), rng.integers(0, 2 * n - 1, 1500)])
    zeros = np.zeros(oy.size, np.int32)
    want, ab = oracle.xcorr_f32_at(left, right, zeros, zeros, oy, ox)
    have = got[0, 0, oy, ox].astype(np.float64)
    assert (np.abs(have - want) <= REL_TOL * ab + 1e-30).all()
    check_line_sums(left, right, got)
