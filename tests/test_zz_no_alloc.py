"""corr_xcorr_f32_noalloc: the cross-correlation for callers that cannot let
a library allocate device memory (applications that reserve all GPU memory
for their own allocator, plug-ins whose host forbids driver allocations,
loops that must never wait on an allocator).  Its split-row scratch is a
fixed array inside the library instead of pool memory.

Checked here, through the C ABI, on two calls in a row:
  * every output of every pair against the fp64 oracle, within the f32
    parity bar (1e-5 * sum|L*R| over that output's own overlap);
  * bit-identity with corr_xcorr_f32 on every pair wherever both run the
    same kernel (same plan, same summation order); the larger-matrix
    tensor-core kernel, whose partial sums need more scratch than the
    array holds, is switched off for that comparison, and checked against
    the oracle alone under the default choice;
  * a banded shape run after a different banded / segmented shape has left
    its own partial sums in the array (a slot the second call failed to
    write would then show up as a wrong value, not as a zero);
  * the larger-matrix tensor-core kernel where its partial tiles fit the
    array (its item counter lives there too);
  * a shape needing more than the array holds is rejected with
    CORR_EUNSUPPORTED before anything runs.
This file is collected last so that a failure here stops a -x run only after
every other test.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import normalized_cross_correlation_u8_gb300 as corr
import oracle

pytestmark = pytest.mark.gpu
REL_TOL = 1e-5
NT = max(1, os.cpu_count() or 1)


def call(fn, L, R, out):
    lib = corr.load()
    lib.corr_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    nl, H, W = L.shape
    return fn(ctypes.c_void_p(L.data_ptr()), nl, ctypes.c_void_p(R.data_ptr()),
              R.shape[0], H, W, ctypes.c_void_p(out.data_ptr()))


def inputs(nl, nr, H, W, seed):
    rng = np.random.default_rng(seed)
    left = rng.uniform(-1, 1, size=(nl, H, W)).astype(np.float32)
    right = rng.uniform(-1, 1, size=(nr, H, W)).astype(np.float32)
    dev = torch.device("cuda", 0)
    return left, right, torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev)


def run_both(L, R, calls=2):
    """corr_xcorr_f32 once, then corr_xcorr_f32_noalloc `calls` times into
    NaN-filled buffers; returns (reference, [noalloc outputs]) on the host."""
    nl, H, W = L.shape
    shape = (nl, R.shape[0], 2 * H - 1, 2 * W - 1)
    lib = corr.load()
    ref = torch.empty(shape, dtype=torch.float32, device=L.device)
    assert call(lib.corr_xcorr_f32, L, R, ref) == 0
    outs = []
    for _ in range(calls):
        got = torch.full(shape, float("nan"), dtype=torch.float32, device=L.device)
        assert call(lib.corr_xcorr_f32_noalloc, L, R, got) == 0
        torch.cuda.synchronize()
        outs.append(got.cpu())
    return ref.cpu(), outs


@pytest.mark.parametrize("nl,nr,H,W", [(1, 1, 256, 256), (1, 2, 130, 257), (1, 1, 24, 800),
                                       (2, 3, 40, 40), (32, 64, 16, 16)])
def test_noalloc_matches_oracle_and_allocating_entry_point(nl, nr, H, W, monkeypatch):
    monkeypatch.setenv("CORR_XCORR_TCL", "0")     # same plan on both entry points
    left, right, L, R = inputs(nl, nr, H, W, 77 + H)
    ref, outs = run_both(L, R)
    exact, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    for got in outs:
        assert torch.equal(got, ref)             # every pair, bit for bit
        g = got.numpy().astype(np.float64)
        assert np.isfinite(g).all()
        err = np.abs(g - exact)
        worst = np.unravel_index(np.argmax(err - REL_TOL * ab), err.shape)
        assert (err <= REL_TOL * ab + 1e-30).all(), \
            f"error {err[worst]} > {REL_TOL} * {ab[worst]} at {worst}"


def test_noalloc_default_choice_against_the_oracle():
    """Default kernel choice: a 256x256 pair takes the larger-matrix
    tensor-core kernel on corr_xcorr_f32 but a kernel that fits the fixed
    array here; both meet the bar."""
    left, right, L, R = inputs(1, 1, 256, 256, 9)
    ref, outs = run_both(L, R)
    exact, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    for got in (ref, *outs):
        err = np.abs(got.numpy().astype(np.float64) - exact)
        assert (err <= REL_TOL * ab + 1e-30).all()


def test_noalloc_runs_the_tensor_core_kernel_where_its_partials_fit():
    """1 x 32 of 64x64 takes the larger-matrix tensor-core kernel on both
    entry points (128 partial tiles, 8 MB, and its item counter in the
    array): bit for bit the same as corr_xcorr_f32, twice in a row (the
    counter is zeroed per call), and within the bar of the oracle, on
    non-negative inputs (the tensor cores' accumulation drifts most there)."""
    assert corr.xcorr_f32_kernel(1, 32, 64, 64) == "tensor_large"
    rng = np.random.default_rng(31)
    left = rng.uniform(0, 1, size=(1, 64, 64)).astype(np.float32)
    right = rng.uniform(0, 1, size=(32, 64, 64)).astype(np.float32)
    dev = torch.device("cuda", 0)
    L, R = torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev)
    ref, outs = run_both(L, R)
    exact, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    for got in outs:
        assert torch.equal(got, ref)
        assert (np.abs(got.numpy().astype(np.float64) - exact) <= REL_TOL * ab + 1e-30).all()


def test_noalloc_after_another_shape_left_data_in_the_array(monkeypatch):
    """Two banded / segmented shapes back to back: the second call's reads
    of the shared array must all be of slots it wrote itself."""
    monkeypatch.setenv("CORR_XCORR_TCL", "0")     # same plan on both entry points
    _, _, L1, R1 = inputs(1, 1, 24, 800, 5)      # three x segments
    assert call(corr.load().corr_xcorr_f32_noalloc, L1, R1,
                torch.empty((1, 1, 47, 1599), dtype=torch.float32, device=L1.device)) == 0
    left, right, L, R = inputs(1, 1, 256, 256, 6)   # two row bands
    ref, outs = run_both(L, R, calls=1)
    assert torch.equal(outs[0], ref)
    exact, ab = oracle.xcorr_f32(left, right, nthreads=NT)
    assert (np.abs(outs[0].numpy().astype(np.float64) - exact) <= REL_TOL * ab + 1e-30).all()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda", 0)
    # one 1024x1024 pair: three x segments of partial sums, 48 MiB > 16 MiB
    L = torch.zeros((1, 1024, 1024), dtype=torch.float32, device=dev)
    R = torch.zeros((1, 1024, 1024), dtype=torch.float32, device=dev)
    out = torch.full((1, 1, 2047, 2047), 7.0, dtype=torch.float32, device=dev)
    assert call(corr.load().corr_xcorr_f32_noalloc, L, R, out) == -2
    torch.cuda.synchronize()
    assert (out == 7.0).all()                  # nothing was launched
