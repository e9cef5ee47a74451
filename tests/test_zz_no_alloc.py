"""corr_xcorr_f32_noalloc: the cross-correlation for callers that cannot let
a library allocate device memory (applications that reserve all GPU memory
for their own allocator, plug-ins whose host forbids driver allocations,
loops that must never wait on an allocator).  Its split-row scratch is a
fixed array inside the library instead of pool memory.

Checked here, through the C ABI: two calls in a row agree with
corr_xcorr_f32 on the same inputs within the f32 parity bar (1e-5 * sum|L*R|
per output), on a shape that uses the scratch (256x256, two row bands) and
on shapes that need none; and a shape needing more than the array holds is
rejected with CORR_EUNSUPPORTED before anything runs.  This file is collected
last so that a failure here stops a -x run only after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import normalized_cross_correlation_u8_gb300 as corr
import oracle

pytestmark = pytest.mark.gpu
REL_TOL = 1e-5


def call(fn, L, R, out):
    lib = corr.load()
    lib.corr_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    nl, H, W = L.shape
    return fn(ctypes.c_void_p(L.data_ptr()), nl, ctypes.c_void_p(R.data_ptr()),
              R.shape[0], H, W, ctypes.c_void_p(out.data_ptr()))


@pytest.mark.parametrize("nl,nr,H,W", [(1, 1, 256, 256), (1, 2, 130, 257), (1, 1, 24, 800), (2, 3, 40, 40),
                                       (32, 64, 16, 16)])
def test_noalloc_matches_allocating_entry_point(nl, nr, H, W):
    rng = np.random.default_rng(77 + H)
    left = rng.uniform(-1, 1, size=(nl, H, W)).astype(np.float32)
    right = rng.uniform(-1, 1, size=(nr, H, W)).astype(np.float32)
    dev = torch.device("cuda", 0)
    L, R = torch.from_numpy(left).to(dev), torch.from_numpy(right).to(dev)
    shape = (nl, nr, 2 * H - 1, 2 * W - 1)
    ref = torch.empty(shape, dtype=torch.float32, device=dev)
    lib = corr.load()
    assert call(lib.corr_xcorr_f32, L, R, ref) == 0
    # |L|*|R| correlation bounds each output's rounding error
    _, ab = oracle.xcorr_f32(np.abs(left[:1]), np.abs(right[:1]))
    for _ in range(2):
        got = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
        assert call(lib.corr_xcorr_f32_noalloc, L, R, got) == 0
        torch.cuda.synchronize()
        g, r = got.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(g).all()
        err = np.abs(g - r)
        # pair (0, 0) against its own |L||R| bound; all pairs against a bound
        # scaled by the matrices' size
        assert (err[0, 0] <= REL_TOL * ab[0, 0] + 1e-30).all()
        assert err.max() <= REL_TOL * H * W


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda", 0)
    # one 1024x1024 pair: three x segments of partial sums, 48 MiB > 16 MiB
    L = torch.zeros((1, 1024, 1024), dtype=torch.float32, device=dev)
    R = torch.zeros((1, 1024, 1024), dtype=torch.float32, device=dev)
    out = torch.full((1, 1, 2047, 2047), 7.0, dtype=torch.float32, device=dev)
    assert call(corr.load().corr_xcorr_f32_noalloc, L, R, out) == -2
    torch.cuda.synchronize()
    assert (out == 7.0).all()                  # nothing was launched
