"""ctypes front end of the C oracle (oracle.c).  TEST INFRASTRUCTURE ONLY.

Argument marshalling only: every number comes from the plain loops in
oracle.c, whose header cites the pages each definition follows:

* u8 normalized cross-correlation -- The CUDA Handbook ch. 15 "Image
  Processing: Normalized Correlation", section 15.5 "Instruction-Level
  Parallelism and DP4A" (the sums SumI, SumISq, SumIT over unsigned pixels).
* f32 full cross-correlation -- "Efficient GPU-accelerated Parallel
  Cross-correlation" artifact README, kernel overview (one overlap per output,
  all shifts, one-to-one / one-to-many / n-to-m).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def open_library(path):
    """Load an oracle shared library from `path` and declare its functions."""
    lib = ctypes.CDLL(path)
    c_int, c_long, vp = ctypes.c_int, ctypes.c_long, ctypes.c_void_p
    lib.oracle_ncc_u8.argtypes = [vp, c_int, c_int, vp, c_int, c_int,
                                  vp, vp, vp, c_int]
    lib.oracle_ncc_u8_at.argtypes = [vp, c_int, c_int, vp, c_int, c_int,
                                     c_long, vp, vp, vp, vp]
    lib.oracle_template_sums.argtypes = [vp, c_int, c_int, vp]
    lib.oracle_xcorr_f32.argtypes = [vp, c_int, vp, c_int, c_int, c_int,
                                     vp, vp, c_int]
    lib.oracle_xcorr_f32_at.argtypes = [vp, c_int, vp, c_int, c_int, c_int,
                                        c_long, vp, vp, vp, vp, vp, vp]
    for f in (lib.oracle_ncc_u8, lib.oracle_ncc_u8_at,
              lib.oracle_template_sums, lib.oracle_xcorr_f32,
              lib.oracle_xcorr_f32_at):
        f.restype = c_int
    return lib


def load():
    """Build (if stale) and load liboracle.so; returns the ctypes handle."""
    global _lib
    if _lib is None:
        _lib = open_library(_build.build())
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc != 0:
        raise OracleError(f"oracle returned {rc}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _u8(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8 or a.ndim != 2:
        raise ValueError("expected a 2-D uint8 array")
    return a


def _f32(a, ndim):
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise ValueError("expected float32")
    if a.ndim == ndim - 1:
        a = a[None]
    if a.ndim != ndim:
        raise ValueError(f"expected {ndim}-D float32")
    return a


def default_threads():
    return max(1, os.cpu_count() or 1)


def ncc_u8(image, tmpl, nthreads=1):
    """All valid offsets.  Returns (sums [3,oh,ow] uint32, coef f64 [oh,ow],
    coef f32 [oh,ow])."""
    image, tmpl = _u8(image), _u8(tmpl)
    h, w = image.shape
    ht, wt = tmpl.shape
    oh, ow = max(h - ht + 1, 0), max(w - wt + 1, 0)
    sums = np.zeros((3, oh, ow), np.uint32)
    c64 = np.zeros((oh, ow), np.float64)
    c32 = np.zeros((oh, ow), np.float32)
    _check(load().oracle_ncc_u8(_ptr(image), w, h, _ptr(tmpl), wt, ht,
                                _ptr(sums), _ptr(c64), _ptr(c32), int(nthreads)))
    return sums, c64, c32


def ncc_u8_at(image, tmpl, xs, ys):
    """Offsets (xs[k], ys[k]).  Returns (sums [3,count] uint32, coef f64)."""
    image, tmpl = _u8(image), _u8(tmpl)
    h, w = image.shape
    ht, wt = tmpl.shape
    xs = np.ascontiguousarray(xs, np.int32)
    ys = np.ascontiguousarray(ys, np.int32)
    n = xs.size
    if ys.size != n:
        raise ValueError("xs and ys differ in length")
    sums = np.zeros((3, n), np.uint32)
    c64 = np.zeros(n, np.float64)
    _check(load().oracle_ncc_u8_at(_ptr(image), w, h, _ptr(tmpl), wt, ht, n,
                                   _ptr(xs), _ptr(ys), _ptr(sums), _ptr(c64)))
    return sums, c64


def template_sums(tmpl):
    """(SumT, SumTSq) of a template."""
    tmpl = _u8(tmpl)
    out = np.zeros(2, np.uint32)
    _check(load().oracle_template_sums(_ptr(tmpl), tmpl.shape[1],
                                       tmpl.shape[0], _ptr(out)))
    return int(out[0]), int(out[1])


def xcorr_f32(left, right, nthreads=1):
    """Every pair and shift.  left [nl,H,W] (or [H,W]), right [nr,H,W].
    Returns (out, abs) as float64 [nl,nr,2H-1,2W-1]."""
    left, right = _f32(left, 3), _f32(right, 3)
    nl, H, W = left.shape
    nr = right.shape[0]
    if right.shape[1:] != (H, W):
        raise ValueError("left and right matrices differ in shape")
    out = np.zeros((nl, nr, 2 * H - 1, 2 * W - 1), np.float64)
    ab = np.zeros_like(out)
    _check(load().oracle_xcorr_f32(_ptr(left), nl, _ptr(right), nr, H, W,
                                   _ptr(out), _ptr(ab), int(nthreads)))
    return out, ab


def xcorr_f32_at(left, right, ls, rs, oys, oxs):
    """Outputs (pair ls[k]*nr+rs[k], row oys[k], column oxs[k]).
    Returns (out, abs) float64 [count]."""
    left, right = _f32(left, 3), _f32(right, 3)
    nl, H, W = left.shape
    nr = right.shape[0]
    arrs = [np.ascontiguousarray(a, np.int32) for a in (ls, rs, oys, oxs)]
    n = arrs[0].size
    if any(a.size != n for a in arrs):
        raise ValueError("index arrays differ in length")
    out = np.zeros(n, np.float64)
    ab = np.zeros(n, np.float64)
    _check(load().oracle_xcorr_f32_at(_ptr(left), nl, _ptr(right), nr, H, W, n,
                                      *[_ptr(a) for a in arrs], _ptr(out),
                                      _ptr(ab)))
    return out, ab
