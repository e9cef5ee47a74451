"""The C-ABI library builds, loads and exports every declared entry point;
argument errors come back as codes before anything reaches the GPU (these
tests make no compute call and need no GPU)."""
import ctypes
import os
import re

import pytest

import normalized_cross_correlation_u8_gb300 as corr
from normalized_cross_correlation_u8_gb300 import _binding

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
FAKE = ctypes.c_void_p(0x100000)    # never dereferenced: every call below fails validation


def declared_functions():
    names = set()
    for fn in sorted(os.listdir(INCLUDE)):
        if fn.endswith(".h"):
            src = open(os.path.join(INCLUDE, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(corr_\w+)\s*\(", src))
    return sorted(names)


def test_headers_declare_functions():
    names = declared_functions()
    assert "corr_ncc_u8" in names and "corr_xcorr_f32" in names
    assert set(names) == set(_binding.EXPORTS), "binding and headers disagree"


@pytest.mark.parametrize("name", declared_functions())
def test_library_exports_declared_symbol(name):
    lib = corr.load()
    assert hasattr(lib, name), f"libcorr.so does not export {name}"


def test_version_and_strerror():
    lib = corr.load()
    assert lib.corr_version() >= 100
    for code in (0, -1, -2, -3):
        assert lib.corr_strerror(code)
    assert lib.corr_strerror(-99) == b"unknown error code"
    assert lib.corr_last_cuda_error() == 0


def test_stream_is_thread_local_setting():
    lib = corr.load()
    lib.corr_set_stream(ctypes.c_void_p(0x1234))
    assert lib.corr_get_stream() == 0x1234
    lib.corr_set_stream(None)
    assert lib.corr_get_stream() is None


def test_ncc_method_setting():
    lib = corr.load()
    assert lib.corr_ncc_get_method() == 1                  # box by default
    assert lib.corr_ncc_set_method(0) == 0
    assert lib.corr_ncc_get_method() == 0
    assert lib.corr_ncc_set_method(2) == -1                # unknown: unchanged
    assert lib.corr_ncc_get_method() == 0
    assert lib.corr_ncc_set_method(1) == 0


@pytest.mark.parametrize("args,code", [
    ((None, 16, 16, FAKE, 4, 4, FAKE, FAKE), -1),            # null image
    ((FAKE, 16, 16, None, 4, 4, FAKE, FAKE), -1),            # null template
    ((FAKE, 16, 16, FAKE, 4, 4, None, None), -1),            # no output at all
    ((FAKE, 0, 16, FAKE, 4, 4, FAKE, FAKE), -1),             # empty image
    ((FAKE, 16, 16, FAKE, 20, 4, FAKE, FAKE), -1),           # template wider
    ((FAKE, 16, 16, FAKE, 4, 17, FAKE, FAKE), -1),           # template taller
    ((FAKE, 16, 16, FAKE, 0, 4, FAKE, FAKE), -1),            # empty template
    ((FAKE, 300, 300, FAKE, 257, 258, FAKE, FAKE), -2),      # odd width, > 66051 pixels
    ((FAKE, 1000, 1000, FAKE, 260, 260, FAKE, FAKE), -2),    # > 66051 pixels
    ((FAKE, 16513, 300, FAKE, 16513, 4, FAKE, FAKE), -2),    # 66052 pixels: SumISq may wrap
    ((FAKE, 369, 300, FAKE, 369, 179, FAKE, FAKE), -1),      # 66051 pixels: accepted; fake buffer
    ((FAKE, 4, 60000, FAKE, 1, 58001, FAKE, FAKE), -2),      # 58001 template words
    ((FAKE, 4, 60000, FAKE, 1, 58000, FAKE, FAKE), -1),      # 58000 words: accepted; fake buffer
    ((FAKE, 16, 16, FAKE, -4, 4, FAKE, FAKE), -1),
])
def test_ncc_argument_errors(args, code):
    assert corr.load().corr_ncc_u8(*args) == code


@pytest.mark.parametrize("args,code", [
    ((FAKE, 16, 16, 15, FAKE, 4, 4, FAKE, FAKE), -1),        # pitch < w
    ((FAKE, 16, 16, 0, FAKE, 4, 4, FAKE, FAKE), -1),
    ((None, 16, 16, 32, FAKE, 4, 4, FAKE, FAKE), -1),        # null image
    ((FAKE, 16, 16, 32, FAKE, 20, 4, FAKE, FAKE), -1),       # template wider
    ((FAKE, 300, 300, 512, FAKE, 257, 258, FAKE, FAKE), -2), # > 66051 pixels
])
def test_ncc_pitched_argument_errors(args, code):
    assert corr.load().corr_ncc_u8_pitched(*args) == code


@pytest.mark.parametrize("args,code", [
    ((None, 1, FAKE, 1, 4, 4, FAKE), -1),
    ((FAKE, 1, FAKE, 1, 4, 4, None), -1),
    ((FAKE, 0, FAKE, 1, 4, 4, FAKE), -1),
    ((FAKE, 1, FAKE, 1, 0, 4, FAKE), -1),
    ((ctypes.c_void_p(0x100002), 1, FAKE, 1, 4, 4, FAKE), -1),   # misaligned float*
    ((FAKE, 70000, FAKE, 70000, 4, 4, FAKE), -2),               # pair count > int
])
def test_xcorr_argument_errors(args, code):
    assert corr.load().corr_xcorr_f32(*args) == code


def test_no_gpu_means_loud_failure():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(RuntimeError):
        corr.ncc_u8(torch.zeros(8, 8, dtype=torch.uint8), torch.zeros(4, 4, dtype=torch.uint8))


def test_xcorr_kernel_choice(monkeypatch):
    """Host-side dispatch (no launch, no GPU needed): the named batches take
    the kernels measured fastest for them, and the environment switches
    force or forbid the tensor-core and warp-per-overlap kernels."""
    for v in ("CORR_XCORR_TC", "CORR_XCORR_TCL", "CORR_XCORR_WARP"):
        monkeypatch.delenv(v, raising=False)
    k = corr.xcorr_f32_kernel
    assert k(32, 64, 16, 16) == "tensor"       # n-to-m of 16x16
    assert k(1, 1, 256, 256) == "tensor_large" # one-to-one
    assert k(1, 128, 64, 64) == "tensor_large" # one-to-many
    assert k(1, 1, 128, 128) == "rows"         # below the larger-matrix rule
    assert k(1, 128, 32, 32) == "bcast"
    assert k(1, 1, 1024, 1024) == "tensor_large"   # 32 row units per item: 512 MB
    assert k(1, 1, 2048, 2048) == "rows_win"   # partial sums would pass 512 MB
    assert k(2, 96, 48, 48) == "tensor_large"  # 1.0e9 products
    assert k(1, 64, 48, 48) == "bcast"         # below the larger-matrix rule
    assert k(1, 1, 1, 4096) == "warp"          # a single long row
    assert k(16, 16, 16, 16) == "tensor"       # 256 pairs of 16x16
    assert k(8, 8, 12, 12) == "tensor"         # 64 pairs of 12x12
    assert k(64, 64, 10, 10) == "tiny"         # H*W < 144
    assert k(32, 64, 8, 8) == "tiny"
    assert k(4, 8, 16, 16) == "rows"           # fewer than 64 pairs
    monkeypatch.setenv("CORR_XCORR_TC", "0")
    assert k(32, 64, 16, 16) == "tiny"
    monkeypatch.setenv("CORR_XCORR_TC", "1")
    assert k(2, 2, 3, 5) == "tensor"
    assert k(1, 1, 17, 16) != "tensor"         # beyond 16 x 16
    monkeypatch.setenv("CORR_XCORR_TCL", "0")
    assert k(1, 1, 256, 256) == "rows"
    monkeypatch.setenv("CORR_XCORR_WARP", "1")
    assert k(1, 1, 40, 64) == "warp"
    with pytest.raises(corr.CorrError):
        k(0, 1, 4, 4)
