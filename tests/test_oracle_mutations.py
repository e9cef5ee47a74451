"""The pins must catch plausible slips in the oracle.

Each case plants one mistake in a copy of oracle/oracle.c (on the CPU, in a
temporary folder), loads that copy in place of the real oracle and runs the
pins of test_oracle_pins.py; at least one pin must fail.  Mistakes planted:
signed pixels, a mirrored template index (byte-order slip), a wrong
accumulated term, a dropped numerator term, a wrong variance term, an
off-by-one window, a wrong shift sign, swapped operands, a dropped absolute
value, and a shifted zero-shift index.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle.oracle as om
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(om.__file__), "oracle.c")

MUTATIONS = {
    "signed_pixel": ("uint32_t p = image[(size_t)(y + j) * w + (x + i)];",
                     "uint32_t p = (uint32_t)(int32_t)(int8_t)image[(size_t)(y + j) * w + (x + i)];"),
    "mirrored_template": ("uint32_t t = tmpl[(size_t)j * wt + i];\n            si += p;",
                          "uint32_t t = tmpl[(size_t)j * wt + (wt - 1 - i)];\n            si += p;"),
    "wrong_term": ("st += p * t;", "st += p * p;"),
    "dropped_numerator_term": ("int64_t num = (int64_t)n * sum_it - (int64_t)sum_i * sum_t;",
                               "int64_t num = (int64_t)n * sum_it;"),
    "wrong_variance": ("int64_t d_i = (int64_t)n * sum_i_sq - (int64_t)sum_i * sum_i;",
                       "int64_t d_i = (int64_t)n * sum_i_sq - (int64_t)sum_i * sum_t;"),
    "window_off_by_one": ("for (int j = 0; j < ht; j++)\n        for (int i = 0; i < wt; i++) {\n            uint32_t p",
                          "for (int j = 0; j < ht; j++)\n        for (int i = 1; i < wt; i++) {\n            uint32_t p"),
    "shift_sign": ("int xr = x - dx;", "int xr = x + dx;"),
    "swapped_operands": ("double p = (double)L[(size_t)y * W + x] * (double)R[(size_t)yr * W + xr];",
                         "double p = (double)R[(size_t)y * W + x] * (double)L[(size_t)yr * W + xr];"),
    "dropped_abs": ("a += fabs(p);", "a += p;"),
    "zero_shift_index": ("oy - (H - 1), ox - (W - 1), &a);", "oy - (H - 1), ox - W, &a);"),
}


def all_pins():
    """Every pin of test_oracle_pins.py, bound to small arguments."""
    yield from (lambda a=a: pins.test_u8_sums_match_library_valid_correlation(*a)
                for a in pins.U8_SHAPES[:5])
    yield pins.test_u8_sums_byte_order_single_hot_byte
    yield pins.test_u8_all_ones_template_and_patch_identities
    yield lambda: pins.test_u8_coef_matches_pearson_corrcoef(9, 13, 5, 8)
    yield pins.test_u8_coef_sign_flip_and_affine
    yield pins.test_u8_coef_exactly_one_at_patch
    yield from (lambda a=a: pins.test_xcorr_matches_scipy_full(*a)
                for a in pins.F32_SHAPES[3:6])
    yield pins.test_xcorr_delta_identities
    yield pins.test_xcorr_sum_flip_and_centre


def build_mutant(name, tmpdir):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} is not unique"
    path = os.path.join(tmpdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmpdir, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                    path, "-o", lib, "-lm"], check=True)
    return lib


def test_unmutated_oracle_passes_every_pin():
    for pin in all_pins():
        pin()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    with tempfile.TemporaryDirectory() as tmp:
        monkeypatch.setattr(om, "_lib", om.open_library(build_mutant(name, tmp)))
        caught = 0
        for pin in all_pins():
            try:
                pin()
            except (AssertionError, oracle.oracle.OracleError):
                caught += 1
        assert caught > 0, f"no pin caught the planted mistake {name!r}"
