"""Write the small text fixtures in this folder from the CPU oracle alone.

Run:  python tests/golden/make_golden.py
Each fixture holds seeded inputs and the oracle's outputs for them.  They pin
the oracle against later edits (a change to its arithmetic must come with a
regenerated fixture and a cited reason) and give the GPU tests tiny, fully
listed cases.  Nothing here calls the CUDA library.

ncc_u8_*.txt  -- sums SumI / SumISq / SumIT and the normalized coefficient
                 (The CUDA Handbook ch. 15, section 15.5).
xcorr_f32_*.txt -- full cross-correlation of every pair and shift
                 ("Efficient GPU-accelerated Parallel Cross-correlation"
                 artifact README, kernel overview).
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CITE_U8 = ("The CUDA Handbook ch. 15 'Image Processing: Normalized Correlation'"
           ", section 15.5 'Instruction-Level Parallelism and DP4A'")
CITE_F32 = ("'Efficient GPU-accelerated Parallel Cross-correlation' artifact "
            "README, kernel overview (one overlap per output, all shifts)")


def arr_lines(name, a, fmt):
    flat = " ".join(fmt % v for v in np.asarray(a).ravel())
    return [f"{name} {' '.join(str(s) for s in np.shape(a))}", flat]


def write_ncc(fname, seed, h, w, ht, wt):
    rng = np.random.default_rng(seed)
    image = rng.integers(0, 256, size=(h, w), dtype=np.uint8)
    tmpl = rng.integers(0, 256, size=(ht, wt), dtype=np.uint8)
    tmpl[0, 0] = 255          # asymmetric, bright corner
    tmpl[-1, -1] = 1
    sums, c64, _ = oracle.ncc_u8(image, tmpl)
    lines = [f"# {CITE_U8}", f"# seed {seed}; written by make_golden.py (oracle only)"]
    lines += arr_lines("image", image, "%d")
    lines += arr_lines("tmpl", tmpl, "%d")
    lines += arr_lines("sums", sums, "%d")
    lines += arr_lines("coef", c64, "%.17g")
    with open(os.path.join(HERE, fname), "w") as f:
        f.write("\n".join(lines) + "\n")


def write_xcorr(fname, seed, nl, nr, H, W):
    rng = np.random.default_rng(seed)
    left = rng.uniform(-1, 1, size=(nl, H, W)).astype(np.float32)
    right = rng.uniform(-1, 1, size=(nr, H, W)).astype(np.float32)
    out, ab = oracle.xcorr_f32(left, right)
    lines = [f"# {CITE_F32}", f"# seed {seed}; written by make_golden.py (oracle only)"]
    lines += arr_lines("left", left, "%.9g")
    lines += arr_lines("right", right, "%.9g")
    lines += arr_lines("out", out, "%.17g")
    lines += arr_lines("abs", ab, "%.17g")
    with open(os.path.join(HERE, fname), "w") as f:
        f.write("\n".join(lines) + "\n")


def read_fixture(path):
    """Parse a fixture into {name: ndarray} (ints stay int64)."""
    out = {}
    with open(path) as f:
        rows = [r.rstrip("\n") for r in f if not r.startswith("#")]
    for head, body in zip(rows[0::2], rows[1::2]):
        name, *shape = head.split()
        shape = tuple(int(s) for s in shape)
        vals = body.split()
        if any(("." in v or "e" in v) for v in vals):
            a = np.array([float(v) for v in vals], np.float64)
        else:
            a = np.array([int(v) for v in vals], np.int64)
        out[name] = a.reshape(shape)
    return out


if __name__ == "__main__":
    write_ncc("ncc_u8_13x10_t8x3.txt", 31, 10, 13, 3, 8)
    write_ncc("ncc_u8_40x21_t12x5.txt", 32, 21, 40, 5, 12)
    write_xcorr("xcorr_f32_2x3_5x7.txt", 33, 2, 3, 5, 7)
    print("written")
