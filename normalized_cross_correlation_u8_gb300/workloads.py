"""Seeded synthetic inputs for the correlation path.

This module only draws input arrays.  It holds none of the correlation
arithmetic, imports neither the CUDA binding nor the oracle, and is the one
piece of code both sides share (tests feed the same arrays to the GPU path and
to the CPU oracle).

The pages measure on no public dataset: the handbook's sample images and the
cross-correlation artifact's benchmark inputs are not reproduced.  Each named
workload below stands in for them with the sizes, value ranges and structure
stated for it (seed = 1000 + workload number; the large u8 image of the fifth
workload uses 1050).
"""
from dataclasses import dataclass, field

import numpy as np


@dataclass
class NccWorkload:
    name: str
    image: np.ndarray            # [h, w] uint8, row-major
    tmpl: np.ndarray             # [ht, wt] uint8
    offset: tuple                # (x, y) the template was copied from
    notes: dict = field(default_factory=dict)

    @property
    def offsets(self):
        h, w = self.image.shape
        ht, wt = self.tmpl.shape
        return (w - wt + 1) * (h - ht + 1)


@dataclass
class XcorrWorkload:
    name: str
    left: np.ndarray             # [nl, H, W] float32
    right: np.ndarray            # [nr, H, W] float32
    notes: dict = field(default_factory=dict)

    @property
    def pairs(self):
        return self.left.shape[0] * self.right.shape[0]

    @property
    def flops(self):
        """2 * (multiply-adds of all true overlaps) = 2 * pairs * (H*W)^2."""
        _, H, W = self.left.shape
        return 2 * self.pairs * (H * W) ** 2


def uniform_u8(rng, h, w):
    """i.i.d. uniform pixels over the whole byte range [0, 255]."""
    return rng.integers(0, 256, size=(h, w), dtype=np.uint8)


def patch(image, x, y, wt, ht):
    return np.ascontiguousarray(image[y:y + ht, x:x + wt])


def gaussian_blur(field_, sigma=3.0, radius=12):
    """Separable Gaussian blur with reflected edges (input synthesis only)."""
    k = np.arange(-radius, radius + 1, dtype=np.float64)
    g = np.exp(-k * k / (2.0 * sigma * sigma))
    g /= g.sum()
    h, w = field_.shape
    p = np.pad(field_, ((0, 0), (radius, radius)), mode="reflect")
    tmp = np.zeros((h, w), np.float64)
    for t in range(2 * radius + 1):
        tmp += g[t] * p[:, t:t + w]
    p = np.pad(tmp, ((radius, radius), (0, 0)), mode="reflect")
    out = np.zeros((h, w), np.float64)
    for t in range(2 * radius + 1):
        out += g[t] * p[t:t + h, :]
    return out


def smooth_u8(rng, h, w, frac_bright=0.30, sigma=3.0, radius=12):
    """Blurred uniform noise mapped to bytes so that about frac_bright of the
    pixels exceed 127 (40 grey levels per standard deviation)."""
    f = gaussian_blur(rng.random((h, w)), sigma, radius)
    z = (f - f.mean()) / f.std()
    q = np.quantile(z, 1.0 - frac_bright)
    return np.clip(np.rint(127.5 + 40.0 * (z - q)), 0, 255).astype(np.uint8)


def ncc_patch_workload(name, seed, w, h, wt, ht):
    """Uniform image; template copied from a seeded valid offset."""
    rng = np.random.default_rng(seed)
    image = uniform_u8(rng, h, w)
    ox = int(rng.integers(0, w - wt + 1))
    oy = int(rng.integers(0, h - ht + 1))
    return NccWorkload(name, image, patch(image, ox, oy, wt, ht), (ox, oy),
                       {"seed": seed, "image": "uniform [0,255]",
                        "template": "exact patch"})


def ncc_smooth_workload(name, seed, w, h, wt, ht, noise=8):
    """Smooth image (30 % of pixels > 127); template = patch + uniform noise
    in [-noise, noise], clamped to [0, 255]."""
    rng = np.random.default_rng(seed)
    image = smooth_u8(rng, h, w)
    ox = int(rng.integers(0, w - wt + 1))
    oy = int(rng.integers(0, h - ht + 1))
    t = patch(image, ox, oy, wt, ht).astype(np.int32)
    t += rng.integers(-noise, noise + 1, size=t.shape, dtype=np.int32)
    tmpl = np.clip(t, 0, 255).astype(np.uint8)
    return NccWorkload(name, image, tmpl, (ox, oy),
                       {"seed": seed, "image": "blurred uniform, sigma 3",
                        "template": f"patch + U[-{noise},{noise}]",
                        "frac_gt_127": float((image > 127).mean())})


def xcorr_workload(name, seed, nl, nr, H, W, dist):
    rng = np.random.default_rng(seed)
    if dist == "uniform":
        left = rng.uniform(-1.0, 1.0, size=(nl, H, W)).astype(np.float32)
        right = rng.uniform(-1.0, 1.0, size=(nr, H, W)).astype(np.float32)
    elif dist == "normal":
        left = rng.standard_normal(size=(nl, H, W)).astype(np.float32)
        right = rng.standard_normal(size=(nr, H, W)).astype(np.float32)
    else:
        raise ValueError(dist)
    return XcorrWorkload(name, left, right, {"seed": seed, "dist": dist})


# --- the named workloads ---------------------------------------------------

def ncc_256():
    """256x256 uniform image, 16x16 exact-patch template (58 081 offsets)."""
    return ncc_patch_workload("ncc_u8_256x256_t16", 1001, 256, 256, 16, 16)


def ncc_1080p():
    """1920x1080 smooth image, 32x32 noisy-patch template (1 981 561 offsets)."""
    return ncc_smooth_workload("ncc_u8_1920x1080_t32", 1002, 1920, 1080, 32, 32)


def ncc_4k():
    """4096x4096 uniform image, 64x64 exact-patch template (16 265 089 offsets)."""
    return ncc_patch_workload("ncc_u8_4096x4096_t64", 1050, 4096, 4096, 64, 64)


def xcorr_one_to_one():
    """One 256x256 pair, uniform [-1, 1]: 511x511 overlaps."""
    return xcorr_workload("xcorr_f32_1to1_256", 1003, 1, 1, 256, 256, "uniform")


def xcorr_one_to_many():
    """One 64x64 left against 128 rights, N(0, 1): 128 x 127x127 overlaps."""
    return xcorr_workload("xcorr_f32_1to128_64", 1004, 1, 128, 64, 64, "normal")


def xcorr_n_to_m():
    """32 lefts x 64 rights of 16x16, uniform [-1, 1]: 2048 x 31x31 overlaps."""
    return xcorr_workload("xcorr_f32_32x64_16", 1005, 32, 64, 16, 16, "uniform")


NCC_WORKLOADS = {"ncc_256": ncc_256, "ncc_1080p": ncc_1080p, "ncc_4k": ncc_4k}
XCORR_WORKLOADS = {"xcorr_1to1": xcorr_one_to_one,
                   "xcorr_1tomany": xcorr_one_to_many,
                   "xcorr_ntom": xcorr_n_to_m}
