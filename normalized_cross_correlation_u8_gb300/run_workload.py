"""Run named workloads through the library, for profiling.

    python -m normalized_cross_correlation_u8_gb300.run_workload NAME[,NAME...] [--reps N]
        [--method box|dp4a]

NAME is one of ncc_256, ncc_1080p, ncc_4k (u8 NCC) or xcorr_1to1,
xcorr_1tomany, xcorr_ntom (f32 cross-correlation); see workloads.py; or
ncc:WxHxWTxHT for a u8 image of W x H with a WT x HT template (seeded
uniform bytes); or xcorr:NLxNRxHxW for an f32 batch of that shape with
seeded uniform [-1, 1) inputs.  --method selects the u8 method.  Each workload's inputs are moved to cuda:0 and the device entry
point is called N times (default 2); nothing is checked or timed, so the
launches can be captured by a profiler in isolation.
"""
import argparse

import numpy as np
import torch

from . import _binding as corr
from . import workloads as wl


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("names")
    p.add_argument("--reps", type=int, default=2)
    p.add_argument("--method", choices=["box", "dp4a"], default=None)
    args = p.parse_args(argv)
    dev = torch.device("cuda", 0)
    for name in args.names.split(","):
        if name in wl.NCC_WORKLOADS or name.startswith("ncc:"):
            if name.startswith("ncc:"):
                ww, h, wt, ht = (int(v) for v in name[len("ncc:"):].split("x"))
                rng = np.random.default_rng(4242)
                image = rng.integers(0, 256, size=(h, ww), dtype=np.uint8)
                tmpl = rng.integers(0, 256, size=(ht, wt), dtype=np.uint8)
            else:
                w = wl.NCC_WORKLOADS[name]()
                image, tmpl = w.image, w.tmpl
            img = torch.from_numpy(image).to(dev)
            tm = torch.from_numpy(tmpl).to(dev)
            (h, ww), (ht, wt) = image.shape, tmpl.shape
            s = torch.empty((3, h - ht + 1, ww - wt + 1), dtype=torch.int32, device=dev)
            c = torch.empty((h - ht + 1, ww - wt + 1), dtype=torch.float32, device=dev)
            for _ in range(args.reps):
                corr.ncc_u8_into(img, tm, s, c, method=args.method)
        elif name in wl.XCORR_WORKLOADS or name.startswith("xcorr:"):
            if name.startswith("xcorr:"):
                nl, nr, H, W = (int(v) for v in name[len("xcorr:"):].split("x"))
                rng = np.random.default_rng(4242)
                left = rng.uniform(-1, 1, size=(nl, H, W)).astype(np.float32)
                right = rng.uniform(-1, 1, size=(nr, H, W)).astype(np.float32)
            else:
                w = wl.XCORR_WORKLOADS[name]()
                left, right = w.left, w.right
            L = torch.from_numpy(left).to(dev)
            R = torch.from_numpy(right).to(dev)
            nl, H, W = left.shape
            out = torch.empty((nl, right.shape[0], 2 * H - 1, 2 * W - 1),
                              dtype=torch.float32, device=dev)
            for _ in range(args.reps):
                corr.xcorr_f32_into(L, R, out)
        else:
            raise SystemExit(f"unknown workload {name!r}")
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
