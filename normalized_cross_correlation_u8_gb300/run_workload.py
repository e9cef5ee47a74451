"""Run named workloads through the library, for profiling.

    python -m normalized_cross_correlation_u8_gb300.run_workload NAME[,NAME...] [--reps N]

NAME is one of ncc_256, ncc_1080p, ncc_4k (u8 NCC) or xcorr_1to1,
xcorr_1tomany, xcorr_ntom (f32 cross-correlation); see workloads.py.  Each
workload's inputs are moved to cuda:0 and the device entry point is called
N times (default 2); nothing is checked or timed, so the launches can be
captured by a profiler in isolation.
"""
import argparse

import torch

from . import _binding as corr
from . import workloads as wl


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("names")
    p.add_argument("--reps", type=int, default=2)
    args = p.parse_args(argv)
    dev = torch.device("cuda", 0)
    for name in args.names.split(","):
        if name in wl.NCC_WORKLOADS:
            w = wl.NCC_WORKLOADS[name]()
            img = torch.from_numpy(w.image).to(dev)
            tm = torch.from_numpy(w.tmpl).to(dev)
            (h, ww), (ht, wt) = w.image.shape, w.tmpl.shape
            s = torch.empty((3, h - ht + 1, ww - wt + 1), dtype=torch.int32, device=dev)
            c = torch.empty((h - ht + 1, ww - wt + 1), dtype=torch.float32, device=dev)
            for _ in range(args.reps):
                corr.ncc_u8_into(img, tm, s, c)
        elif name in wl.XCORR_WORKLOADS:
            w = wl.XCORR_WORKLOADS[name]()
            L = torch.from_numpy(w.left).to(dev)
            R = torch.from_numpy(w.right).to(dev)
            nl, H, W = w.left.shape
            out = torch.empty((nl, w.right.shape[0], 2 * H - 1, 2 * W - 1),
                              dtype=torch.float32, device=dev)
            for _ in range(args.reps):
                corr.xcorr_f32_into(L, R, out)
        else:
            raise SystemExit(f"unknown workload {name!r}")
    torch.cuda.synchronize()
    print("ok")


if __name__ == "__main__":
    main()
