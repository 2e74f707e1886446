"""Run one addmm or conv2d of a chosen shape through the C ABI (for profiling).

    python -m addmm_implicit_im2col_gb300.run_case addmm M N K [--self2d] [--mode default]
    python -m addmm_implicit_im2col_gb300.run_case conv B IC H W OC KH KW stride pad dilation

Inputs are seeded synthetic draws created on the host and copied to the GPU
once; the operation is then launched ``--reps`` times and the CUDA-event time
of each launch is printed.
"""
from __future__ import annotations

import argparse
import sys

import numpy as np


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["addmm", "conv"])
    ap.add_argument("dims", type=int, nargs="+")
    ap.add_argument("--mode", default="default")
    ap.add_argument("--self2d", action="store_true")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)

    import torch

    from . import binding, build, synth
    build.build()
    binding.load()
    dev = torch.device("cuda:0")
    if args.op == "addmm":
        M, N, K = args.dims
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=args.self2d, workload=900,
                                     mat1=("N", 0.0, 1.0), mat2=("N", 0.0, 1.0 / np.sqrt(K)),
                                     self_=("N", 0.0, 1.0))
        S, A, B = (torch.from_numpy(t).to(dev) for t in (s, a, b))
        out = torch.empty((M, N), dtype=torch.float32, device=dev)
        flops = 2.0 * M * N * K

        def fn():
            binding.addmm(S, A, B, mode=args.mode, out=out)
    else:
        B_, IC, H, W, OC, KH, KW, st, pd, dl = args.dims
        x, w, bias = synth.conv_inputs(B_, IC, H, W, OC, KH, KW, workload=901,
                                       x=("N", 0.0, 1.0), w=("N", 0.0, 1.0 / np.sqrt(IC * KH * KW)))
        X, Wt, Bb = (torch.from_numpy(t).to(dev) for t in (x, w, bias))
        OH = binding.conv_out_size(H, KH, st, pd, dl)
        OW = binding.conv_out_size(W, KW, st, pd, dl)
        out = torch.empty((B_, OC, OH, OW), dtype=torch.float32, device=dev)
        flops = 2.0 * OC * B_ * OH * OW * IC * KH * KW

        def fn():
            binding.conv2d(X, Wt, Bb, st, pd, dl, mode=args.mode, out=out)
    for _ in range(args.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        print(f"{args.op} {args.dims} {args.mode} kernel={binding.last_kernel()} "
              f"{ms * 1e3:.1f} us {flops / ms / 1e9:.1f} TFLOP/s", flush=True)
    rc = binding.check_device_error(None)
    if rc != 0:
        print(f"device error: {binding.status_string(rc)}")
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
