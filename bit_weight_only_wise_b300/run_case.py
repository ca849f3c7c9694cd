"""Run one W4A16 / NF4 product of a given shape a few times (for profilers).

    python -m bit_weight_only_wise_b300.run_case --K 5120 --N 55296 --M 1 --dtype bf16 --reps 4

Weights are N(0, 0.02) drawn on the GPU with a seeded torch generator and
quantized by the library (round-to-nearest INT4 g128, or NF4 with --nf4);
activations are N(0, 1).  Prints a checksum of the last output.
"""

from __future__ import annotations

import argparse

import torch

import bit_weight_only_wise_b300 as w4


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--K", type=int, required=True)
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--M", type=int, required=True)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16"])
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--nf4", action="store_true")
    ap.add_argument("--act-order", action="store_true")
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float16
    W = torch.randn(a.K, a.N, device=dev, generator=g) * 0.02
    X = torch.randn(a.M, a.K, device=dev, generator=g).to(dt)
    if a.nf4:
        cb = w4.nf4_codebook(dev)
        qw, am = w4.nf4_quantize(W, cb)
        del W
        run = lambda: w4.nf4_gemm(X, qw, am, cb)  # noqa: E731
    else:
        qw, sc, qz = w4.quantize(W)
        del W
        gi = None
        if a.act_order:
            perm = torch.randperm(a.K, device=dev, generator=g)
            gi = torch.empty(a.K, dtype=torch.int32, device=dev)
            gi[perm] = (torch.arange(a.K, device=dev) // 128).to(torch.int32)
        run = lambda: w4.gemm(X, qw, sc, qz, g_idx=gi)  # noqa: E731
    for _ in range(a.reps):
        Y = run()
    torch.cuda.synchronize()
    print(f"ok K={a.K} N={a.N} M={a.M} {a.dtype} checksum={Y.float().abs().mean().item():.6f}")


if __name__ == "__main__":
    main()
