"""Launch a few GEMV calls on one shape, for profilers (ncu) to capture.

    python -m nvfp4_weight_quantized_gemv_gb300.profile_case --shape attn_qkv --ns 1,4 --reps 2
    python -m nvfp4_weight_quantized_gemv_gb300.profile_case --shape attn_qkv --quantize bf16 --reps 2

With --quantize, the device quantizer runs --reps times on seeded bf16 (or
fp32) weights of the shape instead of the GEMV.

Allocates one weight matrix of the shape (seeded synthetic data, quantized by
the library's host quantizer), then for each n in --ns runs --reps calls,
synchronizing after each.  Prints one line per n with the mean CUDA-event time
of the calls (cold-ish: every call after the first reuses L2-resident weights
unless the shape exceeds L2 -- use bench.py for throughput numbers).
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import nvfp4_weight_quantized_gemv_gb300 as nv  # noqa: E402
import synth  # noqa: E402

SHAPES = {"tiny": (256, 512), "attn_qkv": (14336, 5120), "o_proj": (5120, 6144), "fused_qkv": (16384, 5120)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--shape", default="attn_qkv", choices=list(SHAPES))
    ap.add_argument("--ns", default="1,4")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--variant", default="auto", choices=["auto", "tc", "mma", "simt", "generic"])
    ap.add_argument("--tiling", default="one_pass", choices=["one_pass", "greedy_321"])
    ap.add_argument("--quantize", default=None, choices=["bf16", "fp32"])
    args = ap.parse_args()
    nv.build()
    N, K = SHAPES[args.shape]
    if args.quantize:
        w32 = synth.weights_f32(N, K, 100)
        if args.quantize == "bf16":
            w = torch.from_numpy(synth.to_bf16_bits(w32).view(np.int16)).cuda().view(torch.bfloat16)
        else:
            w = torch.from_numpy(w32).cuda()
        times = []
        for _ in range(args.reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            nv.nvfp4_quantize(w)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
        print(f"quantize {args.quantize} N={N} K={K}: {np.mean(times):.2f} us/call (mean of {args.reps})")
        if nv.nvfp4_device_error() != 0:
            raise SystemExit("device error")
        return
    packed, scale, g = nv.nvfp4_quantize_ref(synth.weights_f32(N, K, 100))
    wp = torch.from_numpy(packed).cuda()
    ws = torch.from_numpy(scale).cuda()
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    variant = {"auto": 0, "mma": 1, "simt": 2, "generic": 3, "tc": 4}[args.variant]
    tiling = nv.TILING_ONE_PASS if args.tiling == "one_pass" else nv.TILING_GREEDY_321
    for n in [int(v) for v in args.ns.split(",")]:
        x = torch.from_numpy(synth.activations_bf16(n, K, 1).view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
        times = []
        for _ in range(args.reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            nv.nvfp4_gemv_batched_ex(wp, ws, gs, x, y, variant=variant, tiling=tiling)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
        print(f"{args.shape} N={N} K={K} n={n}: {np.mean(times):.2f} us/call (mean of {args.reps})")
    if nv.nvfp4_device_error() != 0:
        raise SystemExit("device error")


if __name__ == "__main__":
    main()
