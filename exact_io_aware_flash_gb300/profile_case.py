"""Run the attention kernels on one shape a few times, for profiler captures.

    python -m exact_io_aware_flash_gb300.profile_case --B 2 --H 16 --N 4096 --d 128 --iters 3

Runs `iters` forward + backward calls (causal, bf16 unless --fp16) on seeded
inputs; prints nothing but a completion line.  Used as the target command of
`ncu` captures, which must run on a case small enough to replay quickly.
"""
import argparse
import math

import torch

from . import (backward, build, check_errors, forward, forward_fp8, forward_splitkv,
               quantize_fp8)
from .synth import Shape, make_inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=16)
    ap.add_argument("--Hkv", type=int, default=0)
    ap.add_argument("--N", type=int, default=4096)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--fp16", action="store_true")
    ap.add_argument("--noncausal", action="store_true")
    ap.add_argument("--forward-only", action="store_true")
    ap.add_argument("--atomic", action="store_true",
                    help="backward through fa_backward_atomic (one pass, dQ by atomic adds)")
    ap.add_argument("--fp8", action="store_true", help="e4m3 quantization + forward instead")
    ap.add_argument("--decode", type=int, default=0, metavar="NK",
                    help="split-KV decoding instead: one query row per head against NK keys")
    a = ap.parse_args()
    build.build()
    shape = Shape(a.B, a.H, a.Hkv or a.H, a.N, a.d)
    if a.decode:
        g = torch.Generator(device="cpu").manual_seed(77)
        q = torch.randn(a.B, a.H, 1, a.d, generator=g).to(torch.bfloat16).cuda()
        k, v = (torch.randn(a.B, a.Hkv or a.H, a.decode, a.d, generator=g).to(torch.bfloat16).cuda()
                for _ in range(2))
        for _ in range(a.iters):
            forward_splitkv(q, k, v)
        torch.cuda.synchronize()
        check_errors()
        print(f"profile_case done: decode B{a.B} H{a.H} Nk{a.decode} iters={a.iters}")
        return
    if a.fp8:
        inp = make_inputs(shape, "bf16", seed=77, with_dO=False)
        q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
        signs = torch.ones(a.d, dtype=torch.int8, device="cuda")
        for _ in range(a.iters):
            codes = quantize_fp8(q, k, v, signs)
            forward_fp8(codes, causal=not a.noncausal)
        torch.cuda.synchronize()
        check_errors()
        print(f"profile_case done: fp8 {shape} iters={a.iters}")
        return
    inp = make_inputs(shape, "fp16" if a.fp16 else "bf16", seed=77)
    q, k, v, dO = (inp[n].cuda() for n in ("q", "k", "v", "dO"))
    causal = not a.noncausal
    scale = 1.0 / math.sqrt(a.d)
    for _ in range(a.iters):
        o, lse = forward(q, k, v, causal=causal, scale=scale)
        if not a.forward_only:
            backward(q, k, v, o, lse, dO, causal=causal, scale=scale, deterministic=not a.atomic)
    torch.cuda.synchronize()
    check_errors()
    print(f"profile_case done: {shape} causal={causal} iters={a.iters}")


if __name__ == "__main__":
    main()
