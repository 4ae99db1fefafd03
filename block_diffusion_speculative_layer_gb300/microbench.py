"""Kernel microbenchmarks through the C ABI (device time from CUDA events).

  python -m block_diffusion_speculative_layer_gb300.microbench gemm --M 16 --N 24576 --K 4096 --iters 20
  python -m block_diffusion_speculative_layer_gb300.microbench lmhead --M 16 --N 151936 --K 4096

Inputs are seeded synthetic bf16 (N(0,1) activations, N(0,0.02) weights)
drawn on the GPU by torch.  For small shapes several weight copies are used
in turn so that launches never hit in L2.  The GEMM loop runs inside the
library (df_op_bench_gemm_bf16): no host work between launches.
"""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import block_diffusion_speculative_layer_gb300 as dfl
    from block_diffusion_speculative_layer_gb300 import build

    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["gemm", "lmhead"])
    ap.add_argument("--M", type=int, default=16)
    ap.add_argument("--N", type=int, default=24576)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--token-tile", type=int, default=0)
    a = ap.parse_args()
    build.build()
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(a.M, a.K, device="cuda", generator=g).to(torch.bfloat16)
    nw = max(1, min(4, int(512e6 // (a.N * a.K * 2)) + 1))
    ws = [(torch.randn(a.N, a.K, device="cuda", generator=g) * 0.02).to(torch.bfloat16) for _ in range(nw)]

    if a.op == "gemm":
        for i in range(a.warmup):
            dfl.bench_gemm_bf16(x, ws[i % nw], iters=1, splits=a.splits, token_tile=a.token_tile)
        us = sum(dfl.bench_gemm_bf16(x, ws[i % nw], iters=a.iters, splits=a.splits, token_tile=a.token_tile)
                 for i in range(nw)) / nw
        out_b = 4 * a.M * a.N
    else:
        for i in range(a.warmup):
            dfl.lmhead_argmax_bf16(x, ws[i % nw])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(a.iters):
            dfl.lmhead_argmax_bf16(x, ws[i % nw])
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000.0 / a.iters
        out_b = 8 * a.M
    algo = 2 * a.N * a.K + 2 * a.M * a.K + out_b
    print(json.dumps({"op": a.op, "M": a.M, "N": a.N, "K": a.K, "splits": a.splits, "token_tile": a.token_tile,
                      "us_per_launch": us, "algorithmic_bytes": algo, "GB/s": algo / (us * 1e-6) / 1e9}))


if __name__ == "__main__":
    main()
