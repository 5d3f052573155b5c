"""Timing of the stored layer applied to tokens: gptq_dequant_gemv (a few tokens, against
HBM bandwidth) and gptq_dequant_gemm (many tokens, against the bf16 tensor-core peak).

For each layer shape: random packed codes, scales and zeros (any bit pattern is a valid
code), CUDA events around each launch, the median over the repetitions.
  GEMV: a 256 MB L2 flush before every launch (queued behind a short spin so the host's
        call overhead is not timed); algorithmic bytes m*d*bits/8 (codes) + 8*m*G (scales,
        zeros) + 2*T*d (tokens) + 4*T*m (output).
  GEMM: 2*T*m*d flops (the products of X W_hat^T; the integer operand is formed once per
        call by a separate pass, timed apart); the tokens exceed L2 (T*d*2 bytes).

    python -m post_weight_quantization_gb300.bench_dequant [--reps 50] [--gemm-tokens 65536] [--layers N]

Prints one JSON line per case.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics

import torch

from post_weight_quantization_gb300 import gptq as g

SHAPES = [("llama 4096 x 4096", 4096, 4096), ("llama-7B gate/up 11008 x 4096", 11008, 4096),
          ("llama-7B down 4096 x 11008", 4096, 11008), ("70B gate/up 28672 x 8192", 28672, 8192),
          ("70B down 8192 x 28672", 8192, 28672)]


def peaks() -> tuple[float, float, str]:
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, 1900.0, "fallback"


def packed_layer(m, d, bits, gs, seed):
    dev = torch.device("cuda")
    G = 1 if gs == -1 else d // gs
    wpr = (d * bits + 31) // 32
    gen = torch.Generator(device=dev).manual_seed(seed)
    qweight = torch.randint(-2 ** 31, 2 ** 31 - 1, (m, wpr), dtype=torch.int32, device=dev, generator=gen)
    scales = torch.rand((m, G), device=dev, generator=gen) * 1e-2 + 1e-3
    zeros = torch.randint(0, 2 ** bits, (m, G), device=dev, generator=gen).float()
    return g.QuantizedLayer(qweight, scales, zeros, torch.empty(d, device=dev), bits, gs, d), gen


def time_gemv(m, d, bits, gs, T, reps, flush):
    q, gen = packed_layer(m, d, bits, gs, m + d + T)
    X = torch.randn((T, d), device="cuda", generator=gen).to(torch.bfloat16)
    Y = torch.empty((T, m), dtype=torch.float32, device="cuda")
    times = []
    for i in range(reps + 5):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)   # keeps the GPU busy until the launch below is queued
        e0.record()
        g.gptq_dequant_gemv(q, X, m, Y=Y)
        e1.record()
        torch.cuda.synchronize()
        if i >= 5:
            times.append(e0.elapsed_time(e1) * 1e3)
    g.gptq_device_check()
    G = 1 if gs == -1 else d // gs
    return statistics.median(times), m * d * bits / 8 + 8 * m * G + 2 * T * d + 4 * T * m


def time_gemm(m, d, bits, gs, T, reps, out_bf16):
    q, gen = packed_layer(m, d, bits, gs, m + d)
    X = torch.randn((T, d), device="cuda", generator=gen).to(torch.bfloat16)
    Y = torch.empty((T, m), dtype=torch.bfloat16 if out_bf16 else torch.float32, device="cuda")
    ws = torch.empty(g.gptq_workspace_size(g.GPTQ_WS_DEQUANT_GEMM, m, d), dtype=torch.uint8, device="cuda")
    times = []
    for i in range(reps + 3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.gptq_dequant_gemm(q, X, m, Y=Y, out_bf16=out_bf16, ws=ws)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e3)
    g.gptq_device_check()
    return statistics.median(times)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--bits", type=int, default=4)
    ap.add_argument("--group-size", type=int, default=128)
    ap.add_argument("--gemm-tokens", type=int, default=65536)
    ap.add_argument("--only", choices=["gemv", "gemm"], default=None)
    ap.add_argument("--layers", type=int, default=len(SHAPES), help="the first N layer shapes only")
    args = ap.parse_args()
    hbm, bf16, src = peaks()
    flush = torch.empty(256 << 18, dtype=torch.float32, device="cuda")
    for name, m, d in SHAPES[:args.layers]:
        if args.only != "gemm":
            for T in (1, 8):
                us, nbytes = time_gemv(m, d, args.bits, args.group_size, T, args.reps, flush)
                gbs = nbytes / us / 1e3
                span = d if args.group_size == -1 else args.group_size    # the library's choice of kernel
                tc = (os.environ.get("GPTQ_GEMV_KERNEL") != "fma"
                      and span % (4 * {2: 16, 3: 32, 4: 8, 8: 8}[args.bits]) == 0)
                print(json.dumps({"kernel": "gemv_mma_kernel" if tc else "dequant_gemv_kernel", "layer": name, "m": m, "d": d, "bits": args.bits,
                                  "group_size": args.group_size, "tokens": T, "us": round(us, 2),
                                  "bytes": int(nbytes), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3),
                                  "peak_GB/s": hbm, "peak_source": src, "l2": "256 MB flush before every launch"}),
                      flush=True)
        if args.only != "gemv":
            T = args.gemm_tokens
            us = time_gemm(m, d, args.bits, args.group_size, T, max(5, args.reps // 5), True)
            tf = 2.0 * T * m * d / us / 1e6
            print(json.dumps({"kernel": "dequant_gemm (int operand + dequant_gemm_kernel)", "layer": name, "m": m,
                              "d": d, "bits": args.bits, "group_size": args.group_size, "tokens": T,
                              "out": "bf16", "us": round(us, 1), "flops": 2.0 * T * m * d, "TFLOP/s": round(tf, 1),
                              "frac_bf16": round(tf / bf16, 3), "peak_TFLOP/s": bf16, "peak_source": src,
                              "l2": f"tokens {T * d * 2 / 1e9:.2f} GB, larger than L2"}), flush=True)


if __name__ == "__main__":
    main()
