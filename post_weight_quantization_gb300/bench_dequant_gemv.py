"""Timing of gptq_dequant_gemv (Y = X W_hat^T from the packed layer) against HBM bandwidth.

For each layer shape and token count: random packed codes, scales and zeros (any bit
pattern is a valid code), a 256 MB L2 flush before every launch, CUDA events around
each launch (queued behind a short spin so the host's call overhead is not timed), the
median over the repetitions. Bytes are the algorithmic ones: codes
m*d*bits/8, scales and zeros 8*m*G, tokens 2*T*d, output 4*T*m.

    python -m post_weight_quantization_gb300.bench_dequant_gemv [--reps 50]

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


def peak_hbm() -> tuple[float, str]:
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


def run_case(name, m, d, bits, gs, T, reps, flush):
    dev = torch.device("cuda")
    G = 1 if gs == -1 else d // gs
    wpr = (d * bits + 31) // 32
    gen = torch.Generator(device=dev).manual_seed(m + d + T)
    qweight = torch.randint(-2 ** 31, 2 ** 31 - 1, (m, wpr), dtype=torch.int32, device=dev, generator=gen)
    scales = torch.rand((m, G), device=dev, generator=gen) * 1e-2 + 1e-3
    zeros = torch.randint(0, 2 ** bits, (m, G), device=dev, generator=gen).float()
    q = g.QuantizedLayer(qweight, scales, zeros, torch.empty(d, device=dev), bits, gs, d)
    X = (torch.randn((T, d), device=dev, generator=gen)).to(torch.bfloat16)
    Y = torch.empty((T, m), dtype=torch.float32, device=dev)
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
    us = statistics.median(times)
    nbytes = m * d * bits / 8 + 8 * m * G + 2 * T * d + 4 * T * m
    return us, nbytes


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--bits", type=int, default=4)
    ap.add_argument("--group-size", type=int, default=128)
    args = ap.parse_args()
    peak, src = peak_hbm()
    flush = torch.empty(256 << 18, dtype=torch.float32, device="cuda")
    for name, m, d in SHAPES:
        for T in (1, 8):
            us, nbytes = run_case(name, m, d, args.bits, args.group_size, T, args.reps, flush)
            gbs = nbytes / us / 1e3
            print(json.dumps({"kernel": "dequant_gemv_kernel", "layer": name, "m": m, "d": d, "bits": args.bits,
                              "group_size": args.group_size, "tokens": T, "us": round(us, 2),
                              "bytes": int(nbytes), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak, 3),
                              "peak_GB/s": peak, "peak_source": src, "l2": "256 MB flush before every launch"}))


if __name__ == "__main__":
    main()
