"""Benchmark of the GPTQ per-layer path on GB300.

One step = the whole path for one layer: the Hessian over all calibration tokens
(one bf16 SYRK), damping + Hinv1, and the blocked column loop with packed codes.
Default workload: the Llama-style 4096 x 4096 projection, 4-bit, group 128, with
262144 calibration tokens (128 sequences x 2048), synthetic seeded data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gptq|reference]

Prints one JSON line. The path runs on one GPU: with N > 1 (--gpus or a torchrun
launch) rank 0 prints a line that says so and every rank exits before touching CUDA.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import threading
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GPTQ ms/layer + Mweights/s, 4096² 4-bit g128; SYRK TFLOP/s; % roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------------
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gptq", "reference"], default="gptq")
    ap.add_argument("--workload", default="llama_4096_g128")
    ap.add_argument("--layer", type=int, default=0, help="layer index within the workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--threads", type=int, default=None, help="host threads for input generation")
    ap.add_argument("--tokens", type=int, default=None,
                    help="calibration tokens (default: the workload's); smaller cases are for profiling")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Nominal dense tensor-core ratio TF32 : bf16 on GB300 (1.1 : 2.25 PFLOP/s), applied to
# the measured bf16 peak; FP32 FFMA peak from the unit counts and the maximum SM clock:
# 152 SMs x 128 FP32 lanes x 2 flops per fused multiply-add.
TF32_PER_BF16 = 1.1 / 2.25
SM_COUNT, FP32_LANES_PER_SM = 152, 128


def stage_rooflines(m, d, n, bits, group_size, blocksize, syrk_ms, quantize_ms, peaks, factor_ms=None):
    """Each stage against its own bound (bars for the SYRK and the column loop).

    Hessian SYRK: n*d*(d+1) flops (upper triangle) against the measured bf16 peak.
    Column loop + lazy update (the quantize call): T_roof = max(B / HBM,
    F_lazy / P_tf32 + F_in / P_ffma) with B the algorithmic bytes (W in bf16, the upper
    triangle of Hinv1, codes, scales and zeros, column losses), F_lazy the flops of the
    lazy block updates Err1 @ Hinv1[block, rest] and F_in those of the rank-one updates
    inside the blocks. The path computes every lazy product as three TF32 passes (fp32
    accuracy), so the same bound with 3 F_lazy is given beside it.
    Factor (reported, no bar): the Cholesky of the reversed damped Hessian and the
    inverse of its triangular factor, d^3/3 flops each, against the TF32 peak, with one
    and with three passes per product.
    """
    G = 1 if group_size in (-1, 0) else d // group_size
    f_lazy = f_in = 0.0
    for i1 in range(0, d, blocksize):
        nb = min(blocksize, d - i1)
        f_lazy += 2.0 * m * nb * (d - i1 - nb)
        f_in += 1.0 * m * nb * (nb - 1)
    nbytes = 2.0 * m * d + 4.0 * d * (d + 1) / 2 + m * d * bits / 8 + 8.0 * m * G + 4.0 * d
    hbm = peaks["hbm_gbs"] * 1e9
    p_tf32 = peaks["bf16_tflops"] * 1e12 * TF32_PER_BF16
    p_ffma = SM_COUNT * FP32_LANES_PER_SM * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6
    t_mem = nbytes / hbm
    t1 = max(t_mem, f_lazy / p_tf32 + f_in / p_ffma)
    t3 = max(t_mem, 3 * f_lazy / p_tf32 + f_in / p_ffma)
    syrk_flops = float(n) * d * (d + 1)
    t_syrk = syrk_flops / (peaks["bf16_tflops"] * 1e12)
    out = {
        "syrk": {"ms": round(syrk_ms, 4), "bound_ms": round(t_syrk * 1e3, 4),
                 "frac": round(t_syrk * 1e3 / syrk_ms, 4), "bar": 0.60,
                 "model": "n*d*(d+1) flops / measured bf16 peak"},
        "column_loop_and_lazy_update": {
            "ms": round(quantize_ms, 4), "bound_ms": round(t1 * 1e3, 4), "frac": round(t1 * 1e3 / quantize_ms, 4),
            "bar": 0.50,
            "bound_ms_three_pass": round(t3 * 1e3, 4), "frac_three_pass": round(t3 * 1e3 / quantize_ms, 4),
            "model": "max(bytes / HBM, F_lazy / P_tf32 + F_in / P_ffma)",
            "bytes": int(nbytes), "flops_lazy": f_lazy, "flops_in_block": f_in,
            "p_tf32_tflops": round(p_tf32 / 1e12, 1), "p_ffma_tflops": round(p_ffma / 1e12, 2),
            "peaks": "HBM and bf16 measured; TF32 = bf16 x 1.1/2.25 (nominal ratio); FFMA from unit counts "
                     "and the maximum SM clock"},
    }
    if factor_ms is not None:
        f_fac = 2.0 * d ** 3 / 3
        tf1, tf3 = f_fac / p_tf32, 3 * f_fac / p_tf32
        out["factor"] = {"ms": round(factor_ms, 4), "flops": f_fac, "bound_ms": round(tf1 * 1e3, 4),
                         "frac": round(tf1 * 1e3 / factor_ms, 4), "bound_ms_three_pass": round(tf3 * 1e3, 4),
                         "frac_three_pass": round(tf3 * 1e3 / factor_ms, 4), "bar": None,
                         "model": "(d^3/3 Cholesky + d^3/3 triangular inverse) flops / P_tf32"}
    return out


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return host_cores()


# ----------------------------------------------------------------------------------
# the oracle as it stands, on a bounded sample of the layer
def oracle_sample(wl, layer, X_bits_sample, W_bits_rows, n_total, rows_total):
    """Time the CPU oracle on a bounded sample and scale each stage to the full layer.

    SYRK: the oracle Hessian over the sampled tokens, scaled by n_total / n_sample.
    Factor: the full d x d damping + Cholesky chain (no sampling).
    Column loop: the oracle loop over the sampled rows (rows are independent),
    scaled by rows_total / rows_sample.
    """
    from oracle import gptq_oracle as orc
    from synth import bf16_bits_to_f32

    t0 = time.perf_counter()
    step = 16384        # the oracle's batches, so a large sample never needs one float64 copy
    Hs = orc.hessian(bf16_bits_to_f32(X_bits_sample[i:i + step]) for i in range(0, X_bits_sample.shape[0], step))
    t1 = time.perf_counter()
    Hd, _ = orc.damp(Hs, wl.percdamp)
    perm = orc.act_order_perm(Hs) if wl.act_order else np.arange(Hs.shape[0])
    U = orc.hinv1(Hd[np.ix_(perm, perm)])
    t2 = time.perf_counter()
    W = bf16_bits_to_f32(W_bits_rows).astype(np.float64)[:, perm]
    orc.gptq_columns(W, U, wl.bits, wl.group_size, wl.blocksize)
    t3 = time.perf_counter()
    n_s, r_s = X_bits_sample.shape[0], W_bits_rows.shape[0]
    syrk = (t1 - t0) * n_total / n_s
    factor = t2 - t1
    loop = (t3 - t2) * rows_total / r_s
    return {"syrk_s": syrk, "factor_s": factor, "loop_s": loop, "total_s": syrk + factor + loop,
            "sample_wall_s": t3 - t0, "tokens": n_s, "rows": r_s}


# ----------------------------------------------------------------------------------
class Clocks:
    """nvidia-smi sampled every 100 ms by a reader thread; stop(t0, t1) keeps the samples
    taken inside the timed region [t0, t1] (perf_counter seconds)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled: bool):
        self.proc = None
        self.lines = []
        self.ready = threading.Event()
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
        if self.proc is not None:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            self.ready.wait(timeout=10.0)      # sampler running before the timed region starts

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))
            self.ready.set()

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.25)                       # the sample that closes the window
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        inside = [ln for t, ln in self.lines if t0 <= t <= t1 + 0.15]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in inside:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_traffic(kernel_file: str, key: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(key)
        with open(os.path.join(ROOT, "post_weight_quantization_gb300", "csrc", kernel_file), "rb") as f:
            h = hashlib.sha256(f.read()).hexdigest()[:16]
        if rec and rec.get("source_sha256_16") == h:
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


# ----------------------------------------------------------------------------------
def world_size(args) -> int:
    """GPUs the run was asked for: the larger of --gpus and a torchrun WORLD_SIZE."""
    return max(int(args.gpus), int(os.environ.get("WORLD_SIZE", "1")))


def single_gpu_only_line(n: int) -> dict:
    """The line printed for N > 1: the path and its kernels are built for one GPU (the
    Hessian kernel's paired tiles share activation slabs by cluster multicast, which
    only a one-GPU process may run), so no multi-GPU run is made."""
    return {"metric": METRIC, "n_gpus": n,
            "unavailable": "single-GPU path: the layer runs on one GPU; no multi-GPU or replica mode is built"}


def rate_mweights(steps: int, weights: int, seconds: float) -> float:
    """Throughput of `steps` layers of `weights` weights each in `seconds`."""
    return steps * weights / seconds / 1e6


# ----------------------------------------------------------------------------------
def run_reference(args):
    """The oracle as it stands on the host cores, each step a bounded sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from synth import ActSpec, gen_activations_into, workload
    from synth.workloads import CHUNK
    wl = workload(args.workload)
    layer = wl.layers[args.layer]
    spec = wl.acts[layer.hessian]
    n_sample = min(spec.n, 2 * CHUNK)
    Xs = np.empty((n_sample, spec.d), dtype=np.uint16)
    gen_activations_into(spec, Xs, args.threads, (0, n_sample))
    Wfull = wl.weight(layer, threads=args.threads)
    rows = min(layer.m, 32)
    times = []
    for i in range(args.warmup + args.steps):
        r = oracle_sample(wl, layer, Xs, Wfull[:rows], spec.n, layer.m)
        if i >= args.warmup:
            times.append(r)
    t = statistics.mean(x["total_s"] for x in times)
    wall = statistics.mean(x["sample_wall_s"] for x in times)
    weights = layer.m * layer.d
    value = weights / t / 1e6
    sample = (f"per step: oracle Hessian over {n_sample} of {spec.n} tokens (scaled x{spec.n / n_sample:g}), "
              f"full d={layer.d} factor chain, column loop over {rows} of {layer.m} rows (scaled); "
              f"ms_per_step is the sample's wall time, value the layer rate scaled from it")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "Mweights/s",
            "n_gpus": world_size(args), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall * 1e3, 3),
            "ms_per_layer_scaled": round(t * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": args.workload, "layer": layer.name, "m": layer.m, "d": layer.d,
                       "tokens": spec.n, "bits": wl.bits, "group_size": wl.group_size, "blocksize": wl.blocksize,
                       "act_order": wl.act_order},
            "cpu_baseline": {"value": round(value, 6), "unit": "Mweights/s", "cores": blas_threads(),
                             "host_cores": host_cores(), "blas_threads": blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "Mweights/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "stages_s": {k: round(statistics.mean(x[k] for x in times), 4) for k in ("syrk_s", "factor_s", "loop_s")}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------
def run_gpu(args):
    n_req = world_size(args)
    if n_req > 1:
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(single_gpu_only_line(n_req)), flush=True)
        return
    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from post_weight_quantization_gb300 import gptq as g
    from synth import gen_activations_into, workload
    from synth.workloads import CHUNK

    wl = workload(args.workload)
    layer = wl.layers[args.layer]
    spec = wl.acts[layer.hessian]
    if args.tokens:
        spec = dataclasses.replace(spec, n=int(args.tokens))
    m, d, n = layer.m, layer.d, spec.n

    # ---- inputs: pinned host buffers (also the end-to-end source), then HBM copies
    t_gen = time.perf_counter()
    X_host = torch.empty((n, d), dtype=torch.int16, pin_memory=True)
    gen_activations_into(spec, X_host.numpy().view(np.uint16), args.threads)
    W_bits = wl.weight(layer, threads=args.threads)
    W_host = torch.from_numpy(W_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    t_gen = time.perf_counter() - t_gen
    X = X_host.to(dev)
    W = W_host.to(dev)
    H = torch.empty((d, d), dtype=torch.float32, device=dev)
    U = torch.empty((d, d), dtype=torch.float32, device=dev)
    perm = torch.empty(d, dtype=torch.int32, device=dev) if wl.act_order else None
    ws_f = torch.empty(g.gptq_workspace_size(g.GPTQ_WS_FACTOR, 0, d), dtype=torch.uint8, device=dev)
    ws_q = torch.empty(g.gptq_workspace_size(g.GPTQ_WS_QUANTIZE, m, d, wl.bits, wl.group_size, wl.blocksize),
                       dtype=torch.uint8, device=dev)
    G = 1 if wl.group_size == -1 else d // wl.group_size
    out = g.QuantizedLayer(torch.empty((m, (d * wl.bits + 31) // 32), dtype=torch.int32, device=dev),
                           torch.empty((m, G), dtype=torch.float32, device=dev),
                           torch.empty((m, G), dtype=torch.float32, device=dev),
                           torch.empty(d, dtype=torch.float32, device=dev), wl.bits, wl.group_size, d)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev):
        ev[0].record(stream)
        g.gptq_hessian_accumulate(X, H, alpha=2.0, zero_first=True, stream=stream)
        ev[1].record(stream)
        g.gptq_factor(H, percdamp=wl.percdamp, act_order=wl.act_order, Hinv1=U, perm_out=perm, ws=ws_f,
                      sync=False, stream=stream)
        ev[2].record(stream)
        g.gptq_quantize_layer(W, U, perm, bits=wl.bits, group_size=wl.group_size, blocksize=wl.blocksize, out=out,
                              ws=ws_q, stream=stream)
        ev[3].record(stream)

    def mk():
        return [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    for _ in range(args.warmup):
        flush.zero_()
        step(mk())
    torch.cuda.synchronize()
    g.gptq_device_check()
    g.gptq_factor_status(ws_f) if hasattr(g, "gptq_factor_status") else None

    # ---- timed region
    torch.cuda.synchronize()
    clocks = Clocks(local, not args.no_clocks)
    launches0 = g.gptq_launch_count()
    events = []
    t_wall = time.perf_counter()
    t_region0 = t_wall
    for _ in range(args.steps):
        flush.zero_()                       # L2 flush between steps, outside the step's events
        ev = mk()
        step(ev)
        events.append(ev)
    torch.cuda.synchronize()
    t_region1 = time.perf_counter()
    t_wall = t_region1 - t_wall
    launches = g.gptq_launch_count() - launches0
    clk = clocks.stop(t_region0, t_region1)
    g.gptq_device_check()

    st_ms = {"syrk": [], "factor": [], "quantize": []}
    for ev in events:
        st_ms["syrk"].append(ev[0].elapsed_time(ev[1]))
        st_ms["factor"].append(ev[1].elapsed_time(ev[2]))
        st_ms["quantize"].append(ev[2].elapsed_time(ev[3]))
    step_ms = [a + b + c for a, b, c in zip(st_ms["syrk"], st_ms["factor"], st_ms["quantize"])]
    t_max = sum(step_ms) / 1e3
    weights = m * d
    value = rate_mweights(args.steps, weights, t_max)
    ms_per_step = t_max / args.steps * 1e3
    syrk_ms = statistics.mean(st_ms["syrk"])
    syrk_flops = float(n) * d * (d + 1)
    peaks, peak_src = load_peaks()
    syrk_tflops = syrk_flops / (syrk_ms * 1e-3) / 1e12
    roofline = {"kernel": "syrk_kernel (Hessian, tcgen05 bf16)", "bound": "tensor",
                "achieved": round(syrk_tflops, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(syrk_tflops / peaks["bf16_tflops"], 4),
                "frac_of_sustained": round(syrk_tflops / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]), 4),
                "peak_source": f"{peak_src} (bf16 burst)",
                "traffic": kernel_traffic("syrk_tc.cu", f"syrk_{args.workload}"),
                "algorithmic_flops_per_launch": syrk_flops}

    # ---- end to end through the public host-buffer API
    e2e = None
    if not args.no_e2e:
        pipe = g.HostPipeline(m, d, bits=wl.bits, group_size=wl.group_size, blocksize=wl.blocksize,
                              percdamp=wl.percdamp, act_order=wl.act_order, device=dev)
        for _ in range(max(1, args.warmup)):
            pipe.run(W_host, X_host)
        torch.cuda.synchronize()
        e_ms = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pipe.run(W_host, X_host)
            b.record(stream)
            b.synchronize()
            e_ms.append(a.elapsed_time(b))
        te = sum(e_ms) / 1e3
        g.gptq_device_check()
        e2e = {"value": round(rate_mweights(args.steps, weights, te), 4), "unit": "Mweights/s",
               "ms_per_step": round(te / args.steps * 1e3, 4),
               "h2d_bytes_per_step": pipe.bytes_h2d(n), "d2h_bytes_per_step": pipe.bytes_d2h()}

    # ---- CPU oracle baseline, bounded sample
    cpu = None
    if not args.no_cpu_baseline:
        # about 12 s of host work on 16 cores: every token, the full factor, 1/4 of the rows
        n_s = n
        rows = min(m, max(32, m // 4))
        r = oracle_sample(wl, layer, X_host.numpy().view(np.uint16)[:n_s], W_bits[:rows], n, m)
        cpu = {"value": round(weights / r["total_s"] / 1e6, 6), "unit": "Mweights/s", "cores": blas_threads(),
               "host_cores": host_cores(), "blas_threads": blas_threads(), "kind": "oracle",
               "sample": (f"oracle Hessian over {n_s} of {n} tokens (scaled x{n / n_s:g}), full d={d} factor chain, "
                          f"column loop over {rows} of {m} rows (scaled x{m / rows:g}); "
                          f"sample wall {r['sample_wall_s']:.1f} s"),
               "stages_s": {k: round(r[k], 3) for k in ("syrk_s", "factor_s", "loop_s")}}

    if args.tokens:
        line_note = {"note": f"profiling case: {n} tokens instead of the workload's {wl.acts[layer.hessian].n}"}
    else:
        line_note = {}
    line = {"metric": METRIC, "value": round(value, 4), "unit": "Mweights/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32",
            "data": "synthetic (seeded generators; no dataset or trained weights available)",
            "config": {"workload": args.workload, "layer": layer.name, "m": m, "d": d, "tokens": n,
                       "bits": wl.bits, "group_size": wl.group_size, "blocksize": wl.blocksize,
                       "percdamp": wl.percdamp, "act_order": wl.act_order,
                       "parallelism": "single GPU",
                       "l2": "inputs larger than L2 (X is %.2f GB per step) and a 256 MB L2 flush between "
                             "steps, outside the step's events" % (n * d * 2 / 1e9)},
            "stages_ms": {k: round(statistics.mean(v), 4) for k, v in st_ms.items()},
            "quantize_only_ms": round(statistics.mean(st_ms["factor"]) + statistics.mean(st_ms["quantize"]), 4),
            "syrk_tflops": round(syrk_tflops, 2),
            "stage_rooflines": stage_rooflines(m, d, n, wl.bits, wl.group_size, wl.blocksize, syrk_ms,
                                               statistics.mean(st_ms["quantize"]), peaks,
                                               factor_ms=statistics.mean(st_ms["factor"])),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "wall_s_timed_region": round(t_wall, 4), "input_generation_s": round(t_gen, 2),
            **line_note}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
