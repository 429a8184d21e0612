#!/usr/bin/env python
"""Benchmark of the NVFP4 W4A16 MoE layer (route -> FC1 + SwiGLU -> FC2 -> combine).

One step = one pass of the whole layer over one batch: moe_nvfp4_forward through the
C-ABI (route, gather, FC1, FC2, combine).  Default workload: DeepSeek-class decode,
M=16 tokens, H=7168, I=2048, E=256 experts, top_k=8, synthetic seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

Prints one JSON line on rank 0.  Under torchrun (N > 1) every rank runs its own batch
(weak scaling, no collective on the data path); value = all ranks' tokens / max time.
The reference arm times the CPU oracle on the host cores on a bounded sample of the
same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "decode_m16_h7168_i2048_e256_k8"
METRIC = "MoE layer tokens/s (decode M=16, H=7168, I=2048, E=256, top_k=8, NVFP4 W4A16)"
STAGES = ["route", "gather", "fc1", "fc2", "combine"]
# Files whose code decides the GEMMs' memory traffic: the kernels, the launch
# configurations and schedules, the route's tile lists and the repacked layout.
KERNEL_SOURCE_DIR = "csrc"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--sched", choices=["auto", "decode", "prefill", "prefill_pair"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-soak", action="store_true",
                    help="skip the untimed soak before each timed region (for profiler runs)")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time only the headline workload (not the other decode / prefill ones)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (timing: the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, M: int, ms: float) -> float:
    """Whole-job throughput: every rank processes its own M tokens per step."""
    return world * M / (ms * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained",
                                                                           d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed: edits to comments
    or layout leave the compiled kernels, and so the hash, unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(root: str = None) -> str:
    """Hash of the code (not the comments) of every source file that the profiled
    kernels and their launches are built from."""
    root = root or ROOT
    h = hashlib.sha256()
    d = os.path.join(root, "quantized_moe_grouped_route_gb300", KERNEL_SOURCE_DIR)
    files = [os.path.join(d, n) for n in sorted(os.listdir(d)) if n.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(root, "include", "qmoe.h"))
    for path in files:
        with open(path) as f:
            h.update(os.path.basename(path).encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel sources still
    match the ones that were profiled; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}:{workload}")
    if not ent or ent.get("source_sha") != kernel_source_sha():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in list(self.lines):
            if (t0 is not None and t < t0) or (t1 is not None and t > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_bytes(cfg, ids_cpu):
    """Per-launch algorithmic DRAM bytes of FC1 and FC2 and the layer's weight bytes."""
    import numpy as np
    ids = ids_cpu.numpy().reshape(-1)
    valid = ids[(ids >= 0) & (ids < cfg.E)]
    touched = int(np.unique(valid).size)
    n_valid = int(valid.size)
    H, I = cfg.H, cfg.I
    w13 = touched * (2 * I * H * (0.5 + 1 / 16) + 4)
    w2 = touched * (H * I * (0.5 + 1 / 16) + 4)
    fc1 = w13 + n_valid * H * 2 + n_valid * I * 2          # weights + gathered x + h
    fc2 = w2 + n_valid * I * 2 + n_valid * H * 4           # weights + h + fp32 partials
    return {"touched_experts": touched, "pairs": n_valid, "fc1": fc1, "fc2": fc2,
            "weights": w13 + w2, "flops": 2.0 * n_valid * 3 * H * I}


def run_cpu_oracle(li, n_tokens: int):
    """Time the CPU oracle on the first n_tokens tokens; returns (tokens/s, seconds, threads)."""
    import oracle
    toks = list(range(min(n_tokens, li.cfg.M)))
    threads = oracle.max_threads()
    host = [t.detach().cpu() for t in (li.x, li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2,
                                       li.topk_ids, li.topk_weights)]
    t0 = time.perf_counter()
    oracle.forward(*host, tokens=toks, nthreads=threads)
    dt = time.perf_counter() - t0
    return len(toks) / dt, dt, threads, len(toks)


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    import torch

    from qmoe_inputs.gen import config_by_name, make_inputs
    import oracle
    cfg = config_by_name(args.config)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    li = make_inputs(cfg, dev)
    threads = oracle.max_threads()
    n_tok = max(1, min(cfg.M, threads))
    for _ in range(max(args.warmup, 0)):
        run_cpu_oracle(li, n_tok)
    times = []
    for _ in range(args.steps):
        _, dt, threads, n = run_cpu_oracle(li, n_tok)
        times.append(dt)
    total = sum(times)
    value = args.steps * n_tok / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "M": cfg.M, "H": cfg.H, "I": cfg.I, "E": cfg.E,
                   "top_k": cfg.top_k},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_tok} of {cfg.M} tokens per step (all their top_k slots)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Workloads timed in the same run besides the headline one (one line, "configs" key):
# the other decode shape and both prefill shapes of the pages' workloads.
EXTRA_CONFIGS = ["decode_m1_h7168_i3072_e32_k8", "prefill_zipf_m2048_h4096_i1536_e128_k8",
                 "prefill_m8192_h7168_i2048_e256_k8"]


def is_decode(qmoe, sched, M, top_k, E):
    return sched == qmoe.QMOE_SCHED_DECODE or (sched == qmoe.QMOE_SCHED_AUTO and M * top_k <= 4 * E)


def roofline_entry(cfg, alg, stage_ms, decode, sched_name, peaks):
    """Roofline of the dominant kernel (FC1): HBM bytes on decode, tensor FLOPs on prefill."""
    hbm_gbs, bf16_tf, _, peak_kind = peaks
    if decode:
        ach = alg["fc1"] / (stage_ms["fc1"] * 1e-3) / 1e9
        return {"kernel": f"moe_gemm_kernel<FC1,{sched_name}>", "bound": "hbm", "achieved": ach,
                "peak": hbm_gbs, "unit": "GB/s", "frac": ach / hbm_gbs,
                "peak_kind": f"{peak_kind} (hbm_gbs, burst)",
                "algorithmic_bytes_per_launch": alg["fc1"],
                "traffic": measured_traffic("fc1", cfg.name)}
    fl = 2.0 * alg["pairs"] * 2 * cfg.H * cfg.I
    ach = fl / (stage_ms["fc1"] * 1e-3) / 1e12
    return {"kernel": f"moe_gemm_kernel<FC1,{sched_name}>", "bound": "tensor", "achieved": ach,
            "peak": bf16_tf, "unit": "TFLOP/s", "frac": ach / bf16_tf,
            "peak_kind": f"{peak_kind} (bf16_tflops, burst)", "algorithmic_flops_per_launch": fl,
            "traffic": measured_traffic("fc1", cfg.name)}


def time_workload(cfg, sched, K, warmup, dev, rank, world, barrier, token_seed=None,
                  keep_plain=False, soak=True):
    """Build one workload, warm up, time K forwards (one region, CUDA events on the
    launching stream), then K more with the library's stage events for per-kernel times.
    Returns everything the JSON line reports about it, plus the objects e2e needs."""
    import torch

    from quantized_moe_grouped_route_gb300 import NVFP4MoE, qmoe
    from qmoe_inputs.gen import make_inputs

    li = make_inputs(cfg, dev, token_seed=token_seed)
    torch.cuda.synchronize()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record()
    layer = NVFP4MoE(li.w13, li.s13, li.gs13, li.w2, li.s2, li.gs2)
    r1.record()
    torch.cuda.synchronize()
    repack_ms = r0.elapsed_time(r1)
    M, H, I, E, top_k = cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k
    if not keep_plain:  # only the repacked weights are read from here on
        li.w13 = li.s13 = li.w2 = li.s2 = None
        torch.cuda.empty_cache()
    ws = layer.workspace(M, top_k, sched, dev)
    out = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(events=None):
        if events is None:
            qmoe.moe_nvfp4_forward(li.x, layer.w13c, layer.w13s, layer.gs13, layer.w2c, layer.w2s,
                                   layer.gs2, li.topk_ids, li.topk_weights, out, H=H, I=I, E=E,
                                   sched=sched, workspace=ws, stream=stream)
        else:
            qmoe.moe_nvfp4_forward_events(li.x, layer.w13c, layer.w13s, layer.gs13, layer.w2c,
                                          layer.w2s, layer.gs2, li.topk_ids, li.topk_weights, out,
                                          events, H=H, I=I, E=E, sched=sched, workspace=ws,
                                          stream=stream)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc, flags = qmoe.qmoe_read_error(ws)
    if rc != 0:
        raise RuntimeError(f"{cfg.name}: device error word after warm-up: rc={rc} flags={flags}")
    # an untimed soak of the same steps right before the timed region, so that the clock
    # sampler (every 100 ms) sees this workload's load even when the region is short
    soak0 = time.time()
    while soak and time.time() - soak0 < 0.5:
        for _ in range(10):
            step()
        torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for row in evs:  # torch creates the CUDA event on first record
        for ev in row:
            ev.record()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t0.record()
    for _ in range(K):
        step()
    t1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    ms = t0.elapsed_time(t1) / K
    # per-kernel durations: the same K steps again with the library's stage events (an
    # event between two kernels keeps the later one from starting early, so these are
    # each kernel's own durations); the median of the K steps is reported as well
    for i in range(K):
        step(evs[i])
    torch.cuda.synchronize()
    stage_ms = {s: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
                for j, s in enumerate(STAGES)}
    step_median = statistics.median(evs[i][0].elapsed_time(evs[i][5]) for i in range(K))
    rc, flags = qmoe.qmoe_read_error(ws)
    if rc != 0:
        raise RuntimeError(f"{cfg.name}: device error word after the timed region: rc={rc} "
                           f"flags={flags}")
    return {"li": li, "layer": layer, "ws": ws, "out": out, "stream": stream, "ms": ms,
            "stage_ms": stage_ms, "step_median_ms": step_median, "repack_ms": repack_ms,
            "window": (soak0 if soak else wall0, wall1)}


def ours_arm(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from quantized_moe_grouped_route_gb300 import qmoe
    from qmoe_inputs.gen import config_by_name

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    cfg = config_by_name(args.config)
    sched = {"auto": qmoe.QMOE_SCHED_AUTO, "decode": qmoe.QMOE_SCHED_DECODE,
             "prefill": qmoe.QMOE_SCHED_PREFILL,
             "prefill_pair": qmoe.QMOE_SCHED_PREFILL_PAIR}[args.sched]
    M, H, I, E, top_k = cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k

    sampler = ClockSampler(local)
    sampler.start()
    main = time_workload(cfg, sched, args.steps, args.warmup, dev, rank, world, barrier,
                         token_seed=cfg.seed + 1000 * rank, keep_plain=True,
                         soak=not args.no_soak)
    ms = max_over_ranks(main["ms"], world, dev)
    li, layer, out, stream = main["li"], main["layer"], main["out"], main["stream"]

    # end to end through the public call with host buffers: H2D of the step's inputs
    # from pinned memory, the layer, D2H of the result, all inside the timed region
    K = args.steps
    hx = li.x.cpu().pin_memory()
    hids = li.topk_ids.cpu().pin_memory()
    hw = li.topk_weights.cpu().pin_memory()
    hout = torch.empty(M, H, dtype=torch.bfloat16).pin_memory()
    dx, dids, dw = torch.empty_like(li.x), torch.empty_like(li.topk_ids), torch.empty_like(
        li.topk_weights)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dids.copy_(hids, non_blocking=True)
        dw.copy_(hw, non_blocking=True)
        layer(dx, dids, dw, out=out, sched=sched, stream=stream)
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record()
    for _ in range(K):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / K
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    h2d = hx.numel() * 2 + hids.numel() * 4 + hw.numel() * 4
    d2h = hout.numel() * 2
    rc, flags = qmoe.qmoe_read_error(main["ws"])
    if rc != 0:
        raise RuntimeError(f"device error word after the e2e leg: rc={rc} flags={flags}")

    peaks = load_peaks()
    hbm_gbs = peaks[0]
    alg = algorithmic_bytes(cfg, li.topk_ids.cpu())
    decode = is_decode(qmoe, sched, M, top_k, E)
    sched_name = "decode" if decode else "prefill"
    roof = roofline_entry(cfg, alg, main["stage_ms"], decode, sched_name, peaks)

    # the other workloads of the pages, timed in the same run (rank 0's line reports them;
    # every rank runs them so that the barriers match)
    extra = {}
    if world == 1 and not args.no_extra_configs and args.config == DEFAULT_CONFIG:
        steps_x = max(20, min(K, 50))
        for name in EXTRA_CONFIGS:
            c = config_by_name(name)
            r = time_workload(c, qmoe.QMOE_SCHED_AUTO, steps_x, args.warmup, dev, rank, world,
                              barrier, soak=not args.no_soak)
            a = algorithmic_bytes(c, r["li"].topk_ids.cpu())
            dec = is_decode(qmoe, qmoe.QMOE_SCHED_AUTO, c.M, c.top_k, c.E)
            sn = "decode" if dec else "prefill"
            rf = roofline_entry(c, a, r["stage_ms"], dec, sn, peaks)
            layer_frac = (a["weights"] / (r["ms"] * 1e-3) / 1e9 / hbm_gbs if dec else
                          a["flops"] / (r["ms"] * 1e-3) / 1e12 / peaks[1])
            extra[name] = {
                "M": c.M, "H": c.H, "I": c.I, "E": c.E, "top_k": c.top_k, "sched": sn,
                "steps": steps_x, "ms_per_step": r["ms"], "step_median_ms": r["step_median_ms"],
                "tokens_per_s": c.M / (r["ms"] * 1e-3), "stages_ms": r["stage_ms"],
                "roofline": rf,
                "layer": {"bound": "hbm" if dec else "tensor", "frac": layer_frac,
                          "weight_gbs": a["weights"] / (r["ms"] * 1e-3) / 1e9,
                          "tflops": a["flops"] / (r["ms"] * 1e-3) / 1e12},
                "touched_experts": a["touched_experts"],
                "clocks": sampler.summary(*r["window"]),
                "l2": ("inputs larger than L2: "
                       f"{a['weights'] / 1e9:.2f} GB of touched expert weights per step"),
            }
            del r
            torch.cuda.empty_cache()
    sampler.stop()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        n_tok = max(1, min(M, oracle.max_threads()))
        v, dt, threads, n = run_cpu_oracle(li, n_tok)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} of {M} tokens (all their top_k slots), {dt:.1f} s"}

    value = job_tokens_per_s(world, M, ms)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "M": M, "H": H, "I": I, "E": E, "top_k": top_k,
                   "sched": sched_name, "global_batch": world * M,
                   "l2": f"inputs larger than L2: {alg['weights'] / 1e9:.2f} GB of touched "
                         f"expert weights streamed per step",
                   "parallelism": f"replicas{world}"},
        "e2e": {"value": job_tokens_per_s(world, M, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": qmoe.qmoe_forward_kernel_count(M, top_k, E, sched) * K,
        "roofline": roof,
        "cpu_baseline": cpu,
        "clocks": sampler.summary(*main["window"]),
        "stages_ms": main["stage_ms"],
        "stages_from": "a second pass of the same steps with stage events (kernels serialised)",
        "step_median_ms": main["step_median_ms"],
        "weight_gbs": alg["weights"] / (ms * 1e-3) / 1e9,
        "hbm_frac_layer": alg["weights"] / (ms * 1e-3) / 1e9 / hbm_gbs,
        "tflops": alg["flops"] / (ms * 1e-3) / 1e12,
        "touched_experts": alg["touched_experts"],
        "repack_ms": main["repack_ms"],
        "configs": extra or None,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    return ours_arm(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
