#!/usr/bin/env python
"""Benchmark of the streamed 32-layer NF4-LoRA forward + backward step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload stream512|stream16k|pref1024]
                    [--recompute] [--resident] [--layers L] [--tokens M] [--no-cpu-baseline]
    python bench.py --impl reference ...     # the CPU oracle, timed on the host cores

One step = layer_stack_step over 32 synthetic Llama-3.1-8B-shaped layers: the forward sweep,
the loss and the reverse backward sweep, every layer's packed NF4 image (112.57 MB) copied
from pinned host RAM into one of two VRAM slots, prefetched one layer ahead.  Prints one
JSON line (rank 0).  Under torchrun each rank runs an independent replica of the workload on
its own GPU (weak scaling); the timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "streamed 32-layer NF4-LoRA fwd+bwd tokens/s; % of H2D-BW / tensor-peak roofline"
UNIT = "tokens/s"
WORKLOADS = {
    "stream512": {"M": 512, "name": "32-layer Llama-3.1-8B-shaped NF4 + LoRA(r=64, alpha=16) stack, "
                                    "streamed from pinned host through two VRAM slots, batch 1 x 512 tokens"},
    "stream16k": {"M": 16384, "name": "32-layer Llama-3.1-8B-shaped NF4 + LoRA(r=64, alpha=16) stack, "
                                      "streamed from pinned host through two VRAM slots, batch 8 x 2048 tokens"},
    "pref1024": {"M": 1024, "reference_pass": True,
                 "name": "preference pair (chosen + rejected, 2 x 512 tokens) on the 32-layer Llama-3.1-8B-shaped "
                         "NF4 + LoRA(r=64) stack: policy forward + backward and the adapter-disabled reference "
                         "forward on the same streamed slots"},
}
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def measured_traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu summary, or None once the GEMM
    kernel's sources differ from the ones the counters were taken on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "layer_streamed_nf4_quant_b300", "csrc")
    for f in ("tc_gemm.cu", "tc_gemm.h", "tc_ptx.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    try:
        lines = open(os.path.join(ROOT, "profiles", "tc_gemm_dram_traffic.md")).read().splitlines()
    except OSError:
        return None
    src = next((l.split()[1] for l in lines if l.startswith("kernel_source_sha256")), None)
    if src != h.hexdigest():
        return None
    for l in lines:
        f = l.split()
        if len(f) == 3 and f[0] == "traffic_bytes_per_launch" and f[1] == workload:
            return int(f[2])
    return None


def analytic_step_flops(M, L=32, D=4096, dkv=1024, F=14336, r=64, reference_pass=False):
    """Algorithmic FLOPs of one step: forward, dX and dA/dB of every projection, no recompute;
    plus the adapter-disabled forward when the step runs the reference pass."""
    shapes = [(D, D), (dkv, D), (dkv, D), (F, D), (F, D), (D, D), (D, F)]
    P = sum(n * k for n, k in shapes)
    lora = sum(n + k for n, k in shapes)
    fwd = 2 * M * P + 2 * M * r * lora
    bwd = 2 * M * P + 2 * (2 * M * r * lora)   # dW-free: dY W, and dT, dB, dA, dT A
    ref = 2 * M * P if reference_pass else 0
    return L * (fwd + bwd + ref)


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle

def oracle_layer_sample(store_np, desc, layer, M):
    """One layer of the workload, forward and backward, on the CPU oracle: NF4 decode of the
    layer image plus the fp64 layer math.  Returns seconds."""
    import numpy as np

    import synth
    from layer_streamed_nf4_quant_b300 import PROJ, nf4_packed_bytes
    from oracle import nf4 as onf4
    from oracle import stack as ostack
    t0 = time.perf_counter()
    base = layer * desc.image_bytes
    Wh = {}
    for i, p in enumerate(PROJ):
        n, k = desc.shape(p)
        off = base + desc.image_offsets[i]
        st = onf4.unpack(store_np[off: off + nf4_packed_bytes(n, k)], n, k)
        Wh[p] = onf4.dequantize(st)
    A, B = synth.layer_lora(layer, desc.rank, desc.d_model, desc.d_kv, desc.d_ff)
    f = lambda b: onf4.bf16_value(b).astype(np.float64)  # noqa: E731
    x0 = f(synth.stack_input(M, desc.d_model))
    ostack.stack_forward_backward(x0, [(Wh, {p: f(A[p]) for p in A}, {p: f(B[p]) for p in B})], desc.scale)
    return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


# -------------------------------------------------------------------------------- main

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(pg, value, device):
    """The largest of every rank's value (each rank's time of the same number of steps), or
    the value itself on a single rank."""
    if pg is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, tokens_per_rank, ms_per_step):
    """Tokens per second of the whole job: every rank runs its own replica of the workload
    (weak scaling), timed by the slowest rank."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def run_reference(args, world, rank):
    """The oracle arm: the same workload's step, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401

    import layer_streamed_nf4_quant_b300 as lsn
    from layer_streamed_nf4_quant_b300 import workload
    wl = WORKLOADS[args.workload]
    M = min(wl["M"], 512)
    desc = lsn.StackDesc(n_layers=1)
    store = workload.build_store(desc, pinned=False)
    times = []
    for i in range(args.warmup + args.steps):
        t = oracle_layer_sample(store.numpy(), desc, 0, M)
        if i >= args.warmup:
            times.append(t)
    per_step = statistics.mean(times) * 32 * (wl["M"] / M)
    value = wl["M"] / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "tokens_per_step": wl["M"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": f"each step: layer 0 of 32 (NF4 decode + fp64 forward and backward) at "
                                   f"{M} tokens, scaled x32" + (f" and x{wl['M'] // M} tokens" if wl["M"] != M else "")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lsn", choices=["lsn", "reference"])
    ap.add_argument("--workload", default="stream512", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=32,
                    help="layers of the stack (profiling cases; the metric is defined on 32)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's token count")
    ap.add_argument("--resident", action="store_true",
                    help="read the layers from a resident device store instead of streaming them")
    ap.add_argument("--recompute", action="store_true",
                    help="keep only x_l per layer and recompute each layer in the reverse sweep")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import numpy as np  # noqa: F401
    import torch

    import layer_streamed_nf4_quant_b300 as lsn
    from layer_streamed_nf4_quant_b300 import workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist

    wl = dict(WORKLOADS[args.workload])
    M = args.tokens or wl["M"]
    if args.tokens or args.layers != 32 or args.resident:
        wl["name"] = (f"profiling case: {args.layers}-layer Llama-3.1-8B-shaped NF4 + LoRA(r=64) stack, "
                      f"{M} tokens, {'resident' if args.resident else 'streamed'}")
    desc = lsn.StackDesc(n_layers=args.layers)
    L = desc.n_layers
    t_setup = time.perf_counter()
    store = workload.build_store(desc)
    lora = [workload.lora_blob(desc, l, device=dev) for l in range(L)]
    grads = [torch.empty(desc.lora_elems, dtype=torch.float32, device=dev) for _ in range(L)]
    import synth
    x0_bits = synth.stack_input(M, desc.d_model)
    x0 = workload.bf16_tensor(x0_bits, device=dev)
    x0_host = x0.cpu().pin_memory()
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    loss_host = torch.zeros(1, dtype=torch.float32).pin_memory()
    ref_pass = bool(wl.get("reference_pass"))
    ws = torch.empty(desc.workspace_bytes(M, args.recompute, ref_pass), dtype=torch.uint8, device=dev)
    x_ref = torch.empty((M, desc.d_model), dtype=torch.bfloat16, device=dev) if ref_pass else None
    slots = [torch.empty(desc.image_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    compute = torch.cuda.Stream(device=dev)
    copy = torch.cuda.Stream(device=dev)
    pool = lsn.StreamPool(store, [l * desc.image_bytes for l in range(L)], desc.image_bytes, slots[0], slots[1],
                          copy)
    resident = store.to(dev) if args.resident else None
    setup_s = time.perf_counter() - t_setup

    # host->device bandwidth of this machine on the path the pool uses: back-to-back copies of
    # layer images out of the pinned store into the two slots, on the copy stream (best of
    # 4 trials of 16 copies)
    h2d = []
    n_img = min(L, 16)
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy):
            e0.record(copy)
            for j in range(16):
                l = j % n_img
                slots[j % 2].copy_(store[l * desc.image_bytes:(l + 1) * desc.image_bytes], non_blocking=True)
            e1.record(copy)
        e1.synchronize()
        h2d.append(16 * desc.image_bytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    h2d_gbs = max(h2d)

    def step():
        kw = dict(stream=compute, recompute=args.recompute, reference_pass=ref_pass, x_ref_out=x_ref)
        if resident is not None:
            lsn.layer_stack_step(desc, x0, lora, grads, loss, ws, resident_store=resident, **kw)
        else:
            lsn.layer_stack_step(desc, x0, lora, grads, loss, ws, pool=pool, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    lsn.device_check(compute)

    # ---------------------------------------------------------------- timed region
    pool.reset_stats()
    lsn.profile_read(reset=True)
    lsn.profile_enable(True)
    launches0 = lsn.launch_count()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(compute)
        for _ in range(args.steps):
            step()
        ev1.record(compute)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    launches = lsn.launch_count() - launches0
    lsn.profile_enable(False)
    prof = lsn.profile_read(reset=True)
    lsn.device_check(compute)
    ms = max_over_ranks(pg, ev0.elapsed_time(ev1) / args.steps, dev)
    pstats = pool.stats()
    value = whole_job_rate(world, M, ms)

    # ------------------------------------------------------------------- end to end
    e2e_steps = args.e2e_steps or max(3, args.steps // 2)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(compute):
            x0.copy_(x0_host, non_blocking=True)
        step()
        with torch.cuda.stream(compute):
            loss_host.copy_(loss, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(pg, (time.perf_counter() - t0) * 1e3 / e2e_steps, dev)
    streamed_bytes = 0 if resident is not None else 2 * L * desc.image_bytes

    if rank != 0:
        return 0

    peaks, peak_src = load_peaks()
    exec_flops = prof["gemm_flops"] / args.steps        # executed (includes any recompute)
    step_flops = analytic_step_flops(M, L=L, reference_pass=ref_pass)   # algorithmic
    gemm_tflops = prof["gemm_flops"] / (prof["gemm_ms"] * 1e-3) / 1e12 if prof["gemm_ms"] > 0 else None
    peak_tc = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    t_tensor = step_flops / (peak_tc * 1e12)
    t_h2d = streamed_bytes / (h2d_gbs * 1e9)
    copy_gbs = pstats["bytes_copied"] / (pstats["copy_ms"] * 1e-3) / 1e9 if pstats["copy_ms"] > 0 else None
    t_roof = max(t_tensor, t_h2d)

    cpu = None
    if not args.no_cpu_baseline and world == 1 and L == 32:
        t_layer = oracle_layer_sample(store.numpy(), desc, 0, min(M, 512))
        per_step = t_layer * L * (M / min(M, 512))
        cpu = {"value": M / per_step, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"layer 0 of 32 (NF4 decode + fp64 forward and backward) at {min(M, 512)} tokens, "
                         f"timed once and scaled x32" + (f" and x{M // 512} tokens" if M > 512 else "")}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl["name"], "tokens_per_step": M, "layers": L, "lora_rank": desc.rank,
                   "recompute": bool(args.recompute), "reference_pass": ref_pass,
                   "bytes_streamed_per_step_vs_plain_step":
                       (pstats["bytes_copied"] / args.steps) / (2 * L * desc.image_bytes) if resident is None else 0.0,
                   "streamed_bytes_per_step": streamed_bytes, "l2": "inputs larger than L2 "
                   f"({streamed_bytes / 1e9:.2f} GB of layer images streamed per step)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "tc_gemm_kernel", "achieved": gemm_tflops, "peak": peak_tc,
                     "unit": "TFLOP/s", "frac": (gemm_tflops / peak_tc) if gemm_tflops else None,
                     "traffic": None if (args.tokens or L != 32) else measured_traffic(args.workload),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per GEMM launch, "
                                       "averaged over one layer step's launches",
                     "peak_source": f"bf16_tflops_sustained ({peak_src})",
                     "launches_per_step": prof["gemm_launches"] / args.steps,
                     "gemm_ms_per_step": prof["gemm_ms"] / args.steps},
        "step_roofline": {"t_roof_ms": t_roof * 1e3, "bound": "h2d" if t_h2d >= t_tensor else "tensor",
                          "t_h2d_ms": t_h2d * 1e3, "t_tensor_ms": t_tensor * 1e3, "frac": t_roof / (ms * 1e-3),
                          "h2d_gbs_measured": h2d_gbs, "step_gflop": step_flops / 1e9,
                          "step_gflop_executed": exec_flops / 1e9,
                          "copy_ms_per_step": pstats["copy_ms"] / args.steps,
                          "copy_gbs": copy_gbs},
        "cpu_baseline": cpu,
        "e2e": {"value": world * M / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": x0.numel() * 2 + streamed_bytes, "d2h_bytes_per_step": 4,
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "setup_s": setup_s,
    }
    print(json.dumps(line), flush=True)
    pool.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
