#!/usr/bin/env python
"""Benchmark of the streamed 32-layer NF4-LoRA forward + backward step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload stream512|stream16k|pref1024]
                    [--recompute] [--resident] [--layers L] [--tokens M] [--no-cpu-baseline]
                    [--no-secondary]
    python bench.py --impl reference ...     # the CPU oracle, timed on the host cores

One step = layer_stack_step over 32 synthetic Llama-3.1-8B-shaped layers: the forward sweep,
the loss and the reverse backward sweep, every layer's packed NF4 image (112.57 MB) copied
from pinned host RAM into one of two VRAM slots, prefetched one layer ahead.  Prints one
JSON line (rank 0).

The headline line is batch 1 x 512 tokens (host-link bound).  The default run also times the
same streamed stack at batch 8 x 2048 tokens (tensor bound) and reports it under "secondary"
with its own clocks.  The timed regions run without per-launch instrumentation; the GEMM
kernel's own time comes from a separate pass of the same steps with CUDA events around every
GEMM launch.

--gpus N without a launcher starts N local ranks through torch.distributed.run.  Under a
launcher the ranks train data parallel over tokens: each rank holds the workload's M tokens
of an N x M batch (weak scaling), streams the layers from its own pinned store, takes its
loss means over the N x M tokens, and exchanges each layer's dA/dB (NCCL all-gather, then a
fixed-order sum on the device) while the next layer's backward runs.  The timing is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import socket
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
GEMM_SOURCES = ("tc_gemm.cu", "tc_gemm.h", "tc_ptx.cuh")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def gemm_source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "layer_streamed_nf4_quant_b300", "csrc")
    for f in GEMM_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload):
    """DRAM bytes per GEMM launch from the committed ncu record (profiles/tc_gemm_traffic.json),
    or None once the GEMM kernel's sources differ from the ones the counters were taken on."""
    try:
        with open(os.path.join(ROOT, "profiles", "tc_gemm_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != gemm_source_hash():
        return None
    v = rec.get("traffic_bytes_per_launch", {}).get(workload)
    return int(v) if v is not None else None


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

class OracleLayerSample:
    """One layer of the workload, forward and backward, on the CPU oracle.

    Set-up (untimed): layer 0's seven weights from the seeded generator, quantised and packed
    by the oracle.  Each timed sample: the oracle's NF4 decode of the packed layer (unpack and
    dequantise) plus its fp64 layer forward and backward over `tokens` rows.  Nothing here
    touches the CUDA library."""

    def __init__(self, tokens, layer=0, D=4096, dkv=1024, F=14336, r=64, alpha=16.0):
        import synth
        from oracle import nf4 as onf4
        self.tokens, self.layer, self.scale = tokens, layer, alpha / r
        W = synth.layer_weights(layer, D, dkv, F)
        self.shapes = {p: w.shape for p, w in W.items()}
        self.packed = {p: onf4.pack(onf4.quantize(w)) for p, w in W.items()}
        A, B = synth.layer_lora(layer, r, D, dkv, F)
        f = lambda b: onf4.bf16_value(b).astype("float64")  # noqa: E731
        self.A = {p: f(A[p]) for p in A}
        self.B = {p: f(B[p]) for p in B}
        self.x0 = f(synth.stack_input(tokens, D))

    def run(self):
        from oracle import nf4 as onf4
        from oracle import stack as ostack
        t0 = time.perf_counter()
        Wh = {p: onf4.dequantize(onf4.unpack(self.packed[p], *self.shapes[p])) for p in self.packed}
        ostack.stack_forward_backward(self.x0, [(Wh, self.A, self.B)], self.scale)
        return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


# ------------------------------------------------------------------------- ranks

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def under_launcher():
    return "WORLD_SIZE" in os.environ


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launcher_command(n, argv, port):
    """The torch.distributed.run command that starts n local ranks of this script."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def check_world(gpus, world):
    """The launcher's world size must be the --gpus the run was asked for."""
    if world != gpus:
        raise SystemExit(f"bench.py: --gpus {gpus} but the launcher started {world} ranks")


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
    """Tokens per second of the whole job: every rank processes its own tokens_per_rank of the
    global batch (weak scaling), timed by the slowest rank."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


# ----------------------------------------------------------------------- oracle arm

def run_reference(args, world, rank):
    """The oracle arm: the same workload, timed on the host cores (rank 0 only).  Each step is
    a bounded sample of the workload step -- one of its 32 layers, forward and backward, at
    up to 512 of its tokens -- and the line's value extrapolates it to the whole step."""
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    M = wl["M"]
    Ms = min(M, 512)
    sample = OracleLayerSample(Ms)
    times = []
    t_run0 = time.perf_counter()
    for i in range(args.warmup + args.steps):
        t = sample.run()
        if i >= args.warmup:
            times.append(t)
    run_s = time.perf_counter() - t_run0
    t_sample = statistics.mean(times)
    scale_up = 32 * (M / Ms)
    per_step = t_sample * scale_up
    value = M / per_step
    desc = (f"layer 0 of 32 (oracle NF4 decode + fp64 forward and backward) at {Ms} tokens; "
            f"value = tokens / (sample time x {scale_up:g})")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_sample * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "tokens_per_step": M},
        "step_is_sample": True, "layers_timed": 1, "tokens_timed": Ms, "extrapolated": True,
        "extrapolated_ms_per_full_step": per_step * 1e3, "timed_s": sum(times), "run_s": run_s,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- host link

def numa_node_of(dev_index):
    """NUMA node and CPU list of the GPU's PCI device (None if the system does not say)."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        base = f"/sys/bus/pci/devices/{bdf}"
        node = int(open(f"{base}/numa_node").read().strip())
        cpus = open(f"{base}/local_cpulist").read().strip()
    except Exception:
        return None, None
    return (node if node >= 0 else None), cpus


def parse_cpulist(s):
    out = set()
    for part in s.split(","):
        if "-" in part:
            a, b = part.split("-")
            out.update(range(int(a), int(b) + 1))
        elif part:
            out.add(int(part))
    return out


def h2d_probe(torch, dev, store, layer_bytes, n_layers, slots, copy):
    """Host-to-device bandwidth: (a) the pool's own path -- 16 back-to-back layer-image copies
    from the pinned store into the two slots on one copy stream; (b) one 1 GiB pinned buffer
    copied as one transfer; (c) the same 1 GiB as two 512 MiB transfers in flight at once on
    two copy streams.  Best of 4 trials each, GB/s."""
    def timed(fn, nbytes, streams):
        best = 0.0
        for _ in range(4):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = [torch.cuda.Event(enable_timing=True) for _ in streams]
            torch.cuda.synchronize(dev)
            e0.record(streams[0])
            for s in streams[1:]:
                s.wait_event(e0)
            fn()
            for e, s in zip(e1, streams):
                e.record(s)
            torch.cuda.synchronize(dev)
            ms = max(e0.elapsed_time(e) for e in e1)
            best = max(best, nbytes / (ms * 1e-3) / 1e9)
        return best

    n_img = min(n_layers, 16)

    def pool_path():
        with torch.cuda.stream(copy):
            for j in range(16):
                l = j % n_img
                slots[j % 2].copy_(store[l * layer_bytes:(l + 1) * layer_bytes], non_blocking=True)

    out = {"pool_path_gbs": timed(pool_path, 16 * layer_bytes, [copy])}
    gib = 1 << 30
    host = torch.empty(gib, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    dst = torch.empty(gib, dtype=torch.uint8, device=dev)
    copy2 = torch.cuda.Stream(device=dev)

    def one():
        with torch.cuda.stream(copy):
            dst.copy_(host, non_blocking=True)

    def two():
        h = gib // 2
        with torch.cuda.stream(copy):
            dst[:h].copy_(host[:h], non_blocking=True)
        with torch.cuda.stream(copy2):
            dst[h:].copy_(host[h:], non_blocking=True)

    out["one_copy_1GiB_gbs"] = timed(one, gib, [copy])
    out["two_copies_in_flight_gbs"] = timed(two, gib, [copy, copy2])
    del host, dst
    return out


# -------------------------------------------------------------------------- measure

def measure(torch, lsn, dev, desc, M, steps, warmup, pool, resident, lora, ref_pass, recompute, x0_bits, pg,
            e2e_steps, gemm_steps, local, world=1, bwd_weights=0):
    """Warm-up, the timed region (no instrumentation), the GEMM timing pass and the end-to-end
    loop of one workload; returns the measured numbers.  With world > 1 every step is one
    data-parallel step: this rank's M tokens of a world x M batch, each layer's gradients
    exchanged and summed across the ranks while the next layer's backward runs."""
    from layer_streamed_nf4_quant_b300 import workload
    L = desc.n_layers
    grads = [torch.empty(desc.lora_elems, dtype=torch.float32, device=dev) for _ in range(L)]
    x0 = workload.bf16_tensor(x0_bits, device=dev)
    x0_host = x0.cpu().pin_memory()
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    loss_host = torch.zeros(1, dtype=torch.float32).pin_memory()
    ws = torch.empty(desc.workspace_bytes(M, recompute, ref_pass, bwd_weights), dtype=torch.uint8, device=dev)
    x_ref = torch.empty((M, desc.d_model), dtype=torch.bfloat16, device=dev) if ref_pass else None
    compute = torch.cuda.Stream(device=dev)
    dp = lsn.DataParallel(pg, desc, grads, compute) if world > 1 else None

    def step(x=None):
        x = x0 if x is None else x
        kw = dict(stream=compute, recompute=recompute, reference_pass=ref_pass, x_ref_out=x_ref,
                  bwd_weights=bwd_weights)
        if dp is not None:
            kw.update(token_count=world * M, grads_ready=dp.hook)
        if resident is not None:
            lsn.layer_stack_step(desc, x, lora, grads, loss, ws, resident_store=resident, **kw)
        else:
            lsn.layer_stack_step(desc, x, lora, grads, loss, ws, pool=pool, **kw)
        if dp is not None:
            dp.finish()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    lsn.device_check(compute)

    # ------------------------------------------------------------- timed region
    if pool is not None:
        pool.reset_stats()
    launches0 = lsn.launch_count()
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(compute)
        for _ in range(steps):
            step()
        ev1.record(compute)
        torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    launches = lsn.launch_count() - launches0
    lsn.device_check(compute)
    ms = max_over_ranks(pg, ev0.elapsed_time(ev1) / steps, dev)
    pstats = pool.stats() if pool is not None else None

    # ------------------------------------------ GEMM timing pass (events per launch)
    lsn.profile_read(reset=True)
    lsn.profile_enable(True)
    for _ in range(gemm_steps):
        step()
    torch.cuda.synchronize(dev)
    lsn.profile_enable(False)
    prof = lsn.profile_read(reset=True)
    lsn.device_check(compute)

    # ------------------------------------------------------------------ end to end
    # Every step's input comes from pinned host memory and its loss goes back to pinned host
    # memory.  The next step's input is copied on a side stream into the other of two device
    # buffers while the current step runs; a copy into a buffer waits for the step that last
    # read it, and a step waits for its input's copy.
    x0b = [x0, torch.empty_like(x0)]
    copy_in = torch.cuda.Stream(device=dev)
    landed = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(copy_in):
        x0b[0].copy_(x0_host, non_blocking=True)
    landed[0].record(copy_in)
    for i in range(e2e_steps):
        cur, nxt = i % 2, (i + 1) % 2
        if i + 1 < e2e_steps:
            if i >= 1:
                copy_in.wait_event(used[nxt])   # step i - 1 read x0b[nxt]
            with torch.cuda.stream(copy_in):
                x0b[nxt].copy_(x0_host, non_blocking=True)
            landed[nxt].record(copy_in)
        compute.wait_event(landed[cur])
        step(x0b[cur])
        used[cur].record(compute)
        with torch.cuda.stream(compute):
            loss_host.copy_(loss, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(pg, (time.perf_counter() - t0) * 1e3 / e2e_steps, dev)
    out = {"ms": ms, "launches": launches, "pstats": pstats, "prof": prof, "gemm_steps": gemm_steps,
           "e2e_ms": e2e_ms, "e2e_steps": e2e_steps, "clocks": clk.summary(), "x0_bytes": x0.numel() * 2,
           "loss": float(loss_host.item())}
    del ws, grads, x_ref, dp, x0b
    torch.cuda.empty_cache()
    return out


def roofline_fields(m, M, L, ref_pass, h2d_gbs, streamed_bytes, peaks, peak_src, traffic):
    prof = m["prof"]
    exec_flops = prof["gemm_flops"] / m["gemm_steps"]        # executed (includes any recompute)
    step_flops = analytic_step_flops(M, L=L, reference_pass=ref_pass)   # algorithmic
    gemm_ms_step = prof["gemm_ms"] / m["gemm_steps"]
    gemm_tflops = prof["gemm_flops"] / (prof["gemm_ms"] * 1e-3) / 1e12 if prof["gemm_ms"] > 0 else None
    peak_tc = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    t_tensor = step_flops / (peak_tc * 1e12)
    t_h2d = streamed_bytes / (h2d_gbs * 1e9)
    t_roof = max(t_tensor, t_h2d)
    ps = m["pstats"]
    copy_gbs = ps["bytes_copied"] / (ps["copy_ms"] * 1e-3) / 1e9 if ps and ps["copy_ms"] > 0 else None
    ms = m["ms"]
    roof = {"bound": "tensor", "kernel": "tc_gemm_kernel", "achieved": gemm_tflops, "peak": peak_tc,
            "unit": "TFLOP/s", "frac": (gemm_tflops / peak_tc) if gemm_tflops else None, "traffic": traffic,
            "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum per GEMM launch, averaged over "
                              "one layer step's launches (profiles/tc_gemm_traffic.json; null once the kernel "
                              "changed since the counters were taken)",
            "peak_source": f"bf16_tflops_sustained ({peak_src})",
            "timing": f"CUDA events around every GEMM launch in a separate pass of {m['gemm_steps']} steps "
                      "after the timed region",
            "launches_per_step": prof["gemm_launches"] / m["gemm_steps"], "gemm_ms_per_step": gemm_ms_step,
            "gemm_share_of_step": gemm_ms_step / ms}
    step_roof = {"t_roof_ms": t_roof * 1e3, "bound": "h2d" if t_h2d >= t_tensor else "tensor",
                 "t_h2d_ms": t_h2d * 1e3, "t_tensor_ms": t_tensor * 1e3, "frac": t_roof / (ms * 1e-3),
                 "h2d_gbs_measured": h2d_gbs, "step_gflop": step_flops / 1e9,
                 "step_gflop_executed": exec_flops / 1e9,
                 "copy_ms_per_step": ps["copy_ms"] / max(1, m.get("steps", 1)) if ps else None,
                 "copy_gbs": copy_gbs}
    return roof, step_roof


# ----------------------------------------------------------------------------- main

def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lsn", choices=["lsn", "reference"])
    ap.add_argument("--workload", default="stream512", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the 8 x 2048-token measurement that the default run adds")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=32,
                    help="layers of the stack (profiling cases; the metric is defined on 32)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's token count")
    ap.add_argument("--resident", action="store_true",
                    help="read the layers from a resident device store instead of streaming them")
    ap.add_argument("--recompute", action="store_true",
                    help="keep only x_l per layer and recompute each layer in the reverse sweep")
    ap.add_argument("--chunks", type=int, default=1, choices=[1, 2],
                    help="copies per layer image: 2 = [header, q..up] and [o, down] (sub-layer streaming), "
                         "1 = whole-layer copies")
    ap.add_argument("--bwd-weights", type=int, default=0, choices=[0, 1, 2],
                    help="backward GEMMs' W: 0/1 NF4 decoded in the GEMM (default), 2 decoded to bf16 first")
    ap.add_argument("--show-ranks", action="store_true",
                    help="print each rank's world size, rank and device binding as JSON and exit")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.gpus > 1 and not under_launcher():
        # one process per GPU: start the ranks here, one per local GPU
        return subprocess.call(launcher_command(args.gpus, argv, free_port()))
    world, rank, local = dist_setup()
    check_world(args.gpus, world)
    if args.show_ranks:
        print(json.dumps({"rank": rank, "world": world, "local_rank": local, "device": f"cuda:{local}"}),
              flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch

    import layer_streamed_nf4_quant_b300 as lsn
    from layer_streamed_nf4_quant_b300 import workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    wl = dict(WORKLOADS[args.workload])
    M = args.tokens or wl["M"]
    custom = bool(args.tokens or args.layers != 32 or args.resident)
    if custom:
        wl["name"] = (f"profiling case: {args.layers}-layer Llama-3.1-8B-shaped NF4 + LoRA(r=64) stack, "
                      f"{M} tokens, {'resident' if args.resident else 'streamed'}")
    desc = lsn.StackDesc(n_layers=args.layers)
    L = desc.n_layers

    # the pinned store on the GPU's own NUMA node: build it from CPUs of that node
    numa, cpus = numa_node_of(local)
    old_aff = os.sched_getaffinity(0)
    if cpus:
        try:
            os.sched_setaffinity(0, parse_cpulist(cpus) & old_aff or old_aff)
        except OSError:
            pass
    t_setup = time.perf_counter()
    store = workload.build_store(desc)
    lora = [workload.lora_blob(desc, l, device=dev) for l in range(L)]
    import synth
    slots = [torch.empty(desc.image_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    copy = torch.cuda.Stream(device=dev)
    pool = None
    if not args.resident:
        pool = lsn.StreamPool(store, [l * desc.image_bytes for l in range(L)], desc.image_bytes, slots[0],
                              slots[1], copy)
        if args.chunks == 2:
            pool.set_chunks(desc.chunk_offsets())
    resident = store.to(dev) if args.resident else None
    setup_s = time.perf_counter() - t_setup

    link = h2d_probe(torch, dev, store, desc.image_bytes, L, slots, copy)   # its 1 GiB buffer: same node
    os.sched_setaffinity(0, old_aff)
    h2d_gbs = link["pool_path_gbs"]
    link["numa_node"] = numa
    link["note"] = ("pool_path_gbs is the step roofline's denominator: the pool's own copies (112.6 MB layer "
                    "images, pinned store built on the GPU's NUMA node); the 1 GiB probes show what one or two "
                    "transfers in flight reach on this host link")

    ref_pass = bool(wl.get("reference_pass"))
    e2e_steps = args.e2e_steps or max(3, args.steps // 2)
    # data parallel over tokens: this rank's contiguous M rows of a world x M batch
    x0_bits = synth.stack_input(world * M, desc.d_model)[rank * M:(rank + 1) * M]
    main_m = measure(torch, lsn, dev, desc, M, args.steps, args.warmup, pool, resident, lora, ref_pass,
                     args.recompute, x0_bits, pg, e2e_steps, max(2, min(args.steps, 5)), local, world,
                     args.bwd_weights)
    main_m["steps"] = args.steps

    sec = None
    if not args.no_secondary and not custom and world == 1 and args.workload == "stream512" and not args.recompute:
        M2 = WORKLOADS["stream16k"]["M"]
        s_steps = max(10, args.steps // 2)
        sec_m = measure(torch, lsn, dev, desc, M2, s_steps, 3, pool, None, lora, False, False,
                        synth.stack_input(M2, desc.d_model), None, 3, 2, local)
        sec_m["steps"] = s_steps
        sec = (M2, sec_m)

    if rank != 0:
        if pool is not None:
            pool.close()
        return 0

    peaks, peak_src = load_peaks()
    streamed_bytes = 0 if resident is not None else 2 * L * desc.image_bytes
    roof, step_roof = roofline_fields(main_m, M, L, ref_pass, h2d_gbs, streamed_bytes, peaks, peak_src,
                                      None if custom else measured_traffic(args.workload))
    ms = main_m["ms"]
    value = whole_job_rate(world, M, ms)
    ps = main_m["pstats"]

    cpu = None
    if not args.no_cpu_baseline and world == 1 and L == 32:
        Ms = min(M, 512)
        sample = OracleLayerSample(Ms)
        t_layer = sample.run()
        scale_up = L * (M / Ms)
        cpu = {"value": M / (t_layer * scale_up), "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"layer 0 of 32 (oracle NF4 decode + fp64 forward and backward) at {Ms} tokens, "
                         f"timed once ({t_layer:.1f} s) and extrapolated x{scale_up:g}",
               "extrapolated": True, "timed_s": t_layer}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl["name"], "tokens_per_step": M, "layers": L, "lora_rank": desc.rank,
                   "recompute": bool(args.recompute), "reference_pass": ref_pass,
                   "bwd_weights": args.bwd_weights,
                   "bytes_streamed_per_step_vs_plain_step":
                       (ps["bytes_copied"] / args.steps) / (2 * L * desc.image_bytes) if ps else 0.0,
                   "copies_per_layer_image": args.chunks if resident is None else 0,
                   "streamed_bytes_per_step": streamed_bytes, "l2": "inputs larger than L2 "
                   f"({streamed_bytes / 1e9:.2f} GB of layer images streamed per step)",
                   "parallelism": "single GPU" if world == 1 else
                   f"dp{world}: {M} tokens per rank of a {world * M}-token batch, per-layer dA/dB all-gather "
                   "(NCCL) + fixed-order rank sum overlapping the next layer's backward"},
        "roofline": roof,
        "step_roofline": step_roof,
        "h2d_link": link,
        "cpu_baseline": cpu,
        "e2e": {"value": world * M / (main_m["e2e_ms"] * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": main_m["x0_bytes"] + streamed_bytes, "d2h_bytes_per_step": 4,
                "ms_per_step": main_m["e2e_ms"], "steps": main_m["e2e_steps"]},
        "gpu_launches": main_m["launches"],
        "clocks": main_m["clocks"],
        "setup_s": setup_s,
    }
    if sec is not None:
        M2, sm = sec
        r2, s2 = roofline_fields(sm, M2, L, False, h2d_gbs, streamed_bytes, peaks, peak_src,
                                 measured_traffic("stream16k"))
        line["secondary"] = {
            "workload": WORKLOADS["stream16k"]["name"], "tokens_per_step": M2, "value": M2 / (sm["ms"] * 1e-3),
            "unit": UNIT, "ms_per_step": sm["ms"], "steps": sm["steps"], "warmup": 3, "roofline": r2,
            "step_roofline": s2, "clocks": sm["clocks"], "gpu_launches": sm["launches"],
            "e2e": {"value": M2 / (sm["e2e_ms"] * 1e-3), "unit": UNIT, "ms_per_step": sm["e2e_ms"],
                    "steps": sm["e2e_steps"], "h2d_bytes_per_step": sm["x0_bytes"] + streamed_bytes,
                    "d2h_bytes_per_step": 4}}
    print(json.dumps(line), flush=True)
    if pool is not None:
        pool.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
