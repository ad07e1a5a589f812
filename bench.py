"""Benchmark of the QMoE layer forward on GB300.

One step = one full layer forward (routing, grouping, work-lists, fc1 + gated
activation, fc2, weighted combine) over one batch of synthetic tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--mode graph|eager]

Default workload: the int2 GeGLU decode (T=8, hidden=inter=2048, E=8, top-2,
block 128, fractional zero point 1.5, fp16), the shape of the pages' H100
decode figure.  Each rank (torchrun, one GPU each) runs its own replica of
the workload: the layer does not shard, so scaling is weak and no
collective touches the data path.

`--impl reference` times the CPU oracle on this machine's host cores on the same
workload and metric (a deliberately slow reference, not a target).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QMoE layer µs & tokens/s; % HBM roofline (decode), % tensor peak (prefill)"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one fc1
# gemm_kernel launch, from one ncu capture of the current kernel
# (profiles/gemm_kernel_decode_int2_fc1.md, profiles/gemm_kernel_prefill_fc1.md);
# None where no capture of the current kernel exists for the workload.
FC1_TRAFFIC = {"decode_int2": 19_206_144, "prefill_int4": 802_950_656}
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_int2")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="graph", choices=["graph", "eager"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gemm-min-rows", type=int, default=None,
                    help="experts with more rows take the tensor-core grouped GEMM")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process
    group).  Each rank runs an independent replica, so the job's time is the
    slowest rank's."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch (weak scaling)."""
    return world * tokens_per_rank / (ms * 1e-3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(cfg, counts):
    """HBM bytes the layer must move: packed codes + scales + zero points of
    every expert that received rows, plus x, logits and out; and the fc1
    share (fc1 weights of those experts + x + h written)."""
    from qmoe_inputs import DTYPES, expert_fc_bytes
    import torch
    ds = torch.tensor([], dtype=DTYPES[cfg.dtype]).element_size()
    active = int(sum(1 for c in counts if c > 0))
    R = cfg.T * cfg.k
    fc1 = active * expert_fc_bytes(cfg, 1) + cfg.T * cfg.H * ds + R * cfg.I * ds
    layer = active * (expert_fc_bytes(cfg, 1) + expert_fc_bytes(cfg, 2)) + \
        cfg.T * cfg.H * ds * 2 + cfg.T * cfg.E * 4
    return fc1, layer, active


def cpu_baseline(cfg_name, budget_s=20.0):
    """Time the oracle (as it stands) on this host on a bounded sample."""
    import numpy as np
    from oracle import qmoe_oracle as O
    from qmoe_inputs import CONFIGS, make_inputs
    cfg = CONFIGS[cfg_name]
    inp = make_inputs(cfg)
    T = cfg.T
    tokens = np.arange(T) if T <= 64 else np.arange(0, T, max(1, T // 16))[:16]
    t0 = time.perf_counter()
    runs = 0
    while True:
        O.forward(inp, tokens=tokens)
        runs += 1
        if time.perf_counter() - t0 > budget_s / 4 or runs >= 3:
            break
    dt = (time.perf_counter() - t0) / runs
    threads = os.environ.get("OMP_NUM_THREADS") or str(os.cpu_count())
    return {"value": len(tokens) / dt, "unit": "tokens/s", "cores": int(threads),
            "kind": "oracle",
            "sample": f"{len(tokens)} of {T} tokens of {cfg_name}, mean of {runs} run(s), "
                      f"{dt * 1e3:.0f} ms per run"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    from oracle import qmoe_oracle as O
    from qmoe_inputs import CONFIGS, make_inputs
    cfg = CONFIGS[args.workload]
    inp = make_inputs(cfg)
    T = cfg.T
    tokens = np.arange(T) if T <= 64 else np.arange(0, T, max(1, T // 16))[:16]
    for _ in range(args.warmup):
        O.forward(inp, tokens=tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.forward(inp, tokens=tokens)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = len(tokens) / dt
    threads = int(os.environ.get("OMP_NUM_THREADS") or os.cpu_count())
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": cfg.name, "tokens_per_step": len(tokens)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(tokens)} of {T} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import weight_only_quantized_qmoe_gb300 as q
    from weight_only_quantized_qmoe_gb300 import build as qb
    from qmoe_inputs import CONFIGS, DTYPES, make_inputs
    qb.build()

    cfg = CONFIGS[args.workload]
    inp = make_inputs(cfg)
    layer = q.QMoELayer.from_config(cfg)
    if args.gemm_min_rows is not None:
        layer.set_gemm_min_rows(args.gemm_min_rows)
    layer.reserve(cfg.T)
    x, logits = q.load_inputs(layer, inp, device=dev)
    out = torch.empty_like(x)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def make_step(traced):
        """A step callable: the forward replayed from a CUDA graph (or eager),
        with the library's stage events recorded inside it when `traced`."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(q.QMOE_TRACE_NUM_EVENTS)]
        layer.set_trace_events(ev if traced else None)
        with torch.cuda.stream(stream):
            layer.forward(x, logits, out, stream=stream)
        torch.cuda.synchronize()
        graph = None
        if args.mode == "graph":
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                layer.forward(x, logits, out, stream=stream)
            torch.cuda.synchronize()

        def step():
            if graph is not None:
                graph.replay()
            else:
                layer.forward(x, logits, out, stream=stream)
        return step, ev

    # Timed steps: no events inside the forward (recording them between the
    # kernels would break their programmatic launch overlap); one pair of
    # events on the launching stream brackets each step.
    step, _ = make_step(False)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    per_step = []
    t_beg = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            flush.zero_()                      # L2 flush between timed iterations
            t_beg.record(stream)
            step()
            t_end.record(stream)
            stream.synchronize()
            per_step.append(t_beg.elapsed_time(t_end))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()

    # Stage breakdown (and fc1's time for the roofline) from a separate pass
    # with the library's stage events inside the forward.
    tstep, ev = make_step(True)
    stage_ms = [[] for _ in range(q.QMOE_TRACE_NUM_EVENTS - 1)]
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup) + max(5, args.steps // 2)):
            flush.zero_()
            tstep()
            stream.synchronize()
            if i >= max(3, args.warmup):
                for j in range(len(stage_ms)):
                    stage_ms[j].append(ev[j].elapsed_time(ev[j + 1]))
    torch.cuda.synchronize()
    status = layer.poll()
    if status != 0:
        # a bounded device-side wait ran out: the timings are not valid
        print(json.dumps({"error": f"device status {status} after the timed steps"}), file=sys.stderr)
        sys.exit(1)

    ms = max_over_ranks(sum(per_step) / len(per_step), dev)
    value = job_throughput(cfg.T, world, ms)

    # Routing of the run: distinct experts -> algorithmic bytes.
    _, _, _, offs = layer.routing(cfg.T, stream=None)
    torch.cuda.synchronize()
    o = offs.cpu().tolist()
    counts = [o[i + 1] - o[i] for i in range(cfg.E)]
    fc1_bytes, layer_bytes, active = algorithmic_bytes(cfg, counts)
    fc1_stage = statistics.mean(stage_ms[1])
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    min_rows = args.gemm_min_rows if args.gemm_min_rows is not None else 0
    # fc1's roofline: the larger of its HBM time (algorithmic bytes at the
    # measured copy bandwidth) and its tensor time (2 * R * H * 2I FLOPs at
    # the measured bf16 peak) decides what bounds it.
    fc1_flops = 2.0 * cfg.T * cfg.k * cfg.H * 2 * cfg.I
    # counters taken on the default path only (every expert on the GEMM)
    traffic = FC1_TRAFFIC.get(cfg.name) if (min_rows == 0 and cfg.dtype != "f32") else None
    if fc1_flops / (bf16_peak * 1e12) > fc1_bytes / (hbm_peak * 1e9):
        achieved_t = fc1_flops / (fc1_stage * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved_t, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": achieved_t / bf16_peak, "traffic": traffic,
                    "kernel": "fc1 (gemm_kernel, tcgen05 grouped GEMM)", "flops_per_launch": fc1_flops,
                    "peak_kind": peak_kind + " bf16 burst"}
    else:
        achieved = fc1_bytes / (fc1_stage * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": traffic,
                    "kernel": "fc1 (gemm_kernel)" if cfg.T > min_rows and cfg.dtype != "f32"
                    else "fc1 (decode_mma_kernel)", "bytes_per_launch": fc1_bytes,
                    "peak_kind": peak_kind}

    # End-to-end through the public host-buffer entry point (pinned memory).
    ds = torch.tensor([], dtype=DTYPES[cfg.dtype]).element_size()
    xh = inp["x"].pin_memory()
    lh = inp["logits"].pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.set_trace_events(None)
    for _ in range(3):
        layer.forward_host(xh, lh, oh, stream=stream)
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        layer.forward_host(xh, lh, oh, stream=stream)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = max_over_ranks(statistics.mean(e2e_ms), dev)

    # Kernels one forward launches (the library's launch sequence): routing
    # (fused with grouping for T <= 64, else route + group), the x gather and
    # one GEMM per projection when the grouped GEMM runs, one decode-class
    # kernel per projection when any expert can take that class (a positive
    # threshold, or fp32 / T below it), and the combine.
    gemm_on = cfg.dtype != "f32" and cfg.T > min_rows
    decode_on = not gemm_on or min_rows > 0
    launches_per_step = ((1 if cfg.T <= 64 else 2) + (3 if gemm_on else 0) + (2 if decode_on else 0) + 1)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": cfg.name, "tokens": cfg.T, "hidden": cfg.H, "inter": cfg.I,
                   "experts": cfg.E, "top_k": cfg.k, "bits": [cfg.bits1, cfg.bits2],
                   "block_size": cfg.B, "zp": cfg.zp_mode, "act": cfg.act,
                   "mode": args.mode, "l2": "flushed between timed steps (258 MB write)",
                   "us_per_layer": ms * 1e3, "active_experts": active,
                   "stage_us_traced": {n: statistics.mean(v) * 1e3 for n, v in
                                       zip(["route_group", "fc1", "fc2", "combine"], stage_ms)},
                   "layer_bytes": layer_bytes,
                   "layer_hbm_frac": layer_bytes / (ms * 1e-3) / 1e9 / hbm_peak},
        "roofline": roofline,
        "clocks": clk,
        "e2e": {"value": job_throughput(cfg.T, world, e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.H * ds + cfg.T * cfg.E * 4,
                "d2h_bytes_per_step": cfg.T * cfg.H * ds},
        "gpu_launches": launches_per_step * args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
