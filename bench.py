"""Benchmark of the QMoE layer forward on GB300.

One step = one full layer forward (routing, grouping, work-lists, fc1 + gated
activation, fc2, weighted combine) over one batch of synthetic tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--mode graph|eager]

Default workload: the int2 GeGLU decode (T=8, hidden=inter=2048, E=8, top-2,
block 128, fractional zero point 1.5, fp16), the shape of the pages' H100
decode figure.  The same line carries a `workloads` block with the
many-expert int4 decode, the mixed int3/int4 decode and the int4 prefill,
each with its µs per layer, tokens/s, roofline fraction and oracle baseline.  Each rank (torchrun, one GPU each) runs its own replica of
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

L2_BYTES = 129 * 1024 * 1024
# Every workload the line reports besides the headline one; the tiny case is
# a parity case only.
WORKLOADS = ["decode_int2", "decode_many_expert_int4", "mixed_int3_int4", "prefill_int4"]
# DRAM traffic of a kernel is reported only from an ncu capture of the exact
# sources being run: lines "<kernel> <workload> <sources sha256[:16]> <bytes
# per launch>" in this file, written from an ncu capture of those sources.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


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
    ap.add_argument("--path", default="auto", choices=["auto", "fused", "separate"],
                    help="launch sequence: the library's automatic choice (default), the single "
                         "launch wherever it applies, or the separate kernels")
    ap.add_argument("--deterministic", action="store_true",
                    help="slot-ordered combine on the tensor-core path at every size "
                         "(qmoe_set_deterministic; default: automatic, ordered up to 64 tokens)")
    ap.add_argument("--l2", default="rotate", choices=["rotate", "flush"],
                    help="keep the timed steps' inputs out of the L2 by rotating over copies of the layer "
                         "larger than the L2 together (default), or by flushing it before each step")
    ap.add_argument("--only-headline", action="store_true",
                    help="time only --workload (no `workloads` block)")
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
    fc2 = active * expert_fc_bytes(cfg, 2) + R * cfg.I * ds + cfg.T * cfg.H * ds
    layer = active * (expert_fc_bytes(cfg, 1) + expert_fc_bytes(cfg, 2)) + \
        cfg.T * cfg.H * ds * 2 + cfg.T * cfg.E * 4
    return {"fc1": fc1, "fc2": fc2, "layer": layer, "active": active}


def algorithmic_flops(cfg):
    """Multiply-adds x 2 of the two projections over the T*k routed rows."""
    R = cfg.T * cfg.k
    n1 = 2 * cfg.I if cfg.act in ("swiglu", "geglu") else cfg.I
    fc1 = 2.0 * R * cfg.H * n1
    fc2 = 2.0 * R * cfg.I * cfg.H
    return {"fc1": fc1, "fc2": fc2, "layer": fc1 + fc2}


def sources_sha() -> str:
    """sha256[:16] of the CUDA sources and the C header the library is built from."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_quantized_qmoe_gb300", "csrc")
    for f in sorted(os.listdir(csrc)) + ["../../../include/qmoe.h"]:
        path = os.path.normpath(os.path.join(csrc, f))
        if os.path.isfile(path):
            with open(path, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from an ncu capture of
    these exact sources, else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    sha = sources_sha()
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and parts[0] == kernel and parts[1] == workload and parts[2] == sha:
                return int(parts[3])
    return None


def oracle_sample_tokens(cfg, rt, max_experts=8):
    """A bounded sample of tokens for the oracle: tokens in order until their
    routes touch `max_experts` distinct experts (the oracle's cost is the
    dequantisation of every expert it touches)."""
    import numpy as np
    seen, tokens = set(), []
    for t in range(cfg.T):
        new = set(int(e) for e in rt["ids"][t])
        if tokens and len(seen | new) > max_experts:
            break
        seen |= new
        tokens.append(t)
    return np.array(tokens)


def time_oracle(cfg_name, runs=1):
    """The oracle (as it stands) on this host on a bounded sample of the
    workload: tokens/s, and the cores it actually kept busy (process CPU
    time over wall time)."""
    from oracle import qmoe_oracle as O
    from qmoe_inputs import CONFIGS, make_inputs
    cfg = CONFIGS[cfg_name]
    inp = make_inputs(cfg)
    tokens = oracle_sample_tokens(cfg, O.routing(inp))
    w0, c0 = time.perf_counter(), time.process_time()
    for _ in range(runs):
        O.forward(inp, tokens=tokens)
    wall, cpu = time.perf_counter() - w0, time.process_time() - c0
    dt = wall / runs
    return {"value": len(tokens) / dt, "unit": "tokens/s", "cores": max(1, round(cpu / wall)),
            "cores_busy": round(cpu / wall, 2), "kind": "oracle",
            "sample": f"{len(tokens)} of {cfg.T} tokens of {cfg_name} (routes touching <= 8 experts), "
                      f"{runs} run(s), {dt * 1e3:.0f} ms per run"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import qmoe_oracle as O
    from qmoe_inputs import CONFIGS, make_inputs
    cfg = CONFIGS[args.workload]
    inp = make_inputs(cfg)
    tokens = oracle_sample_tokens(cfg, O.routing(inp))
    for _ in range(args.warmup):
        O.forward(inp, tokens=tokens)
    w0, c0 = time.perf_counter(), time.process_time()
    for _ in range(args.steps):
        O.forward(inp, tokens=tokens)
    wall, cpu = time.perf_counter() - w0, time.process_time() - c0
    dt = wall / max(1, args.steps)
    value = len(tokens) / dt
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": cfg.name, "tokens_per_step": len(tokens)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": max(1, round(cpu / wall)),
                         "kind": "oracle",
                         "sample": f"{len(tokens)} of {cfg.T} tokens per step (routes touching <= 8 experts)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PATH_NAMES = {1: "separate kernels", 2: "single launch"}


def launches_per_step(cfg, path, min_rows):
    """Kernels one forward launches: the single launch, or the separate
    sequence -- routing (fused with grouping for T <= 64; else route +
    group, + a scatter of the permutation past 1024 routes), one GEMM per
    projection when the grouped GEMM runs (+ the x gather for T <= 64; above,
    fc1 gathers itself), one decode-class kernel per projection when any
    expert can take that class, and the combine."""
    if path == 2:
        return 1
    gemm_on = cfg.dtype != "f32" and cfg.T > min_rows
    decode_on = not gemm_on or min_rows > 0
    R = cfg.T * cfg.k
    routing = 1 if cfg.T <= 64 else (3 if R > 1024 and cfg.k <= 32 else 2)
    gemm = (2 + (1 if cfg.T <= 64 else 0)) if gemm_on else 0
    return routing + gemm + (2 if decode_on else 0) + 1


def replicas_for(cfg, args):
    """Copies of the layer (weights, x, logits) the timed steps rotate over so
    that between two uses of one copy the other copies stream at least twice
    the L2's size: every step then reads inputs the L2 does not hold."""
    if args.l2 != "rotate":
        return 1
    from qmoe_inputs import expert_fc_bytes
    per = cfg.E * (expert_fc_bytes(cfg, 1) + expert_fc_bytes(cfg, 2))
    return 1 + -(-2 * L2_BYTES // per)


def measure(q, cfg, args, dev, stream, flush, steps, warmup, fused=1, min_rows=0):
    """Time one workload: graph-replayed (or eager) forwards, CUDA events on
    the launching stream around each step.  The primary figure rotates over
    enough copies of the layer that no step finds its inputs in the L2; a
    second figure runs one copy with the L2 flushed (a 258 MB write) before
    every step, which also evicts the kernels' code.  Then a traced pass for
    the per-stage times of the separate kernels, and the host-buffer entry
    point end to end."""
    import torch
    from qmoe_inputs import DTYPES, make_inputs
    inp = make_inputs(cfg)
    nrep = replicas_for(cfg, args)
    reps = []
    for _ in range(nrep):
        layer = q.QMoELayer.from_config(cfg)
        layer.set_fused_decode(fused)
        layer.set_gemm_min_rows(min_rows)
        if args.deterministic:
            layer.set_deterministic(1)   # else the layer's automatic choice
        layer.reserve(cfg.T)
        x, logits = q.load_inputs(layer, inp, device=dev)
        reps.append((layer, x, logits, torch.empty_like(x)))
    layer, x, logits, out = reps[0]

    def make_step(traced, rep):
        lay, xx, lg, oo = rep
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(q.QMOE_TRACE_NUM_EVENTS)]
        lay.set_trace_events(ev if traced else None)
        with torch.cuda.stream(stream):
            lay.forward(xx, lg, oo, stream=stream)
        torch.cuda.synchronize()
        graph = None
        if args.mode == "graph":
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                lay.forward(xx, lg, oo, stream=stream)
            torch.cuda.synchronize()

        def step():
            if graph is not None:
                graph.replay()
            else:
                lay.forward(xx, lg, oo, stream=stream)
        return step, ev

    def timed(step_fns, n, flush_each):
        """Per-step device times of n steps.  Flushed: each step after its
        own flush, one step per host round trip (the flush keeps the device
        busy while the host enqueues the step).  Rotating: the steps are
        enqueued back to back with an event between each two, after warm-up
        steps in the same queue, so the device never waits on the host."""
        with torch.cuda.stream(stream):
            for i in range(max(3, warmup)):
                if flush_each:
                    flush.zero_()
                step_fns[i % len(step_fns)]()
        torch.cuda.synchronize()
        per = []
        if flush_each:
            t_beg = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                for i in range(n):
                    flush.zero_()              # L2 flush between timed iterations
                    t_beg.record(stream)
                    step_fns[i % len(step_fns)]()
                    t_end.record(stream)
                    stream.synchronize()
                    per.append(t_beg.elapsed_time(t_end))
        else:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            lead = max(3, warmup)
            with torch.cuda.stream(stream):
                for i in range(lead):          # keeps the queue ahead of the host
                    step_fns[(i - lead) % len(step_fns)]()
                for i in range(n):
                    ev[i].record(stream)
                    step_fns[i % len(step_fns)]()
                ev[n].record(stream)
            stream.synchronize()
            per = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
        torch.cuda.synchronize()
        return per

    # Timed steps: no events inside the forward (between the separate kernels
    # they would break the programmatic launch overlap).
    steps_fns = [make_step(False, r)[0] for r in reps]
    path = layer.last_path()
    if nrep > 1:
        per_step = timed(steps_fns, steps, False)      # copy i % nrep at step i
        per_flushed = timed(steps_fns[:1], steps, True)
    else:
        per_step = timed(steps_fns, steps, True)
        per_flushed = per_step

    # the same rotated forwards captured back to back in one graph (as a
    # model's layers run): no graph launch or event between two forwards
    seq_ms = None
    if args.mode == "graph" and nrep > 1:
        S = 24
        seq = torch.cuda.CUDAGraph()
        with torch.cuda.graph(seq, stream=stream):
            for i in range(S):
                lay, xx, lg, oo = reps[i % nrep]
                lay.forward(xx, lg, oo, stream=stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            seq.replay()
            e0.record(stream)
            for _ in range(2):
                seq.replay()
            e1.record(stream)
        stream.synchronize()
        seq_ms = e0.elapsed_time(e1) / (2 * S)
        del seq

    stages = None
    if path == 1:
        tstep, ev = make_step(True, reps[0])
        stage_ms = [[] for _ in range(q.QMOE_TRACE_NUM_EVENTS - 1)]
        with torch.cuda.stream(stream):
            for i in range(3 + max(5, steps // 2)):
                flush.zero_()
                tstep()
                stream.synchronize()
                if i >= 3:
                    for j in range(len(stage_ms)):
                        stage_ms[j].append(ev[j].elapsed_time(ev[j + 1]))
        torch.cuda.synchronize()
        stages = {n: statistics.mean(v) * 1e3 for n, v in
                  zip(["route_group", "fc1", "fc2", "combine"], stage_ms)}
        layer.set_trace_events(None)
    for lay, _, _, _ in reps:
        status = lay.poll()
        if status != 0:
            print(json.dumps({"error": f"{cfg.name}: device status {status} after the timed steps"}), file=sys.stderr)
            sys.exit(1)

    _, _, _, offs = layer.routing(cfg.T, stream=None)
    torch.cuda.synchronize()
    o = offs.cpu().tolist()
    counts = [o[i + 1] - o[i] for i in range(cfg.E)]

    # end to end through the host-buffer entry point (pinned memory), rotating
    # over the same copies
    ds = torch.tensor([], dtype=DTYPES[cfg.dtype]).element_size()
    xh = inp["x"].pin_memory()
    lh = inp["logits"].pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    for lay, _, _, _ in reps:
        lay.forward_host(xh, lh, oh, stream=stream)
    e2e_ms = []
    for i in range(steps):
        lay = reps[i % nrep][0]
        if nrep == 1:
            flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        lay.forward_host(xh, lh, oh, stream=stream)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    for lay, _, _, _ in reps:
        lay.close()
    reps.clear()
    return {"ms": statistics.mean(per_step), "ms_median": statistics.median(per_step), "path": path,
            "ms_l2_flushed": statistics.mean(per_flushed), "replicas": nrep, "ms_in_sequence": seq_ms,
            "stages_us": stages, "counts": counts, "e2e_ms": statistics.mean(e2e_ms),
            "h2d": cfg.T * cfg.H * ds + cfg.T * cfg.E * 4, "d2h": cfg.T * cfg.H * ds}


def l2_note(cfg, m):
    from qmoe_inputs import expert_fc_bytes
    if m["replicas"] == 1:
        return "flushed between timed steps (258 MB write)"
    per = cfg.E * (expert_fc_bytes(cfg, 1) + expert_fc_bytes(cfg, 2))
    return (f"inputs larger than L2: {m['replicas']} copies of the layer (weights, x, logits; "
            f"{per * m['replicas'] / 2**20:.0f} MB of weights) rotated step by step")


def roofline_of(cfg, m, hbm_peak, bf16_peak, peak_kind):
    """Roofline of the dominant kernel of a measured workload.

    Single launch: the one kernel is the whole layer (time = the timed step).
    Separate kernels: fc1's grouped GEMM (or decode kernel), timed by the
    traced pass.  Each takes the bound whose floor is larger: HBM (algorithmic
    bytes at the measured copy bandwidth) or tensor (FLOPs at the measured
    bf16 peak)."""
    by = algorithmic_bytes(cfg, m["counts"])
    fl = algorithmic_flops(cfg)
    if m["path"] == 2:
        kernel, bytes_, flops_, ms, tkey = "fused_decode_kernel (single launch)", by["layer"], fl["layer"], m["ms"], \
            "fused_decode_kernel"
    else:
        kernel, bytes_, flops_ = "fc1 gemm_kernel (tcgen05 grouped GEMM)", by["fc1"], fl["fc1"]
        ms, tkey = m["stages_us"]["fc1"] * 1e-3, "gemm_kernel_fc1"
    if flops_ / (bf16_peak * 1e12) > bytes_ / (hbm_peak * 1e9):
        ach = flops_ / (ms * 1e-3) / 1e12
        r = {"bound": "tensor", "achieved": ach, "peak": bf16_peak, "unit": "TFLOP/s", "frac": ach / bf16_peak,
             "flops_per_launch": flops_, "peak_kind": peak_kind + " bf16 burst"}
    else:
        ach = bytes_ / (ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
             "bytes_per_launch": bytes_, "peak_kind": peak_kind}
    r["traffic"] = measured_traffic(tkey, cfg.name)
    r["kernel"] = kernel
    r["launch_us"] = ms * 1e3
    return r, by, fl


def workload_summary(cfg, m, hbm_peak, bf16_peak, peak_kind, world):
    roof, by, fl = roofline_of(cfg, m, hbm_peak, bf16_peak, peak_kind)
    d = {"us_per_layer": m["ms"] * 1e3, "tokens_per_s": job_throughput(cfg.T, world, m["ms"]),
         "l2": l2_note(cfg, m), "us_per_layer_l2_flushed": m["ms_l2_flushed"] * 1e3,
         "us_per_layer_in_graph_sequence": m["ms_in_sequence"] * 1e3 if m["ms_in_sequence"] else None,
         "path": PATH_NAMES.get(m["path"], "?"), "active_experts": by["active"],
         "layer_bytes": by["layer"], "layer_flops": fl["layer"],
         "layer_hbm_frac": by["layer"] / (m["ms"] * 1e-3) / 1e9 / hbm_peak,
         "layer_tensor_frac": fl["layer"] / (m["ms"] * 1e-3) / 1e12 / bf16_peak,
         "roofline": roof,
         "e2e_tokens_per_s": job_throughput(cfg.T, world, m["e2e_ms"])}
    if m["stages_us"]:
        st = m["stages_us"]
        d["stage_us_traced"] = st
        d["fc1_frac"] = (fl["fc1"] / (st["fc1"] * 1e-6) / 1e12 / bf16_peak if cfg.T > 64 else
                         by["fc1"] / (st["fc1"] * 1e-6) / 1e9 / hbm_peak)
        d["fc2_frac"] = (fl["fc2"] / (st["fc2"] * 1e-6) / 1e12 / bf16_peak if cfg.T > 64 else
                         by["fc2"] / (st["fc2"] * 1e-6) / 1e9 / hbm_peak)
    return d


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
    from qmoe_inputs import CONFIGS
    qb.build()

    cfg = CONFIGS[args.workload]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    fused = {"auto": 2, "fused": 1, "separate": 0}[args.path]
    min_rows = args.gemm_min_rows if args.gemm_min_rows is not None else 0

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    head = measure(q, cfg, args, dev, stream, flush, args.steps, args.warmup, fused, min_rows)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    others = {}
    if not args.only_headline:
        for name in WORKLOADS:
            if name == cfg.name:
                continue
            others[name] = measure(q, CONFIGS[name], args, dev, stream, flush, max(10, args.steps // 2),
                                   args.warmup, fused, min_rows)
    clk = clocks.stop()

    ms = max_over_ranks(head["ms"], dev)
    value = job_throughput(cfg.T, world, ms)
    roof, by, fl = roofline_of(cfg, head, hbm_peak, bf16_peak, peak_kind)
    e2e = max_over_ranks(head["e2e_ms"], dev)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": cfg.name, "tokens": cfg.T, "hidden": cfg.H, "inter": cfg.I,
                   "experts": cfg.E, "top_k": cfg.k, "bits": [cfg.bits1, cfg.bits2],
                   "block_size": cfg.B, "zp": cfg.zp_mode, "act": cfg.act,
                   "mode": args.mode, "l2": l2_note(cfg, head),
                   "us_per_layer_l2_flushed": head["ms_l2_flushed"] * 1e3,
                   "us_per_layer_in_graph_sequence": (head["ms_in_sequence"] * 1e3
                                                      if head["ms_in_sequence"] else None),
                   "path": PATH_NAMES.get(head["path"], "?"),
                   "us_per_layer": ms * 1e3, "active_experts": by["active"],
                   "layer_bytes": by["layer"],
                   "layer_hbm_frac": by["layer"] / (ms * 1e-3) / 1e9 / hbm_peak},
        "roofline": roof,
        "clocks": clk,
        "e2e": {"value": job_throughput(cfg.T, world, e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": head["h2d"], "d2h_bytes_per_step": head["d2h"]},
        "gpu_launches": launches_per_step(cfg, head["path"], min_rows) * args.steps,
    }
    if head["stages_us"]:
        line["config"]["stage_us_traced"] = head["stages_us"]
    if others or not args.only_headline:
        wl = {cfg.name: workload_summary(cfg, head, hbm_peak, bf16_peak, peak_kind, world)}
        for name, m in others.items():
            wl[name] = workload_summary(CONFIGS[name], m, hbm_peak, bf16_peak, peak_kind, world)
        line["workloads"] = wl
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(cfg.name)
        if "workloads" in line:
            for name in line["workloads"]:
                line["workloads"][name]["cpu_baseline"] = (line["cpu_baseline"] if name == cfg.name
                                                           else time_oracle(name))
    if rank == 0:
        print(json.dumps(line), flush=True)
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
