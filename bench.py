"""Benchmark of the shape-driven fp16 GEMM + M=1 decode GEMV on GB300.

Default run (`python bench.py [--gpus N] [--steps K] [--warmup W]`):

  one step = the whole hot path over one batch of synthetic input:
    * fp16 GEMM C = A.B for every square size M=N=K in {256, 512, 768, 1024,
      1536, 2048, 2560, 3072, 3584, 4096}, tile chosen by pick_tile;
    * the M=1 decode GEMV, K=4096, N=12288, bf16 weights and q8 weights,
      each from one of 8 rotating weight buffers (so every launch streams
      its weights from HBM).
  The step's working set (~1.6 GB) is far larger than the 129 MB L2, so no
  explicit flush is needed between timed steps.

  value = FLOPs of all timed steps on all ranks / the slowest rank's timed
  wall time (CUDA events on the launching stream, barrier + synchronise on
  both sides), in TFLOP/s.  Rank 0 prints one JSON line.

After the timed region rank 0 runs the configurations' own protocols, each
after at least 1 s of warm-up and under its own clock sampler (--no-legs skips
them).  Each answers one question with a prediction written before it was run:
  decode_protocol  does the M=1 decode stream at >= 80 % of HBM?  200 graph-
                   replayed launches x 10, 8 rotating buffers; predicted bf16
                   93-98 %, q8 80-88 % of the measured copy bandwidth.
  gemm_protocol    what fraction of the dense peak per square size?  200
                   graph-replayed launches x 5 + one eager loop; predicted
                   4096^3 78-86 %; falsified below 70 % or if graph and eager
                   differ by > 5 % from 1536^3 up.
  pick_check       is pick_tile within 5 % of the fastest feasible tile (the
                   square sizes and the K-scan shapes)?
                   every feasible tile cold, 5 shuffled passes x 8 launches;
                   predicted average <= 1 %, worst <= 5 %.
  kscan            does K = 2048 (32 k-tiles) camp memory channels on GB300?
                   M=N=2048, K 1920..2304, 128x128, stagger off/on, cold and
                   warm; predicted no dip at 2048 beyond 3 % and the stagger
                   within +-3 %.
  large            8192^3 / 12288^3 / 16384^3 with pick_tile, graph-replayed;
                   predicted 80-90 / 78-90 / 72-86 % of the burst peak.

Other modes (--mode): `sweep` times every feasible tile per square size and
reports pick_tile's slowdown against the best; `kscan` the K-scan with the
stagger on and off; `decode` the decode protocol (200 launches x 10
repeats); `large` the 8192..16384 squares.  They print one JSON line each.

`--impl reference` times the CPU oracle (the only implementation the pages'
method has here) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import random
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fp16 GEMM TFLOP/s per size (% tensor peak); M=1 decode µs and HBM GB/s"
SWEEP = [256, 512, 768, 1024, 1536, 2048, 2560, 3072, 3584, 4096]
KSCAN = [1920, 1984, 2048, 2112, 2176, 2304]
LARGE = [8192, 12288, 16384]
DEC_K, DEC_N, DEC_BUFFERS = 4096, 12288, 8
WORKLOAD = ("square fp16 GEMM sweep M=N=K in {256,512,768,1024,1536,2048,2560,3072,3584,4096} "
            "(pick_tile) + M=1 decode GEMV K=4096 N=12288, bf16 and q8 arms, 8 rotating weight buffers")


# ---------------------------------------------------------------------------------------------
# workload arithmetic
# ---------------------------------------------------------------------------------------------


def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def gemm_bytes(M, N, K):
    """Compulsory DRAM bytes of one fp16 GEMM: read A and B once, write C once."""
    return 2.0 * (M * K + K * N + M * N)


def decode_bytes(K, N, fmt, scale_bytes=2, group=32):
    """Bytes one decode GEMV must move: weights (+ scales), x (bf16) and y (fp32)."""
    if fmt == "bf16":
        w = 2 * K * N
    else:
        w = K * N + (K // group) * N * scale_bytes
    return w + 2 * K + 4 * N


def decode_weight_bytes(K, N, fmt, scale_bytes=2, group=32):
    return 2 * K * N if fmt == "bf16" else K * N + (K // group) * N * scale_bytes


def step_flops():
    return sum(gemm_flops(n, n, n) for n in SWEEP) + 2 * (2.0 * DEC_K * DEC_N)


# ---------------------------------------------------------------------------------------------
# distributed bookkeeping (replicas only: no data-path collective)
# ---------------------------------------------------------------------------------------------


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend):
    import torch.distributed as dist

    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29500")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return world, rank


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank_per_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    return units_per_rank_per_step * steps * world / max_seconds


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
                "temperature.gpu,utilization.gpu")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while the timed region runs."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="sdt_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        return parse_clock_csv(open(self.path).read() if self.path and os.path.exists(self.path) else "")


def _num(v):
    try:
        return float(v)
    except ValueError:
        return None


def parse_clock_csv(text: str):
    """Summary of nvidia-smi samples (CLOCK_FIELDS, csv, no header, no units).  Samples
    "under load" are those with GPU utilisation >= 50 % when the column is there, else
    those with the SM clock above half its maximum."""
    rows = []
    for line in text.splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]), power=_num(parts[3]),
                             active=parts[4], hw=parts[5], hw_thermal=parts[6], sw_thermal=parts[7],
                             sw_power=parts[8], temp=_num(parts[9]) if len(parts) > 9 else None,
                             util=_num(parts[10]) if len(parts) > 10 else None))
        except ValueError:
            continue
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    if any(r["util"] is not None for r in rows):
        load = [r for r in rows if r["util"] is not None and r["util"] >= 50]
    else:
        load = [r for r in rows if r["sm"] > 0.5 * r["sm_max"]]
    sel = load or rows
    reasons = set()
    for r in rows:
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    pw = [r["power"] for r in sel if r["power"] is not None]
    tp = [r["temp"] for r in rows if r["temp"] is not None]
    out = {"sm_mhz": statistics.median(r["sm"] for r in sel), "sm_max_mhz": max(r["sm_max"] for r in rows),
           "sm_mhz_min_under_load": min(r["sm"] for r in sel), "reasons": sorted(reasons), "samples": len(rows),
           "samples_under_load": len(load), "power_w_max": max(pw) if pw else None,
           "power_w_median_under_load": statistics.median(pw) if pw else None}
    if tp:
        out["temp_c_max"] = max(tp)
    return out


def gpu_state(gpu_index: int):
    """One query of the GPU's temperature, power, clocks and utilisation (read only)."""
    fields = "temperature.gpu,power.draw,clocks.sm,clocks.mem,pstate,utilization.gpu"
    try:
        r = subprocess.run(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={fields}",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
    except (OSError, subprocess.SubprocessError):
        return None
    parts = [p.strip() for p in r.stdout.strip().split(",")]
    if r.returncode != 0 or len(parts) < 6:
        return None
    return {"temp_c": _num(parts[0]), "power_w": _num(parts[1]), "sm_mhz": _num(parts[2]),
            "mem_mhz": _num(parts[3]), "pstate": parts[4], "util_pct": _num(parts[5]),
            "t": round(time.time(), 1)}


# ---------------------------------------------------------------------------------------------
# peaks
# ---------------------------------------------------------------------------------------------


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "tflops": p["bf16_tflops"],
                "tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample (also the correctness gate for the sampled rows)
# ---------------------------------------------------------------------------------------------


def _u16(t):
    import numpy as np
    import torch

    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_sample_plan(budget_flops: float):
    """Rows of each sweep size the oracle computes, about budget_flops in total."""
    per = budget_flops / len(SWEEP)
    plan = []
    for n in SWEEP:
        rows = int(max(1, min(n, round(per / (2.0 * n * n)))))
        plan.append((n, rows))
    return plan


def cpu_baseline_leg(host_inputs, gpu_outputs, budget_flops, check=True):
    """Time the oracle on sampled rows of every GEMM and on one full decode of each arm.

    host_inputs: {n: (A, B)} CPU fp16 tensors, plus "dec_bf16": (x, W), "dec_q8": (x, q, s)
    gpu_outputs: {n: C (CPU fp16 tensor)}, "dec_bf16": y, "dec_q8": y (CPU fp32) or None
    Returns (baseline dict, gate dict).
    """
    import numpy as np

    import oracle

    threads = oracle.max_threads()
    flops = 0.0
    seconds = 0.0
    worst = 0.0
    gate_ok = True
    parts = []
    for n, rows in oracle_sample_plan(budget_flops):
        A, B = host_inputs[n]
        sel = np.linspace(0, n - 1, rows).round().astype(np.int64) if rows < n else None
        t0 = time.perf_counter()
        ref = oracle.gemm(_u16(A), _u16(B), rows=sel)
        seconds += time.perf_counter() - t0
        flops += gemm_flops(ref.shape[0], n, n)
        parts.append(f"{n}^3:{ref.shape[0]} rows")
        if check and gpu_outputs is not None:
            C = gpu_outputs[n].double().numpy()
            got = C if sel is None else C[sel]
            err = np.abs(got - ref).max()
            rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
            worst = max(worst, err / (1e-3 * math.sqrt(n)))
            if not (np.isfinite(got).all() and err <= 1e-3 * math.sqrt(n) and rel <= 1e-3):
                gate_ok = False
    x, W = host_inputs["dec_bf16"]
    t0 = time.perf_counter()
    yb = oracle.gemv_bf16(_u16(x), _u16(W))
    x, q, s = host_inputs["dec_q8"]
    yq = oracle.gemv_q8(_u16(x), q.numpy(), _u16(s))
    seconds += time.perf_counter() - t0
    flops += 2 * 2.0 * DEC_K * DEC_N
    parts.append("decode bf16+q8 full")
    if check and gpu_outputs is not None:
        for key, ref in (("dec_bf16", yb), ("dec_q8", yq)):
            got = gpu_outputs[key].double().numpy()
            err = np.abs(got - ref).max()
            rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
            worst = max(worst, err / (1e-3 * math.sqrt(DEC_K)))
            if not (np.isfinite(got).all() and err <= 1e-3 * math.sqrt(DEC_K) and rel <= 1e-3):
                gate_ok = False
    baseline = {"value": flops / seconds / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": "; ".join(parts) + f" ({flops / 1e9:.1f} GFLOP, {seconds:.1f} s, fp64 C oracle)"}
    # the same oracle on one thread, on 32 evenly spaced rows of the 2048^3 product
    n1 = 2048 if 2048 in host_inputs else max(k for k in host_inputs if isinstance(k, int))
    A, B = host_inputs[n1]
    sel = np.linspace(0, n1 - 1, 32).round().astype(np.int64)
    t0 = time.perf_counter()
    oracle.gemm(_u16(A), _u16(B), rows=sel, threads=1)
    t1 = time.perf_counter() - t0
    baseline["one_thread"] = {"value": gemm_flops(32, n1, n1) / t1 / 1e12, "unit": "TFLOP/s",
                              "sample": f"{n1}^3: 32 rows ({gemm_flops(32, n1, n1) / 1e9:.2f} GFLOP, {t1:.2f} s)"}
    gate = {"passed": gate_ok, "worst_err_over_bound": worst} if check else None
    return baseline, gate


# ---------------------------------------------------------------------------------------------
# the default step on the GPU
# ---------------------------------------------------------------------------------------------


def make_host_inputs(rank=0):
    import torch

    from shape_driven_tile_gb300 import inputs

    host = {}
    for n in SWEEP:
        host[n] = (inputs.uniform((n, n), seed=inputs.seed_for(1, 0, base=1000 * rank)),
                   inputs.uniform((n, n), seed=inputs.seed_for(1, 1, base=1000 * rank)))
    x = inputs.uniform((DEC_K,), seed=inputs.seed_for(3, 0, base=1000 * rank), dtype=torch.bfloat16)
    Wb = [inputs.uniform((DEC_N, DEC_K), seed=inputs.seed_for(3, 1, base=1000 * rank + 17 * i),
                         dtype=torch.bfloat16) for i in range(DEC_BUFFERS)]
    Q = [inputs.q8_weights(DEC_N, DEC_K, seed=inputs.seed_for(3, 1, base=1000 * rank + 17 * i + 5))
         for i in range(DEC_BUFFERS)]
    host["dec_bf16"] = (x, Wb[0])
    host["dec_q8"] = (x, Q[0][0], Q[0][1])
    return host, x, Wb, Q


def run_default(args):
    import torch

    import shape_driven_tile_gb300 as sdt

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    world, rank = dist_init("nccl")
    peaks = load_peaks()
    state_before = gpu_state(local)

    host, x_h, Wb_h, Q_h = make_host_inputs(rank)
    A = {n: host[n][0].to(dev) for n in SWEEP}
    B = {n: host[n][1].to(dev) for n in SWEEP}
    C = {n: torch.empty((n, n), dtype=torch.float16, device=dev) for n in SWEEP}
    x = x_h.to(dev)
    Wb = [w.to(dev) for w in Wb_h]
    Wq = [q.to(dev) for q, _ in Q_h]
    Sq = [s.to(dev) for _, s in Q_h]
    yb = torch.empty(DEC_N, dtype=torch.float32, device=dev)
    yq = torch.empty(DEC_N, dtype=torch.float32, device=dev)
    tiles = {n: sdt.tile_info(sdt.pick_tile(n, n, n))["name"] for n in SWEEP}
    stream = torch.cuda.current_stream()
    # The GEMMs are gemm_f16_ws calls with one workspace: a two-CTA tile may then split the
    # contraction of a partly empty last round (here 4096^3, and 8192^3 and 12288^3 of the
    # large leg); --gemm-ws off makes them plain gemm_f16 calls.
    gws = sdt.gemm_workspace(dev) if args.gemm_ws == "on" else None
    # The timed loop calls the C ABI directly with the operands' device pointers, so that
    # Python-side argument checks do not leave the GPU idle between the small GEMMs.
    L = sdt.lib()
    gemv_b, gemv_q = L.gemv_m1_bf16, L.gemv_m1_q8
    wsa = (gws.data_ptr(), gws.numel()) if gws is not None else None
    gemm_c = L.gemm_f16_ws if gws is not None else L.gemm_f16

    def launch_args(sp, ws=True):
        # launches on a side stream get no workspace: calls that share one must not overlap
        w = (wsa if ws else (None, 0)) if gws is not None else ()
        return ([(n, n, n, A[n].data_ptr(), B[n].data_ptr(), C[n].data_ptr(), *w, sp) for n in SWEEP],
                [(DEC_K, DEC_N, x.data_ptr(), w.data_ptr(), yb.data_ptr(), sp) for w in Wb],
                [(DEC_K, DEC_N, x.data_ptr(), q.data_ptr(), s_.data_ptr(), yq.data_ptr(), sp) for q, s_ in zip(Wq, Sq)])

    args_on = {stream.cuda_stream: launch_args(stream.cuda_stream)}
    dom_j = len(SWEEP) - 1  # the 4096^3 launch: largest share of the step

    def step(i, ev=None, on=None):
        # ev: events around every launch (instrumented step).  Any event between two
        # launches stops the second from overlapping its set-up with the first
        # (programmatic dependent launch), so most timed steps carry no events.
        # on: the stream the launches go to (a capturing stream for the graphs).
        on = on or stream
        gemm_args, pb, pq = args_on.setdefault(on.cuda_stream, launch_args(on.cuda_stream))
        rc = 0
        for j, a in enumerate(gemm_args):
            if ev is not None:
                ev[j].record(on)
            rc |= gemm_c(*a)
        if ev is not None:
            ev[len(SWEEP)].record(on)
        rc |= gemv_b(*pb[i % DEC_BUFFERS])
        if ev is not None:
            ev[len(SWEEP) + 1].record(on)
        rc |= gemv_q(*pq[i % DEC_BUFFERS])
        if ev is not None:
            ev[len(SWEEP) + 2].record(on)
        if rc:
            raise sdt.SdtError(rc, (L.sdt_last_error() or b"").decode())

    # Concurrent form of a step (graph-replayed steps, --concurrent-steps): the four small GEMMs
    # (<= 1024^3, 8 to 144 CTAs each, launch-bound) on one side stream and the two
    # decode GEMVs on another, beside the large GEMMs on the main stream -- a fork and
    # a join per step.  The launches and buffers are the serial step's; only their
    # order on the device changes (the problems are independent).
    SMALL = [n for n in SWEEP if n <= 1024]
    side_small = torch.cuda.Stream(device=dev)
    side_dec = torch.cuda.Stream(device=dev)

    def step_concurrent(i, on):
        fork = torch.cuda.Event()
        fork.record(on)
        side_small.wait_event(fork)
        side_dec.wait_event(fork)
        g_main, _, _ = args_on.setdefault(on.cuda_stream, launch_args(on.cuda_stream))
        g_small, _, _ = args_on.setdefault(side_small.cuda_stream, launch_args(side_small.cuda_stream, ws=False))
        _, pb, pq = args_on.setdefault(side_dec.cuda_stream, launch_args(side_dec.cuda_stream))
        rc = 0
        for j, n in enumerate(SWEEP):
            if n in SMALL:
                rc |= gemm_c(*g_small[j])
        rc |= gemv_b(*pb[i % DEC_BUFFERS])
        rc |= gemv_q(*pq[i % DEC_BUFFERS])
        for j, n in enumerate(SWEEP):
            if n not in SMALL:
                rc |= gemm_c(*g_main[j])
        for side in (side_small, side_dec):
            join = torch.cuda.Event()
            join.record(side)
            on.wait_event(join)
        if rc:
            raise sdt.SdtError(rc, (L.sdt_last_error() or b"").decode())

    launches_per_step = len(SWEEP) + 2
    t_warm = time.perf_counter()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    warmup_s = time.perf_counter() - t_warm
    sdt.check_device_status()

    # correctness gate + CPU baseline (rank 0): results of one step vs the oracle on the sample
    gate, baseline = None, None
    if rank == 0:
        step(0)
        torch.cuda.synchronize()
        outs = {n: C[n].cpu() for n in SWEEP}
        outs["dec_bf16"] = yb.cpu()
        outs["dec_q8"] = yq.cpu()
        calib, _ = cpu_baseline_leg(host, None, budget_flops=2e9, check=False)
        budget = min(args.cpu_budget_s * calib["value"] * 1e12, 400e9)
        baseline, gate = cpu_baseline_leg(host, outs, budget_flops=budget)
        if not gate["passed"]:
            print(json.dumps({"metric": METRIC, "error": "correctness gate failed", "gate": gate}))
            sys.exit(3)

    # timed region: every INSTR-th step is instrumented around every launch
    INSTR = 10
    nev = launches_per_step + 1
    plan = step_schedule(args.steps, INSTR, DEC_BUFFERS, graphed=not args.no_graph)
    inst_idx = [first for kind, first, _ in plan if kind == "instrumented"]
    events = {i: [torch.cuda.Event(enable_timing=True) for _ in range(nev)] for i in inst_idx}
    # The other nine steps in ten carry no events at all, so their launches overlap
    # through programmatic dependent launch, and they run as one CUDA graph of nine
    # steps (captured once per decode-buffer offset), so no host launch gap lands
    # between them; the dominant kernel's duration comes from the instrumented steps.
    graphs = {}
    for kind, first, _ in plan:
        if kind == "graph" and first % DEC_BUFFERS not in graphs:
            cap = torch.cuda.Stream(device=dev)
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                for j in range(INSTR - 1):
                    if args.concurrent_steps:
                        step_concurrent(first + j, cap)
                    else:
                        step(first + j, on=cap)
            stream.wait_stream(cap)
            graphs[first % DEC_BUFFERS] = g
    if graphs:
        torch.cuda.synchronize()
        for g in graphs.values():  # one untimed replay each
            g.replay()
        torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        # clock warm-up right before the timed region (the oracle leg above left the GPU
        # idle): whole steps back to back for at least --clock-warmup-s seconds
        warm_graph = graphs.get(0)
        clock_warm_s = warm_for(args.clock_warmup_s, (lambda: warm_graph.replay()) if warm_graph is not None
                                else (lambda: step(0)))
        barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for kind, first, count in plan:
            if kind == "instrumented":
                step(first, events[first])
            elif kind == "graph":
                graphs[first % DEC_BUFFERS].replay()  # steps first .. first+count-1, same buffers
            else:
                step(first)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier()
    elapsed_s = start.elapsed_time(stop) / 1e3
    sdt.check_device_status()
    max_s = max_over_ranks(elapsed_s, device=dev)

    # per-kernel durations from the events inside the timed region
    per = {n: [] for n in SWEEP}
    dec_b, dec_q = [], []
    for ev in events.values():
        for j, n in enumerate(SWEEP):
            per[n].append(ev[j].elapsed_time(ev[j + 1]))
        dec_b.append(ev[len(SWEEP)].elapsed_time(ev[len(SWEEP) + 1]))
        dec_q.append(ev[len(SWEEP) + 1].elapsed_time(ev[len(SWEEP) + 2]))
    dom_ms = per[SWEEP[dom_j]]

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    e2e = run_e2e(args, dev, host, Wb_h, Q_h, stream, gws)

    # the decode protocol (after the timed region): 200 back-to-back launches x 10 repeats
    dec_proto = None
    ev_cost = event_pair_cost(stream, dev) if rank == 0 else None
    if rank == 0:
        with ClockSampler(local) as dclk:
            dec_proto = decode_protocol(x, Wb, Wq, Sq, yb, peaks, stream)
        dec_proto["clocks"] = dclk.summary()

    # the configurations' own protocols (after the timed region, rank 0)
    legs = run_legs(L, A, B, C, tiles, peaks, stream, dev, local, wsa) if rank == 0 and not args.no_legs else {}
    if rank == 0:
        sdt.check_device_status()
    state_after = gpu_state(local)

    if rank != 0:
        return
    value = aggregate_value(step_flops(), args.steps, world, max_s) / 1e12
    per_size = []
    for n in SWEEP:
        ms = statistics.mean(per[n])
        tf = gemm_flops(n, n, n) / (ms / 1e3) / 1e12
        per_size.append({"size": n, "tile": tiles[n], "us": round(ms * 1e3, 2), "tflops": round(tf, 1),
                         "pct_peak": round(100 * tf / peaks["tflops"], 1)})
    dec = {}
    for name, lst, fmt in (("bf16", dec_b, "bf16"), ("q8", dec_q, "q8")):
        us = statistics.mean(lst) * 1e3
        gbs = decode_bytes(DEC_K, DEC_N, fmt) / (us / 1e6) / 1e9
        dec[name] = {"us": round(us, 2), "us_min": round(min(lst) * 1e3, 2), "us_max": round(max(lst) * 1e3, 2),
                     "gbs": round(gbs, 1), "pct_hbm": round(100 * gbs / peaks["hbm_gbs"], 1)}
    # dominant kernel: the largest share of the step, timed in every step
    shares = {n: statistics.mean(per[n]) for n in SWEEP}
    dom = SWEEP[dom_j]
    largest_share = max(shares, key=shares.get)  # 4096 in every unprofiled run so far
    achieved = gemm_flops(dom, dom, dom) / (statistics.mean(dom_ms) / 1e3) / 1e12
    traffic = load_traffic(f"gemm_{dom}")
    clock = clocks.summary()
    gemm_name = "gemm_f16_ws" if gws is not None else "gemm_f16"
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_s * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (step working set %.0f MB, L2 129 MB)"
                   % (step_working_set() / 1e6), "parallelism": f"replicas x{world}"},
        "timing": {"per_size_and_decode": f"instrumented steps (every {INSTR}th, queued behind a graph replay, "
                   "events around every launch; a decode launch there follows the GEMMs, so it cannot overlap a "
                   "previous decode)",
                   "roofline": f"events around the 4096^3 launch in the instrumented steps ({len(inst_idx)} of "
                               f"{args.steps}); the other steps carry no events",
                   "launch": "eager" if args.no_graph else "instrumented steps eager, the nine steps before "
                             "each of them replayed as one CUDA graph",
                   "concurrency": "serial" if (not args.concurrent_steps or args.no_graph) else
                                  "graph-replayed steps: the GEMMs up to 1024^3 and the two decode GEMVs on two side "
                                  "streams beside the larger GEMMs (fork and join per step); instrumented steps serial",
                   "clock_warmup": f"{clock_warm_s:.2f} s of whole steps right before the timed region",
                   "clocks": "nvidia-smi every 50 ms over the clock warm-up and the timed region",
                   "event_pair_around_one_element_fill_us": ev_cost},
        "roofline": {"bound": "tensor", "kernel": f"{gemm_name} {dom}^3 ({tiles[dom]}{last_round_note(dom, tiles[dom], gws)})",
                     "largest_share_in_step": f"{gemm_name} {largest_share}^3",
                     "achieved": round(achieved, 1), "peak": peaks["tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["tflops"], 4), "peak_source": peaks["source"] + " bf16 burst",
                     "peak_sustained": peaks["tflops_sustained"],
                     "frac_sustained": round(achieved / peaks["tflops_sustained"], 4),
                     "traffic": traffic, **({"traffic_note": traffic_note(f"gemm_{dom}")} if traffic is None else {})},
        "cpu_baseline": baseline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clock,
        "roofline_decode": {
            "bound": "hbm", "kernel": "gemv_m1 bf16 and q8, K=4096 N=12288 (decode protocol, best repeat)",
            "achieved": {a: dec_proto[a]["gbs_best"] for a in ("bf16", "q8")}, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": {a: round(dec_proto[a]["gbs_best"] / peaks["hbm_gbs"], 4) for a in ("bf16", "q8")},
            "peak_source": peaks["source"] + " copy bandwidth",
            "traffic": {a: load_traffic(f"gemv_{a}") for a in ("bf16", "q8")}},
        "per_size": per_size,
        "decode": dec,
        "decode_protocol": dict(dec_proto, protocol="1 s warm, 200 graph-replayed launches x 10 repeats, "
                                "8 rotating buffers, after the timed region"),
        **legs,
        "gate": gate,
        "receipt": receipt(dev, warmup_s, clock_warm_s, state_before, state_after),
    }
    print(json.dumps(out), flush=True)


def event_pair_cost(stream, dev, reps=50):
    """What an event pair costs around a launch on this GPU: min and median of `reps` pairs
    of timing events around a one-element fill kernel (after the timed region).  Every
    launch of an instrumented step carries such a pair, so this is the part of the per-size
    and decode figures there that is launch and event latency rather than the kernel."""
    import torch

    t = torch.empty(1, device=dev)
    for _ in range(5):
        t.fill_(1.0)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    for e0, e1 in pairs:
        e0.record(stream)
        t.fill_(1.0)
        e1.record(stream)
    torch.cuda.synchronize()
    us = sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in pairs)
    return {"min": round(us[0], 2), "median": round(us[len(us) // 2], 2)}


def step_schedule(steps, instr, buffers, graphed=True):
    """How the timed steps run: a list of (kind, first step, count) in step order.
    Every `instr`-th step (instr-1, 2 instr-1, ...; the last step when there are fewer
    than instr) is "instrumented" (events around each launch); the instr-1 steps before
    each of them are one "graph" replay (a graph captured once per first-step decode
    buffer, first % buffers), so an instrumented step is queued behind a replay and its
    first launch does not wait for the host; anything else is an "eager" step.  Each
    step index appears exactly once."""
    inst = {i for i in range(steps) if i % instr == instr - 1} or ({steps - 1} if steps else set())
    plan, i = [], 0
    while i < steps:
        if i in inst:
            plan.append(("instrumented", i, 1))
            i += 1
        elif graphed and i % instr == 0 and i + instr - 1 in inst:
            plan.append(("graph", i, instr - 1))
            i += instr - 1
        else:
            plan.append(("eager", i, 1))
            i += 1
    return plan


def receipt(dev, warmup_s, clock_warmup_s=None, before=None, after=None):
    """What the numbers were measured on: device, driver, runtime, library sources, the
    warm-up, and the GPU's temperature, power and clocks before and after the run."""
    import torch

    import shape_driven_tile_gb300 as sdt

    props = torch.cuda.get_device_properties(dev)
    driver = None
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                            f"--id={dev.index or 0}"], capture_output=True, text=True, timeout=20)
        driver = r.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    return {"gpu": props.name, "sm_count": sdt.device_sm_count(), "driver": driver,
            "cuda_runtime": torch.version.cuda, "torch": torch.__version__,
            "kernel_sources": {k: kernel_source_digest(k) for k in SOURCES},
            "warmup_s": round(warmup_s, 3),
            "clock_warmup_s": None if clock_warmup_s is None else round(clock_warmup_s, 3),
            "gpu_before": before, "gpu_after": after, "host_cores": len(os.sched_getaffinity(0))}


def step_working_set():
    gemm = sum(3 * 2 * n * n for n in SWEEP)
    dec = DEC_BUFFERS * (decode_weight_bytes(DEC_K, DEC_N, "bf16") + decode_weight_bytes(DEC_K, DEC_N, "q8"))
    return gemm + dec


SOURCES = {  # the CUDA sources each recorded kernel is built from
    "gemm": lambda name: name.startswith("gemm") or name in ("ptx.cuh", "launch.cuh"),
    "gemv": lambda name: name in ("gemv.cu", "ptx.cuh", "launch.cuh"),
}


def kernel_source_digest(kind="gemm"):
    """Digest of the CUDA sources of one kernel family; recorded ncu traffic is stale once it changes."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "shape_driven_tile_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")) and SOURCES[kind](name):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def load_traffic(kernel_key):
    """DRAM bytes per launch from an ncu capture (profiles/traffic.json), or None when the
    record is missing or was taken on different kernel sources."""
    if not os.path.exists(TRAFFIC):
        return None
    with open(TRAFFIC) as f:
        t = json.load(f)
    e = t.get(kernel_key)
    kind = kernel_key.split("_")[0]
    if not isinstance(e, dict) or kind not in SOURCES or e.get("source_digest") != kernel_source_digest(kind):
        return None
    return e.get("bytes")


def traffic_note(kernel_key):
    """Why load_traffic gave None: no record, or a record taken on other sources (its
    digest beside the current one); None when the record is in use."""
    if load_traffic(kernel_key) is not None:
        return None
    kind = kernel_key.split("_")[0]
    e = None
    if os.path.exists(TRAFFIC):
        with open(TRAFFIC) as f:
            e = json.load(f).get(kernel_key)
    if not isinstance(e, dict):
        return "no ncu record for this launch"
    return (f"the ncu record ({e.get('bytes')} bytes) was taken on sources {e.get('source_digest')}; "
            f"the current ones are {kernel_source_digest(kind)}")


def record_traffic(args):
    """Store the DRAM bytes of one launch from an ncu CSV (--metrics dram__bytes_read.sum,
    dram__bytes_write.sum, one captured launch) under --key in profiles/traffic.json, with
    the digest of the sources the kernel was built from."""
    import csv

    with open(args.ncu_csv) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rows = list(csv.DictReader(lines))
    vals, kernel = {}, None
    for r in rows:
        name, unit, v = r.get("Metric Name"), r.get("Metric Unit", ""), r.get("Metric Value", "")
        if name in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(unit, 1)
            vals[name] = float(v.replace(",", "")) * scale
            kernel = r.get("Kernel Name")
    if len(vals) != 2:
        raise SystemExit(f"{args.ncu_csv}: no dram__bytes_read/write.sum rows")
    t = {}
    if os.path.exists(TRAFFIC):
        with open(TRAFFIC) as f:
            t = json.load(f)
    kind = args.key.split("_")[0]
    t[args.key] = {"bytes": int(round(vals["dram__bytes_read.sum"] + vals["dram__bytes_write.sum"])),
                   "read": int(round(vals["dram__bytes_read.sum"])), "write": int(round(vals["dram__bytes_write.sum"])),
                   "kernel": (kernel or "")[:120], "source_digest": kernel_source_digest(kind),
                   "how": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one launch: " + args.ncu_csv}
    with open(TRAFFIC, "w") as f:
        json.dump(t, f, indent=1)
    print(json.dumps({"mode": "record-traffic", args.key: t[args.key]}))


def last_round_note(n, tile, gws):
    """How a two-CTA tile runs the last round of an n^3 launch (empty for other tiles)."""
    import shape_driven_tile_gb300 as sdt

    if not tile.startswith("2cta"):
        return ""
    ts, items, sp, long_k = sdt.pair_tail_plan(n, n, n, tile, sdt.device_sm_count(),
                                               sdt.lib().sdt_device_smem_optin(), workspace=gws is not None)
    if items == ts:
        return ""
    if sp:
        return f"; last round: {(items - ts) // sp} tiles x {sp} k-ranges (split 0: {long_k} k-tiles)"
    return f"; last round: {(items - ts) // 2} tiles as half-width items"


def _packed(specs, make):
    """One buffer (make(nbytes) -> uint8 tensor) holding tensors of the given shapes and
    dtypes at 256-byte aligned offsets; returns the buffer and a view per key."""
    import torch

    offs, total = {}, 0
    for key, shape, dtype in specs:
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        offs[key] = (total, nbytes, shape, dtype)
        total += (nbytes + 255) // 256 * 256
    buf = make(total)
    return buf, {key: buf[o:o + nb].view(dtype).view(shape) for key, (o, nb, shape, dtype) in offs.items()}


def run_e2e(args, dev, host, Wb_h, Q_h, stream, gws=None):
    """Same metric through the public API with pinned host buffers: every step copies its
    inputs host -> device, runs the step and copies every result device -> host, all inside
    the timed region.  A step's inputs sit in one pinned staging buffer and go over in one
    copy, its results come back in one copy, as a serving loop that batches its transfers
    would run it; the copies of neighbouring steps overlap the compute on three streams
    (inputs of step i+1 in, step i computed, results of step i-1 out), each with two
    buffer sets ordered by events."""
    import torch

    import shape_driven_tile_gb300 as sdt

    steps = max(3, min(args.steps, args.e2e_steps))
    x_h = host["dec_bf16"][0]
    in_specs = ([(("A", n), (n, n), torch.float16) for n in SWEEP] + [(("B", n), (n, n), torch.float16) for n in SWEEP]
                + [("x", tuple(x_h.shape), x_h.dtype), ("W", tuple(Wb_h[0].shape), Wb_h[0].dtype),
                   ("q", tuple(Q_h[0][0].shape), Q_h[0][0].dtype), ("s", tuple(Q_h[0][1].shape), Q_h[0][1].dtype)])
    out_specs = [(("C", n), (n, n), torch.float16) for n in SWEEP] + [("yb", (DEC_N,), torch.float32),
                                                                      ("yq", (DEC_N,), torch.float32)]
    pinned = lambda nbytes: torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    on_dev = lambda nbytes: torch.empty(nbytes, dtype=torch.uint8, device=dev)
    # host inputs: two staging buffers (the decode weights alternate between two sets)
    hin = []
    for k in range(2):
        buf, v = _packed(in_specs, pinned)
        for n in SWEEP:
            v[("A", n)].copy_(host[n][0])
            v[("B", n)].copy_(host[n][1])
        v["x"].copy_(x_h)
        v["W"].copy_(Wb_h[k])
        v["q"].copy_(Q_h[k][0])
        v["s"].copy_(Q_h[k][1])
        hin.append(buf)
    sets = []
    for _ in range(2):
        din, dv = _packed(in_specs, on_dev)
        dout, ov = _packed(out_specs, on_dev)
        hout, hv = _packed(out_specs, pinned)
        sets.append({"din": din, "dv": dv, "dout": dout, "ov": ov, "hout": hout, "hv": hv,
                     # step i's input copy done / compute done / result copy done
                     "in": torch.cuda.Event(), "comp": torch.cuda.Event(), "out": torch.cuda.Event()})
    h2d = hin[0].numel()
    d2h = sets[0]["dout"].numel()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s_c = stream

    def e2e_step(i):
        b = sets[i % 2]
        dv, ov = b["dv"], b["ov"]
        with torch.cuda.stream(s_in):
            s_in.wait_event(b["comp"])  # step i-2 no longer reads this set's inputs
            b["din"].copy_(hin[i % 2], non_blocking=True)
            b["in"].record(s_in)
        s_c.wait_event(b["in"])
        s_c.wait_event(b["out"])  # step i-2's results have left this set's outputs
        for n in SWEEP:
            if gws is None:
                sdt.gemm_f16(dv[("A", n)], dv[("B", n)], ov[("C", n)], stream=s_c)
            else:
                sdt.gemm_f16_ws(dv[("A", n)], dv[("B", n)], ov[("C", n)], workspace=gws, stream=s_c)
        sdt.gemv_m1(dv["x"], dv["W"], y=ov["yb"], stream=s_c)
        sdt.gemv_m1(dv["x"], dv["q"], dv["s"], y=ov["yq"], stream=s_c)
        b["comp"].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["comp"])
            b["hout"].copy_(b["dout"], non_blocking=True)
            b["out"].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        e2e_step(i)
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    barrier()
    # the last step's results against a device-only run of the same step
    last = sets[(steps - 1) % 2]
    ref = {n: torch.empty((n, n), dtype=torch.float16, device=dev) for n in SWEEP}
    for n in SWEEP:
        if gws is None:
            sdt.gemm_f16(last["dv"][("A", n)], last["dv"][("B", n)], ref[n])
        else:
            sdt.gemm_f16_ws(last["dv"][("A", n)], last["dv"][("B", n)], ref[n], workspace=gws)
    torch.cuda.synchronize()
    ok = all(torch.equal(last["hv"][("C", n)], ref[n].cpu()) for n in SWEEP)
    world = dist_env()[0]
    max_s = max_over_ranks(secs, device=dev)
    return {"value": round(aggregate_value(step_flops(), steps, world, max_s) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(max_s * 1e3 / steps, 3), "results_match_device_run": ok,
            "overlap": "inputs of step i+1 in, step i computed, results of step i-1 out, on three streams; one "
                       "copy each way per step (the step's inputs and results in one pinned staging buffer each)"}


# ---------------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------------------------


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    host, _, _, _ = make_host_inputs(0)
    # size each step so that warmup + steps stay within about three minutes
    calib_flops = 2e9
    base, _ = cpu_baseline_leg(host, None, calib_flops, check=False)
    per_step_s = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    budget = max(2e8, per_step_s * base["value"] * 1e12)
    for _ in range(args.warmup):
        cpu_baseline_leg(host, None, budget, check=False)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        b, _ = cpu_baseline_leg(host, None, budget, check=False)
        vals.append(b)
    secs = time.perf_counter() - t0
    value = statistics.mean(b["value"] for b in vals)
    out = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / max(1, args.steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD + " -- oracle on a bounded sample per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": vals[0]["cores"], "kind": "oracle",
                         "sample": vals[0]["sample"]},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------------------------
# measurement modes
# ---------------------------------------------------------------------------------------------


def L2Flush(dev):
    """A read of 4x the L2 size before each timed launch (shape_driven_tile_gb300.tune.L2Flush)."""
    from shape_driven_tile_gb300 import tune

    return tune.L2Flush(dev)


def time_cold(fn, reps, flush, stream):
    """Mean device time of fn over reps launches, each after an L2 flush (events bracket fn only)."""
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    ts = [e0.elapsed_time(e1) for e0, e1 in evs]
    return statistics.mean(ts), min(ts), max(ts)


def run_sweep(args):
    """Every feasible tile per square size (plus K-scan shapes); pick_tile's slowdown."""
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    peaks = load_peaks()
    shapes = [(n, n, n) for n in (args.sizes or SWEEP)]
    if args.with_kscan:
        shapes += [(2048, 2048, k) for k in KSCAN if k != 2048]
    for sh in args.shapes or []:
        M, N, K = (int(v) for v in sh.lower().split("x"))
        shapes.append((M, N, K))
    # bring the clocks up before the first (smallest, launch-bound) shape is timed
    W = (torch.rand((4096, 4096), device=dev) * 2 - 1).half()
    Wc = torch.empty_like(W)
    t_end = time.time() + 1.0
    while time.time() < t_end:
        for _ in range(20):
            sdt.gemm_f16(W, W, Wc)
        torch.cuda.synchronize()
    del W, Wc
    rows = load_resume(args.resume, shapes)
    done = {tuple(r["shape"]) for r in rows}
    for (M, N, K) in shapes:
        if (M, N, K) in done:
            continue
        A = (torch.rand((M, K), device=dev) * 2 - 1).half()
        B = (torch.rand((K, N), device=dev) * 2 - 1).half()
        C = torch.empty((M, N), device=dev, dtype=torch.float16)
        res = {}
        feas = sdt.feasible_tiles(M, N, K)
        for t in feas:
            for _ in range(3):
                sdt.gemm_f16_with_tile(A, B, C, tile=t)
        # three passes over the tiles, each in a fresh shuffled order; a tile keeps its best
        # pass mean, so the device's drift does not favour whichever tile is timed first
        rng = random.Random(M * 1000003 + N * 1009 + K)
        order = list(feas)
        for _ in range(3):
            rng.shuffle(order)
            for t in order:
                name = sdt.tile_info(t)["name"]
                mean, lo, hi = time_cold(lambda: sdt.gemm_f16_with_tile(A, B, C, tile=t),
                                         max(1, args.reps // 3), flush, stream)
                res[name] = min(mean, res.get(name, mean))
        pick = sdt.tile_info(sdt.pick_tile(M, N, K))["name"]
        best = min(res, key=res.get)
        fl = gemm_flops(M, N, K)
        rows.append({"shape": [M, N, K], "pick": pick, "best": best,
                     "slowdown": round(res[pick] / res[best] - 1, 4),
                     "tflops": {k: round(fl / (v / 1e3) / 1e12, 1) for k, v in res.items()},
                     "us": {k: round(v * 1e3, 2) for k, v in res.items()}})
        print(json.dumps(rows[-1]), flush=True)
        append_resume(args.resume, rows[-1])
        del A, B, C
    sdt.check_device_status()
    if args.table_out:
        write_tune_table(args.table_out, [(*r["shape"], {"tile": r["best"]}) for r in rows], "the tile sweep")
    slow = [r["slowdown"] for r in rows]
    print(json.dumps({"mode": "sweep", "shapes": len(rows), "pick_avg_slowdown": round(statistics.mean(slow), 4),
                      "pick_worst_slowdown": round(max(slow), 4), "peak_tflops": peaks["tflops"],
                      "timing": f"best of 3 shuffled passes, each the mean of {max(1, args.reps // 3)} launches "
                                "with L2 flushed before each"}), flush=True)


def load_resume(path, shapes):
    """Rows of an interrupted sweep (one JSON object per line, as the sweep prints them)
    for the shapes still asked for; a missing file is an empty start."""
    rows = []
    if not path or not os.path.exists(path):
        return rows
    want = {tuple(sh) for sh in shapes}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line:
                continue
            try:
                r = json.loads(line)
            except json.JSONDecodeError:
                continue  # a line cut short when the run stopped
            if isinstance(r, dict) and tuple(r.get("shape", ())) in want and "us" in r:
                rows.append(r)
    return rows


def append_resume(path, row):
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(row) + "\n")
            f.flush()
            os.fsync(f.fileno())


def run_ktile(args):
    """The per-k-tile time of one CTA: every one-CTA tile on one output tile with a long K
    (65536, 1024 k-tiles), ring depths 4, 8 and the tile's own, cold L2.  A time that does
    not move with the ring depth or the bytes per k-tile is the tensor pipe's pace."""
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    K = 65536
    rows = []
    for t in sdt.tiles():
        if t["cta_group"] != 1 or t["name"].startswith("p"):
            continue
        M, N = (t["BN"], t["BM"]) if t["skinny"] else (t["BM"], t["BN"])
        A = (torch.rand((M, K), device=dev) * 2 - 1).bfloat16()
        B = (torch.rand((N, K), device=dev) * 2 - 1).bfloat16().t()
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        row = {"tile": t["name"], "M": M, "N": N, "K": K,
               "bytes_per_ktile": (t["BM"] + t["BN"]) * 64 * 2}
        for depth in (4, 8, 0):
            os.environ["SDT_STAGES"] = str(depth) if depth else ""
            fn = lambda: sdt.gemm_ex(A, B, C, tile=t["name"])
            fn()
            mean = time_cold(fn, max(3, args.reps // 4), flush, stream)[0]
            row[f"ns_per_ktile_depth{depth or t['stages']}"] = round(mean * 1e6 / (K // 64), 1)
        os.environ.pop("SDT_STAGES", None)
        rows.append(row)
        print(json.dumps(row), flush=True)
        del A, B, C
    sdt.check_device_status()
    print(json.dumps({"mode": "ktile", "rows": len(rows), "timing": "mean of cold launches, L2 flushed before each"}),
          flush=True)


def run_kscan(args):
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    tile = sdt.tile_id(args.tile or "128x128")
    out = []
    for K in KSCAN:
        A = (torch.rand((2048, K), device=dev) * 2 - 1).half()
        B = (torch.rand((K, 2048), device=dev) * 2 - 1).half()
        C = torch.empty((2048, 2048), device=dev, dtype=torch.float16)
        row = {"K": K}
        for st in (0, 1):
            for _ in range(3):
                sdt.gemm_f16_with_tile(A, B, C, tile=tile, stagger=st)
            mean, lo, hi = time_cold(lambda: sdt.gemm_f16_with_tile(A, B, C, tile=tile, stagger=st),
                                     args.reps, flush, stream)
            row[f"stagger{st}_tflops"] = round(gemm_flops(2048, 2048, K) / (mean / 1e3) / 1e12, 1)
        out.append(row)
        print(json.dumps(row), flush=True)
    sdt.check_device_status()
    print(json.dumps({"mode": "kscan", "tile": sdt.tile_info(tile)["name"], "rows": out}), flush=True)


def decode_protocol(x, Wb, Wq, Sq, y, peaks, stream, warm_s=1.0, reps=10, launches=200):
    """The decode protocol of the pages' workload: a warm-up of warm_s seconds, then `reps`
    repeats of `launches` back-to-back launches (captured in a CUDA graph, cycling the
    rotating weight buffers so every launch streams its weights from HBM), timed with
    events on the launching stream.  Returns per arm the min/max per-launch time."""
    import torch

    import shape_driven_tile_gb300 as sdt

    nb = len(Wb)
    res = {}
    for arm in ("bf16", "q8"):
        def launch(i):
            if arm == "bf16":
                sdt.gemv_m1(x, Wb[i % nb], y=y)
            else:
                sdt.gemv_m1(x, Wq[i % nb], Sq[i % nb], y=y)
        t_end = time.time() + warm_s
        i = 0
        while time.time() < t_end:
            launch(i)
            i += 1
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for j in range(launches):
                    launch(j)
        torch.cuda.synchronize()
        times = []
        for r in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / launches)
        del g
        nbytes = decode_bytes(DEC_K, DEC_N, arm)
        res[arm] = {"us_min": round(min(times), 2), "us_max": round(max(times), 2),
                    "gbs_best": round(nbytes / (min(times) / 1e6) / 1e9, 1),
                    "pct_hbm_best": round(100 * nbytes / (min(times) / 1e6) / 1e9 / peaks["hbm_gbs"], 1),
                    "bytes": nbytes}
    return res


# ---------------------------------------------------------------------------------------------
# protocol legs: each configuration measured by the pages' own protocol, after the timed region
# ---------------------------------------------------------------------------------------------


def _chk(rc):
    if rc:
        import shape_driven_tile_gb300 as sdt

        raise sdt.SdtError(rc, (sdt.lib().sdt_last_error() or b"").decode())


def warm_for(seconds, fn):
    """Runs fn() back to back until `seconds` of wall time have passed, synchronising
    after every batch of eight (so the time is GPU time, not queued launches); returns
    the wall time spent."""
    import torch

    t0 = time.perf_counter()
    while True:
        for _ in range(8):
            fn()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if dt >= seconds:
            return dt


def graph_of(launch, count, dev):
    """A CUDA graph of `count` calls launch(i, stream_handle), captured on a side stream."""
    import torch

    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for i in range(count):
            launch(i, cap.cuda_stream)
    torch.cuda.current_stream(dev).wait_stream(cap)
    torch.cuda.synchronize()
    return g


def time_graph(g, count, reps, stream):
    """Per-launch microseconds of each of `reps` replays of a graph of `count` launches
    (CUDA events on `stream`, the stream the replay runs on)."""
    import torch

    out = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / count)
    return out


def gemm_protocol_leg(L, A, B, C, tiles, peaks, stream, dev, launches=200, reps=5, warm_s=1.0, wsa=None):
    """The square sweep by the pages' GEMM protocol ("Beating hipBLASLt on a Gaming GPU",
    "Why these numbers should be trusted"; "mojo-baro", "Square fp16 GEMM vs hipBLASLt"):
    a clock warm-up, then per size `launches` back-to-back launches of gemm_f16 replayed
    from a CUDA graph, `reps` repeats in a shuffled size order, min-max per launch; plus
    one host-issued loop of the same launches between two events (the plain-launch arm
    of the FlyDSL pull request's "Performance")."""
    import torch

    def call(n, sp):
        if wsa is None:
            _chk(L.gemm_f16(n, n, n, A[n].data_ptr(), B[n].data_ptr(), C[n].data_ptr(), sp))
        else:
            _chk(L.gemm_f16_ws(n, n, n, A[n].data_ptr(), B[n].data_ptr(), C[n].data_ptr(), *wsa, sp))

    warm = warm_for(warm_s, lambda: [call(n, stream.cuda_stream) for n in SWEEP])
    graphs = {n: graph_of(lambda i, sp, n=n: call(n, sp), launches, dev) for n in SWEEP}
    times = {n: [] for n in SWEEP}
    rng = random.Random(7)
    for _ in range(reps):
        order = list(SWEEP)
        rng.shuffle(order)
        for n in order:
            times[n] += time_graph(graphs[n], launches, 1, stream)
    eager = {}
    for n in SWEEP:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(launches):
            call(n, stream.cuda_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        eager[n] = e0.elapsed_time(e1) * 1e3 / launches
    del graphs
    rows = []
    for n in SWEEP:
        best = min(times[n])
        tf = gemm_flops(n, n, n) / (best / 1e6) / 1e12
        rows.append({"size": n, "tile": tiles[n], "us_min": round(best, 2), "us_max": round(max(times[n]), 2),
                     "tflops_best": round(tf, 1), "pct_peak_best": round(100 * tf / peaks["tflops"], 1),
                     "eager_us": round(eager[n], 2)})
    return {"rows": rows, "warmup_s": round(warm, 2),
            "protocol": f"{warm_s:g} s warm-up; per size {launches} back-to-back launches replayed from a CUDA graph "
                        f"(every size's operands fit in the 129 MB L2, as in a hot loop), {reps} repeats in shuffled size order, min-max per "
                        f"launch; eager_us: {launches} host-issued launches between two events"}


def large_leg(L, peaks, stream, dev, sizes=None, reps=3, warm_s=1.0, wsa=None):
    """Large squares M=N=K in {8192, 12288, 16384} with pick_tile: a clock warm-up on the
    first size, then per size a CUDA graph of back-to-back launches (about 20 ms) replayed
    `reps` times; operands far larger than L2.  TFLOP/s against the measured burst and
    sustained (power-capped) bf16 peaks."""
    import torch

    import shape_driven_tile_gb300 as sdt

    rows, warm = [], 0.0
    for idx, n in enumerate(sizes or LARGE):
        g = torch.Generator(device=dev).manual_seed(50 + n)
        A = torch.empty((n, n), dtype=torch.float16, device=dev).uniform_(-1, 1, generator=g)
        B = torch.empty((n, n), dtype=torch.float16, device=dev).uniform_(-1, 1, generator=g)
        C = torch.empty((n, n), dtype=torch.float16, device=dev)
        fl = gemm_flops(n, n, n)
        count = max(3, min(20, round(20e-3 / (fl / 1.5e15))))

        def call(sp, n=n, A=A, B=B, C=C):
            if wsa is None:
                _chk(L.gemm_f16(n, n, n, A.data_ptr(), B.data_ptr(), C.data_ptr(), sp))
            else:
                _chk(L.gemm_f16_ws(n, n, n, A.data_ptr(), B.data_ptr(), C.data_ptr(), *wsa, sp))

        if idx == 0:
            warm = warm_for(warm_s, lambda: call(stream.cuda_stream))
        else:
            for _ in range(2):
                call(stream.cuda_stream)
        gr = graph_of(lambda i, sp: call(sp), count, dev)
        us = time_graph(gr, count, reps, stream)
        best = min(us)
        tf = fl / (best / 1e6) / 1e12
        rows.append({"size": n, "tile": sdt.tile_info(sdt.pick_tile(n, n, n))["name"], "us_min": round(best, 1),
                     "us_max": round(max(us), 1), "tflops_best": round(tf, 1),
                     "pct_peak_best": round(100 * tf / peaks["tflops"], 1),
                     "pct_sustained_peak_best": round(100 * tf / peaks["tflops_sustained"], 1),
                     "launches_per_replay": count})
        del gr, A, B, C
        torch.cuda.empty_cache()
    return {"rows": rows, "warmup_s": round(warm, 2),
            "protocol": f"{warm_s:g} s warm-up, per size a graph of back-to-back launches (~20 ms) x {reps} "
                        "repeats, min-max per launch; operands much larger than L2"}


def kscan_leg(L, peaks, stream, dev, tile="128x128", passes=4, launches=8, graph_launches=50, warm_s=1.0):
    """The K-scan of the FlyDSL pull request ("Motivation"; third commit message): M=N=2048,
    K in {1920, 1984, 2048, 2112, 2176, 2304}, one fixed tile, the k-loop stagger off and
    on.  Cold: each launch after an L2 flush, `passes` shuffled passes of `launches`
    launches per setting, best pass mean.  Warm: `graph_launches` back-to-back launches
    replayed from a CUDA graph, best of three."""
    import torch

    import shape_driven_tile_gb300 as sdt

    tid = sdt.tile_id(tile)
    M = N = 2048
    g = torch.Generator(device=dev).manual_seed(31)
    bufs = {}
    for K in KSCAN:
        bufs[K] = (torch.empty((M, K), dtype=torch.float16, device=dev).uniform_(-1, 1, generator=g),
                   torch.empty((K, N), dtype=torch.float16, device=dev).uniform_(-1, 1, generator=g),
                   torch.empty((M, N), dtype=torch.float16, device=dev))

    def call(K, st, sp):
        A, B, C = bufs[K]
        _chk(L.gemm_f16_with_tile(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), sp, tid, st))

    warm = warm_for(warm_s, lambda: [call(K, 1, stream.cuda_stream) for K in KSCAN])
    flush = L2Flush(dev)
    configs = [(K, st) for K in KSCAN for st in (0, 1)]
    cold = {}
    rng = random.Random(11)
    for _ in range(passes):
        rng.shuffle(configs)
        for K, st in configs:
            mean = time_cold(lambda: call(K, st, stream.cuda_stream), launches, flush, stream)[0]
            cold[(K, st)] = min(cold.get((K, st), mean), mean)
    warm_t = {}
    for K, st in configs:
        gr = graph_of(lambda i, sp, K=K, st=st: call(K, st, sp), graph_launches, dev)
        warm_t[(K, st)] = min(time_graph(gr, graph_launches, 3, stream)) / 1e3
        del gr
    rows = []
    for K in KSCAN:
        fl = gemm_flops(M, N, K)
        nK = K // 64
        rows.append({"K": K, "k_tiles": nK, "stagger_applies": nK & (nK - 1) == 0,
                     "cold_tflops": {"off": round(fl / (cold[(K, 0)] / 1e3) / 1e12, 1),
                                     "on": round(fl / (cold[(K, 1)] / 1e3) / 1e12, 1)},
                     "warm_tflops": {"off": round(fl / (warm_t[(K, 0)] / 1e3) / 1e12, 1),
                                     "on": round(fl / (warm_t[(K, 1)] / 1e3) / 1e12, 1)}})
    del bufs, flush
    torch.cuda.empty_cache()
    return {"tile": tile, "rows": rows, "warmup_s": round(warm, 2),
            "protocol": f"{warm_s:g} s warm-up; cold: L2 flushed (512 MB read) before each launch, {passes} shuffled "
                        f"passes x {launches} launches per (K, stagger), best pass mean; warm: {graph_launches} "
                        "graph-replayed launches, best of 3"}


def pick_check_leg(L, A, B, C, tiles, peaks, stream, dev, passes=5, launches=8, warm_s=1.0, kscan=True):
    """pick_tile against every feasible tile on each square size and on the K-scan
    shapes (the FlyDSL pull request's check of pick_tile against the per-shape fastest,
    "Changes" and its first commit message): every feasible tile timed cold (L2 flushed
    before each launch) in `passes` passes of `launches` launches, each pass in a fresh
    shuffled tile order, a tile's time its best pass mean; the pick's slowdown against
    the fastest."""
    import torch

    import shape_driven_tile_gb300 as sdt

    warm = warm_for(warm_s, lambda: [_chk(L.gemm_f16(n, n, n, A[n].data_ptr(), B[n].data_ptr(), C[n].data_ptr(),
                                                     stream.cuda_stream)) for n in SWEEP])
    flush = L2Flush(dev)
    problems = [(n, n, n, A[n], B[n], C[n]) for n in SWEEP]
    if kscan:
        g = torch.Generator(device=dev).manual_seed(71)
        for K in KSCAN:
            if K != 2048:
                problems.append((2048, 2048, K,
                                 torch.empty((2048, K), dtype=torch.float16, device=dev).uniform_(-1, 1, generator=g),
                                 torch.empty((K, 2048), dtype=torch.float16, device=dev).uniform_(-1, 1, generator=g),
                                 torch.empty((2048, 2048), dtype=torch.float16, device=dev)))
    rows = []
    for M, N, K, Am, Bm, Cm in problems:
        feas = sdt.feasible_tiles(M, N, K)
        res = {}
        rng = random.Random(1000 * M + 7 * K)
        order = list(feas)
        for _ in range(passes):
            rng.shuffle(order)
            for t in order:
                fn = lambda t=t: _chk(L.gemm_f16_with_tile(M, N, K, Am.data_ptr(), Bm.data_ptr(), Cm.data_ptr(),
                                                           stream.cuda_stream, t, -1))
                mean = time_cold(fn, launches, flush, stream)[0]
                res[t] = min(res.get(t, mean), mean)
        pick = sdt.pick_tile(M, N, K)
        best = min(res, key=res.get)
        name = lambda t: sdt.tile_info(t)["name"]
        row = {"shape": [M, N, K], "pick": name(pick), "best": name(best),
               "slowdown": round(res[pick] / res[best] - 1, 4),
               "us": {name(t): round(v * 1e3, 2) for t, v in sorted(res.items(), key=lambda kv: kv[1])}}
        if M == N == K:
            row["size"] = M
        rows.append(row)
    del flush, problems
    slow = [r["slowdown"] for r in rows]
    return {"rows": rows, "avg_slowdown": round(statistics.mean(slow), 4), "worst_slowdown": round(max(slow), 4),
            "worst_shape": rows[slow.index(max(slow))]["shape"], "warmup_s": round(warm, 2),
            "protocol": f"{warm_s:g} s warm-up; the square sizes and the K-scan shapes, every feasible tile, L2 "
                        f"flushed (512 MB read) before each launch, {passes} passes x {launches} launches in a fresh "
                        "shuffled tile order per pass, best pass mean per tile"}


def run_legs(L, A, B, C, tiles, peaks, stream, dev, gpu_index, wsa=None):
    """The four protocol legs, each under its own nvidia-smi clock sampler (the GEMM
    protocol and the large squares through gemm_f16_ws with the step's workspace `wsa`
    when one is given, else gemm_f16)."""
    out = {}
    for key, fn in (("gemm_protocol", lambda: gemm_protocol_leg(L, A, B, C, tiles, peaks, stream, dev, wsa=wsa)),
                    ("pick_check", lambda: pick_check_leg(L, A, B, C, tiles, peaks, stream, dev)),
                    ("kscan", lambda: kscan_leg(L, peaks, stream, dev)),
                    ("large", lambda: large_leg(L, peaks, stream, dev, wsa=wsa))):
        t0 = time.perf_counter()
        with ClockSampler(gpu_index) as clk:
            res = fn()
        res["clocks"] = clk.summary()
        res["wall_s"] = round(time.perf_counter() - t0, 2)
        out[key] = res
    return out


def run_decode(args):
    """The decode protocol: 8 rotating buffers, warm-up, 200 timed launches, repeated 10 times."""
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    x = (torch.rand(DEC_K, device=dev) * 2 - 1).bfloat16()
    Wb = [(torch.rand((DEC_N, DEC_K), device=dev) * 2 - 1).bfloat16() for _ in range(DEC_BUFFERS)]
    Wq = [torch.randint(-127, 128, (DEC_N, DEC_K), device=dev, dtype=torch.int8) for _ in range(DEC_BUFFERS)]
    Sq = [(torch.rand((DEC_N, DEC_K // 32), device=dev) * 9e-3 + 1e-3).half() for _ in range(DEC_BUFFERS)]
    y = torch.empty(DEC_N, device=dev)
    res = decode_protocol(x, Wb, Wq, Sq, y, peaks, stream)
    sdt.check_device_status()
    print(json.dumps({"mode": "decode", "K": DEC_K, "N": DEC_N, "hbm_peak_gbs": peaks["hbm_gbs"],
                      "protocol": "1 s warm, 200 graph-replayed launches x 10 repeats, 8 rotating buffers",
                      **res}), flush=True)


def run_p4(args):
    """The GEMM problem matrix of "Iteratively Tuning hipBLASLt TensileLite Kernels"
    ("Experiment Setup": 24 shapes x fp16/bf16 x NN/TN) through gemm_ex with the
    library's pick (one JSON line per problem: latency, tile, roofline fraction);
    with --tune, the monotone coordinate descent of shape_driven_tile_gb300.tune from
    that pick, the latency after every round (the page's Table 2 columns for this
    library's rounds) and the per-round speedups (its Table 3)."""
    import torch

    import shape_driven_tile_gb300 as sdt
    from shape_driven_tile_gb300 import inputs, tune

    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    names = set(args.shapes or [])
    rows = []
    for si, (name, M, N, K) in enumerate(inputs.P4_SHAPES):
        if names and name not in names:
            continue
        for dtype in (torch.float16, torch.bfloat16):
            if args.dtypes and ("f16" if dtype == torch.float16 else "bf16") not in args.dtypes:
                continue
            for layout in ("NN", "TN"):
                if args.layouts and layout not in args.layouts:
                    continue
                A_h, B_h = inputs.p4_operands(M, N, K, layout, seed=inputs.seed_for(6 + si, 0), dtype=dtype)
                A = A_h.to(dev)
                B = B_h.to(dev) if layout == "NN" else B_h.to(dev).t()
                C = torch.empty((M, N), dtype=dtype, device=dev)
                prob = tune.GemmProblem(A, B, C, reps=args.reps)
                start = prob.start()
                if args.tile:  # a given configuration instead of the library's pick
                    start = dict(tune.DEFAULTS, tile=sdt.tile_id(args.tile), splits=args.splits, algo=args.algo)
                row = {"shape": name, "M": M, "N": N, "K": K, "dtype": "f16" if dtype == torch.float16 else "bf16",
                       "layout": layout, "pick": sdt.tile_info(start["tile"])["name"]}
                if args.tile:
                    row["config"] = {"tile": args.tile, "splits": args.splits, "algo": args.algo}
                if args.tune:
                    held, traj = prob.tune()
                    row["rounds"] = {t["round"]: round(t["us"], 2) for t in traj}
                    row["tuned"] = dict(held, tile=sdt.tile_info(held["tile"])["name"])
                    row["speedup"] = round(traj[0]["us"] / traj[-1]["us"], 3)
                    us = traj[-1]["us"]
                else:
                    us = prob.measure(start)
                    if us is None:
                        raise SystemExit(f"configuration {start} is not legal for {name}")
                flops = gemm_flops(M, N, K)
                nbytes = 2 * (M * K + K * N + M * N)
                bound_us = max(flops / (peaks["tflops"] * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9)) * 1e6
                row.update({"us": round(us, 2), "tflops": round(flops / (us / 1e6) / 1e12, 1),
                            "roofline_bound": "tensor" if flops / (peaks["tflops"] * 1e12) >= nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm",
                            "roofline_frac": round(bound_us / us, 3)})
                rows.append(row)
                print(json.dumps(row), flush=True)
                del A, B, C, prob
                torch.cuda.empty_cache()
    sdt.check_device_status()
    out = {"mode": "p4", "problems": len(rows), "timing": f"mean of {args.reps} launches, L2 flushed before each",
           "roofline_frac_median": round(statistics.median(r["roofline_frac"] for r in rows), 3)}
    if args.tune:
        names_r = [k for k in rows[0]["rounds"] if k != "base"]
        per_round = {}
        for i, rn in enumerate(names_r):
            prev = "base" if i == 0 else names_r[i - 1]
            sp = [r["rounds"][prev] / r["rounds"][rn] for r in rows]
            per_round[rn] = {"mean": round(statistics.mean(sp), 3), "median": round(statistics.median(sp), 3),
                             "max": round(max(sp), 3)}
        out["per_round_speedup"] = per_round
        out["overall_speedup"] = {"mean": round(statistics.mean(r["speedup"] for r in rows), 3),
                                  "median": round(statistics.median(r["speedup"] for r in rows), 3),
                                  "max": round(max(r["speedup"] for r in rows), 3)}
        out["monotone"] = all(all(b <= a for a, b in zip(list(r["rounds"].values()),
                                                         list(r["rounds"].values())[1:])) for r in rows)
        if args.table_out:
            out["table"] = write_tune_table(args.table_out, [
                (r["M"], r["N"], r["K"], r["tuned"]) for r in rows
                if r["dtype"] == "f16" and r["layout"] == "NN" and r["tuned"]["splits"] == 1
                and r["tuned"]["algo"] not in (sdt.SPLITK_STREAM, sdt.SPLITK_STREAM_REDUCE)],
                "coordinate descent, bench.py --mode p4 --tune")
    print(json.dumps(out), flush=True)


def write_tune_table(path, entries, how):
    """Freeze tuned configurations for gemm_f16 ("M N K tile stagger raster stages" lines;
    see sdt_load_tune_table); shapes gemm_f16 cannot run with that tile are left out."""
    import shape_driven_tile_gb300 as sdt

    lines = [f"# frozen by {how}; GB300, {time.strftime('%Y-%m-%d')}"]
    for M, N, K, cfg in entries:
        tid = sdt.tile_id(cfg["tile"]) if isinstance(cfg["tile"], str) else cfg["tile"]
        if tid not in sdt.feasible_tiles(M, N, K, smem_limit=232448):
            continue
        lines.append(f"{M} {N} {K} {sdt.tile_info(tid)['name']} {cfg.get('stagger', -1)} "
                     f"{cfg.get('raster', 0)} {cfg.get('stages', 0)}")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return {"path": path, "entries": len(lines) - 1}


def run_large(args):
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    peaks = load_peaks()
    rows = []
    for n in (args.sizes or LARGE):
        A = (torch.rand((n, n), device=dev) * 2 - 1).half()
        B = (torch.rand((n, n), device=dev) * 2 - 1).half()
        C = torch.empty((n, n), device=dev, dtype=torch.float16)
        pick = sdt.pick_tile(n, n, n)
        for _ in range(2):
            sdt.gemm_f16(A, B, C)
        mean, lo, hi = time_cold(lambda: sdt.gemm_f16(A, B, C), args.reps, flush, stream)
        tf = gemm_flops(n, n, n) / (mean / 1e3) / 1e12
        rows.append({"size": n, "tile": sdt.tile_info(pick)["name"], "ms": round(mean, 3), "tflops": round(tf, 1),
                     "pct_peak": round(100 * tf / peaks["tflops"], 1)})
        print(json.dumps(rows[-1]), flush=True)
        del A, B, C
    sdt.check_device_status()
    print(json.dumps({"mode": "large", "rows": rows}), flush=True)


def run_splitk(args):
    """Split-K against the best unsplit tile on small-grid shapes (cold L2)."""
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)
    shapes = [tuple(int(v) for v in s.lower().split("x")) for s in (args.shapes or [])] or [
        (256, 256, 8192), (512, 512, 8192), (1024, 1024, 8192), (256, 4096, 4096), (2048, 512, 8192),
        (1024, 2048, 8192), (512, 512, 4096), (1024, 1024, 4096), (256, 256, 256), (512, 512, 512),
        (1024, 1024, 1024), (768, 768, 768)]
    for (M, N, K) in shapes:
        A = (torch.rand((M, K), device=dev) * 2 - 1).half()
        B = (torch.rand((K, N), device=dev) * 2 - 1).half()
        C = torch.empty((M, N), device=dev, dtype=torch.float16)
        base = {}
        for t in sdt.feasible_tiles(M, N, K):
            for _ in range(3):
                sdt.gemm_f16_with_tile(A, B, C, tile=t)
            base[sdt.tile_info(t)["name"]] = time_cold(lambda: sdt.gemm_f16_with_tile(A, B, C, tile=t),
                                                       args.reps, flush, stream)[0]
        tid, sp = sdt.pick_splitk(M, N, K, sm_count=sdt.device_sm_count())
        res = {}
        for algo in (sdt.SPLITK_REDUCE_KERNEL, sdt.SPLITK_IN_KERNEL):
            for splits in sorted({2, 4, 8, 16, sp}):
                if splits > K // 64 or sdt.splitk_workspace_bytes(M, N, K, tid, splits) == 0:
                    continue
                ws = sdt.splitk_workspace(M, N, K, tid, splits, device=dev)
                fn = lambda: sdt.gemm_f16_splitk(A, B, C, workspace=ws, tile=tid, splits=splits, algo=algo)
                for _ in range(3):
                    fn()
                res[f"{'ik' if algo else 'rk'}x{splits}"] = time_cold(fn, args.reps, flush, stream)[0]
        best_base = min(base, key=base.get)
        best_split = min(res, key=res.get) if res else None
        print(json.dumps({"shape": [M, N, K], "split_tile": sdt.tile_info(tid)["name"], "picked_splits": sp,
                          "best_unsplit": best_base, "best_unsplit_us": round(base[best_base] * 1e3, 2),
                          "split_us": {k: round(v * 1e3, 2) for k, v in res.items()},
                          "speedup_best_split": round(base[best_base] / res[best_split], 3) if res else None}),
              flush=True)
    sdt.check_device_status()


def run_chain(args):
    """Back-to-back launches of one GEMM (or decode GEMV) between two events: the
    per-launch time a stream of dependent-free launches sees (launch overlap included)."""
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    out = {}
    for n in (args.sizes or [256, 512, 768, 1024, 1536, 2048]):
        A = (torch.rand((n, n), device=dev) * 2 - 1).half()
        B = (torch.rand((n, n), device=dev) * 2 - 1).half()
        C = torch.empty((n, n), device=dev, dtype=torch.float16)
        L = sdt.lib()
        a = (n, n, n, A.data_ptr(), B.data_ptr(), C.data_ptr(), stream.cuda_stream)
        for _ in range(10):
            L.gemm_f16(*a)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = args.reps
        e0.record(stream)
        for _ in range(reps):
            L.gemm_f16(*a)
        e1.record(stream)
        torch.cuda.synchronize()
        out[n] = round(e0.elapsed_time(e1) * 1e3 / reps, 2)
    sdt.check_device_status()
    print(json.dumps({"mode": "chain", "pdl": os.environ.get("SDT_PDL", "1"), "us_per_launch": out}), flush=True)


def run_one(args):
    """A few launches of one kernel (for profiler captures): a square GEMM with pick_tile
    (through gemm_f16_ws unless --gemm-ws off, as in the benchmark step), or the decode
    GEMV (--gemv bf16|q8)."""
    import torch

    import shape_driven_tile_gb300 as sdt

    dev = torch.device("cuda", 0)
    if args.gemv:
        x = (torch.rand(DEC_K, device=dev) * 2 - 1).bfloat16()
        if args.gemv == "bf16":
            Ws = [(torch.rand((DEC_N, DEC_K), device=dev) * 2 - 1).bfloat16() for _ in range(2)]
            fn = lambda i: sdt.gemv_m1(x, Ws[i % 2])
        else:
            Ws = [torch.randint(-127, 128, (DEC_N, DEC_K), device=dev, dtype=torch.int8) for _ in range(2)]
            Ss = [(torch.rand((DEC_N, DEC_K // 32), device=dev) * 9e-3 + 1e-3).half() for _ in range(2)]
            fn = lambda i: sdt.gemv_m1(x, Ws[i % 2], Ss[i % 2])
    else:
        n = (args.sizes or [4096])[0]
        A = (torch.rand((n, n), device=dev) * 2 - 1).half()
        B = (torch.rand((n, n), device=dev) * 2 - 1).half()
        C = torch.empty((n, n), device=dev, dtype=torch.float16)
        if args.tile:
            fn = lambda i: sdt.gemm_f16_with_tile(A, B, C, tile=args.tile)
        elif args.gemm_ws == "on":  # as the benchmark step calls it
            ws = sdt.gemm_workspace(dev)
            fn = lambda i: sdt.gemm_f16_ws(A, B, C, workspace=ws)
        else:
            fn = lambda i: sdt.gemm_f16(A, B, C)
    for i in range(args.warmup + args.reps):
        fn(i)
    torch.cuda.synchronize()
    sdt.check_device_status()
    print(json.dumps({"mode": "one", "launches": args.warmup + args.reps,
                      "kernel": args.gemv or f"gemm {(args.sizes or [4096])[0]}^3 {args.tile or 'pick'}",
                      "source_digest": kernel_source_digest("gemv" if args.gemv else "gemm")}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["sdt", "reference"], default="sdt")
    ap.add_argument("--mode", choices=["step", "sweep", "kscan", "decode", "large", "one", "splitk", "chain",
                                       "record-traffic", "p4", "ktile"], default="step")
    ap.add_argument("--tune", action="store_true", help="p4: run the coordinate-descent tuner per problem")
    ap.add_argument("--table-out", help="p4 --tune / sweep: write the winners as a gemm_f16 tune table")
    ap.add_argument("--ncu-csv", help="record-traffic: ncu --csv log of one launch")
    ap.add_argument("--key", help="record-traffic: gemm_4096, gemv_bf16 or gemv_q8")
    ap.add_argument("--gemv", choices=["bf16", "q8"])
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--sizes", type=int, nargs="*")
    ap.add_argument("--tile", help="one/kscan/sweep: the tile; p4: time this tile instead of the pick")
    ap.add_argument("--splits", type=int, default=1, help="p4 with --tile: split count (stream-K: CTA count, 0 = default)")
    ap.add_argument("--algo", type=int, default=0,
                    help="p4 with --tile: 0/1 split-K reduction kernel / in-kernel, 2/3 stream-K fix-up in / after the kernel")
    ap.add_argument("--dtypes", nargs="*", choices=["f16", "bf16"], help="p4: operand types to run (default both)")
    ap.add_argument("--layouts", nargs="*", choices=["NN", "TN"], help="p4: layouts to run (default both)")
    ap.add_argument("--with-kscan", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="default run: launch every timed step eagerly instead of replaying nine-step CUDA graphs")
    ap.add_argument("--resume", help="sweep: append each shape's row to this file and skip shapes already in it")
    ap.add_argument("--shapes", nargs="*", help="extra GEMM shapes MxNxK for --mode sweep; shape names for --mode p4")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--clock-warmup-s", type=float, default=1.0,
                    help="default run: seconds of whole steps right before the timed region")
    ap.add_argument("--concurrent-steps", action="store_true",
                    help="default run: graph-replayed steps issue the GEMMs up to 1024^3 and the decode GEMVs on two "
                         "side streams beside the larger GEMMs (independent problems run at the same time)")
    ap.add_argument("--gemm-ws", choices=["on", "off"], default="on",
                    help="default run: the GEMMs as gemm_f16_ws calls with a workspace (on: a two-CTA tile may split "
                         "its last round in K where the plan says it pays) or as plain gemm_f16 calls (off)")
    ap.add_argument("--no-legs", action="store_true",
                    help="default run: skip the protocol legs after the timed region (gemm_protocol, pick_check, "
                         "kscan, large)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.mode == "record-traffic":
        return record_traffic(args)
    {"step": run_default, "sweep": run_sweep, "kscan": run_kscan, "decode": run_decode,
     "large": run_large, "one": run_one, "splitk": run_splitk, "chain": run_chain, "p4": run_p4,
     "ktile": run_ktile}[args.mode](args)


if __name__ == "__main__":
    main()
