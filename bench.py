#!/usr/bin/env python
"""Benchmark of gated split-KV GQA decode attention on GB300.

One step = one gated decode call (stage 1 + stage 2) over a batch already
resident in HBM.  Default workload: B=64 sequences x 4096 KV positions, Hq=16,
Hkv=2, D=256 (538 MB of K/V rows per call, larger than L2, so no flush is
needed between calls).  Prints ONE JSON line (rank 0):

  value      whole-job achieved HBM GB/s = algorithmic bytes of all ranks' calls
             / max-over-ranks device time (K+V rows + q + gate + out)
  e2e        the same measured from host memory: per step, one copy of the packed
             inputs (q, gate, kv_indptr, kv_indices) from pinned host memory, the
             decode, one copy of out back and a wait, all inside gda_decode_step_host;
             the kernels read the inputs from and write out into pinned host memory
             in place, over the host-device link (without window or sinks;
             otherwise per-tensor copies around gda.decode)
  roofline   stage-1 kernel: algorithmic bytes / its CUDA-event duration vs the
             measured HBM copy bandwidth
  cpu_baseline  the FP64 oracle on the host cores (rank 0, N=1)

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  torchrun --nproc-per-node N --master-addr 127.0.0.1 bench.py --gpus N ...
N > 1 runs independent replicas (each rank its own batch, no collective on the
data path): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "gated decode attention µs/call and achieved HBM GB/s vs GB300 peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = {
    "bf16": ["gda_stage1.cu", "gda_stage1_tma.cu", "gda_device.cuh", "gda_kernels.h"],
    "e4m3": ["gda_stage1_fp8.cu", "gda_device.cuh", "gda_kernels.h"],
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="b64_l4096")
    p.add_argument("--splits", type=int, default=0, help="num_splits (0: automatic)")
    p.add_argument("--variant", type=int, default=0, help="0 auto, 1 mma, 2 simt, 3 tma ring")
    p.add_argument("--no-extra-timing", action="store_true",
                   help="skip the pages'-method and cold-cache timings")
    p.add_argument("--max-len", type=int, default=-1,
                   help="host-known bound on the sequence lengths passed to the decode (-1: the batch's "
                        "longest sequence, as a scheduler knows it; 0: no bound)")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle sample budget (cpu_baseline)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--graph", type=int, default=4,
                   help="calls per captured CUDA graph in the timed region (0: eager launches); the pages "
                        "time 4 calls per graph")
    p.add_argument("--hq", type=int, default=0, help="override the workload's query heads (0: keep)")
    p.add_argument("--hkv", type=int, default=0, help="override the workload's KV heads (0: keep)")
    p.add_argument("--window", type=int, default=0, help="sliding window (0: full attention)")
    p.add_argument("--sinks", type=float, default=None, help="give every query head this sink logit")
    p.add_argument("--kv", choices=["bf16", "e4m3"], default="bf16",
                   help="KV-cache element type: bf16, or e4m3 codes with per-tensor descales (FP8 cache)")
    p.add_argument("--op", choices=["decode", "prep", "prefill", "splits", "splits-cross", "paths"],
                   default="decode",
                   help="decode: the gated decode attention call (default); prep: the step before it "
                        "(Q/K RMSNorm + partial RoPE + KV write) on the workload's batch; prefill: the "
                        "prefill / extend gated SDPA (--workload p1_s4096_causal by default); splits / "
                        "splits-cross / paths: the sweeps behind the split rule and the one-kernel "
                        "dispatch (tables, not a bench line)")
    p.add_argument("--sweep-out", default=None, help="--op splits: also write the table as JSON here")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-workload speeds of the other decode workloads (default run only)")
    p.add_argument("--kernel-only", action="store_true",
                   help="warm-up + K calls and exit (the command profiled under ncu); prints nothing")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29533")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float, device=None) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power = [], [], []
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ helpers

def measured_bf16_peak(sustained: bool = False):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops_sustained" if sustained else "bf16_tflops"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return (1700.0 if sustained else 1900.0), "fallback"


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash(kv: str = "bf16") -> str:
    h = hashlib.sha256()
    for n in KERNEL_SOURCES[kv]:
        with open(os.path.join(ROOT, "gated_gqa_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, units: int, kv: str = "bf16"):
    """DRAM bytes per stage-1 launch from a committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    name = "stage1_%s_traffic.txt" % workload if kv == "bf16" else "stage1_%s_%s_traffic.txt" % (kv, workload)
    path = os.path.join(ROOT, "profiles", name)
    kv_type = kv
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_hash") != kernel_hash(kv_type):
            return None
        per_unit = float(kv["dram_bytes_per_token"])
        return per_unit * units
    except (OSError, KeyError, ValueError):
        return None


def algorithmic_bytes(lengths, hq, hkv, d, kv_bytes=2):
    from gated_gqa_attention_gb300 import workloads
    return workloads.metric_bytes(lengths, hq, hkv, d, kv_bytes)


def stage1_bytes(lengths, hq, hkv, d, kv_bytes=2):
    n = sum(lengths)
    return n * hkv * d * kv_bytes * 2 + len(lengths) * hq * d * 2


def oracle_sample_rate(inp, budget_s: float, nthreads: int = 0):
    """Time the FP64 oracle on the host: full batches until the budget is spent
    (nthreads 0: every core the oracle's OpenMP uses; 1: one core)."""
    import oracle
    w = inp["workload"]
    nbytes = algorithmic_bytes(inp["lengths"], w.hq, w.hkv, w.head_dim, inp["k_pool"].element_size())
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
                      inp["scale"], want=("out",), k_descale=inp["k_descale"], v_descale=inp["v_descale"],
                      nthreads=nthreads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or reps >= 100:
            break
    return nbytes * reps / dt / 1e9, reps, dt, (oracle.max_threads() if nthreads == 0 else nthreads)


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import torch
    import gated_gqa_attention_gb300 as gda
    from gated_gqa_attention_gb300 import workloads

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init(world, "nccl")
    dev_id = local
    gda.load()

    w = workloads.workload(args.workload)
    if args.hq or args.hkv:
        # the workload's lengths and layout with another head geometry
        hq, hkv = args.hq or w.hq, args.hkv or w.hkv
        rl = (w.len_lo, w.len_hi, w.batch) if w.lengths is None else None
        inp = workloads.make(w.lengths if w.lengths is not None else [], seed=w.seed + 1000 * rank, hq=hq, hkv=hkv,
                             head_dim=w.head_dim, layout=w.layout, pool_slots=w.pool_slots, page=w.page,
                             gate_std=w.gate_std, peaky_frac=w.peaky_frac, scale=w.scale, random_lengths=rl,
                             kv=args.kv)
        inp["workload"] = w
    else:
        inp = workloads.make_workload(args.workload, seed=w.seed + 1000 * rank, kv=args.kv)
    lengths = inp["lengths"]
    B, Hq, D = inp["q"].shape
    Hkv = inp["k_pool"].shape[1]
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    out = torch.empty_like(dev["q"])
    # algorithmic bytes: every attended K/V row once, plus q, gate, out (for G > 8 the
    # kernels stream each KV head's rows once per group of 8 query heads, which the
    # achieved fraction then shows)
    att = [min(L, args.window) if args.window > 0 else L for L in lengths]
    kvb = inp["k_pool"].element_size()
    nbytes = algorithmic_bytes(att, Hq, Hkv, D, kvb)
    s1_bytes = stage1_bytes(att, Hq, Hkv, D, kvb)
    kd, vd = inp["k_descale"], inp["v_descale"]
    stream = torch.cuda.current_stream()
    sinks = None if args.sinks is None else torch.full((Hq,), float(args.sinks), dtype=torch.float32, device="cuda")

    max_len = (max(lengths) if len(lengths) else 0) if args.max_len < 0 else args.max_len
    # the library's dispatch rule for the one-kernel cluster path (include/gda.h, max_len)
    small_c = (gda.small_path_cluster(B * Hkv, max_len) if (args.splits <= 0 and args.variant == 0 and
                                                              Hq // Hkv <= 8) else 0)
    small_path = small_c > 0
    # with the bound, the batch's exact total too (a scheduler knows both on the host)
    total_len = int(sum(lengths)) if max_len > 0 else 0

    def call():
        gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                      out=out, workspace=ws, scale=inp["scale"], num_splits=args.splits, variant=args.variant,
                      window=args.window, sinks=sinks, k_descale=kd, v_descale=vd, max_len=max_len,
                      total_len=total_len)

    ws = torch.empty(gda.workspace_bytes(B, Hq, Hkv, D, args.splits), dtype=torch.uint8, device="cuda")
    gda.workspace_init(ws)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    if args.kernel_only:
        for _ in range(args.steps):
            call()
        torch.cuda.synchronize()
        if gda.read_error(ws) != 0:
            raise SystemExit("device error word set")
        return None

    # ---- main timed region: K calls, device time by CUDA events on the launch stream.
    # With --graph R the calls are replayed from a captured CUDA graph of R calls.
    steps = args.steps
    run_steps = None
    if args.graph > 0:
        R = args.graph
        steps = R * max(1, (args.steps + R - 1) // R)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph):
                for _ in range(R):
                    call()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()

        def run_steps():
            for _ in range(steps // R):
                graph.replay()
    else:
        def run_steps():
            for _ in range(steps):
                call()
    try:
        uuid = str(torch.cuda.get_device_properties(dev_id).uuid)
        gpu_sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_sel = str(dev_id)
    sampler = ClockSampler(gpu_sel)
    barrier(dist, dev_id)
    torch.cuda.synchronize()
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_steps()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(dist, dev_id)
    ms_local = e0.elapsed_time(e1)
    ms = max_over_ranks(dist, ms_local, torch.device("cuda", dev_id))
    total_bytes = sum_over_ranks(dist, float(nbytes) * steps, torch.device("cuda", dev_id))
    value = total_bytes / (ms / 1e3) / 1e9
    err = gda.read_error(ws)

    # ---- stage-1 kernel duration (events around stage 1 of each call)
    k1 = min(args.steps, 2000)
    gda.timing_begin(k1)
    for _ in range(k1):
        call()
    n_t, ms_t = gda.timing_end()
    s1_us = ms_t / max(n_t, 1) * 1e3
    achieved = s1_bytes / (s1_us / 1e6) / 1e9
    peak, peak_kind = measured_hbm_peak()

    # ---- the pages' warm method (a CUDA graph of R calls, 14 samples of 50 replays,
    # the median), and a cold figure: 512 MiB (4x L2) read before each timed call (a
    # read leaves clean lines, so no write-back lands in the timed call), then a
    # device-side delay so the call is already enqueued when its start event fires;
    # the median over the calls
    pages_method = None
    if args.graph > 0 and not args.no_extra_timing:
        per = []
        for _ in range(14):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(50):
                graph.replay()
            a1.record(stream)
            torch.cuda.synchronize()
            per.append(a0.elapsed_time(a1) * 1e3 / (50 * args.graph))
        per.sort()
        pages_method = {"us_per_call_median": round(0.5 * (per[6] + per[7]), 3), "samples": 14,
                        "replays_per_sample": 50, "calls_per_replay": args.graph}
    cold = None
    if not args.no_extra_timing:
        flush = torch.ones(64 << 20, dtype=torch.int64, device=dev["q"].device)  # 512 MiB
        cs = []
        for _ in range(30):
            flush.sum()
            torch.cuda._sleep(200000)
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            call()
            c1.record(stream)
            torch.cuda.synchronize()
            cs.append(c0.elapsed_time(c1) * 1e3)
        cs.sort()
        cold = {"us_per_call_median": round(0.5 * (cs[14] + cs[15]), 3), "samples": 30,
                "evicted_bytes_before_each": 512 << 20, "launch": "eager, enqueued ahead"}
        del flush

    # ---- end to end with host buffers: per step, the inputs go from pinned host memory
    # to the device, the decode runs, the result comes back and the host waits for it
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = out_h.numel() * out_h.element_size()
    k_e2e = min(args.steps, 5000)
    step_api = args.window == 0 and args.sinks is None
    if step_api:
        # gda_decode_step_host: one packed block in, the decode, one copy out, one wait
        B_, Hq_, D_ = dev["q"].shape
        nnz_ = dev["kv_indices"].numel()
        _, blk = gda.step_layout(B_, Hq_, D_, nnz_)
        host_in = torch.zeros(blk, dtype=torch.uint8).pin_memory()
        gda.pack_step(host_in, dev["q"], dev["gate"], dev["kv_indptr"], dev["kv_indices"])
        h2d = blk   # read by the kernels in place over the host-device link
        e2e_api = "gda_decode_step_host (inputs read and result written in pinned host memory)"
        # the step's marshalled C call; each step: decode from host_in into out_h, wait
        e2e_step = gda.StepHost(host_in, None, dev["k_pool"], dev["v_pool"], None, out_h, B_, Hq_, nnz_,
                                scale=inp["scale"], num_splits=args.splits, map_in=True, map_out=True,
                                stream=stream, k_descale=kd, v_descale=vd)
    else:
        host = {k: dev[k].cpu().pin_memory() for k in ("q", "gate", "kv_indptr", "kv_indices")}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        e2e_api = "gda_decode (per-tensor copies)"

        def e2e_step():
            for k, t in host.items():
                dev[k].copy_(t, non_blocking=True)
            gda.decode(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                       out=out, scale=inp["scale"], num_splits=args.splits, k_descale=kd, v_descale=vd)
            out_h.copy_(out, non_blocking=True)
            stream.synchronize()   # the host reads the step's result

    for _ in range(3):
        e2e_step()
    barrier(dist, dev_id)
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        e2e_step()
    e2e_s = max_over_ranks(dist, time.perf_counter() - t0, torch.device("cuda", dev_id))
    e2e_total = sum_over_ranks(dist, float(nbytes) * k_e2e, torch.device("cuda", dev_id))
    e2e_value = e2e_total / e2e_s / 1e9

    # ---- the other workloads' speeds (the default bf16 run on one GPU only)
    configs = None
    if (world == 1 and args.kv == "bf16" and args.workload == "b64_l4096" and not (args.hq or args.hkv)
            and args.window == 0 and args.sinks is None and not args.no_configs):
        configs = config_speeds(measured_hbm_peak()[0])

    line = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            v, reps, dt, cores = oracle_sample_rate(inp, args.cpu_seconds)
            cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                   "sample": "%d full pass(es) of workload %s (B=%d) in %.1f s" % (reps, args.workload, B, dt)}
            v1, reps1, dt1, _ = oracle_sample_rate(inp, max(1.0, args.cpu_seconds / 3), nthreads=1)
            cpu["one_core"] = {"value": round(v1, 4), "unit": "GB/s",
                               "sample": "%d full pass(es) in %.1f s on 1 thread" % (reps1, dt1)}
        # the recorded counters are stage 1's; the one-kernel path has none recorded
        traffic = None if small_path else recorded_traffic(args.workload, sum(att) * Hkv, args.kv)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(ms / steps, 6),
            "us_per_call": round(ms / steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if args.kv == "bf16" else "e4m3 KV (f16 MMA, f32 accumulate), bf16 q/gate/out",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "lengths": "%d..%d (total %d)" % (min(lengths), max(lengths),
                                                                                          sum(lengths)),
                       "Hq": Hq, "Hkv": Hkv, "D": D, "num_splits": args.splits or "auto", "kv": args.kv,
                       "variant": ("cluster of %d (one kernel)" % small_c if small_path else
                                   {0: "auto(mma)", 1: "mma", 2: "simt", 3: "tma-ring+mma"}[args.variant]),
                       "max_len_hint": max_len, "total_len_hint": total_len,
                       "bytes_per_call": nbytes,
                       "l2": "inputs larger than L2 (%.0f MB of K/V rows per call), no flush" % (nbytes / 1e6),
                       "parallelism": "replicas x%d" % world, "window": args.window, "sinks": args.sinks,
                       "launch": ("CUDA graph of %d calls, replayed" % args.graph) if args.graph > 0 else "eager"},
            "roofline": {"bound": "hbm", "kernel": ("small_decode (one kernel, %d-CTA clusters)" % small_c if small_path else
                                                    "stage1" if args.kv == "bf16" else "stage1_fp8"),
                         "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                         "traffic": traffic, "algorithmic_bytes": s1_bytes, "avg_us": round(s1_us, 3),
                         "launches_timed": n_t},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": k_e2e, "api": e2e_api,
                    "us_per_step": round(e2e_s / k_e2e * 1e6, 3)},
            "gpu_launches": (1 if small_path else 2) * steps,
            "timing_pages_method": pages_method,
            "cold": cold,
            "configs": configs,
            "clocks": clocks,
            "device_error_word": err,
            "gpu": torch.cuda.get_device_name(dev_id),
        }
    if dist is not None:
        dist.destroy_process_group()
    return line


# ------------------------------------------------------------------ the other workloads

# (workload, KV type, num_splits, what the call is) timed beside the headline
CONFIG_LINES = [
    ("b1_l512", "bf16", 8, "S = 8 as the workload names it (split path, two kernels)"),
    ("b1_l512", "bf16", 0, "automatic with the host-known bound (dispatch)"),
    ("b4_ragged", "bf16", 0, "automatic with the host-known bound (dispatch)"),
    ("b224_ragged", "bf16", 0, "automatic with the host-known bound and total (dispatch)"),
    ("b8_l131072", "bf16", 0, "automatic with the host-known bound and total (dispatch)"),
    ("b64_l4096", "e4m3", 0, "FP8 (e4m3) KV cache, automatic with the host-known bound and total"),
]


def time_graph_us(call, stream, samples=7, target_s=0.02):
    """Median microseconds per call of `call` replayed from a CUDA graph of 4 calls:
    the pages' warm method (kernel window, no host work), with the replays per
    sample sized so one sample lasts about target_s."""
    import torch
    R = 4
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            for _ in range(R):
                call()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    reps = max(5, min(2000, int(target_s / max(t0.elapsed_time(t1) / 1e3, 1e-6))))
    per = []
    for _ in range(samples):
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        per.append(t0.elapsed_time(t1) * 1e3 / (reps * R))
    per.sort()
    return per[len(per) // 2], reps * R


def config_speeds(peak):
    """µs per call and GB/s of every workload other than the headline one, each through
    its default call: the inputs' lengths, layout and peaky rows as the parity tests
    draw them, their values drawn on the device (workloads.make, values_device)."""
    import torch
    import gated_gqa_attention_gb300 as gda
    from gated_gqa_attention_gb300 import workloads
    stream = torch.cuda.current_stream()
    lines = []
    for key, kv, splits, what in CONFIG_LINES:
        d = workloads.make_workload(key, kv=kv, values_device="cuda")
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        lengths = d["lengths"]
        B, Hq, D = dev["q"].shape
        Hkv = dev["k_pool"].shape[1]
        kvb = dev["k_pool"].element_size()
        max_len, total_len = (max(lengths), sum(lengths)) if splits <= 0 else (0, 0)
        small_c = gda.small_path_cluster(B * Hkv, max_len) if splits <= 0 and Hq // Hkv <= 8 else 0
        out = torch.empty_like(dev["q"])
        ws = torch.empty(gda.workspace_bytes(B, Hq, Hkv, D, splits), dtype=torch.uint8, device="cuda")
        gda.workspace_init(ws)

        def call():
            gda.decode_ex(dev["q"], dev["gate"], dev["k_pool"], dev["v_pool"], dev["kv_indptr"], dev["kv_indices"],
                          out=out, workspace=ws, scale=d["scale"], num_splits=splits, k_descale=d["k_descale"],
                          v_descale=d["v_descale"], max_len=max_len, total_len=total_len)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        us, n = time_graph_us(call, stream)
        nbytes = algorithmic_bytes(lengths, Hq, Hkv, D, kvb)
        gbs = nbytes / (us / 1e6) / 1e9
        err = gda.read_error(ws)
        lines.append({"workload": key, "kv": kv, "num_splits": splits or "auto", "call": what,
                      "path": ("one kernel, clusters of %d CTAs" % small_c if small_c else "split path (2 kernels)"),
                      "B": B, "lengths": "%d..%d (total %d)" % (min(lengths), max(lengths), sum(lengths)),
                      "us_per_call": round(us, 3), "GBs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                      "bytes_per_call": nbytes, "calls_timed": n, "device_error_word": err})
        del dev, out, ws, d
        torch.cuda.empty_cache()
    return {"method": "CUDA graph of 4 calls, median of 7 samples (the pages' warm method)",
            "values": "drawn on the device (same recipe, layout and lengths as the parity tests)", "lines": lines}


# ------------------------------------------------------------------ reference arm (the oracle)

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import numpy as np
    import oracle
    from gated_gqa_attention_gb300 import workloads

    inp = workloads.make_workload(args.workload, kv=args.kv)
    w = inp["workload"]
    lengths = inp["lengths"]
    B, G = len(lengths), w.hq // w.hkv
    kvb = inp["k_pool"].element_size()
    groups = [(b, kvh) for b in range(B) for kvh in range(w.hkv)]

    def step(i):
        b, kvh = groups[i % len(groups)]
        pairs = np.array([(b, kvh * G + g) for g in range(G)], dtype=np.int32)
        oracle.decode(inp["q"], inp["gate"], inp["k_pool"], inp["v_pool"], inp["kv_indptr"], inp["kv_indices"],
                      inp["scale"], pairs=pairs, want=("out",), k_descale=inp["k_descale"],
                      v_descale=inp["v_descale"])
        return lengths[b] * w.head_dim * kvb * 2 + G * 3 * w.head_dim * 2

    for i in range(max(args.warmup, 3)):
        step(i)
    t0 = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += step(i)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = ("each step: one (sequence, KV head) group of %d query heads of workload %s, cycling over its %d groups"
              % (G, args.workload, len(groups)))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "Hq": w.hq, "Hkv": w.hkv, "D": w.head_dim, "kv": args.kv},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_prep(args):
    """Time gda_qk_norm_rope_kv_write on the workload's batch (one decode token per
    sequence): rope_dim 64, both norms, graph replay of 4 calls.  Bytes: every row of
    the projection output read once, and q, gate, the K and V rows written."""
    import torch
    import gated_gqa_attention_gb300 as gda
    from gated_gqa_attention_gb300 import workloads

    torch.cuda.set_device(0)
    gda.load()
    w = workloads.workload(args.workload)
    B, Hq, Hkv, D = w.batch, w.hq, w.hkv, w.head_dim
    gen = torch.Generator(device="cpu").manual_seed(7)
    qgkv = torch.randn(B, (2 * Hq + 2 * Hkv) * D, generator=gen).to(torch.bfloat16).cuda()
    wq = torch.rand(D, generator=gen).add(0.5).to(torch.bfloat16).cuda()
    wk = torch.rand(D, generator=gen).add(0.5).to(torch.bfloat16).cuda()
    ang = torch.rand(B, 32, generator=gen) * 6.28
    cos = torch.cat([ang.cos(), ang.cos()], 1).to(torch.bfloat16).cuda()
    sin = torch.cat([ang.sin(), ang.sin()], 1).to(torch.bfloat16).cuda()
    slots_n = max(4 * B, 1024)
    slots = torch.randperm(slots_n, generator=gen)[:B].to(torch.int32).cuda()
    kp = torch.zeros(slots_n, Hkv, D, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    q_out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    g_out = torch.empty_like(q_out)
    call = lambda: gda.qk_norm_rope_kv_write(qgkv, slots, kp, vp, Hq, w_q_norm=wq, w_k_norm=wk, cos=cos, sin=sin,
                                             rope_dim=64, q_out=q_out, gate_out=g_out)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    R = 4
    steps = R * max(1, (args.steps + R - 1) // R)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            for _ in range(R):
                call()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps // R):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    nbytes = 2 * B * (2 * Hq + 2 * Hkv) * D * 2
    gbs = nbytes * steps / (ms / 1e3) / 1e9
    peak, kind = measured_hbm_peak()
    return {"metric": "qk-norm + rope + kv-write µs/call and achieved HBM GB/s (1 GPU)", "op": "prep",
            "value": round(gbs, 2), "unit": "GB/s", "us_per_call": round(ms / steps * 1e3, 3), "steps": steps,
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "rope_dim": 64,
                       "bytes_per_call": nbytes, "launch": "CUDA graph of 4 calls, replayed"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind}}


def run_prefill(args):
    """Time gda_prefill (tcgen05 gated SDPA) on a prefill workload: algorithmic FLOPs
    (4 * D per visible (query, key) pair per query head) over the CUDA-event time of K
    calls replayed from a CUDA graph of 4 (the kernel window, without per-call host
    work; the eager figure is reported beside it); beside it the unfused torch chain
    the cuDNN block page compares with (torch SDPA, then torch sigmoid and multiply)
    on the same inputs, timed the same way, and the FP64 oracle on a sample of rows."""
    import torch
    import gated_gqa_attention_gb300 as gda
    from gated_gqa_attention_gb300 import workloads

    torch.cuda.set_device(0)
    gda.load()
    key = args.workload if args.workload in workloads.PREFILL_BY_NAME else "p1_s4096_causal"
    inp = workloads.make_prefill_workload(key)
    w = inp["workload"]
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, Sq, Hq, D = inp["q"].shape
    Skv, Hkv = inp["k"].shape[1], inp["k"].shape[2]
    out = torch.empty_like(dev["q"])
    flops = workloads.prefill_flops(B, Sq, Skv, Hq, D, w.causal)
    call = lambda: gda.prefill(dev["q"], dev["gate"], dev["k"], dev["v"], out=out, scale=inp["scale"],
                               causal=w.causal)
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 200))
    stream = torch.cuda.current_stream()
    try:
        uuid = str(torch.cuda.get_device_properties(0).uuid)
        gpu_sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_sel = "0"
    sampler = ClockSampler(gpu_sel)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / steps

    def graph_of(fn, R=4):
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g):
                for _ in range(R):
                    fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        return g

    def time_graph(g, calls, R=4):
        reps = max(1, (calls + R - 1) // R)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / (reps * R), reps * R

    graph = graph_of(call)
    ms, steps = time_graph(graph, steps)
    clocks = sampler.stop()
    tflops = flops / (ms / 1e3) / 1e12
    err = gda.prefill_read_error()
    peak, kind = measured_bf16_peak()

    # the unfused torch chain on the same inputs: SDPA ([B, H, S, D]), sigmoid, multiply
    qt, kt, vt = (dev[n].transpose(1, 2) for n in ("q", "k", "v"))
    gt = dev["gate"]
    off = Skv - Sq

    def torch_chain():
        if w.causal and off > 0:
            mask = torch.ones(Sq, Skv, dtype=torch.bool, device="cuda").tril(diagonal=off)
            o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=inp["scale"],
                                                                 enable_gqa=True)
        else:
            o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=w.causal, scale=inp["scale"],
                                                                 enable_gqa=True)
        return o.transpose(1, 2) * torch.sigmoid(gt)
    torch_ms, torch_launch = None, "CUDA graph of 4 calls, replayed"
    try:
        for _ in range(3):
            torch_chain()
        torch.cuda.synchronize()
        n_t = max(1, min(steps, 50))
        try:
            torch_ms, _ = time_graph(graph_of(torch_chain), n_t)
        except RuntimeError:  # not capturable here: eager calls instead
            torch_launch = "eager"
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(n_t):
                torch_chain()
            t1.record(stream)
            torch.cuda.synchronize()
            torch_ms = t0.elapsed_time(t1) / n_t
    except RuntimeError as e:  # a backend that declines the shape
        torch_ms = "unavailable: %s" % str(e).splitlines()[0][:120]

    cpu = None
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        rng = np.random.default_rng(0)
        n_rows, t0c, done = 0, time.perf_counter(), 0.0
        while time.perf_counter() - t0c < min(args.cpu_seconds, 10.0):
            rows = np.stack([rng.integers(0, B, 64), rng.integers(0, Sq, 64), rng.integers(0, Hq, 64)], 1)
            oracle.prefill(inp["q"], inp["gate"], inp["k"], inp["v"], inp["scale"], causal=w.causal,
                           rows=rows.astype(np.int32), want=("out",))
            n_rows += 64
            for bb, ii, _ in rows:
                done += 4.0 * D * (min(Skv, ii + (Skv - Sq) + 1) if w.causal else Skv)
        dt = time.perf_counter() - t0c
        cpu = {"value": round(done / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
               "sample": "%d random (b, i, h) query rows of workload %s in %.1f s" % (n_rows, key, dt)}
    return {"metric": "prefill gated SDPA TFLOP/s (algorithmic) vs GB300 bf16 peak (1 GPU)", "op": "prefill",
            "value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4), "steps": steps,
            "eager_ms_per_call": round(eager_ms, 4),
            "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16 (tcgen05, f32 accumulate)",
            "data": "synthetic",
            "config": {"workload": key, "B": B, "Sq": Sq, "Skv": Skv, "Hq": Hq, "Hkv": Hkv, "D": D,
                       "causal": w.causal, "flops_per_call": flops, "launch": "CUDA graph of 4 calls, replayed"},
            "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "peak_kind": kind},
            "torch_chain_ms": torch_ms, "torch_chain_launch": torch_launch,
            "speedup_vs_torch_chain": (round(torch_ms / ms, 3) if isinstance(torch_ms, float) else None),
            "cpu_baseline": cpu, "clocks": clocks, "device_error_word": err, "gpu_launches": steps}


# ------------------------------------------------------------------ sweeps behind the dispatch rules

def _per_call_us(f, calls=200):
    """Microseconds per call of f replayed from a CUDA graph of 4 calls."""
    import torch
    for _ in range(5):
        f()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            for _ in range(4):
                f()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls // 4):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls * 1e3


def _sweep_batch(B, L, seed, hq=16, hkv=2, d=256):
    """Equal-length batch made on the device (timing only): N(0, 1) q, gate and K/V
    rows, slots a random permutation of the pool."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    n = B * L
    slots = n + 64
    mk = lambda *sh: torch.randn(*sh, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    q, gate = mk(B, hq, d), mk(B, hq, d)
    k_pool, v_pool = mk(slots, hkv, d), mk(slots, hkv, d)
    indptr = (torch.arange(B + 1, device="cuda", dtype=torch.int64) * L).to(torch.int32)
    indices = torch.randperm(slots, generator=g, device="cuda")[:n].to(torch.int32)
    return q, gate, k_pool, v_pool, indptr, indices


SWEEP_SPLITS = (1, 2, 4, 8, 16, 32, 64, 128)


def _sweep_batch8(B, L, seed):
    """An equal-length batch over an e4m3 cache (the workloads module's recipe, values
    drawn on the device): q, gate, k_pool, v_pool, kv_indptr, kv_indices, k_descale,
    v_descale, scale."""
    import torch
    from gated_gqa_attention_gb300 import workloads
    d = workloads.make([L] * B, seed=seed, layout="perm", pool_slots=B * L + 64, values_device="cuda", kv="e4m3")
    dv = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    return (dv["q"], dv["gate"], dv["k_pool"], dv["v_pool"], dv["kv_indptr"], dv["kv_indices"], d["k_descale"],
            d["v_descale"], d["scale"])


def run_split_sweep(args):
    """The split-count sweep ("chosen per (B, length) from measured time", FreeToken PR
    #781): for B equal-length sequences, B in {1 .. 128} and L in {512 .. 32768} (B L <=
    2^21), the µs per call with every explicit split count S in 1 .. 128, with the
    automatic schedule planned on the device (no length bound), and with the full
    dispatch (the longest length and the total passed: the one-kernel path where it
    applies, else the rule on the host).  Prints a table; --sweep-out writes JSON."""
    import torch
    import gated_gqa_attention_gb300 as gda
    torch.cuda.set_device(0)
    gda.load()
    HQ, HKV, D = 16, 2, 256
    rows = []
    print("%4s %6s | %s | %9s %9s %6s | %9s" % ("B", "L", " ".join("%8s" % ("S=%d" % s) for s in SWEEP_SPLITS),
                                                "best S", "auto", "a/best", "dispatch"))
    for B in (1, 2, 4, 8, 16, 32, 64, 128):
        for L in (512, 2048, 8192, 32768):
            if B * L > (1 << 21):
                continue
            if args.kv == "e4m3":
                q, gate, kp, vp, indptr, idx, kd, vd, sc = _sweep_batch8(B, L, seed=1000 + B + L)
            else:
                q, gate, kp, vp, indptr, idx = _sweep_batch(B, L, seed=1000 + B + L)
                kd, vd, sc = 1.0, 1.0, D ** -0.5
            out = torch.empty_like(q)
            t = {}
            for S in SWEEP_SPLITS + (0,):
                ws = torch.empty(gda.workspace_bytes(B, HQ, HKV, D, S), dtype=torch.uint8, device="cuda")
                gda.workspace_init(ws)
                t[S] = _per_call_us(lambda: gda.decode_ex(q, gate, kp, vp, indptr, idx, out=out, workspace=ws,
                                                          scale=sc, k_descale=kd, v_descale=vd, num_splits=S),
                                    calls=100)
            ws = torch.empty(gda.workspace_bytes(B, HQ, HKV, D, 0), dtype=torch.uint8, device="cuda")
            gda.workspace_init(ws)
            disp = _per_call_us(lambda: gda.decode_ex(q, gate, kp, vp, indptr, idx, out=out, workspace=ws,
                                                      scale=sc, k_descale=kd, v_descale=vd, max_len=L,
                                                      total_len=B * L), calls=100)
            best = min(SWEEP_SPLITS, key=lambda s: t[s])
            rows.append({"B": B, "L": L, "us_by_splits": {str(s): round(t[s], 3) for s in SWEEP_SPLITS},
                         "best_splits": best, "best_us": round(t[best], 3), "auto_us": round(t[0], 3),
                         "dispatch_us": round(disp, 3), "cluster": gda.small_path_cluster(B * HKV, L)})
            print("%4d %6d | %s | %4d %4.1f %9.2f %6.3f | %9.2f" % (
                B, L, " ".join("%8.2f" % t[s] for s in SWEEP_SPLITS), best, t[best], t[0], t[0] / t[best], disp),
                flush=True)
            del q, gate, kp, vp, indptr, idx, out, ws
            torch.cuda.empty_cache()
    if args.sweep_out:
        with open(args.sweep_out, "w") as f:
            json.dump(rows, f, indent=1)


# (B, L, S): S the one-wave uniform count near the rule's bounds
SPLIT_CROSS = [(64, 3072, 1), (64, 4096, 1), (64, 5120, 1), (64, 6144, 1), (32, 6144, 2), (32, 8192, 2),
               (32, 10240, 2), (16, 12288, 4), (16, 16384, 4), (16, 20480, 4), (8, 2048, 8), (8, 2048, 9),
               (8, 32768, 8), (8, 32768, 9), (4, 2048, 16), (4, 2048, 19), (4, 32768, 16), (4, 32768, 19),
               (2, 32768, 32), (2, 32768, 38), (1, 32768, 64), (1, 32768, 76), (48, 4096, 1), (48, 8192, 1),
               (24, 8192, 3), (24, 8192, 2)]


def run_split_cross(args):
    """Explicit uniform splits against the automatic schedule around the rule's bounds
    (positions per CTA near 3072; the power of two below the wave bound against the
    bound itself; waves that leave CTAs idle)."""
    import torch
    import gated_gqa_attention_gb300 as gda
    torch.cuda.set_device(0)
    gda.load()
    HQ, HKV, D = 16, 2, 256
    for B, L, S in SPLIT_CROSS:
        if args.kv == "e4m3":
            q, gate, kp, vp, indptr, idx, kd, vd, sc = _sweep_batch8(B, L, seed=5)
        else:
            q, gate, kp, vp, indptr, idx = _sweep_batch(B, L, seed=5)
            kd, vd, sc = 1.0, 1.0, D ** -0.5
        out = torch.empty_like(q)
        t = {}
        for s in (0, S):
            ws = torch.empty(gda.workspace_bytes(B, HQ, HKV, D, s), dtype=torch.uint8, device="cuda")
            gda.workspace_init(ws)
            t[s] = _per_call_us(lambda: gda.decode_ex(q, gate, kp, vp, indptr, idx, out=out, workspace=ws,
                                                      scale=sc, k_descale=kd, v_descale=vd, num_splits=s),
                                calls=200)
        print("B %3d L %6d per-CTA %6d | auto %8.2f | S=%3d %8.2f | S/auto %.3f" % (
            B, L, (HKV * B * L + 151) // 152, t[0], S, t[S], t[S] / t[0]), flush=True)
        del q, gate, kp, vp, indptr, idx, out, ws
        torch.cuda.empty_cache()


def run_paths(args):
    """The decode's one-kernel cluster path against the split path: B in {1 .. 64} and
    equal lengths L in {128 .. 2048}, the µs per call with the length bound (the
    one-kernel path where the library takes it), without it (split path, split count
    planned on the device), and on the split path with the bound and the total (split
    count from the host rule); the cluster size the library chose beside them."""
    import torch
    import gated_gqa_attention_gb300 as gda
    from gated_gqa_attention_gb300 import workloads
    torch.cuda.set_device(0)
    gda.load()
    print("%3s %5s %9s %12s %10s %13s %6s" % ("B", "L", "cluster C", "one-kernel", "split", "split (host)",
                                               "ratio"))
    for B in (1, 4, 8, 12, 16, 24, 32, 48, 64):
        for L in (128, 256, 512, 1024, 2048):
            inp = workloads.make([L] * B, seed=7, layout="perm", pool_slots=max(4096, B * L + 100))
            d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
            out = torch.empty_like(d["q"])
            _, Hq, D = d["q"].shape
            Hkv = d["k_pool"].shape[1]
            ws = torch.empty(gda.workspace_bytes(B, Hq, Hkv, D, 0), dtype=torch.uint8, device="cuda")
            gda.workspace_init(ws)
            t = {}
            for ml in (L, 0):
                t[ml] = _per_call_us(lambda: gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"],
                                                           d["kv_indices"], out=out, workspace=ws, scale=inp["scale"],
                                                           max_len=ml))
            th = _per_call_us(lambda: gda.decode_ex(d["q"], d["gate"], d["k_pool"], d["v_pool"], d["kv_indptr"],
                                                    d["kv_indices"], out=out, workspace=ws, scale=inp["scale"],
                                                    max_len=L, total_len=B * L, variant=gda.VARIANT_MMA))
            print("%3d %5d %9d %9.2f us %7.2f us %10.2f us %6.2f" % (B, L, gda.small_path_cluster(B * Hkv, L), t[L],
                                                                    t[0], th, t[L] / min(t[0], th)), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.op in ("splits", "splits-cross", "paths"):
        {"splits": run_split_sweep, "splits-cross": run_split_cross, "paths": run_paths}[args.op](args)
        return
    if args.op in ("prep", "prefill"):
        line = run_prep(args) if args.op == "prep" else run_prefill(args)
        print(json.dumps(line), flush=True)
        return
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
