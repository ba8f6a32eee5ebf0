#!/usr/bin/env python3
"""Benchmark of the multi-LoRA delta hot path on GB300.

One step = one pass of the LoRA delta over every layer instance of a
workload for one batch, replayed as a CUDA graph.  The default run measures
all five workloads in one process: the headline line is the largest
single-GPU one (Mistral-7B-shaped prefill, about 33.8k rows through the
seven projections of one layer), and ``per_config`` carries the other four
(tiny; Llama-3.2-3B-shaped decode as a 28-layer graph; the mixed continuous
batch as a 32-layer graph; the 70B-shaped stress batch).  Throughput counts
a token once per layer call: value = tokens x layers / step time.

Timing: W untimed replays, then K timed replays with a CUDA event between
consecutive replays; ``ms_per_step`` is the median replay (``ms_per_step_mean``
the mean over the K).  L2 honesty: the step's inputs (adapter stores, x, y)
are replicated into enough rotating sets that consecutive steps touch more
than 4x the L2 size (one set suffices when a step alone is that large).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(plain fp64 C, the correctness reference) on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import signal
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "all"
HEADLINE = "mistral7b_prefill"            # the largest workload that fits one GPU
PER_CONFIG = ["tiny", "llama3b_decode", "mixed", "stress70b"]
# layer instances per step: Llama-3.2-3B has 28 decoder layers; the mixed
# batch is Mistral-7B-shaped (32 layers)
LAYERS = {"llama3b_decode": 28, "mixed": 32}
# workloads whose rows are decode tokens: their chain of calls is also timed
# behind a base GEMM per call
DECODE_WORKLOADS = ("llama3b_decode", "mixed")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--seqs", type=int, default=None,
                    help="prefill sequences of the linear-layer workload (default 32; fewer for profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle sample budget")
    return ap.parse_args(argv)


# ----------------------------------------------------------- ranks ----

def dist_setup(backend: str):
    import torch.distributed as dist
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return rank, local, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, ws: int, device="cpu") -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, ws: int, device="cpu") -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------ accounting ----

def algorithmic_bytes(wl, group) -> int:
    """Compulsory bytes of one lora_apply call: each distinct adapter slot used
    by an active row read once (A and B' at the slot rank), x of the active
    rows read, y slices of the active rows read and written, plus the ids."""
    act = wl.ids >= 0
    n_act = int(act.sum())
    n_adapters = int(np.unique(wl.ids[act]).size)
    w_bytes = sum(wl.r_slot * (group.h_in + w) * 2 for _, w in group.projs)
    return n_adapters * w_bytes + n_act * group.h_in * 2 + n_act * group.ld_y * 2 * 2 + wl.n_rows * 4


def useful_flops(wl, group) -> int:
    act = wl.ids >= 0
    r = wl.ranks[wl.ids[act]].astype(np.int64)
    return int(sum(2 * (r * (group.h_in + w)).sum() for _, w in group.projs))


def src_digest(files) -> str:
    """sha256 (16 hex digits) over the named kernel sources under csrc/."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lora_serving_gb300", "csrc")
    for f in sorted(files):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


# Kernels a lora_apply call launches on each workload (the route of csrc/abi.cu).
ROUTE_KERNELS = {
    "tiny": "shrink_rowwise + expand_rowwise (prefill), bgmv_fused_kernel (decode)",
    "llama3b_decode": "bgmv_fused_kernel",
    "mistral7b_prefill": "sgmv_shrink_tc_kernel + sgmv_expand_tc_kernel",
    "mixed": "sgmv_shrink_tc_kernel + sgmv_expand_tc_kernel (prefill), bgmv_fused_kernel (decode)",
    "stress70b": "bgmv_group_shrink_kernel + bgmv_group_expand_kernel",
}

# DRAM traffic per lora_apply call from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum over the call's launches), keyed by workload; per
# step for the merge and linear-layer workloads (linear_tc_kernel's launches
# only for the linear layer); valid only while the listed kernel sources
# hash to `src`.
NCU_TRAFFIC = {
    "llama3b_decode": {"files": ['bgmv_fused.cu', 'decode_common.cuh', 'common.cuh', 'cluster.cuh'], "src": "c3d91c968f69f3f4",
             "bytes_per_call": 3442240},
    "stress70b": {"files": ['bgmv_grouped.cu', 'decode_common.cuh', 'common.cuh', 'cluster.cuh'], "src": "5d6b34e0b472f189",
             "bytes_per_call": 987991680},
    "mistral7b_prefill": {"files": ['sgmv_tc.cu', 'tc_common.cuh', 'tmap.cpp', 'common.cuh', 'cluster.cuh'], "src": "8bc12fda24a1f2bd",
             "bytes_per_call": 2061036160},
    "merge_mistral7b": {"files": ['merge.cu', 'merge_tc.cu', 'tc_common.cuh', 'tmap.cpp', 'common.cuh', 'cluster.cuh'], "src": "868105680b61064e",
             "bytes_per_step": 6934772736},
    "linear_mistral7b_prefill": {"files": ['linear_tc.cu', 'tc_common.cuh', 'tmap.cpp', 'common.cuh', 'cluster.cuh'], "src": "f30119a4aaa30b0e",
             "bytes_per_step": 13868097280},
    "mixed": {"files": ['sgmv_tc.cu', 'tc_common.cuh', 'tmap.cpp', 'bgmv_fused.cu', 'decode_common.cuh', 'common.cuh', 'cluster.cuh'], "src": "cf39137e5cbe5700",
             "bytes_per_call": 113187840},
    # captured on 2 layers, scaled to the 28 of a step (every layer has the same shapes)
    "linear_llama3b_decode": {"files": ['linear_swap.cu', 'bgmv_grouped.cu', 'tc_common.cuh', 'tmap.cpp', 'decode_common.cuh', 'common.cuh', 'cluster.cuh'],
             "src": "eda5c99cc28c95a4", "bytes_per_step": 1603022848},
}


def recorded_traffic(name, layers=None):
    """Recorded DRAM bytes per step of a merge or linear-layer workload, or
    None once its kernel sources have changed (or for another layer count)."""
    tr = NCU_TRAFFIC.get(name)
    if not tr or tr.get("src") != src_digest(tr["files"]):
        return None
    if layers is not None and layers != MERGE_LAYERS:
        return None
    return tr["bytes_per_step"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
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
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------ CPU oracle ----

_ORACLE_INPUTS = {}


def cpu_oracle_rate(wl_name: str, budget_s: float, layers: int, single_core: bool = True):
    """Times the fp64 oracle (as it stands) on layer calls of the workload,
    rows split across all host cores; returns (tokens/s per layer call, info).
    With `single_core`, info also holds the rate of the same oracle on one
    core (timed over a quarter of the budget) and the host CPU's model."""
    import concurrent.futures as cf
    import oracle as O
    from lora_serving_gb300 import synth

    cores = os.cpu_count() or 1
    if _ORACLE_INPUTS.get("name") != wl_name:   # inputs drawn once per workload, outside the timing
        wl = synth.get(wl_name).materialise("delta")
        ads = {}
        for g in wl.groups:
            for pname, _ in g.projs:
                A = [wl.A[(g.name, pname, k)] for k in range(wl.n_slots)]
                B = [wl.B[(g.name, pname, k)] for k in range(wl.n_slots)]
                sc = [O.scale(float(wl.alphas[k]), int(wl.ranks[k]), bool(wl.rslora[k]))
                      for k in range(wl.n_slots)]
                ads[(g.name, pname)] = O.Adapters(A, B, sc)
        _ORACLE_INPUTS.clear()
        _ORACLE_INPUTS.update(name=wl_name, wl=wl, ads=ads)
    wl, ads = _ORACLE_INPUTS["wl"], _ORACLE_INPUTS["ads"]
    # rows per layer call: all of them for small batches, a row block for large ones
    T = wl.n_rows
    blocks = np.array_split(np.arange(T), min(T, cores)) if T else []

    def run_block(rows):
        for g in wl.groups:
            y = wl.y[g.name][rows].copy()
            for (pname, _), off in zip(g.projs, g.offsets):
                y = O.apply_projection(wl.ids[rows], wl.x[g.name][rows], y, off, ads[(g.name, pname)])
        return len(rows)

    # warm (builds the oracle library) then time whole layer calls until the budget
    run_block(blocks[0][:1])
    done_rows = 0
    calls = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        if T <= 4096:
            while True:
                done_rows += sum(ex.map(run_block, blocks))
                calls += 1
                if time.perf_counter() - t0 >= budget_s:
                    break
            sample = f"{calls} layer call(s) of all {T} rows (all groups of one layer)"
        else:
            # large batches: a random subset of rows, one block per core
            rng = np.random.default_rng(0)
            sub = np.sort(rng.choice(T, min(T, 64 * cores), replace=False))
            done_rows = sum(ex.map(run_block, np.array_split(sub, cores)))
            sample = f"{sub.size} sampled rows of {T} (all groups of one layer), scaled per row"
    dt = time.perf_counter() - t0
    rate = done_rows / dt
    if not single_core:
        return rate, {"cores": cores, "sample": sample, "seconds": round(dt, 3)}
    # the same oracle on one core, over a quarter of the budget (at most 64 rows per pass)
    one = (np.arange(T) if T <= 4096 else sub)[:64]
    n1, t1 = 0, time.perf_counter()
    while True:
        n1 += run_block(one)
        if time.perf_counter() - t1 >= budget_s / 4:
            break
    rate1 = n1 / (time.perf_counter() - t1)
    return rate, {"cores": cores, "sample": sample, "seconds": round(dt, 3),
                  "single_core_value": round(rate1, 2), "cpu_model": host_cpu_model()}


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


# ------------------------------------------------- merge / unmerge ----
# Merged weights for single-tenant serving: W <- bf16(W +/- B'A) for every
# projection weight of MERGE_LAYERS Mistral-7B-shaped layers, one adapter of
# rank MERGE_RANK.  A step merges then unmerges every weight once.

MERGE_WORKLOAD = "merge_mistral7b"
MERGE_LAYERS = 4
MERGE_RANK = 64
MERGE_SHAPES = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
                ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]   # (name, out, h_in)


def merge_bytes(out: int, h_in: int, r: int) -> int:
    """Algorithmic bytes of one merge: W read and written, A and B' read once."""
    return 2 * 2 * out * h_in + 2 * r * (out + h_in)


def cpu_oracle_merge_rate(budget_s: float):
    """The fp64 oracle's merge on one q-shaped weight, row blocks over all cores."""
    import concurrent.futures as cf
    import oracle as O
    rng = np.random.default_rng(0)
    out, h_in, r = 4096, 4096, MERGE_RANK
    W = O.f64_to_bf16(rng.standard_normal((out, h_in)))
    A = O.f64_to_bf16(rng.standard_normal((r, h_in)) * 0.02)
    Bp = O.f64_to_bf16(rng.standard_normal((out, r)) * 0.02)
    cores = os.cpu_count() or 1
    O.merge(W[:1], A, Bp[:1], 1)   # builds the library
    rows = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        start = 0
        while time.perf_counter() - t0 < budget_s and start < out:
            blocks = [(start + i * 8, start + (i + 1) * 8) for i in range(cores)]
            rows += sum(ex.map(lambda b: O.merge(W[b[0]:b[1]], A, Bp[b[0]:b[1]], 1).shape[0], blocks))
            start += 8 * cores
    dt = time.perf_counter() - t0
    return rows * h_in / dt, {"cores": cores, "sample": f"{rows} rows of a {out}x{h_in} weight, rank {r}",
                              "seconds": round(dt, 3)}


def run_merge(args, rank, local, ws):
    import torch
    from lora_serving_gb300 import abi, build
    build()
    abi.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(7 + rank)
    r = MERGE_RANK
    layers = args.layers or MERGE_LAYERS
    weights = []
    for _ in range(layers):
        for name, out, h_in in MERGE_SHAPES:
            W = torch.randn(out, h_in, generator=g, device=dev).to(torch.bfloat16)
            A = (torch.randn(r, h_in, generator=g, device=dev) * 0.02).to(torch.bfloat16)
            B = (torch.randn(out, r, generator=g, device=dev) * 0.02).to(torch.bfloat16)
            weights.append((W, A, B))
    elems = sum(W.numel() for W, _, _ in weights)
    bytes_step = 2 * sum(merge_bytes(W.shape[0], W.shape[1], r) for W, _, _ in weights)

    Ws, As, Bs = [w for w, _, _ in weights], [a for _, a, _ in weights], [b for _, _, b in weights]

    def step():
        abi.lora_merge_batch(Ws, As, Bs, 1)
        abi.lora_merge_batch(Ws, As, Bs, -1)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    l0 = abi.lora_kernel_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    launches_per_step = abi.lora_kernel_launch_count() - l0
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0.record(cur)
    for _ in range(args.steps):
        graph.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    ms_local = e0.elapsed_time(e1)
    clk = clocks.stop()
    barrier(ws)
    ms = max_over_ranks(ms_local, ws, device=dev if ws > 1 else "cpu")
    units = sum_over_ranks(2.0 * elems * args.steps, ws, device=dev if ws > 1 else "cpu")
    peak, peak_kind = peaks()
    achieved = bytes_step / (ms_local / args.steps / 1e3) / 1e9
    out = {
        "metric": "LoRA merge/unmerge: weight elements updated per second",
        "value": round(units / (ms / 1e3), 1), "unit": "weights/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": MERGE_WORKLOAD, "layers": layers, "rank": r,
                   "weights": {n: [o, h] for n, o, h in MERGE_SHAPES}, "elements": elems,
                   "l2": f"{bytes_step / 2 / 1e9:.2f} GB of weights per pass (L2 "
                         f"{torch.cuda.get_device_properties(dev).L2_cache_size / 1e6:.0f} MB)",
                   "timing": "CUDA graph of one batched merge then one batched unmerge of every weight; CUDA events",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"kernel": "merge_tc_kernel", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "per": "step", "bytes_per_step": bytes_step, "traffic": recorded_traffic(MERGE_WORKLOAD, layers)},
        "clocks": clk,
        "gpu_launches": int(launches_per_step * args.steps),
        "e2e": None,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, info = cpu_oracle_merge_rate(args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(rate, 1), "unit": "weights/s", "cores": info["cores"],
                               "kind": "oracle", "sample": info["sample"]}
    return out


# ----------------------------------------------------- linear layer ----
# The LoRA linear layer: one Mistral-7B-shaped layer of the prefill batch
# (32 sequences of 64-2048 tokens over 16 adapters of ranks 8-64) through
# lora_linear for the q/k/v, o, gate/up and down groups, the base product
# and every row's delta in one accumulator.  Inputs: seeded bf16, base
# weights N(0, 1/h_in) (the synthetic recipe).  Context numbers: the same
# base products through cuBLAS (torch.matmul) without the delta, and cuBLAS
# followed by lora_apply adding the delta in place (the unfused layer).

LINEAR_WORKLOAD = "linear_mistral7b_prefill"
LINEAR_BASE = "mistral7b_prefill"


def linear_flops(wl, group) -> int:
    """Algorithmic FLOPs of one lora_linear call: 2 T h_in n_out for the base
    product plus 2 r (h_in + w) per active row and projection (true ranks)."""
    return 2 * wl.n_rows * group.h_in * group.ld_y + useful_flops(wl, group)


def tensor_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops_sustained"]), float(d["bf16_tflops"]), "measured"
    return 1700.0, 1900.0, "fallback"


_LINEAR_CPU = None


def cpu_oracle_linear_rate(budget_s: float):
    """The fp64 oracle's linear layer (all four groups of one layer) on rows of
    the prefill batch, row blocks over all host cores; returns rows per second."""
    import concurrent.futures as cf
    import oracle as O
    from lora_serving_gb300 import synth
    global _LINEAR_CPU
    cores = os.cpu_count() or 1
    if _LINEAR_CPU is None:   # inputs drawn once, outside the timed region
        wl = synth.get(LINEAR_BASE)
        rng = np.random.default_rng(0)
        rows = np.sort(rng.choice(wl.n_rows, size=min(wl.n_rows, 4 * cores), replace=False))
        wl.materialise("delta")
        sub = {g.name: wl.x[g.name][rows] for g in wl.groups}
        Ws = {g.name: wl.base_weight(g.name) for g in wl.groups}
        ads = {}
        for g in wl.groups:
            for pname, _ in g.projs:
                ads[(g.name, pname)] = O.Adapters(
                    [wl.A[(g.name, pname, k)] for k in range(wl.n_slots)],
                    [wl.B[(g.name, pname, k)] for k in range(wl.n_slots)],
                    [O.scale(float(wl.alphas[k]), int(wl.ranks[k]), bool(wl.rslora[k])) for k in range(wl.n_slots)])
        wl.x.clear()
        _LINEAR_CPU = (wl, rows, sub, Ws, ads)
    wl, rows, sub, Ws, ads = _LINEAR_CPU

    def run_rows(idx):
        for g in wl.groups:
            y = np.zeros((len(idx), g.ld_y), np.uint16)
            for (pname, w), off in zip(g.projs, g.offsets):
                y = O.linear_projection(wl.ids[rows[idx]], sub[g.name][idx], Ws[g.name][off:off + w], y, off,
                                        ads[(g.name, pname)])
        return len(idx)

    done = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        pos = 0
        while time.perf_counter() - t0 < budget_s and pos < rows.size:
            blocks = [np.arange(i, min(i + 1, rows.size)) for i in range(pos, min(pos + cores, rows.size))]
            done += sum(ex.map(run_rows, blocks))
            pos += len(blocks)
    dt = time.perf_counter() - t0
    return done / dt, {"cores": cores, "sample": f"{done} rows of the {wl.n_rows}-row prefill batch, all four "
                                                 f"groups of one layer", "seconds": round(dt, 3)}


def linear_e2e(args, wl, groups, store, dev):
    """The linear layer through the public call with host buffers: per step
    one host->device copy of every group's x (staged in one pinned buffer)
    and of the ids, the four lora_linear calls, and one device->host copy of
    every y; each step a CUDA graph, steps alternating over two streams with
    their own buffers, workspaces and metadata."""
    import torch
    names = [g.name for g in wl.groups]
    sizes_x = {n: wl.x[n].size for n in names}
    sizes_y = {g.name: wl.n_rows * g.ld_y for g in wl.groups}
    n_x, n_y = sum(sizes_x.values()), sum(sizes_y.values())
    h_x = torch.empty(n_x, dtype=torch.bfloat16).pin_memory()
    flat = h_x.view(torch.int16).numpy()
    off = 0
    for n in names:
        flat[off:off + sizes_x[n]] = wl.x[n].reshape(-1).view(np.int16)
        off += sizes_x[n]
    h_ids = torch.from_numpy(wl.ids.copy()).pin_memory()
    lanes = []
    for _ in range(2):
        dx = torch.empty(n_x, dtype=torch.bfloat16, device=dev)
        dy = torch.empty(n_y, dtype=torch.bfloat16, device=dev)
        xv, yv, ox, oy = {}, {}, 0, 0
        for g in wl.groups:
            xv[g.name] = dx[ox:ox + sizes_x[g.name]].view(wl.n_rows, g.h_in)
            yv[g.name] = dy[oy:oy + sizes_y[g.name]].view(wl.n_rows, g.ld_y)
            ox += sizes_x[g.name]
            oy += sizes_y[g.name]
        lanes.append({"stream": torch.cuda.Stream(device=dev), "dx": dx, "dy": dy, "x": xv, "y": yv,
                      "out": torch.empty(n_y, dtype=torch.bfloat16).pin_memory(),
                      "meta": store.BatchMeta(wl.ids, wl.n_prefill, wl.n_slots, device=dev),
                      "ws": {g.name: store.workspace_for(wl.n_rows, len(g.projs), wl.r_slot, device=dev)
                             for g in wl.groups}})

    def step(ln):
        ln["meta"].ids.copy_(h_ids, non_blocking=True)
        ln["dx"].copy_(h_x, non_blocking=True)
        for g in wl.groups:
            store.linear(ln["y"][g.name], ln["x"][g.name], groups[g.name]["W"], groups[g.name]["st"], ln["meta"],
                         ln["ws"][g.name])
        ln["out"].copy_(ln["dy"], non_blocking=True)

    graphs = []
    for ln in lanes:
        with torch.cuda.stream(ln["stream"]):
            step(ln)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=ln["stream"]):
            step(ln)
        graphs.append(gr)
    torch.cuda.synchronize()

    def run(count):
        for i in range(count):
            with torch.cuda.stream(lanes[i % 2]["stream"]):
                graphs[i % 2].replay()

    n = max(4, min(args.steps, 10))
    run(2)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for ln in lanes:
        ln["stream"].wait_event(e0)
    run(n)
    for ln in lanes:
        main.wait_stream(ln["stream"])
    e1.record(main)
    torch.cuda.synchronize()
    ems = e0.elapsed_time(e1)
    return {"value": round(wl.n_rows * n / (ems / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(n_x * 2 + h_ids.numel() * 4), "d2h_bytes_per_step": int(n_y * 2),
            "steps": n, "ms_per_step": round(ems / n, 4), "copies_per_step": 3, "streams": 2,
            "timing": "each step's copies and calls as a CUDA graph; steps alternate over two streams"}


def run_linear(args, rank, local, ws):
    import torch
    from lora_serving_gb300 import abi, build, store, synth
    build()
    abi.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = synth.get(LINEAR_BASE, **({"n_seqs": args.seqs} if args.seqs else {}))
    wl.materialise("delta")
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    meta = store.BatchMeta(wl.ids, wl.n_prefill, wl.n_slots, device=dev)
    groups = {}
    for g in wl.groups:
        groups[g.name] = {
            "st": store.GroupStore.from_workload(wl, g.name, device=dev),
            "x": to_dev(wl.x[g.name]), "W": to_dev(wl.base_weight(g.name)),
            "y": torch.empty(wl.n_rows, g.ld_y, dtype=torch.bfloat16, device=dev),
            "ws": store.workspace_for(wl.n_rows, len(g.projs), wl.r_slot, device=dev)}
    flops_call = {g.name: linear_flops(wl, g) for g in wl.groups}
    flops_step = sum(flops_call.values())

    def fused():
        for g in wl.groups:
            d = groups[g.name]
            store.linear(d["y"], d["x"], d["W"], d["st"], meta, d["ws"])

    def cublas_base():
        for g in wl.groups:
            d = groups[g.name]
            torch.matmul(d["x"], d["W"].t(), out=d["y"])

    def unfused():
        for g in wl.groups:
            d = groups[g.name]
            torch.matmul(d["x"], d["W"].t(), out=d["y"])
            store.apply(d["y"], d["x"], d["st"], meta, d["ws"])

    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    l0 = None
    for name_v, fn in (("fused", fused), ("cublas_base", cublas_base), ("unfused", unfused)):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        if name_v == "fused":
            l0 = abi.lora_kernel_launch_count()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        if name_v == "fused":
            launches_per_step = abi.lora_kernel_launch_count() - l0
        graphs[name_v] = gr
    torch.cuda.synchronize()

    def timed(gr, steps, warm):
        for _ in range(warm):
            gr.replay()
        torch.cuda.synchronize()
        barrier(ws)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        torch.cuda.synchronize()
        e0.record(cur)
        for _ in range(steps):
            gr.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        barrier(ws)
        return e0.elapsed_time(e1)

    other = {}
    for name_v in ("cublas_base", "unfused"):
        n_v = max(5, args.steps // 4)
        other[name_v] = round(timed(graphs[name_v], n_v, args.warmup) / n_v, 4)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ms_local = timed(graphs["fused"], args.steps, args.warmup)
    clk = clocks.stop()
    ms = max_over_ranks(ms_local, ws, device=dev if ws > 1 else "cpu")
    units = sum_over_ranks(float(wl.n_rows * args.steps), ws, device=dev if ws > 1 else "cpu")
    sustained, burst, kind = tensor_peaks()
    achieved = flops_step / (ms_local / args.steps / 1e3) / 1e12
    out = {
        "metric": "LoRA linear layer tokens/s (base product + per-row delta, one Mistral-7B layer)",
        "value": round(units / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {
            "workload": LINEAR_WORKLOAD, "tokens": wl.n_rows, "segments": len(wl.seg_lens), "n_slots": wl.n_slots,
            "r_slot": wl.r_slot, "groups": {g.name: [g.h_in, g.ld_y] for g in wl.groups},
            "l2": "inputs larger than L2 (x, W and y of a group are 0.3-2 GB each)",
            "timing": "CUDA graph of the four lora_linear calls of one layer; CUDA events",
            "ms_per_step_context": {"cublas_base_only": other["cublas_base"],
                                    "cublas_base_then_lora_apply": other["unfused"]},
            "parallelism": f"replicas x{ws}",
        },
        "roofline": {"kernel": "linear_tc_kernel (+ sgmv_shrink_tc_kernel per call)", "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": sustained, "unit": "TFLOP/s",
                     "frac": round(achieved / sustained, 4), "frac_of_burst": round(achieved / burst, 4),
                     "peak_source": f"{kind} bf16_tflops_sustained (burst {burst})", "per": "step",
                     "flops_per_step": flops_step,
                     "traffic": recorded_traffic(LINEAR_WORKLOAD) if not args.seqs else None},
        "clocks": clk,
        "gpu_launches": int(launches_per_step * args.steps),
    }
    if not args.no_e2e:
        out["e2e"] = linear_e2e(args, wl, groups, store, dev)
    if args.seqs:
        out["config"]["seqs"] = args.seqs
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, info = cpu_oracle_linear_rate(args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(rate, 2), "unit": "tokens/s", "cores": info["cores"],
                               "kind": "oracle", "sample": info["sample"]}
    return out


# ------------------------------------------- linear layer, decode ----
# The LoRA linear layer on the Llama-3.2-3B-shaped decode batch (64 tokens,
# 8 adapters of rank 16): 28 layer instances x (q/k/v, o) lora_linear calls
# per step, each layer's base weights its own (1.4 GB, beyond L2).  Context
# in the same run: the base products alone through cuBLAS, and cuBLAS then
# lora_apply (the unfused layer, two roundings).

LINEAR_DECODE_WORKLOAD = "linear_llama3b_decode"


def linear_decode_bytes(wl, group) -> int:
    """Algorithmic (compulsory) bytes of one decode-sized lora_linear call:
    the group's base weight, the adapters the batch uses (A and B' once),
    x read once and y written once (every row: base rows get the base
    product)."""
    act = wl.ids >= 0
    n_adapters = int(np.unique(wl.ids[act]).size)
    w_lora = sum(wl.r_slot * (group.h_in + w) * 2 for _, w in group.projs)
    return (group.ld_y * group.h_in * 2 + n_adapters * w_lora + wl.n_rows * group.h_in * 2
            + wl.n_rows * group.ld_y * 2)


def run_linear_decode(args, rank, local, ws):
    import torch
    from lora_serving_gb300 import abi, build, store, synth
    torch.cuda.set_device(local)
    build()
    abi.load()
    dev = torch.device("cuda", local)
    name = "llama3b_decode"
    layers = args.layers or LAYERS[name]
    base = synth.get(name)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    meta = store.BatchMeta(base.ids, 0, base.n_slots, device=dev)
    ws_buf = {g.name: store.workspace_for(base.n_rows, len(g.projs), base.r_slot, device=dev) for g in base.groups}
    inst = []
    for l in range(layers):
        wl = synth.get(name)
        wl.materialise("delta", layer=l)
        inst.append({g.name: {"st": store.GroupStore.from_workload(wl, g.name, device=dev),
                              "x": to_dev(wl.x[g.name]), "W": to_dev(wl.base_weight(g.name, layer=l)),
                              "y": torch.empty(base.n_rows, g.ld_y, dtype=torch.bfloat16, device=dev)}
                     for g in base.groups})

    def fused():
        for it in inst:
            for g in base.groups:
                d = it[g.name]
                store.linear(d["y"], d["x"], d["W"], d["st"], meta, ws_buf[g.name])

    def cublas_base():
        for it in inst:
            for g in base.groups:
                d = it[g.name]
                torch.matmul(d["x"], d["W"].t(), out=d["y"])

    def unfused():
        for it in inst:
            for g in base.groups:
                d = it[g.name]
                torch.matmul(d["x"], d["W"].t(), out=d["y"])
                store.apply(d["y"], d["x"], d["st"], meta, ws_buf[g.name], flags=abi.LORA_APPLY_X_READY)

    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    launches = 0
    for name_v, fn in (("fused", fused), ("cublas_base", cublas_base), ("unfused", unfused)):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        l0 = abi.lora_kernel_launch_count()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            fn()
        if name_v == "fused":
            launches = abi.lora_kernel_launch_count() - l0
        graphs[name_v] = gr
    torch.cuda.synchronize()
    other = {}
    for name_v in ("cublas_base", "unfused"):
        _, per = time_replays(lambda i: graphs[name_v].replay(), max(10, args.steps // 2), args.warmup, ws)
        other[name_v] = round(statistics.median(per), 5)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    _, per = time_replays(lambda i: graphs["fused"].replay(), args.steps, args.warmup, ws)
    clk = clocks.stop()
    med_local = statistics.median(per)
    med = max_over_ranks(med_local, ws, device=dev if ws > 1 else "cpu")
    units = sum_over_ranks(float(base.n_rows * layers), ws, device=dev if ws > 1 else "cpu")
    bytes_step = layers * sum(linear_decode_bytes(base, g) for g in base.groups)
    achieved = bytes_step / (med_local / 1e3) / 1e9
    peak, peak_kind = peaks()
    out = {
        "metric": "LoRA linear layer tokens/s (base product + per-row delta, decode batch)",
        "value": round(units / (med / 1e3), 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(med, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": LINEAR_DECODE_WORKLOAD, "tokens": base.n_rows, "layers": layers,
                   "groups": {g.name: [g.h_in, g.ld_y] for g in base.groups}, "n_slots": base.n_slots,
                   "r_slot": base.r_slot, "us_per_layer": round(med / layers * 1e3, 3),
                   "l2": "every layer's base weights its own (1.4 GB per step)",
                   "timing": "CUDA graph of the step's lora_linear calls; median replay",
                   "us_per_layer_context": {"cublas_base_only": round(other["cublas_base"] / layers * 1e3, 3),
                                            "cublas_base_then_lora_apply": round(other["unfused"] / layers * 1e3, 3)},
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"kernel": "linear_swap_kernel (+ bgmv_group_shrink_kernel per call)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs", "per": "step", "bytes_per_step": bytes_step,
                     "traffic": recorded_traffic(LINEAR_DECODE_WORKLOAD) if layers == LAYERS[name] else None},
        "clocks": clk,
        "gpu_launches": int(launches * args.steps),
        "e2e": None,
    }
    return out


# ---------------------------------------------------------- slots ----
# Adapter slot manager: loading adapters into GPU slots.  Llama-3.2-3B q/k/v/o
# adapters of rank 16 (640 KiB prepared), SLOTS_N slots, a pool of SLOTS_POOL
# registered adapters; a step acquires a batch of SLOTS_N adapters none of
# which is resident (every one a load), then a batch of resident ones (all hits).

SLOTS_WORKLOAD = "slots_llama3b"
SLOTS_N, SLOTS_POOL, SLOTS_RANK = 8, 64, 16
SLOTS_PROJS = [(3072, 3072), (3072, 1024), (3072, 1024), (3072, 3072)]   # (h_in, width): q, k, v, o


def run_slots(args, rank, local, ws):
    import torch
    from lora_serving_gb300 import abi, build
    build()
    abi.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    r_slot = SLOTS_RANK
    A_st = [torch.zeros(SLOTS_N, r_slot, h, dtype=torch.bfloat16, device=dev) for h, _ in SLOTS_PROJS]
    B_st = [torch.zeros(SLOTS_N, w, r_slot, dtype=torch.bfloat16, device=dev) for _, w in SLOTS_PROJS]
    m = abi.SlotManager([h for h, _ in SLOTS_PROJS], [w for _, w in SLOTS_PROJS], SLOTS_N, r_slot, SLOTS_POOL,
                        A_stores=A_st, B_stores=B_st)
    rng = np.random.default_rng(3 + rank)
    for k in range(SLOTS_POOL):
        A = [(rng.standard_normal((SLOTS_RANK, h)) * 0.02).astype(np.float32).view(np.uint32) >> 16
             for h, _ in SLOTS_PROJS]
        B = [(rng.standard_normal((w, SLOTS_RANK)) * 0.02).astype(np.float32).view(np.uint32) >> 16
             for _, w in SLOTS_PROJS]
        m.register(k, [a.astype(np.uint16) for a in A], [b.astype(np.uint16) for b in B], SLOTS_RANK, 32.0)
    stream = torch.cuda.current_stream(dev)
    adapter_bytes = sum(2 * r_slot * (h + w) for h, w in SLOTS_PROJS)
    batch = 0

    def step():
        nonlocal batch
        ids = np.arange(batch * SLOTS_N, (batch + 1) * SLOTS_N) % SLOTS_POOL   # none resident
        batch += 1
        m.acquire(ids, stream=stream)
        return ids

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(ws)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    last = None
    l0 = abi.lora_kernel_launch_count()
    for _ in range(args.steps):
        last = step()
    launches = abi.lora_kernel_launch_count() - l0
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms_local = e0.elapsed_time(e1)
    # host cost of a batch whose adapters are all resident (no copies)
    t1 = time.perf_counter()
    for _ in range(1000):
        m.acquire(last, stream=stream)
    hit_us = (time.perf_counter() - t1) / 1000 * 1e6
    barrier(ws)
    ms = max_over_ranks(ms_local, ws, device=dev if ws > 1 else "cpu")
    loads = sum_over_ranks(float(SLOTS_N * args.steps), ws, device=dev if ws > 1 else "cpu")
    st = m.stats()
    m.close()
    # the host-to-device link, measured here: one 256 MiB copy from pinned memory, best of 5
    src = torch.empty(128 << 20, dtype=torch.bfloat16).pin_memory()
    dst = torch.empty(128 << 20, dtype=torch.bfloat16, device=dev)
    best = float("inf")
    for _ in range(5):
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        dst.copy_(src, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        best = min(best, c0.elapsed_time(c1))
    link_gbs = src.numel() * 2 / (best / 1e3) / 1e9
    achieved = SLOTS_N * adapter_bytes * args.steps / (ms_local / 1e3) / 1e9
    return {
        "metric": "adapter loads into GPU slots per second", "value": round(loads / (ms / 1e3), 1),
        "unit": "loads/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": SLOTS_WORKLOAD, "slots": SLOTS_N, "pool": SLOTS_POOL, "rank": SLOTS_RANK,
                   "adapter_bytes": adapter_bytes, "projections": SLOTS_PROJS,
                   "timing": "CUDA events around the acquires of a step's all-miss batches (one gather kernel each)",
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"kernel": "slot_copy_kernel", "bound": "host link", "achieved": round(achieved, 1),
                     "peak": round(link_gbs, 1), "unit": "GB/s", "frac": round(achieved / link_gbs, 4),
                     "peak_source": "one 256 MiB pinned host-to-device copy measured in this run", "traffic": None},
        "h2d": {"achieved_gbs": round(achieved, 1),
                "pieces_per_load": 2 * len(SLOTS_PROJS), "host_wall_ms_per_step": round(wall / args.steps * 1e3, 4)},
        "acquire_all_hits_us": round(hit_us, 2),
        "stats": st,
        "gpu_launches": int(launches),
        "e2e": None,
    }


# ------------------------------------------------- standalone calls ----
# The four standalone entry points on the Llama-3.2-3B-shaped decode batch:
# per layer and group, one shrink over the group's rank-stacked A store (v
# fp32 [T][n_proj * r_slot]) then one expand per projection.  BGMV takes the
# per-token ids; SGMV the gather form (rows grouped by adapter through a
# permutation).  28 layer instances per step, as the decode workload.

STANDALONE_WORKLOAD = "standalone_llama3b"


def run_standalone(args, rank, local, ws):
    import torch
    from lora_serving_gb300 import abi, build, store, synth
    torch.cuda.set_device(local)
    build()
    abi.load()
    dev = torch.device("cuda", local)
    name = "llama3b_decode"
    layers = args.layers or LAYERS[name]
    base = synth.get(name)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    host = []
    for l in range(layers):
        wl = synth.get(name)
        wl.materialise("accumulate", layer=l)
        host.append(wl)
    meta = store.BatchMeta(base.ids, 0, base.n_slots, device=dev)
    m = meta.host
    inst0 = [Instance(h, store, to_dev) for h in host]
    set_bytes = sum(i.nbytes() for i in inst0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(4 * l2 / set_bytes))
    sets = [inst0] + [[Instance(h, store, to_dev) for h in host] for _ in range(n_sets - 1)]
    stacked = [[{g.name: torch.cat(inst.stores[g.name].A, dim=1).contiguous() for g in base.groups} for inst in st]
               for st in sets]
    T, r = base.n_rows, base.r_slot
    v = {g.name: torch.empty(T, len(g.projs) * r, dtype=torch.float32, device=dev) for g in base.groups}

    def step(s, form):
        for inst, A_st in zip(sets[s], stacked[s]):
            for g in base.groups:
                R = len(g.projs) * r
                st = inst.stores[g.name]
                if form == "bgmv":
                    abi.lora_bgmv_shrink(v[g.name], inst.x[g.name], A_st[g.name], meta.ids, h_in=g.h_in, r_slot=R,
                                         n_slots=base.n_slots)
                else:
                    abi.lora_sgmv_shrink(v[g.name], inst.x[g.name], A_st[g.name], meta.gseg_starts, meta.gseg_slot,
                                         m["n_gsegs"], meta.perm, T, h_in=g.h_in, r_slot=R, n_slots=base.n_slots,
                                         max_seg_len=m["max_gseg_len"])
                for pj, ((_, w), off) in enumerate(zip(g.projs, g.offsets)):
                    if form == "bgmv":
                        abi.lora_bgmv_expand(inst.y[g.name], off, w, v[g.name], st.B[pj], meta.ids, r_slot=r,
                                             n_slots=base.n_slots, v_col=pj * r)
                    else:
                        abi.lora_sgmv_expand(inst.y[g.name], off, w, v[g.name], st.B[pj], meta.gseg_starts,
                                             meta.gseg_slot, m["n_gsegs"], meta.perm, T, r_slot=r,
                                             n_slots=base.n_slots, max_seg_len=m["max_gseg_len"], v_col=pj * r)

    stream = torch.cuda.Stream(device=dev)
    res = {}
    clk = None
    for form in ("sgmv", "bgmv"):
        with torch.cuda.stream(stream):
            for s_ in range(n_sets):
                step(s_, form)
        torch.cuda.synchronize()
        l0 = abi.lora_kernel_launch_count()
        gs = []
        for s_ in range(n_sets):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                step(s_, form)
            gs.append(gr)
        launches = (abi.lora_kernel_launch_count() - l0) // n_sets
        clocks = ClockSampler(local) if form == "bgmv" else None
        if clocks:
            clocks.start()
            time.sleep(0.3)
        _, per = time_replays(lambda i: gs[i % n_sets].replay(), args.steps, args.warmup, ws)
        if clocks:
            clk = clocks.stop()
        res[form] = (statistics.median(per), launches)
        del gs
    calls = layers * len(base.groups)
    act = int((base.ids >= 0).sum())
    # a call's algorithmic bytes: the lora_apply bytes plus the fp32 v the
    # standalone form writes and reads back
    bytes_call = [algorithmic_bytes(base, g) + 2 * act * len(g.projs) * r * 4 for g in base.groups]
    bpc = sum(bytes_call) / len(bytes_call)
    peak, peak_kind = peaks()
    med, launches = res["bgmv"]
    med = max_over_ranks(med, ws, device=dev if ws > 1 else "cpu")
    call_ms = med / calls
    achieved = bpc / (call_ms / 1e3) / 1e9
    sg_ms, sg_launches = res["sgmv"]
    units = sum_over_ranks(float(T * layers), ws, device=dev if ws > 1 else "cpu")
    return {
        "metric": "standalone BGMV shrink+expand tokens/s (token x layer calls per second)",
        "value": round(units / (med / 1e3), 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(med, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": STANDALONE_WORKLOAD, "tokens": T, "layers": layers, "r_slot": r,
                   "groups": {g.name: [w for _, w in g.projs] for g in base.groups},
                   "calls": "per group: one shrink over the rank-stacked A, one expand per projection",
                   "l2": f"{n_sets} rotating input set(s) x {set_bytes / 1e6:.0f} MB (L2 {l2 / 1e6:.0f} MB)",
                   "timing": "CUDA graph of the step; median replay",
                   "sgmv_gather_form": {"ms_per_step": round(sg_ms, 5),
                                        "us_per_call": round(sg_ms / calls * 1e3, 3),
                                        "frac": round(bpc / (sg_ms / calls / 1e3) / 1e9 / peak, 4),
                                        "launches_per_step": sg_launches},
                   "parallelism": f"replicas x{ws}"},
        "roofline": {"kernel": "lora_bgmv_shrink + lora_bgmv_expand kernels", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs", "per": "group call (shrink + expands)",
                     "bytes_per_call": round(bpc), "call_us": round(call_ms * 1e3, 3), "traffic": None},
        "clocks": clk,
        "gpu_launches": int(launches * args.steps),
        "e2e": None,
    }


# --------------------------------------------------------- GPU arm ----

class Instance:
    """Device inputs of one layer instance: stores, x and y per group."""

    def __init__(self, wl, store_mod, to_dev):
        self.stores = {g.name: store_mod.GroupStore.from_workload(wl, g.name) for g in wl.groups}
        self.x = {g.name: to_dev(wl.x[g.name]) for g in wl.groups}
        self.y = {g.name: to_dev(wl.y[g.name]) for g in wl.groups}

    def nbytes(self):
        n = 0
        for st in self.stores.values():
            n += sum(a.numel() * 2 for a in st.A) + sum(b.numel() * 2 for b in st.B)
        n += sum(t.numel() * 2 for t in self.x.values()) + sum(t.numel() * 2 for t in self.y.values())
        return n


def time_replays(run_step, steps, warm, ws):
    """W untimed steps, then K timed ones with a CUDA event between
    consecutive steps, bracketed by a barrier and a synchronise on both
    sides.  Returns (total ms, per-step ms list)."""
    import torch
    for i in range(warm):
        run_step(i)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(ws)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    ev[0].record(cur)
    for i in range(steps):
        run_step(warm + i)
        ev[i + 1].record(cur)
    torch.cuda.synchronize()
    barrier(ws)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[steps]), per


def measure_delta(name, args, rank, local, ws, *, with_e2e=True, cpu_seconds=None, layers=None,
                  sample_clocks=True):
    """The LoRA delta of one workload through lora_apply: one line's worth of
    figures (value, roofline, orderings, clocks, and optionally e2e and the
    oracle's host rate)."""
    import torch
    from lora_serving_gb300 import abi, store, synth

    dev = torch.device("cuda", local)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    layers = layers or LAYERS.get(name, 1)
    base = synth.get(name)
    # host inputs of every layer instance (weights differ per layer)
    host = []
    for l in range(layers):
        wl = synth.get(name)
        wl.materialise("accumulate", layer=l)
        host.append(wl)
    meta = store.BatchMeta(base.ids, base.n_prefill, base.n_slots, device=dev)
    ws_buf = {g.name: store.workspace_for(base.n_rows, len(g.projs), base.r_slot, device=dev) for g in base.groups}
    inst0 = [Instance(h, store, to_dev) for h in host]
    set_bytes = sum(i.nbytes() for i in inst0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = max(1, math.ceil(4 * l2 / set_bytes))
    sets = [inst0] + [[Instance(h, store, to_dev) for h in host] for _ in range(n_sets - 1)]
    if not with_e2e:
        host = None

    calls_per_step = layers * len(base.groups)

    # Dependency model of the timed step: each call's y is treated as the
    # output of the kernel just before it (as the base GEMM's output is in a
    # model layer) and x as produced earlier (LORA_APPLY_X_READY).  The
    # other orderings are timed too and reported beside the headline.
    variants = {"x_ready": abi.LORA_APPLY_X_READY, "default": 0, "no_pdl": abi.LORA_APPLY_NO_PDL,
                "independent": abi.LORA_APPLY_X_READY | abi.LORA_APPLY_Y_READY}

    def step(s, flags):
        for inst in sets[s]:
            for g in base.groups:
                store.apply(inst.y[g.name], inst.x[g.name], inst.stores[g.name], meta, ws_buf[g.name],
                            flags=flags)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for s in range(n_sets):  # eager warm-up (first-call attributes) before capture
            step(s, 0)
    torch.cuda.synchronize()
    graphs = {}
    l0 = abi.lora_kernel_launch_count()
    for name_v, fl in variants.items():
        graphs[name_v] = []
        for s in range(n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(s, fl)
            graphs[name_v].append(g)
    launches_per_step = (abi.lora_kernel_launch_count() - l0) // (n_sets * len(variants))
    torch.cuda.synchronize()

    def replay(gs):
        return lambda i: gs[i % n_sets].replay()

    other = {}
    n_other = max(10, args.steps // 2)
    for name_v in ("default", "no_pdl", "independent"):
        _, per = time_replays(replay(graphs[name_v]), n_other, args.warmup, ws)
        other[name_v] = round(statistics.median(per), 5)
    del graphs["default"], graphs["no_pdl"], graphs["independent"]

    # A model layer puts a base GEMM (x W^T, here cuBLAS) before each delta:
    # the chain timed with and without the delta gives the delta's marginal
    # cost per call behind a kernel that does not start it early.
    gemm_ctx = floor = None
    if name in DECODE_WORKLOADS:
        gemm_ctx = gemm_chain(base, sets[0], meta, ws_buf, store, abi, dev, args, ws, stream)
        floor = y_rmw_chain(base, sets, n_sets, args, ws, stream)

    clocks = ClockSampler(local) if sample_clocks else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    total_ms, per = time_replays(replay(graphs["x_ready"]), args.steps, args.warmup, ws)
    clk = clocks.stop() if clocks else None
    med_local = statistics.median(per)
    med = max_over_ranks(med_local, ws, device=dev if ws > 1 else "cpu")
    tokens = base.n_rows
    units = sum_over_ranks(float(tokens * layers), ws, device=dev if ws > 1 else "cpu")
    value = units / (med / 1e3)

    # roofline of the delta: every launch in the step belongs to a lora_apply
    # call; algorithmic bytes per call / the call's share of the step
    bytes_call = [algorithmic_bytes(base, g) for g in base.groups]
    bytes_per_call = sum(bytes_call) / len(bytes_call)
    call_ms = med_local / calls_per_step
    achieved = bytes_per_call / (call_ms / 1e3) / 1e9
    peak, peak_kind = peaks()
    tr = NCU_TRAFFIC.get(name)
    traffic = tr["bytes_per_call"] if tr and tr.get("src") == src_digest(tr["files"]) else None

    out = {
        "metric": "SGMV/BGMV LoRA-delta tokens/s (token x layer calls per second)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(med, 5),
        "ms_per_step_mean": round(max_over_ranks(total_ms, ws, device=dev if ws > 1 else "cpu") / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)",
        "data": "synthetic",
        "config": {
            "workload": name, "tokens": tokens, "n_prefill": base.n_prefill, "layers": layers,
            "groups": {g.name: [w for _, w in g.projs] for g in base.groups},
            "hidden": base.groups[0].h_in, "n_slots": base.n_slots, "r_slot": base.r_slot,
            "active_rows": int((base.ids >= 0).sum()),
            "l2": f"{n_sets} rotating input set(s) x {set_bytes / 1e6:.0f} MB (L2 {l2 / 1e6:.0f} MB)",
            "timing": "CUDA graph of the step replayed; a CUDA event between replays on the launching stream; "
                      "median replay",
            "dependency": "x_ready: each call's y treated as the preceding kernel's output, x as earlier",
            "ms_per_step_other_orderings": other,
            "parallelism": f"replicas x{ws}",
        },
        "roofline": {
            "kernel": ROUTE_KERNELS.get(name, "lora_apply"), "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs",
            "per": "lora_apply call", "launches_per_call": round(launches_per_step / calls_per_step, 3),
            "bytes_per_call": round(bytes_per_call), "call_us": round(call_ms * 1e3, 3),
            "traffic": traffic,
        },
        "clocks": clk,
        "gpu_launches": launches_per_step * args.steps,
    }
    if gemm_ctx:
        out["config"]["behind_base_gemm"] = gemm_ctx
    if floor:
        out["config"]["chain_floor"] = floor

    if with_e2e:
        out["e2e"] = run_e2e(args, base, host, sets[0], meta, ws_buf, store, dev, layers)

    if rank == 0 and ws == 1 and cpu_seconds:
        rate, info = cpu_oracle_rate(name, cpu_seconds, layers)
        out["cpu_baseline"] = {"value": round(rate, 2), "unit": "tokens/s", "cores": info["cores"],
                               "kind": "oracle", "sample": info["sample"],
                               "single_core_value": info["single_core_value"], "cpu_model": info["cpu_model"]}
    del sets, inst0, graphs, ws_buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def gemm_chain(base, inst, meta, ws_buf, store, abi, dev, args, ws, stream):
    """Each layer call behind a base GEMM that writes its y (cuBLAS, x W^T):
    the step with the GEMMs alone, and with lora_apply (X_READY) after each
    GEMM.  The difference per call is the delta's marginal cost in a layer."""
    import torch
    g_w = torch.Generator(device=dev).manual_seed(11)
    Ws = [{g.name: (torch.randn(g.ld_y, g.h_in, generator=g_w, device=dev) / math.sqrt(g.h_in)).to(torch.bfloat16)
           for g in base.groups} for _ in inst]

    def step(with_delta):
        for li, it in enumerate(inst):
            for g in base.groups:
                torch.matmul(it.x[g.name], Ws[li][g.name].t(), out=it.y[g.name])
                if with_delta:
                    store.apply(it.y[g.name], it.x[g.name], it.stores[g.name], meta, ws_buf[g.name],
                                flags=abi.LORA_APPLY_X_READY)

    graphs = {}
    for key in (False, True):
        with torch.cuda.stream(stream):
            step(key)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(key)
        graphs[key] = gr
    n = max(10, args.steps // 2)
    _, per0 = time_replays(lambda i: graphs[False].replay(), n, args.warmup, ws)
    _, per1 = time_replays(lambda i: graphs[True].replay(), n, args.warmup, ws)
    calls = len(inst) * len(base.groups)
    t0, t1 = statistics.median(per0), statistics.median(per1)
    del graphs, Ws
    return {"ms_per_step_gemm_only": round(t0, 5), "ms_per_step_gemm_then_delta": round(t1, 5),
            "delta_us_per_call": round((t1 - t0) / calls * 1e3, 3),
            "note": "cuBLAS x W^T writes y, then lora_apply (X_READY) adds the delta; weights of "
                    f"{len(inst)} layer instance(s), one input set"}


def y_rmw_chain(base, sets, n_sets, args, ws, stream):
    """Context for a chain of dependent calls: the same step with each call
    replaced by one plain torch kernel that reads and writes the call's y
    (y *= 1, in place) -- what any design with one kernel per call pays
    before it does any LoRA work."""
    import torch

    def step(s):
        for inst in sets[s]:
            for g in base.groups:
                inst.y[g.name].mul_(1)

    graphs = []
    for s in range(n_sets):
        with torch.cuda.stream(stream):
            step(s)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(s)
        graphs.append(gr)
    n = max(10, args.steps // 2)
    _, per = time_replays(lambda i: graphs[i % n_sets].replay(), n, args.warmup, ws)
    calls = len(sets[0]) * len(base.groups)
    t = statistics.median(per)
    del graphs
    return {"ms_per_step_y_rmw_only": round(t, 5), "us_per_call": round(t / calls * 1e3, 3),
            "note": "each call replaced by torch's in-place y *= 1 over the call's whole y (all rows): "
                    "a dependent chain of one plain read-modify-write kernel per call"}


def run_all(args, rank, local, ws):
    """The default line: the headline workload in full (e2e, oracle
    baseline), the other four workloads in per_config."""
    import torch
    from lora_serving_gb300 import abi, build
    torch.cuda.set_device(local)
    if rank == 0:
        build()
    barrier(ws)
    build()
    abi.load()
    cpu = None if args.no_cpu_baseline else args.cpu_seconds
    out = measure_delta(HEADLINE, args, rank, local, ws, with_e2e=not args.no_e2e, cpu_seconds=cpu)
    per = {}
    keep = ("value", "unit", "ms_per_step", "ms_per_step_mean", "roofline", "clocks", "gpu_launches",
            "cpu_baseline")
    for name in PER_CONFIG:
        line = measure_delta(name, args, rank, local, ws, with_e2e=False,
                             cpu_seconds=None if cpu is None else max(1.0, cpu / 4))
        d = {k: line[k] for k in keep if k in line}
        d["config"] = line["config"]
        per[name] = d
    out["per_config"] = per
    # The rows beyond the delta itself (merge / unmerge, adapter slot loads,
    # the standalone calls, the LoRA linear layer in both forms), each with
    # its own metric, trimmed: no e2e and no oracle leg.
    extra = {}
    trimmed = argparse.Namespace(**{**vars(args), "no_e2e": True, "no_cpu_baseline": True, "layers": None,
                                    "seqs": None})
    for wname, fn in ((MERGE_WORKLOAD, run_merge), (SLOTS_WORKLOAD, run_slots),
                      (STANDALONE_WORKLOAD, run_standalone), (LINEAR_DECODE_WORKLOAD, run_linear_decode),
                      (LINEAR_WORKLOAD, run_linear)):
        line = fn(trimmed, rank, local, ws)
        extra[wname] = {k: line[k] for k in ("metric", "value", "unit", "ms_per_step", "roofline", "clocks",
                                             "gpu_launches", "config") if k in line}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out["extra_workloads"] = extra
    out["gpu_launches"] = (out["gpu_launches"] + sum(d["gpu_launches"] for d in per.values())
                           + sum(d.get("gpu_launches", 0) for d in extra.values()))
    out["gpu_launches_note"] = "timed launches of the headline, of every per_config line and of extra_workloads"
    return out


def run_ours(args, rank, local, ws):
    import torch
    from lora_serving_gb300 import abi, build
    torch.cuda.set_device(local)
    if rank == 0:
        build()
    barrier(ws)
    build()
    abi.load()
    return measure_delta(args.workload, args, rank, local, ws, with_e2e=not args.no_e2e,
                         cpu_seconds=None if args.no_cpu_baseline else args.cpu_seconds, layers=args.layers)


def run_e2e(args, base, host, inst, meta, ws_buf, store, dev, layers):
    """Same metric through the public call with host buffers.  A step's inputs
    (x and y_in of every layer call) are staged in one pinned host buffer, as
    a serving loop would stage a batch: per step one host->device copy of it
    (and one of the ids), lora_apply on views of the device copy, and one
    device->host copy of every y.  Consecutive steps alternate between two
    streams, each with its own device buffer, workspaces and metadata, so one
    step's copies overlap the other's kernels (the copy engines and the SMs
    work side by side, as in a pipelined serving loop)."""
    import torch
    from lora_serving_gb300 import abi
    keys = [(l, g.name) for l in range(layers) for g in base.groups]
    xs = [host[l].x[gn] for l, gn in keys]
    ys = [host[l].y[gn] for l, gn in keys]
    n_x = sum(a.size for a in xs)
    n_y = sum(a.size for a in ys)
    h_in = torch.empty(n_x + n_y, dtype=torch.bfloat16).pin_memory()   # [all x | all y_in]
    h_flat = h_in.view(torch.int16).numpy()
    off = 0
    for a in xs + ys:
        h_flat[off:off + a.size] = a.reshape(-1).view(np.int16)
        off += a.size
    h_ids = torch.from_numpy(base.ids.copy()).pin_memory()

    lanes = []
    for _ in range(2):
        d_buf = torch.empty(n_x + n_y, dtype=torch.bfloat16, device=dev)
        views, off = {}, 0
        for key, a in zip(keys, xs):
            views[("x",) + key] = d_buf[off:off + a.size].view(a.shape)
            off += a.size
        for key, a in zip(keys, ys):
            views[("y",) + key] = d_buf[off:off + a.size].view(a.shape)
            off += a.size
        lanes.append({
            "stream": torch.cuda.Stream(device=dev), "buf": d_buf, "views": views,
            "out": torch.empty(n_y, dtype=torch.bfloat16).pin_memory(),
            "meta": store.BatchMeta(base.ids, base.n_prefill, base.n_slots, device=dev),
            "ws": {g.name: store.workspace_for(base.n_rows, len(g.projs), base.r_slot, device=dev)
                   for g in base.groups}})
    h2d = (n_x + n_y) * 2 + h_ids.numel() * 4
    d2h = n_y * 2

    def step(i):
        ln = lanes[i % 2]
        with torch.cuda.stream(ln["stream"]):
            ln["meta"].ids.copy_(h_ids, non_blocking=True)
            ln["buf"].copy_(h_in, non_blocking=True)
            for l, gn in keys:
                store.apply(ln["views"][("y", l, gn)], ln["views"][("x", l, gn)], inst[l].stores[gn], ln["meta"],
                            ln["ws"][gn], flags=abi.LORA_APPLY_X_READY)
            ln["out"].copy_(ln["buf"][n_x:], non_blocking=True)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    # each lane's step (its copies and lora_apply calls) captured once as a
    # CUDA graph, as the device-side measurement does: the replays carry no
    # per-call host cost
    graphs = []
    for k, ln in enumerate(lanes):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=ln["stream"]):
            step(k)
        graphs.append(g)
    torch.cuda.synchronize()

    def run(count):
        for i in range(count):
            ln = lanes[i % 2]
            with torch.cuda.stream(ln["stream"]):
                graphs[i % 2].replay()

    n = max(4, min(args.steps, 20))
    run(4)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for ln in lanes:
        ln["stream"].wait_event(e0)
    run(n)
    for ln in lanes:
        main.wait_stream(ln["stream"])
    e1.record(main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"value": round(base.n_rows * layers * n / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n,
            "ms_per_step": round(ms / n, 4), "copies_per_step": 3, "streams": 2,
            "timing": "each step's copies and calls as a CUDA graph; steps alternate over two streams"}


def run_reference(args, rank, ws):
    """The CPU oracle timed on the machine's host cores, as the reference arm."""
    if rank != 0:
        return None
    name = HEADLINE if args.workload == "all" else args.workload
    if name == STANDALONE_WORKLOAD:   # the same delta, through the oracle's per-row path
        name = "llama3b_decode"
    if name == LINEAR_DECODE_WORKLOAD:
        return {"impl": "reference", "unavailable": "the oracle's linear layer is timed on the prefill workload "
                                                    "(--workload linear_mistral7b_prefill)"}
    layers = args.layers or LAYERS.get(name, 1)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    if name == SLOTS_WORKLOAD:
        # the slot manager moves bytes, it computes nothing: the host-side
        # counterpart is the same adapter loads done by memory copies
        rng = np.random.default_rng(3)
        adapter_elems = [SLOTS_RANK * h for h, _ in SLOTS_PROJS] + [w * SLOTS_RANK for _, w in SLOTS_PROJS]
        pool = [[rng.integers(0, 1 << 16, n, dtype=np.uint16) for n in adapter_elems] for _ in range(SLOTS_POOL)]
        slots = [[np.empty(n, np.uint16) for n in adapter_elems] for _ in range(SLOTS_N)]
        vals = []
        t0 = time.perf_counter()
        batch = 0
        for _ in range(args.steps):
            loads = 0
            ts = time.perf_counter()
            while time.perf_counter() - ts < per_step:
                for k in range(SLOTS_N):
                    for dst, src in zip(slots[k], pool[(batch * SLOTS_N + k) % SLOTS_POOL]):
                        np.copyto(dst, src)
                    loads += 1
                batch += 1
            vals.append(loads / (time.perf_counter() - ts))
        value = statistics.median(vals)
        return {
            "impl": "reference", "metric": "adapter loads into GPU slots per second",
            "value": round(value, 1), "unit": "loads/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": {"workload": name, "slots": SLOTS_N, "rank": SLOTS_RANK},
            "cpu_baseline": {"value": round(value, 1), "unit": "loads/s", "cores": 1, "kind": "host memory copies",
                             "sample": f"batches of {SLOTS_N} adapter loads for {per_step:.1f} s per step"},
            "e2e": {"value": round(value, 1), "unit": "loads/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "seconds": round(time.perf_counter() - t0, 2),
        }
    if name == LINEAR_WORKLOAD:
        vals, info = [], None
        t0 = time.perf_counter()
        for _ in range(args.steps):
            rate, info = cpu_oracle_linear_rate(per_step)
            vals.append(rate)
        value = statistics.median(vals)
        return {
            "impl": "reference",
            "metric": "LoRA linear layer tokens/s (base product + per-row delta, one Mistral-7B layer)",
            "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": {"workload": name},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": info["cores"], "kind": "oracle",
                             "sample": info["sample"]},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "seconds": round(time.perf_counter() - t0, 2),
        }
    if name == MERGE_WORKLOAD:
        vals, info = [], None
        t0 = time.perf_counter()
        for _ in range(args.steps):
            rate, info = cpu_oracle_merge_rate(per_step)
            vals.append(rate)
        value = statistics.median(vals)
        return {
            "impl": "reference", "metric": "LoRA merge/unmerge: weight elements updated per second",
            "value": round(value, 1), "unit": "weights/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": {"workload": name, "rank": MERGE_RANK},
            "cpu_baseline": {"value": round(value, 1), "unit": "weights/s", "cores": info["cores"], "kind": "oracle",
                             "sample": info["sample"]},
            "e2e": {"value": round(value, 1), "unit": "weights/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "seconds": round(time.perf_counter() - t0, 2),
        }
    vals = []
    info = None
    t0 = time.perf_counter()
    cpu_oracle_rate(name, 0.0, layers, single_core=False)  # warm-up: builds the oracle, one layer call
    for _ in range(args.steps):
        rate, info = cpu_oracle_rate(name, per_step, layers, single_core=False)
        vals.append(rate)
    total = time.perf_counter() - t0
    value = statistics.median(vals)
    from lora_serving_gb300 import synth
    base = synth.get(name)
    return {
        "impl": "reference",
        "metric": "SGMV/BGMV LoRA-delta tokens/s (token x layer calls per second)",
        "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * base.n_rows * layers / value, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "tokens": base.n_rows, "layers": layers, "n_slots": base.n_slots,
                   "r_slot": base.r_slot},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": info["cores"], "kind": "oracle",
                         "sample": info["sample"], "cpu_model": host_cpu_model()},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "seconds": round(total, 2),
    }


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        rank, local, ws = dist_setup("gloo")
        out = run_reference(args, rank, ws)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
        return 0
    rank, local, ws = dist_setup("nccl")
    if args.workload == MERGE_WORKLOAD:
        out = run_merge(args, rank, local, ws)
    elif args.workload == LINEAR_WORKLOAD:
        out = run_linear(args, rank, local, ws)
    elif args.workload == SLOTS_WORKLOAD:
        out = run_slots(args, rank, local, ws)
    elif args.workload == STANDALONE_WORKLOAD:
        out = run_standalone(args, rank, local, ws)
    elif args.workload == LINEAR_DECODE_WORKLOAD:
        out = run_linear_decode(args, rank, local, ws)
    elif args.workload == "all":
        out = run_all(args, rank, local, ws)
    else:
        out = run_ours(args, rank, local, ws)
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
