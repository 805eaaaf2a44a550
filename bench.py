#!/usr/bin/env python3
"""CRISP sparse prefill benchmark on one synthetic Llama-3.1-8B-shaped layer.

Workload (default): 32 query / 8 kv heads, head_dim 128, 524,288 tokens,
bf16, every head sink-type with 2 slashes and 32 needle columns (seed 5).
One step = one pass of the whole hot path over the layer: block masses of
the proxy map (fused: the map is never stored), C_struct routing, VS
selection, pooled estimate and PE selection, mask + schedule, block-sparse
attention. The unfused map path (map write, then the mass pass) is timed
separately after the step. Inputs (6 GiB) are larger than L2, so no flush
between steps; for workloads whose inputs fit in L2 (--config gqa4x1-2k) a
512 MiB buffer is written before each timed step, outside its events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl crisp|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs its own replica
of the layer on its own GPU (no data-path collective; the path shards by kv
head group with no exchange); timing is the max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B = 128
METRIC = "sparse prefill ms/layer"
UNIT = "ms/layer"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["crisp", "reference"], default="crisp")
    ap.add_argument("--config", default="llama8b-512k", help="gqa4x1-2k, llama8b-32k, qwen7b-128k, llama8b-256k-L0..llama8b-256k-L3, llama8b-512k")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="run the chosen workload's recipe at this many tokens instead (small profiling cases)")
    ap.add_argument("--also", default="qwen7b-128k",
                    help="a second workload timed in the same process and reported under 'also' ('' for none)")
    ap.add_argument("--alpha", default="1/1")
    ap.add_argument("--pe-mode", choices=["gamma", "noise"], default="gamma",
                    help="PE selection rule: gamma coverage (the pages' rule) or the noise floor")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense-attention baseline launch")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-map", action="store_true", help="skip the map-reading route/select timing")
    ap.add_argument("--sweep", choices=["lengths", "alpha", "pe", "flex"], default=None,
                    help="instead of the step: sparse layer vs dense attention over sequence lengths (the "
                         "llama8b-32k recipe, 2k-128k), over alpha (llama8b-512k), PE gamma vs noise-floor rule "
                         "(llama8b-32k), or CRISP vs the FlexPrefill rules it replaces and the two ablations "
                         "(llama8b-512k and llama8b-32k)")
    return ap.parse_args(argv)


def workload_config(w, args, world):
    """The config keys both arms report for a workload (identical in both)."""
    return {"workload": w.name, "hq": w.hq, "hkv": w.hkv, "seq_len": w.n, "head_dim": 128, "block": B,
            "alpha": args.alpha, "tau": "1/5", "gamma": "19/20", "kmin_blocks": 8, "pe_mode": args.pe_mode,
            "parallelism": f"replicas x{world}"}


def workload(synth, name, seq_len=0):
    """A named workload; llama8b-256k-L0..L3 are the layers of the 4-layer
    stack. seq_len > 0: the same recipe at that length (named '<name>@<n>')."""
    if name.startswith("llama8b-256k-L"):
        w = synth.WORKLOADS["llama8b-256k-stack"].layer(int(name[len("llama8b-256k-L"):]))
    else:
        w = synth.WORKLOADS[name]
    if seq_len:
        w = synth.Workload(**{**w.__dict__, "name": f"{w.name}@{seq_len}", "n": seq_len})
    return w


# --------------------------------------------------------------- distributed
def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a host float over all ranks (NCCL with a device, else gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while running (SM clock, reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
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
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- accounting
def num_blocks(n: int) -> int:
    """128-token blocks of an n-token layer (the last one short when 128 does not divide n)."""
    return (n + B - 1) // B


def selected_pairs(rowbits: np.ndarray, n: int) -> int:
    """(row, key) pairs of the selected blocks of an n-token layer:
    len(qb)*len(kb) below the diagonal block, len(qb)(len(qb)+1)/2 on it (the
    causal half); len = B except a short last block."""
    nb = num_blocks(n)
    bits = np.unpackbits(rowbits.view(np.uint8), axis=-1, bitorder="little")[..., :nb]  # [hq][nb][nb]
    ln = np.minimum(B, n - B * np.arange(nb)).astype(np.int64)
    wgt = np.tril(np.outer(ln, ln), -1) + np.diag(ln * (ln + 1) // 2)
    return int((bits.sum(axis=0).astype(np.int64) * wgt).sum())


def profiled_traffic(sources, profile: str, w, blocks: int):
    """DRAM bytes per attention launch from a committed ncu summary, and how
    they were obtained. The summary holds the counters of one launch on a
    small case of a workload's recipe and that case's selected key blocks;
    a run of the same recipe at any length gets the per-block figure times
    its own selected blocks (the summary states why that scaling holds).
    None when a source that decides the traffic (the kernel, its work order)
    has changed since the counters were taken (sha256 over the files in
    order), or when the run's recipe is another one."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, profile)).read()
        src = b"".join(open(os.path.join(ROOT, f), "rb").read() for f in sources)
    except OSError:
        return None, "no profile"
    fields = dict(line.split(": ", 1) for line in text.splitlines() if ": " in line and " " not in line.split(": ")[0])
    if fields.get("source_sha256", "").strip() != hashlib.sha256(src).hexdigest():
        return None, "kernel changed since the counters were taken"
    try:
        captured = fields["workload"].strip()
        per_launch = int(fields["traffic_bytes_per_launch"])
        per_block = float(fields["traffic_bytes_per_selected_block"]) if "traffic_bytes_per_selected_block" in fields \
            else None
    except (KeyError, ValueError):
        return None, "profile incomplete"
    if w.name == captured:
        return per_launch, f"measured on this workload ({captured})"
    if per_block is not None and w.name.split("@")[0] == captured.split("@")[0]:
        return int(round(per_block * blocks)), (f"{per_block:.0f} B per selected block measured on {captured}, "
                                                f"times this run's {blocks} selected blocks")
    return None, f"profile is for another recipe ({captured})"


# The attention kernel and the kernel that writes its work order.
TRAFFIC_SOURCES = ("dynamic_sparse_prefill_crisp_gb300/csrc/attention.cu",
                   "dynamic_sparse_prefill_crisp_gb300/csrc/mask.cu")
TRAFFIC_PROFILE = "profiles/attention_llama8b_512k_traffic.md"


def measured_peaks():
    """(HBM GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, kind). A kernel
    timed by its own events inside a step of tens of ms is a burst: the burst
    figure is its denominator; the sustained one is reported beside it."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p.get("hbm_gbs", 6800.0), p.get("bf16_tflops", 1900.0), p.get("bf16_tflops_sustained", 1700.0), \
            "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------ CPU baseline
def cpu_sample(w, q, k, v, params_alpha, nthreads=None):
    """The fp64 oracle on a bounded sample of the layer: the full proxy /
    route / selection for the query heads of kv group 0 and attention for 128
    query rows of each of those heads; extrapolated to the whole layer."""
    import oracle
    G = w.hq // w.hkv
    heads = list(range(G))
    nb = num_blocks(w.n)
    t0 = time.perf_counter()
    P = oracle.proxy_map(q[heads], k[:1], nthreads=nthreads).astype(np.float32)
    vm, sm = oracle.vs_masses(P)
    _, _, route = oracle.route(P)
    vb, sb = oracle.select_vs(vm, sm, route, alpha=params_alpha)
    if (route == 0).any():
        pbar = oracle.pe_map(q[heads], k[:1], nthreads=nthreads).astype(np.float32)
    else:
        pbar = np.zeros((len(heads), nb, nb), np.float32)
    pe = oracle.select_pe(pbar, route)
    rb = oracle.build_mask(route, vb, sb, pe)
    t_select = time.perf_counter() - t0
    rng = np.random.default_rng(0)
    rows = 128
    hh = np.repeat(np.arange(len(heads)), rows).astype(np.int32)
    tt = rng.integers(0, w.n, hh.size).astype(np.int32)
    t1 = time.perf_counter()
    oracle.attention_rows(q[heads], k[:1], v[:1], hh, tt, rowbits=rb, nthreads=nthreads)
    t_attn = time.perf_counter() - t1
    # Pairs visited by the sampled rows vs by every row of the sampled heads.
    counts = np.unpackbits(rb.view(np.uint8), axis=-1, bitorder="little")[..., :nb]
    sampled_keys = sum(int(counts[h, t // B, : t // B].sum()) * B + (t % B + 1) for h, t in zip(hh, tt))
    all_pairs = selected_pairs(rb, w.n)
    layer_s = (t_select + t_attn * all_pairs / max(sampled_keys, 1)) * (w.hq / len(heads))
    return {
        "layer_ms": layer_s * 1e3,
        "sample": (f"oracle proxy map, C_struct route, VS/PE selection and mask for the {len(heads)} query heads of "
                   f"kv head 0 over all {w.n} keys ({t_select:.2f} s), plus fp64 attention for {hh.size} random query "
                   f"rows of those heads ({t_attn:.2f} s); scaled by selected (row,key) pairs to all rows and by "
                   f"{w.hq}/{len(heads)} to all heads"),
        "seconds": t_select + t_attn,
    }


def cpu_full_layer(w, q, k, v, params_alpha):
    """The whole layer through the fp64 oracle on one core (small layers)."""
    import oracle
    nb = num_blocks(w.n)
    t0 = time.perf_counter()
    P = oracle.proxy_map(q, k, nthreads=1).astype(np.float32)
    vm, sm = oracle.vs_masses(P, nthreads=1)
    _, _, route = oracle.route(P, nthreads=1)
    vb, sb = oracle.select_vs(vm, sm, route, alpha=params_alpha)
    pbar = oracle.pe_map(q, k, nthreads=1).astype(np.float32)
    pe = oracle.select_pe(pbar, route, nthreads=1)
    rb = oracle.build_mask(route, vb, sb, pe)
    hh, tt = np.meshgrid(np.arange(w.hq), np.arange(w.n), indexing="ij")
    oracle.attention_rows(q, k, v, hh.ravel().astype(np.int32), tt.ravel().astype(np.int32), rowbits=rb, nthreads=1)
    del nb
    return (time.perf_counter() - t0) * 1e3


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import synth
    w = workload(synth, args.config, args.seq_len)
    alpha = tuple(int(x) for x in args.alpha.split("/"))
    q, k, v = w.generate()
    cores = os.cpu_count() or 1
    times, secs = [], []
    sample = None
    for i in range(args.warmup + args.steps):
        r = cpu_sample(w, q, k, v, alpha, nthreads=cores)
        sample = r["sample"]
        if i >= args.warmup:
            times.append(r["layer_ms"])
            secs.append(r["seconds"])
    ms = statistics.mean(times)
    cpu = {"value": ms, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample, "extrapolated": True,
           "sample_seconds_per_step": statistics.mean(secs)}
    line = {"impl": "reference", "metric": METRIC, "value": ms, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args, 1),
            "host": "fp64 oracle on the host cores (the reference is prose: the oracle stands in for it)",
            "extrapolated": True,
            "extrapolation": ("each step times the oracle on a bounded sample of the layer (sample_seconds_per_step "
                              "of wall time) and scales it to a whole layer by selected (row, key) pairs and by "
                              "heads; value and ms_per_step are that scaled figure, not wall time"),
            "sample_seconds_per_step": statistics.mean(secs),
            "cpu_baseline": cpu,
            "e2e": {"value": ms, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm
# our kernel launches per step: proxy statistics 2, fused masses 2, route 1,
# select_vs 1, pe_pool 2, select_pe 1, mask+schedule 2, attention 1
LAUNCHES_PER_STEP = 12
STAGES = ["proxy_masses", "route", "select_vs", "pe_pool", "select_pe", "mask", "attention"]


def host_facts(ptrs):
    """Host-side facts behind the e2e number: CPUs, NUMA nodes, the GPU's
    node and the node of each pinned buffer's pages (/proc/self/numa_maps)."""
    facts = {"cpus": os.cpu_count()}
    try:
        facts["numa_nodes"] = len([d for d in os.listdir("/sys/devices/system/node") if d.startswith("node")])
    except OSError:
        facts["numa_nodes"] = None
    try:
        bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader", "-i",
                              os.environ.get("LOCAL_RANK", "0")], capture_output=True, text=True, timeout=20)
        bus_id = bus.stdout.strip().lower()
        if len(bus_id.split(":")[0]) > 4:  # nvidia-smi prints an 8-digit domain; sysfs uses 4
            bus_id = bus_id[len(bus_id.split(":")[0]) - 4:]
        with open(f"/sys/bus/pci/devices/{bus_id}/numa_node") as f:
            facts["gpu_numa_node"] = int(f.read())
    except (OSError, ValueError, subprocess.SubprocessError):
        facts["gpu_numa_node"] = None
    try:
        spans = []
        with open("/proc/self/maps") as f:
            for line in f:
                lo, hi = (int(x, 16) for x in line.split()[0].split("-"))
                spans.append((lo, hi))
        nodes = {}
        with open("/proc/self/numa_maps") as f:
            numa = {int(line.split()[0], 16): line.split()[1:] for line in f}
        for name, ptr in ptrs.items():
            hit = [lo for lo, hi in spans if lo <= ptr < hi]
            fields = numa.get(hit[0], []) if hit else []
            nodes[name] = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in fields
                           if kv.startswith("N") and "=" in kv and kv.split("=")[1].isdigit()}
        facts["pinned_pages_per_node"] = nodes
    except (OSError, ValueError, IndexError):
        facts["pinned_pages_per_node"] = None
    return facts


class Layer:
    """Device buffers and the step calls of one workload (inputs in HBM)."""

    def __init__(self, crisp, torch, w, params, dev, stream):
        self.w, self.params, self.stream = w, params, stream
        hq, hkv, n = w.hq, w.hkv, w.n
        nb = num_blocks(n)
        W = (nb + 31) // 32
        # Inputs: generated on the host into pinned buffers (also the e2e source).
        self.qh = torch.empty((hq, n, 128), dtype=torch.int16, pin_memory=True)
        self.kh = torch.empty((hkv, n, 128), dtype=torch.int16, pin_memory=True)
        self.vh = torch.empty((hkv, n, 128), dtype=torch.int16, pin_memory=True)
        t0 = time.perf_counter()
        w.generate(*(t.numpy().view(np.uint16) for t in (self.qh, self.kh, self.vh)))
        self.gen_s = time.perf_counter() - t0
        self.qd = self.qh.to(dev).view(torch.bfloat16)
        self.kd = self.kh.to(dev).view(torch.bfloat16)
        self.vd = self.vh.to(dev).view(torch.bfloat16)
        self.out = torch.empty((hq, n, 128), dtype=torch.bfloat16, device=dev)
        s = self.shape = crisp.make_shape(hq, hkv, n, self.qd, self.kd, self.out)
        self.ws = torch.empty(crisp.workspace_size(s), dtype=torch.uint8, device=dev)
        crisp.workspace_init(self.ws)
        E = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)
        self.vmass, self.smass, self.rmass = E((hq, nb), torch.int64), E((hq, nb), torch.int64), E((hq,), torch.int64)
        self.cstruct, self.total, self.route = E((hq,), torch.int64), E((hq,), torch.int64), E((hq,), torch.uint8)
        self.vbits, self.sbits = E((hq, W), torch.int32), E((hq, W), torch.int32)
        self.pbar = E((hq, nb, nb), torch.float32)
        self.pebits, self.rowbits = E((hq, nb, W), torch.int32), E((hq, nb, W), torch.int32)
        self.counts, self.order = E((hq, nb), torch.int32), E((hq * nb,), torch.int32)
        st, ws, p = stream, self.ws, params
        self.calls = [
            lambda: crisp.proxy_masses(s, self.qd, self.kd, self.vmass, self.smass, self.rmass, ws, st),
            lambda: crisp.route_cstruct_masses(s, p, self.vmass, self.rmass, self.cstruct, self.total, self.route,
                                               ws, st),
            lambda: crisp.select_vs_masses(s, p, self.vmass, self.smass, self.route, self.vbits, self.sbits, ws, st),
            lambda: crisp.pe_pool(s, self.qd, self.kd, self.route, self.pbar, ws, st),
            lambda: crisp.select_pe(s, p, self.pbar, self.route, self.pebits, ws, st),
            lambda: crisp.build_mask(s, self.route, self.vbits, self.sbits, self.pebits, self.rowbits, self.counts,
                                     self.order, ws, st),
            lambda: crisp.sparse_prefill_mask(s, self.qd, self.kd, self.vd, self.rowbits, self.order, self.out, ws,
                                              st),
        ]

    def step(self, events=None):
        for i, c in enumerate(self.calls):
            if events is not None:
                events[i].record(self.stream)
            c()
        if events is not None:
            events[-1].record(self.stream)


def time_steps(torch, layer, args, world, local, dev):
    """W warm-up steps, then K steps timed with CUDA events (per stage too),
    inside a barrier and synchronize on both sides, clocks sampled."""
    import dynamic_sparse_prefill_crisp_gb300 as crisp
    for _ in range(args.warmup):
        layer.step()
    torch.cuda.synchronize()
    st = crisp.read_status(layer.ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {crisp.status_string(st)}")
    w = layer.w
    in_bytes = (w.hq + 2 * w.hkv) * w.n * 128 * 2
    l2_bytes = 129 * 2**20
    flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev) if in_bytes < 2 * l2_bytes else None
    l2_note = (f"inputs ({in_bytes / 2**30:.2f} GiB) larger than L2; no flush" if flush is None else
               f"inputs ({in_bytes / 2**20:.1f} MiB) smaller than L2: 512 MiB written before each timed step")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(layer.calls) + 1)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    if flush is None:
        start.record(layer.stream)
        for i in range(args.steps):
            layer.step(ev[i])
        end.record(layer.stream)
    else:
        # Inputs smaller than L2: a 512 MiB write evicts them before each
        # step, outside the timed intervals (the step total is the sum).
        for i in range(args.steps):
            flush.zero_()
            layer.step(ev[i])
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if flush is None:
        ms_total = start.elapsed_time(end)
    else:
        ms_total = sum(ev[i][0].elapsed_time(ev[i][-1]) for i in range(args.steps))
    ms_total = max_over_ranks(ms_total, world, dev)
    stage_ms = {name: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                for j, name in enumerate(STAGES)}
    st = crisp.read_status(layer.ws)
    if st != 0:
        raise RuntimeError(f"device status after timing: {crisp.status_string(st)}")
    return ms_total / args.steps, stage_ms, clk, l2_note


def attention_roofline(layer, stage_ms, peaks):
    """The attention kernel's selected-block FLOP rate against the burst bf16
    peak (the sustained figure beside it), and the layer's work counts."""
    w = layer.w
    rb = layer.rowbits.cpu().numpy().view(np.uint32)
    pairs = selected_pairs(rb, w.n)
    blocks = int(layer.counts.cpu().numpy().astype(np.int64).sum())
    flops = 4 * 128 * pairs
    dense_pairs = w.hq * w.n * (w.n + 1) // 2
    hbm, burst, sustained, kind = peaks
    tf = flops / (stage_ms["attention"] * 1e-3) / 1e12
    routes = layer.route.cpu().numpy()
    return {"pairs": pairs, "blocks": blocks, "flops": flops, "dense_pairs": dense_pairs, "tflops": tf,
            "density": pairs / dense_pairs, "routes": {"vs": int(routes.sum()), "pe": int((routes == 0).sum())},
            "frac_burst": tf / burst, "frac_sustained": tf / sustained, "kind": kind}


def dense_run(torch, crisp, layer, attn_ms, ms_per_step):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w, st = layer.w, layer.stream
    e0.record(st)
    crisp.dense_prefill(layer.shape, layer.qd, layer.kd, layer.vd, layer.out, layer.ws, st)
    e1.record(st)
    torch.cuda.synchronize()
    d_ms = e0.elapsed_time(e1)
    dense_pairs = w.hq * w.n * (w.n + 1) // 2
    # put the sparse output back (the e2e check compares against it)
    crisp.sparse_prefill_mask(layer.shape, layer.qd, layer.kd, layer.vd, layer.rowbits, layer.order, layer.out,
                              layer.ws, st)
    return {"ms": d_ms, "tflops": 4 * 128 * dense_pairs / (d_ms * 1e-3) / 1e12, "attention_speedup": d_ms / attn_ms,
            "layer_speedup": d_ms / ms_per_step}


def map_path(torch, crisp, layer, stage_ms, hbm_peak):
    """The survey's map-reading calls on the same inputs, after the step: the
    proxy map written to HBM, C_struct routing from it, VS selection from it
    (each reads the whole map once). Their masses, routes and bitsets must
    equal the step's."""
    w, s, st, ws, p = layer.w, layer.shape, layer.stream, layer.ws, layer.params
    dev = layer.qd.device
    pmap = torch.empty((w.hq, B, num_blocks(w.n) * B), dtype=torch.float32, device=dev)
    E = lambda t: torch.empty_like(t)
    cs, tot, route = E(layer.cstruct), E(layer.total), E(layer.route)
    vm, sm, vb, sb = E(layer.vmass), E(layer.smass), E(layer.vbits), E(layer.sbits)
    ue = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    t = {"proxy": [], "route": [], "select": []}
    for _ in range(3):
        ue[0].record(st)
        crisp.proxy_map(s, layer.qd, layer.kd, pmap, ws, st)
        ue[1].record(st)
        crisp.route_cstruct(s, p, pmap, cs, tot, route, ws, st)
        ue[2].record(st)
        crisp.select_vs(s, p, pmap, route, vm, sm, vb, sb, ws, st)
        ue[3].record(st)
        torch.cuda.synchronize()
        t["proxy"].append(ue[0].elapsed_time(ue[1]))
        t["route"].append(ue[1].elapsed_time(ue[2]))
        t["select"].append(ue[2].elapsed_time(ue[3]))
    for a, b in ((cs, layer.cstruct), (tot, layer.total), (route, layer.route), (vm, layer.vmass), (sm, layer.smass),
                 (vb, layer.vbits), (sb, layer.sbits)):
        assert torch.equal(a, b), "the map-reading calls differ from the fused step"
    med = {k: statistics.median(v) for k, v in t.items()}
    map_bytes = 4 * w.hq * B * num_blocks(w.n) * B
    proxy_bytes = map_bytes + 2 * (2 * w.hkv * w.n * 128) + 2 * w.hq * B * 128
    gbs = lambda b, ms: b / (ms * 1e-3) / 1e9
    del pmap
    return {"proxy_map_ms": med["proxy"], "route_cstruct_ms": med["route"], "select_vs_ms": med["select"],
            "proxy_map_gbs": gbs(proxy_bytes, med["proxy"]), "route_cstruct_gbs": gbs(map_bytes, med["route"]),
            "select_vs_gbs": gbs(map_bytes, med["select"]), "peak_gbs": hbm_peak,
            "route_cstruct_frac": gbs(map_bytes, med["route"]) / hbm_peak,
            "select_vs_frac": gbs(map_bytes, med["select"]) / hbm_peak,
            "route_select_frac": gbs(2 * map_bytes, med["route"] + med["select"]) / hbm_peak,
            "bytes_note": "each call reads the fp32 map once (4*hq*128*ld bytes)",
            "fused_saving_ms": med["proxy"] + med["route"] + med["select"]
            - (stage_ms["proxy_masses"] + stage_ms["route"] + stage_ms["select_vs"])}


def e2e_run(torch, crisp, layer, args, world, local, dev):
    """End to end through the public API with HOST buffers: one call of
    crisp_prefill_layer_host per step, which uploads q, k, v from pinned host
    memory, runs the whole layer and downloads the output, one kv group at a
    time with the copies overlapped with the compute."""
    s, st = layer.shape, layer.stream
    lws = torch.empty(crisp.layer_workspace_size(s), dtype=torch.uint8, device=dev)
    crisp.workspace_init(lws)
    oh = torch.empty(tuple(layer.out.shape), dtype=torch.int16, pin_memory=True)
    qx, kx, vx = torch.empty_like(layer.qd), torch.empty_like(layer.kd), torch.empty_like(layer.vd)
    ox = torch.empty_like(layer.out)
    pipe = crisp.HostPipeline()
    facts = host_facts({"q": layer.qh.data_ptr(), "k": layer.kh.data_ptr(), "v": layer.vh.data_ptr(),
                        "out": oh.data_ptr()})

    def copy_probe():
        # one 1 GiB upload and one 1 GiB download between pinned and device memory
        nel = min(layer.qh.numel(), 2**29)
        src, dst = layer.qh.view(-1)[:nel], qx.view(torch.int16).view(-1)[:nel]
        c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        c0.record(st)
        dst.copy_(src, non_blocking=True)
        c1.record(st)
        oh.view(-1)[:nel].copy_(dst, non_blocking=True)
        c2.record(st)
        torch.cuda.synchronize()
        return {"h2d": nel * 2 / (c0.elapsed_time(c1) * 1e-3) / 1e9, "d2h": nel * 2 / (c1.elapsed_time(c2) * 1e-3) / 1e9,
                "bytes": nel * 2}

    def e2e_step():
        crisp.prefill_layer_host(pipe, s, layer.params, layer.qh, layer.kh, layer.vh, oh, qx, kx, vx, ox, lws, st)

    probe_before = copy_probe()
    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    # Three windows of K steps; the value is their median (the host-side
    # copy path of a shared machine varies between windows, so all three
    # are reported).
    windows = []
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(args.steps):
            e2e_step()
        b.record(st)
        torch.cuda.synchronize()
        windows.append(max_over_ranks(a.elapsed_time(b) / args.steps, world, dev))
    clk = clocks.stop()
    if crisp.read_status(lws) != 0:
        raise RuntimeError("device status after e2e")
    assert torch.equal(oh.view(torch.bfloat16).to(dev), layer.out), "e2e output differs from the device-resident run"
    probe_after = copy_probe()
    pipe.close()
    h2d = (layer.qh.numel() + layer.kh.numel() + layer.vh.numel()) * 2
    return {"value": statistics.median(windows) / world, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": oh.numel() * 2, "api": "crisp_prefill_layer_host",
            "windows_ms": [round(x / world, 3) for x in windows],
            "host_buffers_pinned": all(t.is_pinned() for t in (layer.qh, layer.kh, layer.vh, oh)), "clocks": clk,
            "copy_gbs_before": probe_before, "copy_gbs_after": probe_after,
            "copy_bound_ms": (h2d / probe_before["h2d"] + oh.numel() * 2 / probe_before["d2h"]) / 1e6,
            "host": facts}


def cpu_baseline(layer, alpha):
    w = layer.w
    r = cpu_sample(w, *(t.numpy().view(np.uint16) for t in (layer.qh, layer.kh, layer.vh)), alpha,
                   nthreads=os.cpu_count())
    cpu = {"value": r["layer_ms"], "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": r["sample"],
           "extrapolated": True, "sample_seconds": r["seconds"]}
    if w.n <= 8192:  # small layers: also the whole layer through the oracle on one core, no sampling
        cpu["full_layer_1core_ms"] = cpu_full_layer(w, *(t.numpy().view(np.uint16) for t in (layer.qh, layer.kh,
                                                                                               layer.vh)), alpha)
    return cpu


def run_crisp(args):
    import torch
    import dynamic_sparse_prefill_crisp_gb300 as crisp
    import synth
    from dynamic_sparse_prefill_crisp_gb300 import build as crisp_build

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    if rank == 0:
        crisp_build.build()
    barrier(world)
    dev = torch.device("cuda", local)
    alpha = tuple(int(x) for x in args.alpha.split("/"))
    pe_mode = crisp.PE_GAMMA if args.pe_mode == "gamma" else crisp.PE_NOISE
    params = crisp.params_default(alpha=alpha, pe_mode=pe_mode)
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    hbm_peak, burst_peak, sustained_peak, peak_kind = peaks

    w = workload(synth, args.config, args.seq_len)
    layer = Layer(crisp, torch, w, params, dev, stream)
    ms_per_step, stage_ms, clk, l2_note = time_steps(torch, layer, args, world, local, dev)
    roof = attention_roofline(layer, stage_ms, peaks)
    traffic, traffic_how = profiled_traffic(TRAFFIC_SOURCES, TRAFFIC_PROFILE, w, roof["blocks"])
    mp = None if args.no_map else map_path(torch, crisp, layer, stage_ms, hbm_peak)
    dense = None if args.no_dense else dense_run(torch, crisp, layer, stage_ms["attention"], ms_per_step)
    e2e = None if args.no_e2e else e2e_run(torch, crisp, layer, args, world, local, dev)
    cpu = cpu_baseline(layer, alpha) if rank == 0 and world == 1 and not args.no_cpu else None
    gen_s = layer.gen_s
    del layer
    torch.cuda.empty_cache()

    # The other workload the metric is quoted on, same process, same timing.
    also = None
    if args.also and args.also != args.config and not args.seq_len:
        w2 = workload(synth, args.also)
        l2 = Layer(crisp, torch, w2, params, dev, stream)
        ms2, stages2, clk2, l2note2 = time_steps(torch, l2, args, world, local, dev)
        roof2 = attention_roofline(l2, stages2, peaks)
        dense2 = None if args.no_dense else dense_run(torch, crisp, l2, stages2["attention"], ms2)
        cpu2 = cpu_baseline(l2, alpha) if rank == 0 and world == 1 and not args.no_cpu else None
        also = {"config": workload_config(w2, args, world), "l2_note": l2note2, "ms_per_layer": ms2,
                "stages_ms": {k: round(v, 4) for k, v in stages2.items()}, "routes": roof2["routes"],
                "density": roof2["density"], "eff_tflops": roof2["tflops"],
                "roofline": {"bound": "tensor", "kernel": "attention_kernel", "achieved": roof2["tflops"],
                             "peak": burst_peak, "unit": "TFLOP/s", "frac": roof2["frac_burst"],
                             "frac_sustained": roof2["frac_sustained"],
                             "peak_kind": f"bf16 dense, {peak_kind} burst"},
                "dense": dense2, "clocks": clk2, "cpu_baseline": cpu2,
                "gpu_launches": LAUNCHES_PER_STEP * args.steps}
        del l2
        torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": ms_per_step / world, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, planted sink/slash/needle structure)",
            "config": workload_config(w, args, world),
            "l2_note": l2_note,
            "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "routes": roof["routes"],
            "density": roof["density"],
            "eff_tflops": roof["tflops"],
            "roofline": {"bound": "tensor", "kernel": "attention_kernel", "achieved": roof["tflops"],
                         "peak": burst_peak, "unit": "TFLOP/s", "frac": roof["frac_burst"], "traffic": traffic,
                         "traffic_source": TRAFFIC_PROFILE, "traffic_how": traffic_how,
                         "peak_kind": f"bf16 dense, {peak_kind} burst (the kernel is timed alone by its own "
                                      f"events inside a ~{ms_per_step:.0f} ms step)",
                         "peak_sustained": sustained_peak, "frac_sustained": roof["frac_sustained"],
                         "algorithmic_flops": roof["flops"], "selected_blocks": roof["blocks"]},
            "map_path": mp,
            "dense": dense,
            "e2e": e2e,
            "also": also,
            "gpu_launches": LAUNCHES_PER_STEP * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "gen_seconds": gen_s,
        }
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------- sweeps
def time_layer(w, params, reps, dense=True):
    """One layer through crisp_prefill_layer (device-resident inputs; the
    routing and selection rules follow params) and dense attention on the
    same inputs; CUDA events, median of reps after one warm-up."""
    import torch
    import dynamic_sparse_prefill_crisp_gb300 as crisp
    q, k, v = w.generate()
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    qd, kd, vd = dev(q), dev(k), dev(v)
    hq, hkv, n = w.hq, w.hkv, w.n
    nb = num_blocks(n)
    W = (nb + 31) // 32
    out = torch.empty((hq, n, 128), dtype=torch.bfloat16, device="cuda")
    s = crisp.make_shape(hq, hkv, n, qd, kd, out)
    ws = torch.empty(crisp.layer_workspace_size(s), dtype=torch.uint8, device="cuda")
    crisp.workspace_init(ws)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    layer_ms = timed(lambda: crisp.prefill_layer(s, params, qd, kd, vd, out, ws))
    if crisp.read_status(ws) != 0:
        raise RuntimeError("device status after the sweep layer")
    views = crisp.layer_views(s, ws)

    def grab(name, shape, dtype):
        t = torch.empty(shape, dtype=dtype, device="cuda")
        off = views[name] - ws.data_ptr()
        t.view(torch.uint8).view(-1).copy_(ws[off:off + t.numel() * t.element_size()])
        return t.cpu().numpy()

    rb = grab("rowbits", (hq, nb, W), torch.int32).view(np.uint32)
    route = grab("route", (hq,), torch.uint8)
    counts = grab("counts", (hq, nb), torch.int32)
    pairs = selected_pairs(rb, n)
    dense_pairs = hq * n * (n + 1) // 2
    r = {"seq_len": n, "layer_ms": layer_ms, "density": pairs / dense_pairs, "routes_vs": int(route.sum()),
         "blocks_per_row": float(counts.mean())}
    if dense:
        r["dense_ms"] = timed(lambda: crisp.dense_prefill(s, qd, kd, vd, out, ws))
        r["speedup_vs_dense"] = r["dense_ms"] / layer_ms
    return r


def run_sweep(args):
    import torch
    import dynamic_sparse_prefill_crisp_gb300 as crisp
    import synth
    from dynamic_sparse_prefill_crisp_gb300 import build as crisp_build
    crisp_build.build()
    torch.cuda.set_device(0)
    rows = []
    if args.sweep == "lengths":
        base = synth.WORKLOADS["llama8b-32k"]
        for n in (2048, 4096, 8192, 16384, 32768, 65536, 131072):
            w = synth.Workload(**{**base.__dict__, "name": f"llama8b-recipe-{n}", "n": n})
            rows.append(time_layer(w, crisp.params_default(), reps=5))
        workload = "llama8b-32k recipe (32 q / 8 kv heads, half sink-type, half diffuse) at 2k-128k tokens"
    elif args.sweep == "alpha":
        w = synth.WORKLOADS["llama8b-512k"]
        for i, a in enumerate(((1, 1), (5, 4), (3, 2))):
            r = time_layer(w, crisp.params_default(alpha=a), reps=3, dense=(i == 0))
            r["alpha"] = f"{a[0]}/{a[1]}"
            rows.append(r)
        d = rows[0]["dense_ms"]
        for r in rows:
            r["speedup_vs_dense"] = d / r["layer_ms"]
        workload = "llama8b-512k (512k tokens, 32 q / 8 kv heads)"
    elif args.sweep == "flex":
        variants = [("CRISP (C_struct, noise floor alpha 1)", crisp.params_default()),
                    ("CRISP alpha 5/4", crisp.params_default(alpha=(5, 4))),
                    ("FlexPrefill rules gamma 0.95 (JSD routing, coverage on VS heads)",
                     crisp.params_default(route_mode=crisp.ROUTE_JSD, vs_mode=crisp.VS_GAMMA, vs_gamma=(95, 100))),
                    ("FlexPrefill rules gamma 0.97",
                     crisp.params_default(route_mode=crisp.ROUTE_JSD, vs_mode=crisp.VS_GAMMA, vs_gamma=(97, 100))),
                    # the pages' two ablations: each of CRISP's two changes alone
                    ("routing only (C_struct routing, coverage 0.95 on VS heads)",
                     crisp.params_default(vs_mode=crisp.VS_GAMMA, vs_gamma=(95, 100))),
                    ("sink-aware selection only (JSD routing, noise floor on VS heads)",
                     crisp.params_default(route_mode=crisp.ROUTE_JSD))]
        for cfg in ("llama8b-512k", "llama8b-32k"):
            w = synth.WORKLOADS[cfg]
            for i, (label, p) in enumerate(variants):
                r = time_layer(w, p, reps=3, dense=(i == 0))
                r.update(workload=cfg, rules=label)
                rows.append(r)
            d = rows[-len(variants)]["dense_ms"]
            for r in rows[-len(variants):]:
                r["speedup_vs_dense"] = d / r["layer_ms"]
        workload = ("llama8b-512k (all heads sink-type) and llama8b-32k (half diffuse); same kernels, rules differ; "
                    "the last two rows are the pages' ablations")
    else:
        w = synth.WORKLOADS["llama8b-32k"]
        for mode in (crisp.PE_GAMMA, crisp.PE_NOISE):
            r = time_layer(w, crisp.params_default(pe_mode=mode), reps=5, dense=(mode == crisp.PE_GAMMA))
            r["pe_mode"] = "gamma 19/20" if mode == crisp.PE_GAMMA else "noise floor (alpha 1)"
            rows.append(r)
        workload = "llama8b-32k (32k tokens, 16 sink-type + 16 diffuse heads)"
    print(json.dumps({"sweep": args.sweep, "workload": workload, "unit": "ms", "rows": rows}), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_crisp(args)


if __name__ == "__main__":
    sys.exit(main())
