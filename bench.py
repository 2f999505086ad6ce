#!/usr/bin/env python3
"""Benchmark of the fused FSDP FlatParameter shard step on GB300.

Default workload: one rank's step of the Llama-7B-shaped model (32 blocks of
202,383,360 params + a root unit of 262,148,096; W = 8 virtual ranks,
local-rank mode). One step = one fsdp_shard_step_grouped call over all 33
units: reduce-scatter of the rank's slice of the 8 bf16 gradients, Adam on the
rank's fp32 master/m/v shard, bf16 cast, and all-gather of the 7 other ranks'
bf16 shards into the 33 full bf16 FlatParameters. Algorithmic bytes per shard
element: 2W (gradients) + 24 (state read+write) + 2 (own bf16) + 4(W-1)
(other shards read + written) = 70 at W = 8.

Prints one JSON line (rank 0). Options pick other workloads for measurement
notes; the default is the headline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-e2e] [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused FSDP shard-step HBM GB/s and params/s, % of GB300 HBM peak"
UNIT = "GB/s"
KERNEL_SOURCES = ["fully_sharded_gb300/csrc/segment_kernel.cuh", "fully_sharded_gb300/csrc/abi.cu",
                  "fully_sharded_gb300/csrc/host_internal.h", "fully_sharded_gb300/csrc/tma_kernel.cuh"]
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "tma_kernel_llama7b_local_rank.md")


# ------------------------------------------------------------------ helpers

def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def virtual_rank(rank: int, world_size_virtual: int) -> int:
    """The virtual FSDP rank a GPU process steps: independent partitions, one per process."""
    return rank % world_size_virtual


def max_over_ranks(x: float, dist) -> float:
    """Slowest rank's time (no-op without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_ranks_ok(ok: bool, dist) -> bool:
    """True when every rank reports ok (no-op without a process group): ranks agree before a
    step that would otherwise leave a failed rank out of the next collective."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return bool(ok)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(t.item())


def whole_job_gbs(bytes_per_step_per_rank: int, nproc: int, ms_per_step: float) -> float:
    """Aggregate algorithmic GB/s: every rank's bytes over the slowest rank's step time."""
    return bytes_per_step_per_rank * nproc / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on this kernel source."""
    if not os.path.exists(TRAFFIC_PROFILE):
        return None
    text = open(TRAFFIC_PROFILE).read()
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_wl = re.search(r"workload:\s*(\S+)", text)
    m_b = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not (m_src and m_b and m_wl) or m_src.group(1) != kernel_source_hash() or m_wl.group(1) != workload:
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- workloads

def build_local_rank(wl, rank, torch, fs, synth, row_numel=0):
    """Device buffers of one rank's step over all units (local-rank mode). `row_numel`:
    the length of each gradient row of the pool (at least the largest unit's padded
    size, which is the default)."""
    from synth import workloads as wls
    W = wl.world_size
    lays = [fs.fsdp_flatten_layout(wls.numels(u), W)[0] for u in wl.units]
    S_tot = sum(l.shard_numel for l in lays)
    pad_tot = sum(l.padded_numel for l in lays)
    maxpad = max([l.padded_numel for l in lays] + [row_numel])
    dev = torch.device("cuda")
    # gradient pool: 2 unit-sets of W rows (units alternate between them)
    slots = min(2, len(lays))
    pool = [torch.empty((W, maxpad), dtype=torch.int16, device=dev) for _ in range(slots)]
    for s in range(slots):
        for k in range(W):
            synth.fill_(pool[s][k], wls.key_grad(wl, s, k, 0), wl.sigma_grad)
    master = torch.empty(S_tot, device=dev)
    exp_avg = torch.empty(S_tot, device=dev)
    exp_avg_sq = torch.empty(S_tot, device=dev)
    others = torch.empty((W, S_tot), dtype=torch.int16, device=dev)
    full = torch.empty(pad_tot, dtype=torch.int16, device=dev)
    units = []
    so = po = 0
    for u, lay in enumerate(lays):
        S, padded, P = lay.shard_numel, lay.padded_numel, lay.numel
        sl = slice(so, so + S)
        synth.fill_(master[sl], wls.key_master(wl, u), wl.sigma_master, idx0=rank * S, n_valid=P)
        for buf, key in ((exp_avg, wls.key_exp_avg(wl, u)), (exp_avg_sq, wls.key_exp_avg_sq(wl, u))):
            if wl.sigma_state:
                synth.fill_(buf[sl], key, wl.sigma_state, idx0=rank * S, absval=True, n_valid=P)
            else:
                buf[sl].zero_()
        oth = [None] * W
        for k in range(W):
            if k != rank:
                synth.fill_(others[k, sl], wls.key_shard(wl, u), wl.sigma_master, idx0=k * S, n_valid=P)
                oth[k] = others[k, sl]
        units.append(dict(layout=lay, grads=[pool[u % slots][k, :padded] for k in range(W)],
                          master=[master[sl]], exp_avg=[exp_avg[sl]], exp_avg_sq=[exp_avg_sq[sl]],
                          other_shards=oth, full_out=[full[po:po + padded]]))
        so += S
        po += padded
    torch.cuda.synchronize()
    bytes_per_step = (6 * W + 22) * S_tot
    info = dict(units=len(lays), W=W, rank=rank, params=sum(l.numel for l in lays),
                shard_elems=S_tot, bytes_per_step=bytes_per_step, elems_per_step=S_tot,
                mode="local-rank")
    bufs = dict(pool=pool, master=master, exp_avg=exp_avg, exp_avg_sq=exp_avg_sq, others=others,
                full=full)
    return units, info, bufs


def build_all_ranks(wl, F, torch, fs, synth):
    """Device buffers of the all-ranks step (every rank's state updated, every group gathered)."""
    from synth import workloads as wls
    W = wl.world_size
    R = W // F
    dev = torch.device("cuda")
    units = []
    keep = []
    S_sum = pad_sum = 0
    for u, shapes in enumerate(wl.units):
        lay = fs.fsdp_flatten_layout(wls.numels(shapes), W, F)[0]
        S, padded, P = lay.shard_numel, lay.padded_numel, lay.numel
        grads = torch.empty((W, padded), dtype=torch.int16, device=dev)
        for k in range(W):
            synth.fill_(grads[k], wls.key_grad(wl, u, k, 0), wl.sigma_grad, n_valid=P)
        st = [torch.empty((R, padded), device=dev) for _ in range(3)]
        for g in range(R):
            synth.fill_(st[0][g], wls.key_master(wl, u), wl.sigma_master, n_valid=P)
            for j, key in ((1, wls.key_exp_avg(wl, u)), (2, wls.key_exp_avg_sq(wl, u))):
                if wl.sigma_state:
                    synth.fill_(st[j][g], key, wl.sigma_state, absval=True, n_valid=P)
                else:
                    st[j][g].zero_()
        full = torch.empty((R, padded), dtype=torch.int16, device=dev)
        ranks = range(W)
        units.append(dict(layout=lay, grads=[grads[k] for k in range(W)],
                          master=[st[0][r // F, (r % F) * S:(r % F + 1) * S] for r in ranks],
                          exp_avg=[st[1][r // F, (r % F) * S:(r % F + 1) * S] for r in ranks],
                          exp_avg_sq=[st[2][r // F, (r % F) * S:(r % F + 1) * S] for r in ranks],
                          other_shards=None, full_out=[full[g] for g in range(R)]))
        keep.append((grads, st, full))
        S_sum += S
        pad_sum += padded
    torch.cuda.synchronize()
    # per padded element: W bf16 gradient reads, and per replica the fp32 master/m/v
    # read + write (24) and the bf16 write into its group's full buffer (2)
    bytes_per_step = (2 * W + 26 * R) * pad_sum
    info = dict(units=len(wl.units), W=W, F=F, R=R, params=sum(u["layout"].numel for u in units),
                padded_elems=pad_sum, bytes_per_step=bytes_per_step, elems_per_step=pad_sum,
                mode="all-ranks")
    return units, info, keep


def sweep_workload(n, W):
    """One FlatParameter of n elements at W ranks (the size sweep of the 7B configuration)."""
    from synth.workloads import Workload
    return Workload("sweep", 6, [[(n,)]], W, sigma_state=1e-4)


def build_sweep(n, W, torch, fs, synth):
    return build_all_ranks(sweep_workload(n, W), W, torch, fs, synth)


# ------------------------------------------------------------ the GPU arm

def bench_line(info, workload_name, nproc, steps, warmup, ms_per_step, local_ms, launches_per_step,
               tma_launches, l2_bytes, clocks, peak=None):
    """The JSON line of the GPU arm. `ms_per_step`: the slowest rank's time per step;
    `local_ms`: this rank's time for all `steps` (its launches' mean duration gives the
    roofline's achieved bandwidth); `peak`: (GB/s, "measured"|"fallback"), read from
    MEASURED_PEAKS.json when not given."""
    bytes_step = info["bytes_per_step"]
    value = whole_job_gbs(bytes_step, nproc, ms_per_step)
    peak, peak_kind = measured_peaks() if peak is None else peak
    mean_launch_ms = local_ms / (steps * launches_per_step)  # this rank's launches
    achieved = bytes_step / launches_per_step / (mean_launch_ms * 1e-3) / 1e9
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": nproc,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": workload_name,
            "W": info["W"],
            "units": info["units"],
            "params": info["params"],
            "elems_per_step": info["elems_per_step"],
            "algorithmic_bytes_per_step": bytes_step,
            "mode": info["mode"],
            "parallelism": "W=%d virtual ranks in one GPU's HBM; %d GPU process(es), each an independent "
                           "step, no data-path collective" % (info["W"], nproc),
            "l2": ("inputs larger than L2: %.1f GB touched per step vs %.0f MB L2"
                   % (bytes_step / 1e9, l2_bytes / 1e6) if bytes_step > 2 * l2_bytes else
                   "working set %.0f MB is within 2x the %.0f MB L2: L2-resident, not an HBM figure"
                   % (bytes_step / 1e6, l2_bytes / 1e6)),
            "storage": "bf16 gradients/params, fp32 master/m/v",
        },
        "params_per_s": round(info["elems_per_step"] * nproc / (ms_per_step * 1e-3), 1),
        "pct_of_hbm_peak": round(100.0 * value / nproc / peak, 2),
        "pct_of_nominal_8tbs": round(100.0 * value / nproc / 8000.0, 2),
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": peak_kind,
            "kernel": ("fsdp::tma_kernel<%d>" % (16 if info["W"] == 16 else 8) if tma_launches == launches_per_step
                       else "fsdp::segment_kernel<%d>" % (info["W"] if info["W"] in (1, 2, 4, 8, 16) else 0)),
            "traffic": profiled_traffic(workload_name),
        },
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
    }


def run_ours(args):
    import torch
    import fully_sharded_gb300 as fs
    import synth
    from synth import workloads as wls

    rank, world, local_rank = env_rank()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    name = args.workload
    if name == "llama7b":
        wl = wls.LLAMA7B
        row_numel = 0
        if args.units:
            # the first units, with the gradient rows as far apart as in the whole step
            row_numel = max(fs.fsdp_flatten_layout(wls.numels(u), wl.world_size)[0].padded_numel
                            for u in wl.units)
            wl = wls.Workload(wl.name, wl.config_id, wl.units[:args.units], wl.world_size,
                              sigma_state=wl.sigma_state)
        vrank = virtual_rank(rank, wl.world_size)
        units, info, bufs = build_local_rank(wl, vrank, torch, fs, synth, row_numel)
        rb, re = vrank, vrank + 1
        workload_name = "llama7b_local_rank" + ("_units%d" % args.units if args.units else "")
    elif name in ("llama_block", "gpt2_small", "tiny_mlp"):
        wl = wls.ALL[name]
        units, info, bufs = build_all_ranks(wl, wl.world_size, torch, fs, synth)
        rb, re = 0, wl.world_size
        workload_name = name + "_all_ranks"
    elif name.startswith("hybrid"):
        F = int(name.split("_F")[1]) if "_F" in name else 16
        wl = wls.HYBRID
        units, info, bufs = build_all_ranks(wl, F, torch, fs, synth)
        rb, re = 0, wl.world_size
        workload_name = "hybrid_W16_F%d" % F
    elif name.startswith("sweep"):
        # sweep_<n>_W<w>, or sweep_<n>_W<w>_F<f> for a hybrid step (F | W, R = W / F replicas)
        parts = name.split("_")
        n, W = int(float(parts[1])), int(parts[2][1:])
        F = int(parts[3][1:]) if len(parts) > 3 else W
        units, info, bufs = build_all_ranks(sweep_workload(n, W), F, torch, fs, synth)
        rb, re = 0, W
        workload_name = name
    else:
        raise SystemExit("unknown workload %s" % name)
    batch = fs.UnitBatch(units)
    launches_per_step, tma_launches = fs.fsdp_shard_step_grouped_plan(batch, rb, re)
    stream = torch.cuda.Stream()

    # warm-up
    t = 1
    for _ in range(args.warmup):
        fs.fsdp_shard_step_grouped(batch, rb, re, fs.AdamHyper(step=t), stream=stream)
        t += 1
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(visible[local_rank].strip() if len(visible) > local_rank and visible[local_rank].strip()
                          else torch.cuda.current_device())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    fs.fsdp_device_status(clear=True)
    clocks.start()
    time.sleep(0.3)
    # one event pair around the whole timed region: events between launches would
    # stop consecutive launches from overlapping (programmatic dependent launch)
    stream.record_event(start)
    for i in range(args.steps):
        fs.fsdp_shard_step_grouped(batch, rb, re, fs.AdamHyper(step=t), stream=stream)
        t += 1
    stream.record_event(stop)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if fs.fsdp_device_status() != 0:
        raise RuntimeError("a bounded device wait ran out during the timed steps: blocks stopped early, "
                           "so the timing is not of the whole step")
    if dist:
        dist.barrier()
    local_ms = start.elapsed_time(stop)
    total_ms = max_over_ranks(local_ms, dist)
    ms_per_step = total_ms / args.steps
    nproc = world
    # L2 size as the device reports it (129 MB on GB300 when the property is absent)
    l2 = float(getattr(torch.cuda.get_device_properties(local_rank), "L2_cache_size", 0) or 129e6)
    line = bench_line(info, workload_name, world, args.steps, args.warmup, ms_per_step, local_ms,
                      launches_per_step, tma_launches, l2, clk)
    if ms_per_step < 1.0 and launches_per_step == 1:
        # short steps: where host cost per call can matter, report it apart from the device time
        line["host_us"] = host_breakdown(torch, fs, batch, rb, re, stream)
    if not args.no_e2e and name == "llama7b" and not args.units:
        line["e2e"] = e2e_local_rank(args, torch, fs, synth, wls.LLAMA7B, units, info, bufs, rb, stream,
                                     nproc, dist)
    # the oracle baseline: rank 0 of a one-GPU run only
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        if name == "llama7b":
            line["cpu_baseline"] = cpu_baseline(units, info, bufs, rb, torch, seconds=args.cpu_seconds)
        else:
            line["cpu_baseline"] = cpu_baseline_all_ranks(units, torch, seconds=min(args.cpu_seconds, 3.0))
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def host_breakdown(torch, fs, batch, rb, re, stream, reps=200, graph_launches=20):
    """Per-call cost of fsdp_shard_step_grouped, host and device apart (microseconds):
    `binding`: the Python call (marshalling + the library call), `library`: the C call
    made directly through ctypes less a bare ctypes call of the same signature
    (validation, descriptor tables and the kernel launch), `ctypes_call`: that bare call
    (zero units: it returns after checking its arguments), each the median of `reps`
    calls timed one at a time with the device idle before each (so that no call waits
    for room in the launch queue), and `device_per_launch`: one launch's device time,
    from a CUDA graph of `graph_launches` launches replayed (no host work between them)."""
    import ctypes
    hp = fs.AdamHyper(step=1)
    st = stream.cuda_stream
    lib = fs._lib

    def per_call(fn):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        torch.cuda.synchronize()
        return statistics.median(ts) * 1e6

    binding = per_call(lambda: fs.fsdp_shard_step_grouped(batch, rb, re, hp, stream=stream))
    args = (batch.array, batch.n, rb, re, ctypes.byref(hp), st)
    direct = per_call(lambda: lib.fsdp_shard_step_grouped(*args))
    bare_args = (batch.array, 0, rb, re, ctypes.byref(hp), st)
    bare = per_call(lambda: lib.fsdp_shard_step_grouped(*bare_args))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(graph_launches):
            fs.fsdp_shard_step_grouped(batch, rb, re, hp, stream=stream)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    replays = 10
    stream.record_event(a)
    with torch.cuda.stream(stream):
        for _ in range(replays):
            g.replay()
    stream.record_event(b)
    torch.cuda.synchronize()
    device = a.elapsed_time(b) * 1e3 / (replays * graph_launches)
    del g
    return {"binding": round(binding, 2), "library": round(direct - bare, 2), "ctypes_call": round(bare, 2),
            "device_per_launch": round(device, 2), "calls": reps,
            "note": "host: median of %d calls, each alone with the device idle before it; device: a CUDA "
                    "graph of %d launches replayed %d times" % (reps, graph_launches, replays)}


def pipeline_setup(torch, fs, units, info, rank, n_slots):
    """Pinned host gradient slices of every unit (W x S each, unit-major), pinned result
    buffers and a staging pool of n_slots slots, for fsdp_pipeline_step."""
    W = info["W"]
    lays = [u["layout"] for u in units]
    S_tot = info["shard_elems"]
    host_g = torch.empty(W * S_tot, dtype=torch.int16, pin_memory=True)
    host_out = torch.empty(S_tot, dtype=torch.int16, pin_memory=True)
    punits = []
    so = 0
    for u, lay in enumerate(lays):
        S = lay.shard_numel
        g = host_g[W * so:W * (so + S)]
        for k in range(W):
            g[k * S:(k + 1) * S].copy_(units[u]["grads"][k][rank * S:(rank + 1) * S])
        punits.append(dict(layout=lay, grad_slices=g, master=units[u]["master"][0],
                           exp_avg=units[u]["exp_avg"][0], exp_avg_sq=units[u]["exp_avg_sq"][0],
                           other_shards=units[u]["other_shards"], full_out=units[u]["full_out"][0],
                           shard_out=host_out[so:so + S]))
        so += S
    slot = max(l.padded_numel for l in lays)
    staging = torch.empty(n_slots * slot, dtype=torch.int16, device="cuda")
    return fs.PipelineBatch(punits), staging, slot, (host_g, host_out)


def time_pipeline(torch, fs, batch, staging, slot, n_slots, rank, steps, warmup, dist, compute, copy):
    t = 10_000
    for _ in range(max(1, warmup)):
        fs.fsdp_pipeline_step(batch, rank, staging, slot, n_slots, fs.AdamHyper(step=t), compute=compute,
                              copy=copy)
        t += 1
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        fs.fsdp_pipeline_step(batch, rank, staging, slot, n_slots, fs.AdamHyper(step=t), compute=compute,
                              copy=copy)
        t += 1
    torch.cuda.synchronize()
    return max_over_ranks((time.perf_counter() - t0) * 1e3 / steps, dist)


def e2e_local_rank(args, torch, fs, synth, wl, units, info, bufs, rank, stream, nproc, dist):
    """Same metric through the public API with host buffers.

    Per step, fsdp_pipeline_step copies each unit's inputs (the rank's slice of
    each of the W gradients) from pinned host memory into a staging slot,
    steps the unit, and reads the step's result (the rank's new bf16 shard)
    back to pinned host memory. Two slots: unit u+1's copy overlaps unit u's
    step (prefetch 1)."""
    W = info["W"]
    S_tot = info["shard_elems"]
    # the inputs' page-locked host buffers (2 W + 2 bytes per shard element per rank): every
    # rank must have them before any rank enters the timed, synchronised steps
    err = None
    try:
        batch, staging, slot, keep = pipeline_setup(torch, fs, units, info, rank, 2)
    except (RuntimeError, MemoryError) as e:
        err = str(e).splitlines()[0][:160] if str(e) else type(e).__name__
    if not all_ranks_ok(err is None, dist):
        return {"value": None, "unit": UNIT, "h2d_bytes_per_step": 2 * W * S_tot, "d2h_bytes_per_step": 2 * S_tot,
                "unavailable": "page-locked host buffers for the step's inputs could not be allocated on every "
                               "rank" + (": " + err if err else "")}
    k = max(1, min(args.steps, args.e2e_steps))
    copy = torch.cuda.Stream()
    # three blocks of K steps, the best one reported: the host link is shared with work
    # outside this process, which stalls some blocks (all three are in the record)
    blocks = [time_pipeline(torch, fs, batch, staging, slot, 2, rank, k, args.warmup if b == 0 else 1, dist,
                            stream, copy) for b in range(3)]
    ms = min(blocks)
    # the same steps once more, each timed on its own (synchronized before and after):
    # steps far above the median are the host link busy with work outside this process
    per_step = []
    for i in range(k):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fs.fsdp_pipeline_step(batch, rank, staging, slot, 2, fs.AdamHyper(step=20_000 + i), compute=stream,
                              copy=copy)
        torch.cuda.synchronize()
        per_step.append((time.perf_counter() - t0) * 1e3)
    h2d_bytes, d2h_bytes = 2 * W * S_tot, 2 * S_tot
    link = host_link(torch, copy)
    floor_ms = h2d_bytes / (link["h2d_GB_per_s"] * 1e9) * 1e3
    link.update({"floor_ms": round(floor_ms, 2), "frac_of_floor": round(floor_ms / ms, 4)})
    if nproc == 1:  # one process: the host's link and memory are not shared with other ranks
        # the results go back while inputs still come in: during those bytes each direction
        # runs at the two-way rate, the rest of the inputs at the one-way rate
        both = host_link_both_ways(torch, copy, torch.cuda.Stream())
        floor2_ms = (d2h_bytes / (both / 2 * 1e9) + (h2d_bytes - d2h_bytes) / (link["h2d_GB_per_s"] * 1e9)) * 1e3
        link.update({"both_ways_GB_per_s_total": both, "floor_two_way_ms": round(floor2_ms, 2),
                     "frac_of_floor_two_way": round(floor2_ms / ms, 4)})
        link["host_memory"] = host_memory_bandwidth(torch)
    link["placement"] = host_placement(torch, {"grad_slices": keep[0], "shard_out": keep[1]})
    return {"value": round(whole_job_gbs(info["bytes_per_step"], nproc, ms), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "ms_per_step": round(ms, 3),
            "steps": k, "blocks_ms": [round(b, 3) for b in blocks], "host_link": link,
            "per_step_ms": {"median": round(statistics.median(per_step), 2), "min": round(min(per_step), 2),
                            "max": round(max(per_step), 2)},
            "note": "host wall clock around K fsdp_pipeline_step calls (2 staging slots), pinned host "
                    "buffers, best of three blocks (blocks_ms); per_step_ms: K more calls, each timed "
                    "alone; host_link: pinned copy "
                    "bandwidth measured right after, floor_ms = the step's H2D bytes at the one-way "
                    "rate, floor_two_way_ms = its D2H bytes at the two-way rate (both directions "
                    "loaded) plus the remaining H2D bytes at the one-way rate; host_link.placement: "
                    "NUMA nodes, the GPU's node and the nodes of the pinned buffers' pages; "
                    "host_link.host_memory: the host's own read, write and copy bandwidth"}


def host_placement(torch, buffers):
    """Where page-locked host buffers live relative to the GPU, as the OS reports it (nothing
    is changed): the host's NUMA nodes and their CPUs, the GPU's NUMA node (sysfs, by the
    device's PCI address) and, per buffer, the pages on each node of the mappings that hold
    it, and their page size (/proc/self/maps and /proc/self/numa_maps). `buffers`: name ->
    host tensor."""
    import glob
    out = {"numa_nodes": {}}
    for n in sorted(glob.glob("/sys/devices/system/node/node[0-9]*")):
        try:
            out["numa_nodes"][os.path.basename(n)] = open(n + "/cpulist").read().strip()
        except OSError:
            pass
    try:
        p = torch.cuda.get_device_properties(torch.cuda.current_device())
        pci = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        out["gpu_pci"] = pci
        out["gpu_numa_node"] = int(open("/sys/bus/pci/devices/%s/numa_node" % pci).read().strip())
    except (OSError, AttributeError, ValueError, RuntimeError):
        out["gpu_numa_node"] = None
    try:
        spans = []
        for line in open("/proc/self/maps"):
            a, b = line.split()[0].split("-")
            spans.append((int(a, 16), int(b, 16)))
        info = {}
        for line in open("/proc/self/numa_maps"):
            f = line.split()
            info[int(f[0], 16)] = f[1:]
        bufs = {}
        for name, t in buffers.items():
            lo, hi = t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()
            pages, kb, mapped = {}, set(), 0
            for a, b in spans:
                if b <= lo or a >= hi or a not in info:
                    continue
                mapped += b - a
                for field in info[a]:
                    k, _, v = field.partition("=")
                    if k.startswith("N") and k[1:].isdigit():
                        pages[k] = pages.get(k, 0) + int(v)
                    elif k == "kernelpagesize_kB":
                        kb.add(int(v))
            # the counts cover the whole mappings that hold the buffer (they may hold more)
            bufs[name] = {"mapping_pages_per_node": pages, "page_kB": sorted(kb), "bytes": hi - lo,
                          "mapping_bytes": mapped}
        out["buffers"] = bufs
    except OSError as e:
        out["buffers"] = {"unavailable": str(e)[:120]}
    return out


def host_memory_bandwidth(torch, nbytes=1 << 31, reps=3):
    """The host's own memory bandwidth as this process sees it, with torch's CPU threads
    (GB/s, best of `reps`): a read (sum of a buffer), a write (fill) and a copy (its read and
    write bytes both counted). The copy engines' host-side traffic competes for the same
    memory: a host-to-device copy reads it, a device-to-host copy writes it."""
    a = torch.empty(nbytes // 4, dtype=torch.float32)
    a.fill_(1.0)
    b = torch.empty_like(a)

    def best(fn, nb):
        t = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            t = min(t, time.perf_counter() - t0)
        return round(nb / t / 1e9, 1)

    out = {"read_GB_per_s": best(lambda: a.sum(), nbytes), "write_GB_per_s": best(lambda: b.fill_(2.0), nbytes),
           "copy_GB_per_s": best(lambda: b.copy_(a), 2 * nbytes), "threads": torch.get_num_threads()}
    del a, b
    return out


def host_link(torch, stream, nbytes=1 << 31, reps=3):
    """Pinned host <-> device copy bandwidth (GB/s), best of `reps` single copies of `nbytes`
    on `stream`: the bound of a step whose inputs arrive from host memory."""
    host = torch.empty(nbytes // 2, dtype=torch.int16, pin_memory=True)
    host.zero_()
    dev = torch.empty(nbytes // 2, dtype=torch.int16, device="cuda")
    out = {}
    for name, dst, src in (("h2d_GB_per_s", dev, host), ("d2h_GB_per_s", host, dev)):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(stream):
                dst.copy_(src, non_blocking=True)
            stream.synchronize()
            best = min(best, time.perf_counter() - t0)
        out[name] = round(nbytes / best / 1e9, 1)
    del host, dev
    return out


def host_link_both_ways(torch, h2d, d2h, nbytes=3 << 30, reps=3):
    """Pinned host <-> device copy bandwidth with both directions at once (GB/s summed over
    the two), best of `reps`: one copy of `nbytes` each way, on two streams."""
    hs = torch.empty(nbytes // 2, dtype=torch.int16, pin_memory=True)
    hs.zero_()
    hd = torch.empty(nbytes // 2, dtype=torch.int16, pin_memory=True)
    ds = torch.zeros(nbytes // 2, dtype=torch.int16, device="cuda")
    dd = torch.empty(nbytes // 2, dtype=torch.int16, device="cuda")
    best = float("inf")
    for _ in range(reps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(h2d):
            dd.copy_(hs, non_blocking=True)
        with torch.cuda.stream(d2h):
            hd.copy_(ds, non_blocking=True)
        torch.cuda.synchronize()
        best = min(best, time.perf_counter() - t0)
    del hs, hd, ds, dd
    return round(2 * nbytes / best / 1e9, 1)


def run_unfused(args):
    """The step's parts as separate calls, timed on the Llama block (W = 8, all ranks):
    fsdp_reduce_scatter_ranks (every rank's fp32 gradient shard, one launch),
    fsdp_adam_shard_step_grouped (every rank's Adam with its bf16 shard, one launch) and
    fsdp_all_gather of the 8 shards, and the same parts one rank per launch; against the
    fused step on the same buffers. Also fsdp_pack_flat of the block's nine fp32 tensors."""
    import torch
    import fully_sharded_gb300 as fs
    import synth
    from synth import workloads as wls
    torch.cuda.set_device(0)
    # the Llama block, or (--unfused-elems n) one FlatParameter of n elements at W = 8: a
    # case small enough for a many-pass profile
    wl = sweep_workload(args.unfused_elems, 8) if args.unfused_elems else wls.LLAMA_BLOCK
    W = wl.world_size
    units, info, keep = build_all_ranks(wl, W, torch, fs, synth)
    u = units[0]
    lay = u["layout"]
    S, padded = lay.shard_numel, lay.padded_numel
    gshard = torch.empty((W, S), device="cuda")
    bshard = torch.empty((W, S), dtype=torch.int16, device="cuda")
    full = u["full_out"][0]
    stream = torch.cuda.Stream()

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.record_event(a)
        for _ in range(reps):
            fn()
        stream.record_event(b)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    hp = fs.AdamHyper(step=1)
    # one launch per part: every rank's reduce-scatter, every rank's Adam, the gather
    rs = lambda: fs.fsdp_reduce_scatter_ranks(u["grads"], lay, 0, W, [gshard[r] for r in range(W)],  # noqa
                                              stream=stream)
    adam_batch = fs.AdamShardBatch([dict(master=u["master"][r], exp_avg=u["exp_avg"][r],
                                         exp_avg_sq=u["exp_avg_sq"][r], grad_shard=gshard[r],
                                         bf16_shard_out=bshard[r]) for r in range(W)])
    ad = lambda: fs.fsdp_adam_shard_step_grouped(adam_batch, hp, stream=stream)  # noqa
    ag = lambda: fs.fsdp_all_gather([bshard[r] for r in range(W)], lay, full, stream=stream)  # noqa
    # the same parts one rank per launch (8 + 8 + 1 launches)
    rs1 = lambda: [fs.fsdp_reduce_scatter(u["grads"], lay, r, gshard[r], stream=stream) for r in range(W)]  # noqa
    ad1 = lambda: [fs.fsdp_adam_shard_step(u["master"][r], u["exp_avg"][r], u["exp_avg_sq"][r], gshard[r],  # noqa
                                           hp, bshard[r], stream=stream) for r in range(W)]
    batch = fs.UnitBatch(units)
    fused = lambda: fs.fsdp_shard_step_grouped(batch, 0, W, hp, stream=stream)  # noqa
    n = args.steps
    t_rs, t_ad, t_ag, t_fused = timed(rs, n), timed(ad, n), timed(ag, n), timed(fused, n)
    t_rs1, t_ad1 = timed(rs1, n), timed(ad1, n)
    b_rs, b_ad, b_ag = (2 * W + 4) * padded, (4 + 24 + 2) * padded, 4 * padded
    # a2: pack the nine fp32 tensors of the block into the flat master
    numels = wls.numels(wl.units[0])
    tensors = [torch.empty(n_, device="cuda").normal_() for n_ in numels]
    lay2, offs = fs.fsdp_flatten_layout(numels, W)
    flat = torch.empty(lay2.padded_numel, device="cuda")
    t_pack = timed(lambda: fs.fsdp_pack_flat(tensors, lay2, offs, flat, stream=stream), n)
    peak, _ = measured_peaks()
    row = lambda ms, b: {"ms": round(ms, 4), "GB_per_s": round(b / (ms * 1e-3) / 1e9, 1),  # noqa
                         "frac_of_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4)}
    oracle_base = None if args.no_cpu_baseline else oracle_parts_baseline(W, 1 << 17)
    print(json.dumps({
        "workload": ("sweep_%d_W8_unfused" % args.unfused_elems) if args.unfused_elems
        else "llama_block_all_ranks_unfused", "W": W, "padded_elems": padded,
        "reduce_scatter_ranks": row(t_rs, b_rs), "adam_shard_step_grouped": row(t_ad, b_ad),
        "all_gather": row(t_ag, b_ag),
        "unfused_total": row(t_rs + t_ad + t_ag, b_rs + b_ad + b_ag), "unfused_launches": 3,
        "per_rank_launches": {"reduce_scatter_x8": row(t_rs1, b_rs), "adam_shard_step_x8": row(t_ad1, b_ad),
                              "unfused_total": row(t_rs1 + t_ad1 + t_ag, b_rs + b_ad + b_ag),
                              "unfused_launches": 2 * W + 1},
        "fused": row(t_fused, (2 * W + 26) * padded),
        "fused_speedup": round((t_rs + t_ad + t_ag) / t_fused, 3),
        "pack_f32": row(t_pack, 8 * lay2.numel),
        "bytes_per_element": {"unfused": 2 * W + 38, "fused": 2 * W + 26}, "cpu_baseline": oracle_base}), flush=True)


def run_offload(args):
    """Optimizer-state offload: the 7B local-rank step with the rank's fp32 master, m and v
    in page-locked host memory, against the same step with the state in HBM. Two forms:
    zero-copy (the fused kernel reads and writes the mapped host memory over the link) and
    staged (fsdp_offload_step: copy engines move each unit's state in and out on their own
    streams, both link directions at once, and the kernel steps it in HBM)."""
    import torch
    import fully_sharded_gb300 as fs
    import synth
    from synth import workloads as wls
    torch.cuda.set_device(0)
    wl = wls.LLAMA7B
    units, info, bufs = build_local_rank(wl, 0, torch, fs, synth)
    stream = torch.cuda.Stream()

    def timed(batch, steps):
        for t in range(1, 4):
            fs.fsdp_shard_step_grouped(batch, 0, 1, fs.AdamHyper(step=t), stream=stream)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.record_event(a)
        for t in range(steps):
            fs.fsdp_shard_step_grouped(batch, 0, 1, fs.AdamHyper(step=10 + t), stream=stream)
        stream.record_event(b)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    ms_hbm = timed(fs.UnitBatch(units), args.steps)
    host = {n: bufs[n].cpu().pin_memory() for n in ("master", "exp_avg", "exp_avg_sq")}
    so = 0
    off_units = []
    for u in units:
        S = u["layout"].shard_numel
        off_units.append(dict(u, master=[host["master"][so:so + S].data_ptr()],
                              exp_avg=[host["exp_avg"][so:so + S].data_ptr()],
                              exp_avg_sq=[host["exp_avg_sq"][so:so + S].data_ptr()]))
        so += S
    ms_host = timed(fs.UnitBatch(off_units), max(2, args.steps // 10))
    S_tot = info["shard_elems"]
    # staged: each unit's state copied in on one stream, stepped in HBM, copied back on another
    staged_units = []
    so = 0
    for u in units:
        S = u["layout"].shard_numel
        staged_units.append(dict(layout=u["layout"], grads=u["grads"], master=host["master"][so:so + S],
                                 exp_avg=host["exp_avg"][so:so + S], exp_avg_sq=host["exp_avg_sq"][so:so + S],
                                 other_shards=u["other_shards"], full_out=u["full_out"][0]))
        so += S
    staged_batch = fs.OffloadBatch(staged_units)
    slot = (max(u["layout"].shard_numel for u in units) + 3) // 4 * 4
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    staged = {}
    for n_slots in (2, 3):
        staging = torch.empty(n_slots * 3 * slot, device="cuda")

        def step(t):
            fs.fsdp_offload_step(staged_batch, 0, staging, slot, n_slots, fs.AdamHyper(step=t),
                                 compute=stream, h2d=h2d, d2h=d2h)

        for t in range(1, 3):
            step(t)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(2, args.steps // 10)
        stream.record_event(a)
        for t in range(n):
            step(10 + t)
        stream.record_event(b)  # the call orders `stream` after its last copy back
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / n
        staged["slots_%d" % n_slots] = {
            "ms_per_step": round(ms, 3), "GB_per_s": round(info["bytes_per_step"] / (ms * 1e-3) / 1e9, 1),
            "host_link_GB_per_s": round(24 * S_tot / (ms * 1e-3) / 1e9, 1),
            "staging_bytes": staging.numel() * 4}
        del staging
    best = min(v["ms_per_step"] for v in staged.values())
    # the staged step moves 12 B per shard element each way, both directions at once
    both = host_link_both_ways(torch, h2d, d2h)
    floor_ms = 12 * S_tot / (both / 2 * 1e9) * 1e3
    # a pipeline cannot keep both directions busy from start to end: the first unit's state
    # arrives before anything goes back, the last unit's goes back after everything came in
    # (each at its one-way rate); the rest moves at the two-way rate
    link1 = host_link(torch, h2d)
    first, last = 12 * units[0]["layout"].shard_numel, 12 * units[-1]["layout"].shard_numel
    fill_drain_ms = (first / (link1["h2d_GB_per_s"] * 1e9) + last / (link1["d2h_GB_per_s"] * 1e9)
                     + max(12 * S_tot - first, 12 * S_tot - last) / (both / 2 * 1e9)) * 1e3
    oracle_base = None if args.no_cpu_baseline else cpu_baseline(units, info, bufs, 0, torch, seconds=3.0)
    print(json.dumps({
        "workload": "llama7b_local_rank_state_offload", "W": wl.world_size, "shard_elems": S_tot,
        "cpu_baseline": oracle_base,
        "state_in_hbm": {"ms_per_step": round(ms_hbm, 3),
                         "GB_per_s": round(info["bytes_per_step"] / (ms_hbm * 1e-3) / 1e9, 1)},
        "state_in_host_memory": {"ms_per_step": round(ms_host, 3),
                                 "GB_per_s": round(info["bytes_per_step"] / (ms_host * 1e-3) / 1e9, 1),
                                 "host_link_bytes_per_step": 24 * S_tot,
                                 "host_link_GB_per_s": round(24 * S_tot / (ms_host * 1e-3) / 1e9, 1)},
        "state_in_host_memory_staged": staged,
        "host_link_both_ways": {"GB_per_s_total": both, "floor_ms": round(floor_ms, 2),
                                "staged_frac_of_floor": round(floor_ms / best, 4),
                                "one_way_GB_per_s": link1,
                                "floor_with_fill_and_drain_ms": round(fill_drain_ms, 2),
                                "staged_frac_of_floor_with_fill_and_drain": round(fill_drain_ms / best, 4)},
        "gpu_memory_saved_bytes": 12 * S_tot,
        "slowdown": round(ms_host / ms_hbm, 2),
        "staged_slowdown": round(best / ms_hbm, 2),
        "staged_speedup_over_zero_copy": round(ms_host / best, 2)}), flush=True)


def run_state(args):
    """The optimizer-state entry points timed on the Llama block (W = 8): the ZeRO-1 step of rank 0
    (full all-reduce average kept, then the rank's Adam and gather) against the fused
    local-rank step on the same buffers, and the full-state gather + unflatten of the
    fp32 master (8 shards -> flat -> 9 tensors)."""
    import torch
    import fully_sharded_gb300 as fs
    import synth
    from synth import workloads as wls
    torch.cuda.set_device(0)
    wl = wls.Workload("llama_block_local", 2, [wls.LLAMA_BLOCK_UNIT], 8, sigma_state=1e-4)
    units, info, bufs = build_local_rank(wl, 0, torch, fs, synth)
    u = units[0]
    lay = u["layout"]
    W, S, padded = lay.world_size, lay.shard_numel, lay.padded_numel
    avg = torch.empty(padded, device="cuda")
    stream = torch.cuda.Stream()

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.record_event(a)
        for _ in range(reps):
            fn()
        stream.record_event(b)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    hp = fs.AdamHyper(step=1)
    batch = fs.UnitBatch(units)
    t_fused = timed(lambda: fs.fsdp_shard_step_grouped(batch, 0, 1, hp, stream=stream), args.steps)
    t_zero1 = timed(lambda: fs.fsdp_zero1_step(u["grads"], lay, 0, avg, u["master"][0], u["exp_avg"][0],
                                               u["exp_avg_sq"][0], u["other_shards"], u["full_out"][0], hp,
                                               stream=stream), args.steps)
    b_fused = (6 * W + 22) * S
    b_zero1 = (2 * W + 4) * padded + (4 + 24 + 2) * S + 4 * (W - 1) * S
    # full state dict of the fp32 master: gather W shards, unflatten into the 9 tensors
    shards = [torch.empty(S, device="cuda") for _ in range(W)]
    flat = torch.empty(padded, device="cuda")
    numels = wls.numels(wl.units[0])
    _, offs = fs.fsdp_flatten_layout(numels, W)
    outs = [torch.empty(n, device="cuda") for n in numels]
    t_gather = timed(lambda: fs.fsdp_all_gather_state(shards, lay, flat, stream=stream), args.steps)
    t_unpack = timed(lambda: fs.fsdp_unpack_flat(flat, lay, offs, outs, stream=stream), args.steps)
    peak, _ = measured_peaks()
    row = lambda ms, b: {"ms": round(ms, 4), "GB_per_s": round(b / (ms * 1e-3) / 1e9, 1),  # noqa
                         "frac_of_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4)}
    oracle_base = None
    if not args.no_cpu_baseline:
        oracle_base = {"local_step": cpu_baseline(units, info, bufs, 0, torch, seconds=2.0, n_s=1 << 20),
                       "parts": oracle_parts_baseline(W, 1 << 17)}
    print(json.dumps({"workload": "llama_block_rank0_state", "W": W, "shard_elems": S,
                      "fused_local_step": row(t_fused, b_fused), "zero1_step": row(t_zero1, b_zero1),
                      "zero1_over_fused_time": round(t_zero1 / t_fused, 3),
                      "gather_state_f32": row(t_gather, 8 * padded), "unpack_f32": row(t_unpack, 8 * padded),
                      "cpu_baseline": oracle_base}),
          flush=True)


def run_pipeline(args):
    """Prefetch depth 0 / 1 / 2 of fsdp_pipeline_step on the 7B local-rank workload: step
    time with the inputs arriving from pinned host memory, and the staging pool's bytes
    against the accountant's transient term 2 U (1 + prefetch)."""
    import torch
    import fully_sharded_gb300 as fs
    import synth
    from synth import workloads as wls
    rank, world, local_rank = env_rank()
    torch.cuda.set_device(local_rank)
    wl = wls.LLAMA7B
    vrank = virtual_rank(rank, wl.world_size)
    units, info, bufs = build_local_rank(wl, vrank, torch, fs, synth)
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    res = {}
    U = max(u["layout"].padded_numel for u in units)
    for n_slots in (1, 2, 3):
        batch, staging, slot, keep = pipeline_setup(torch, fs, units, info, vrank, n_slots)
        ms = time_pipeline(torch, fs, batch, staging, slot, n_slots, vrank, args.steps, args.warmup, None,
                           compute, copy)
        acc = fs.fsdp_account(info["params"], U, wl.world_size, wl.world_size, n_slots - 1)
        res["prefetch_%d" % (n_slots - 1)] = {
            "ms_per_step": round(ms, 3), "GB_per_s": round(info["bytes_per_step"] / (ms * 1e-3) / 1e9, 2),
            "staging_bytes": staging.numel() * 2, "accountant_transient_bytes": acc["transient_bytes"]}
        del batch, staging, keep
        torch.cuda.empty_cache()
    base = res["prefetch_0"]["ms_per_step"]
    link = host_link(torch, copy)
    h2d_bytes, d2h_bytes = 2 * wl.world_size * info["shard_elems"], 2 * info["shard_elems"]
    link["floor_ms"] = round(h2d_bytes / (link["h2d_GB_per_s"] * 1e9) * 1e3, 2)
    both = host_link_both_ways(torch, copy, compute)
    link["both_ways_GB_per_s_total"] = both
    link["floor_two_way_ms"] = round((d2h_bytes / (both / 2 * 1e9) + (h2d_bytes - d2h_bytes)
                                      / (link["h2d_GB_per_s"] * 1e9)) * 1e3, 2)
    oracle_base = None if args.no_cpu_baseline else cpu_baseline(units, info, bufs, vrank, torch, seconds=3.0)
    print(json.dumps({"workload": "llama7b_local_rank_pipeline", "W": wl.world_size, "rank": vrank,
                      "cpu_baseline": oracle_base,
                      "host_link": link,
                      "units": info["units"], "largest_unit_params": U,
                      "h2d_bytes_per_step": 2 * wl.world_size * info["shard_elems"],
                      "results": res,
                      "speedup_prefetch_1": round(base / res["prefetch_1"]["ms_per_step"], 3),
                      "speedup_prefetch_2": round(base / res["prefetch_2"]["ms_per_step"], 3)}), flush=True)


# -------------------------------------------------------- CPU oracle (baseline)

def oracle_sample_inputs(units, rank, n_s, torch):
    """Unit 0 of the workload restricted to the first n_s elements of the rank's shard,
    copied to the host: gradients' rank slices, state and the other ranks' shards."""
    import numpy as np
    u = units[0]
    W = len(u["grads"])
    S = u["layout"].shard_numel
    n_s = min(n_s, S)
    grads = np.zeros((W, W * n_s), dtype=np.uint16)
    for k in range(W):
        grads[k, rank * n_s:(rank + 1) * n_s] = (
            u["grads"][k][rank * S:rank * S + n_s].cpu().numpy().view(np.uint16))
    master = u["master"][0][:n_s].cpu().numpy().copy()
    m = u["exp_avg"][0][:n_s].cpu().numpy().copy()
    v = u["exp_avg_sq"][0][:n_s].cpu().numpy().copy()
    others = [None if o is None else o[:n_s].cpu().numpy().view(np.uint16).copy()
              for o in u["other_shards"]]
    return grads, master, m, v, others, n_s


def run_oracle_step(ora, grads, master, m, v, others, rank, n_s, step):
    import numpy as np
    W = grads.shape[0]
    full = [np.zeros(W * n_s, np.uint16)]
    ora.shard_step(list(grads), W, rank, rank + 1, [master], [m], [v], others, full,
                   lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=step)


def cpu_baseline(units, info, bufs, rank, torch, seconds=10.0, n_s=1 << 22):
    import oracle
    ora = oracle.load()
    grads, master, m, v, others, n_s = oracle_sample_inputs(units, rank, n_s, torch)
    W = info["W"]
    per = (6 * W + 22) * n_s
    t0 = time.perf_counter()
    reps = 0
    while True:
        run_oracle_step(ora, grads, master, m, v, others, rank, n_s, reps + 1)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    out = {"value": round(per * reps / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": "unit 0 (one Llama block) of the workload, first %d elements of rank %d's "
                     "shard (W=%d), %d repetitions in %.1f s; same algorithmic bytes per element"
                     % (n_s, rank, W, reps, dt),
           "cpu": cpu_model()}
    out["all_cores"] = cpu_baseline_all_cores(ora, grads, master, m, v, others, rank, n_s, per, seconds)
    return out


def oracle_sample_all_ranks(units, n_s):
    """Unit 0 of an all-ranks workload (any F) cut to the first n_s elements of every
    position's shard: a unit of padded length F * n_s with the same W, F and work per
    element, copied to the host (gradient rows, every rank's state)."""
    import numpy as np
    u = units[0]
    lay = u["layout"]
    W, F, S = lay.world_size, lay.shard_factor, lay.shard_numel
    n_s = max(1, min(n_s, S))
    grads = np.empty((W, F * n_s), np.uint16)
    for k in range(W):
        row = u["grads"][k]
        for p in range(F):
            grads[k, p * n_s:(p + 1) * n_s] = row[p * S:p * S + n_s].cpu().numpy().view(np.uint16)
    state = [[t[:n_s].cpu().numpy().copy() for t in u[name]] for name in ("master", "exp_avg", "exp_avg_sq")]
    return grads, state, W, F, n_s


def cpu_baseline_all_ranks(units, torch, seconds=3.0, elems=1 << 20):
    """The oracle on one core, timed on a sample of unit 0 of an all-ranks (or hybrid) workload:
    about `elems` padded elements; GB/s at the workload's algorithmic bytes per element."""
    import numpy as np
    import oracle
    ora = oracle.load()
    F = units[0]["layout"].shard_factor
    grads, (master, m, v), W, F, n_s = oracle_sample_all_ranks(units, max(1, elems // F))
    R = W // F
    per = (2 * W + 26 * R) * F * n_s
    full = [np.zeros(F * n_s, np.uint16) for _ in range(R)]
    t0 = time.perf_counter()
    reps = 0
    while True:
        ora.shard_step(list(grads), F, 0, W, master, m, v, None, full, lr=1e-3, beta1=0.9, beta2=0.999,
                       eps=1e-8, step=reps + 1)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(per * reps / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "unit 0 of the workload cut to the first %d elements of every position's shard "
                      "(W=%d, F=%d: %d padded elements), every rank stepped, %d repetitions in %.1f s; "
                      "same algorithmic bytes per element" % (n_s, W, F, F * n_s, reps, dt),
            "cpu": cpu_model()}


def oracle_rate(fn, bytes_per_call, seconds):
    """One-core GB/s of an oracle call at its algorithmic bytes: repeated for about `seconds`."""
    t0 = time.perf_counter()
    reps = 0
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return round(bytes_per_call * reps / (time.perf_counter() - t0) / 1e9, 4)


def oracle_parts_baseline(W, n, seconds=1.0, seed=0):
    """The oracle's separate calls on a seeded sample of n elements per shard (W ranks), one
    core: reduce-scatter for one rank, Adam with the bf16 cast, the all-gather of W bf16 shards,
    the gather of W fp32 shards (as bytes), and pack / unpack of two fp32 tensors; GB/s at each
    call's algorithmic bytes."""
    import numpy as np
    import oracle
    ora = oracle.load()
    rng = np.random.default_rng(seed)
    bf = lambda x: (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731
    grads = [bf(rng.standard_normal(W * n) * 1e-3) for _ in range(W)]
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float32)
    v = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    shards16 = [bf(rng.standard_normal(n) * 0.02) for _ in range(W)]
    shards32 = [rng.standard_normal(n).astype(np.float32).view(np.uint16) for _ in range(W)]
    tensors = [rng.standard_normal(W * n // 2).astype(np.float32) for _ in range(2)]
    flat = np.concatenate(tensors)
    out = {
        "reduce_scatter_GB_per_s": oracle_rate(lambda: ora.reduce_scatter(grads, W, 1), (2 * W + 4) * n, seconds),
        "adam_GB_per_s": oracle_rate(lambda: ora.adam(p, m, v, g, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                                      step=1), 30 * n, seconds),
        "all_gather_GB_per_s": oracle_rate(lambda: ora.all_gather(shards16), 4 * W * n, seconds),
        "gather_state_f32_GB_per_s": oracle_rate(lambda: ora.all_gather(shards32), 8 * W * n, seconds),
        "pack_f32_GB_per_s": oracle_rate(lambda: ora.pack(tensors, W * n), 8 * W * n, seconds),
        "unpack_f32_GB_per_s": oracle_rate(lambda: ora.unpack(flat, [t.shape for t in tensors]), 8 * W * n, seconds),
    }
    out.update({"unit": UNIT, "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                "sample": "seeded arrays of %d elements per shard, W = %d; each call repeated for %.1f s"
                          % (n, W, seconds)})
    return out


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def cpu_model():
    """The host CPU as /proc/cpuinfo names it (Arm cores by their part number)."""
    arm_parts = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
                 "0xd49": "Arm Neoverse-N2", "0xd8e": "Arm Neoverse-N3", "0xd84": "Arm Neoverse-V3"}
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for line in text.splitlines():
        if line.startswith("model name"):
            return line.split(":", 1)[1].strip()
    for line in text.splitlines():
        if line.startswith("CPU part"):
            part = line.split(":", 1)[1].strip()
            return arm_parts.get(part, "Arm CPU part " + part)
    return "unknown"


def cpu_baseline_all_cores(ora, grads, master, m, v, others, rank, n_s, per, seconds):
    """The same oracle step run by one thread per host core, each on its own copy of the
    sample's state (the C oracle runs without the interpreter lock, so the threads run in
    parallel); the gradient rows and other ranks' shards are shared read-only."""
    import threading
    cores = host_cores()
    counts = [0] * cores

    def work(i):
        mp, mm, mv = master.copy(), m.copy(), v.copy()
        t_end = time.perf_counter() + seconds
        while True:
            run_oracle_step(ora, grads, mp, mm, mv, others, rank, n_s, counts[i] + 1)
            counts[i] += 1
            if time.perf_counter() >= t_end:
                break

    threads = [threading.Thread(target=work, args=(i,)) for i in range(cores)]
    t0 = time.perf_counter()
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    dt = time.perf_counter() - t0
    return {"value": round(per * sum(counts) / dt / 1e9, 4), "unit": UNIT, "cores": cores,
            "sample": "the same sample, one thread per core on its own copy of the state, %d steps "
                      "in %.1f s" % (sum(counts), dt)}


# ----------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle timed on the host cores on a bounded sample of the same workload."""
    rank, world, _ = env_rank()
    if rank != 0:
        return
    import numpy as np
    import oracle
    import synth
    from synth import workloads as wls
    ora = oracle.load()  # the oracle alone: the CUDA library is not loaded on this arm
    wl = wls.LLAMA7B
    W = wl.world_size
    _, _, _, S = ora.flatten_layout(wls.numels(wl.units[0]), W)
    n_s = args.ref_sample
    r = 0
    grads = np.zeros((W, W * n_s), dtype=np.uint16)
    for k in range(W):
        grads[k, r * n_s:(r + 1) * n_s] = synth.normal_bf16(wls.key_grad(wl, 0, k, 0), n_s,
                                                             wl.sigma_grad, idx0=r * S)
    master = synth.normal_f32(wls.key_master(wl, 0), n_s, wl.sigma_master, idx0=r * S)
    m = synth.normal_f32(wls.key_exp_avg(wl, 0), n_s, wl.sigma_state, idx0=r * S, absval=True)
    v = synth.normal_f32(wls.key_exp_avg_sq(wl, 0), n_s, wl.sigma_state, idx0=r * S, absval=True)
    others = [None if k == r else synth.normal_bf16(wls.key_shard(wl, 0), n_s, wl.sigma_master,
                                                    idx0=k * S) for k in range(W)]
    for i in range(args.warmup):
        run_oracle_step(ora, grads, master, m, v, others, r, n_s, i + 1)
    t0 = time.perf_counter()
    for i in range(args.steps):
        run_oracle_step(ora, grads, master, m, v, others, r, n_s, args.warmup + i + 1)
    dt = time.perf_counter() - t0
    per = (6 * W + 22) * n_s
    value = per * args.steps / dt / 1e9
    sample = ("unit 0 (one Llama block) of the Llama-7B local-rank workload, first %d elements of "
              "rank 0's shard (W=8) per step" % n_s)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "llama7b_local_rank", "W": W, "mode": "local-rank",
                   "sample_elems_per_step": n_s},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama7b")
    ap.add_argument("--units", type=int, default=0, help="llama7b: only the first N units (gradient rows spaced as in the whole step)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-sample", type=int, default=1 << 21)
    ap.add_argument("--unfused-elems", type=int, default=0,
                    help="unfused: one FlatParameter of this many elements at W = 8 instead of the Llama block")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    _, world, _ = env_rank()
    if args.gpus != world:
        raise SystemExit("--gpus %d but %d process(es): run N > 1 GPUs as python -m torch.distributed.run "
                         "--nproc-per-node N bench.py --gpus N" % (args.gpus, world))
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "pipeline":
        run_pipeline(args)
    elif args.workload == "unfused":
        run_unfused(args)
    elif args.workload == "offload":
        run_offload(args)
    elif args.workload == "state":
        run_state(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
