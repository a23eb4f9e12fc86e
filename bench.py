#!/usr/bin/env python3
"""Benchmark of the paged decode step on GB300: slot-mapped append of one
token per sequence, then paged decode attention, on the LLaMA-3-8B-shaped
layer (B=32, 32/8 heads, head_dim 128, block size 16, context lengths
uniform in [128, 2048], pool +10 %, random physical block order, fp16 values
from N(0, 1)).

Prints one JSON line.  `value` is the step's algorithmic bytes (unique K/V
rows read + Q + O + block tables + context lengths + the append's reads and
writes) divided by the mean device time of one step, in GB/s.  Steps run as
CUDA-graph replays with timing events inside the graph; L2 is flushed
before every step (a 2x-L2 buffer is written, then a second one is read so
that L2 holds clean lines), outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the CPU oracle (plain C, double) on the host cores
instead, on bounded samples of the same workload.  Under torchrun with N > 1
every rank runs an independent replica on its own GPU (the path has no
exchange step); the slowest rank's time sets the aggregate.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attention achieved HBM GB/s (% of GB300 peak); decode steps/sec"
UNIT = "GB/s"
WORKLOAD = 2
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=WORKLOAD, help=argparse.SUPPRESS)
    ap.add_argument("--partition", type=int, default=0,
                    help="tokens per split-K partition (0 = the library's choice)")
    ap.add_argument("--graph-steps", type=int, default=100,
                    help="steps captured per CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU-oracle sample length for cpu_baseline")
    ap.add_argument("--prefix-shared", action="store_true",
                    help="use the prefix-aware entry point (workloads with shared prefixes)")
    ap.add_argument("--kv-dtype", choices=["fp16", "fp8"], default="fp16",
                    help="cache element type: fp16, or E4M3 codes with per-tensor scales")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence: > 1 times the multi-token causal call "
                         "(speculative verify) instead of the decode step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# multi-process plumbing (one replica per GPU)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of `value` over all ranks (identity for one process)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_ms: float, units_per_rank: float, world: int, device=None):
    """(slowest rank's ms per step, whole-job units per second)."""
    ms = reduce_max(per_rank_ms, world, device)
    return ms, world * units_per_rank / (ms * 1e-3)


# ----------------------------------------------------------------------------
# measured peaks, clocks
# ----------------------------------------------------------------------------

def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_selector(torch, device) -> str:
    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    return str(device.index or 0)


# ----------------------------------------------------------------------------
# byte accounting
# ----------------------------------------------------------------------------

def workload_bytes(batch, kv_bytes=2):
    from paged_kv_cache_213_gb300 import workloads as wl
    s = wl.stats(batch, kv_bytes)
    attn = s["unique_kv"] + s["qo"] + s["meta"]
    return {"step": s["step_unique"], "attention": attn, "append": s["append"],
            "logical_step": s["step_logical"], "stats": s}


# decoder layers of the model each workload is shaped like; the whole-model
# figure (steps/sec divided by layers) is context only: attention alone
MODEL_LAYERS = {1: 1, 2: 32, 3: 32, 4: 32, 5: 80}


def pcts(xs):
    """p10 / p50 / p90 of a list of times in ms."""
    ys = sorted(xs)
    at = lambda f: ys[min(len(ys) - 1, int(round(f * (len(ys) - 1))))]  # noqa: E731
    return {"p10": round(at(0.1), 5), "p50": round(at(0.5), 5), "p90": round(at(0.9), 5)}


def source_sha():
    h = hashlib.sha256()
    for name in ("decode_balanced.cu", "mma_tile.cuh", "pkv_ptx.cuh", "shared_prefix.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_213_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: int):
    """DRAM bytes per attention launch from the committed ncu summary, when it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_attention_llama3-8b.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:") or line.startswith("source_sha:") \
                or line.startswith("workload:"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    try:
        if vals.get("source_sha") != source_sha() or int(vals.get("workload", -1)) != workload:
            return None
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------

def oracle_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step_sample(batch, seqs, threads):
    """Run the oracle's append + decode for the sequences `seqs` (all heads);
    returns (seconds, bytes of that sample)."""
    import oracle
    B, H = batch.num_seqs, batch.n_q_heads
    mask = np.zeros((B, H), dtype=bool)
    mask[list(seqs)] = True
    t0 = time.perf_counter()
    kc, vc = batch.k_cache, batch.v_cache
    if batch.has_append:
        keep = np.isin(np.arange(batch.slot_mapping.shape[0]), list(seqs))
        slots = np.where(keep, batch.slot_mapping, -1)
        kc, vc = oracle.append(batch.k_new, batch.v_new, slots, kc, vc, batch.block_size)
    oracle.decode(batch.q, kc, vc, batch.block_tables, batch.context_lens, batch.scale,
                  batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.block_size,
                  mask=mask, num_threads=threads)
    dt = time.perf_counter() - t0
    per_tok = 2 * batch.n_kv_heads * batch.head_dim * 2
    toks = int(sum(int(batch.context_lens[b]) for b in seqs))
    nbytes = toks * per_tok + len(seqs) * H * batch.head_dim * 2 * 2
    if batch.has_append:
        nbytes += len(seqs) * (2 * 2 * batch.n_kv_heads * batch.head_dim * 2 + 8)
    return dt, nbytes


def cpu_baseline(batch, seconds):
    threads = oracle_threads()
    total_t, total_b, steps = 0.0, 0, 0
    everything = range(batch.num_seqs)
    while total_t < seconds or steps == 0:
        dt, nb = oracle_step_sample(batch, everything, threads)
        total_t += dt
        total_b += nb
        steps += 1
    return {"value": total_b / total_t / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{steps} full step(s) of the workload (append + attention, all "
                      f"{batch.num_seqs} sequences x {batch.n_q_heads} heads), double "
                      f"precision, {threads} OpenMP threads, {total_t:.1f} s"}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (this benchmark has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")

    import paged_kv_cache_213_gb300 as pkv
    from paged_kv_cache_213_gb300 import workloads as wl
    pkv.library()  # raises if the CUDA library is not built

    batch = wl.workload(args.workload, poison=False)
    fp8 = args.kv_dtype == "fp8"
    nq = max(1, args.q_len)
    multi = nq > 1
    if multi:
        # n new tokens per sequence, already in the cache: an attention-only step
        # whose Q and O carry n rows per sequence
        batch.slot_mapping = batch.k_new = batch.v_new = None
        rng_q = np.random.default_rng(20300 + args.workload)
        q_multi = rng_q.standard_normal((batch.num_seqs * nq, batch.n_q_heads,
                                         batch.head_dim)).astype(np.float16)
    nbytes = workload_bytes(batch, 1 if fp8 else 2)
    if multi:
        extra = 2 * (nq - 1) * batch.num_seqs * batch.n_q_heads * batch.head_dim * 2
        for key in ("step", "attention", "logical_step"):
            nbytes[key] += extra

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    q, kc, vc = t(q_multi if multi else batch.q), t(batch.k_cache), t(batch.v_cache)
    k_scale = v_scale = 1.0
    if fp8:
        # per-tensor scales max|x| / 448; the caches' E4M3 codes made by torch
        # (input preparation, outside the timed path)
        def amax(*xs):
            return max(float(np.max(np.abs(x.astype(np.float32)))) for x in xs)
        k_scale = np.float32(amax(batch.k_cache, *([batch.k_new] if batch.has_append else [])) / 448)
        v_scale = np.float32(amax(batch.v_cache, *([batch.v_new] if batch.has_append else [])) / 448)
        kc = (kc.float() / float(k_scale)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        vc = (vc.float() / float(v_scale)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    bt, cl = t(batch.block_tables), t(batch.context_lens)
    has_append = batch.has_append
    if has_append:
        kn, vn, sm = t(batch.k_new), t(batch.v_new), t(batch.slot_mapping)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    B, H, Hk, D, bs = batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, \
        batch.block_size
    mcl = batch.max_context_len
    P, ws_bytes = pkv.decode_plan(B, H, Hk, D, bs, batch.max_blocks_per_seq, mcl,
                                  args.partition)
    if fp8:
        P, ws_bytes = 0, pkv.decode_plan_fp8(B, H, Hk, D, bs, batch.max_blocks_per_seq, mcl)
    if multi:
        qstart = t(np.arange(B + 1, dtype=np.int32) * nq)
        P, ws_bytes = pkv.multi_plan(B, B * nq, nq, H, Hk, D, bs, batch.max_blocks_per_seq, mcl,
                                     args.partition)
    # the balanced split (P == 0) merges in-kernel; fixed partitions add a merge kernel
    launches_per_step = (1 if has_append else 0) + 1 + (1 if ws_bytes > 0 and P > 0 else 0)
    groups = None
    if args.prefix_shared and batch.meta.get("shared") and not fp8:
        offs, pref, gmax, pmax = wl.prefix_groups(batch)
        groups = (t(offs), t(pref), gmax, pmax)
        ws_bytes = pkv.prefix_shared_plan(B, H, Hk, D, bs, batch.max_blocks_per_seq, mcl,
                                          len(pref), gmax, pmax)
        launches_per_step = (1 if has_append else 0) + 2
    work = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=device)

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_w = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
    flush_r = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
    sink = torch.empty(1, dtype=torch.float32, device=device)

    def flush():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=sink[0])

    def append():
        if has_append and fp8:
            pkv.paged_kv_append_fp8(kn, vn, sm, kc, vc, k_scale, v_scale, err_word=err)
        elif has_append:
            pkv.paged_kv_append(kn, vn, sm, kc, vc, err_word=err)

    def attend():
        if multi:
            pkv.paged_decode_attention_multi(q, kc, vc, bt, cl, qstart, batch.scale, H, Hk, D,
                                             bs, nq, max_context_len=mcl, partition_tokens=P,
                                             out=out, workspace=work if ws_bytes > 0 else None,
                                             err_word=err)
            return
        if fp8:
            pkv.paged_decode_attention_fp8(q, kc, vc, bt, cl, batch.scale, k_scale, v_scale, H,
                                           Hk, D, bs, max_context_len=mcl, out=out,
                                           workspace=work, err_word=err)
            return
        if groups is not None:
            pkv.paged_decode_attention_prefix_shared(
                q, kc, vc, bt, cl, batch.scale, H, Hk, D, bs, groups[0], groups[1], groups[2],
                groups[3], max_context_len=mcl, out=out, workspace=work, err_word=err)
            return
        pkv.paged_decode_attention(q, kc, vc, bt, cl, batch.scale, H, Hk, D, bs,
                                   max_context_len=mcl, partition_tokens=P, out=out,
                                   workspace=work if ws_bytes > 0 else None, err_word=err)

    def step():
        """append + attention: one library call when the step has an append on
        the default (fp16, one query token) path, so that the attention's
        prologue overlaps the append."""
        if has_append and not fp8 and not multi and groups is None:
            pkv.paged_decode_step(kn, vn, sm, q, kc, vc, bt, cl, batch.scale, H, Hk, D, bs,
                                  max_context_len=mcl, partition_tokens=P, out=out,
                                  workspace=work if ws_bytes > 0 else None, err_word=err)
        else:
            append()
            attend()

    # host-pinned copies of the per-step inputs for the end-to-end leg
    # The per-step inputs live as 256-byte-aligned views of one device buffer,
    # mirrored by one pinned host buffer: the end-to-end leg moves them with a
    # single host-to-device copy per step.
    stage_host = stage_dev = None
    if not args.no_e2e:
        names = [("q", q), ("bt", bt), ("cl", cl)] + \
            ([("kn", kn), ("vn", vn), ("sm", sm)] if has_append else [])
        offs, total = [], 0
        for _, a in names:
            offs.append(total)
            total += (a.numel() * a.element_size() + 255) // 256 * 256
        stage_dev = torch.zeros(total, dtype=torch.uint8, device=device)
        stage_host = torch.zeros(total, dtype=torch.uint8).pin_memory()
        views = {}
        for (name, a), off in zip(names, offs):
            nb = a.numel() * a.element_size()
            v = stage_dev[off:off + nb].view(a.dtype).view(a.shape)
            v.copy_(a)
            stage_host[off:off + nb].copy_(a.cpu().contiguous().view(-1).view(torch.uint8))
            views[name] = v
        q, bt, cl = views["q"], views["bt"], views["cl"]
        if has_append:
            kn, vn, sm = views["kn"], views["vn"], views["sm"]
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d_bytes = total
        d2h_bytes = out_host.numel() * out_host.element_size()

    def e2e_inputs():
        stage_dev.copy_(stage_host, non_blocking=True)

    # eager warm-up (also sets kernel attributes before any capture)
    for _ in range(max(3, args.warmup)):
        flush()
        step()
    torch.cuda.synchronize()
    if pkv.get_error(err) != 0:
        raise SystemExit(f"bench.py: device error word {pkv.get_error(err)}")

    S = max(1, min(args.graph_steps, args.steps))
    try:
        Ev = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        Ev()
        in_graph_events = True
    except TypeError:
        in_graph_events = False

    def capture(body):
        """Graph of S steps; each step = flush, then `body` between events."""
        g = torch.cuda.CUDAGraph()
        evs = [[Ev() for _ in range(body.n_events)] for _ in range(S)]
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.graph(g, stream=side):
            for i in range(S):
                flush()
                body(evs[i])
        torch.cuda.synchronize()
        return g, evs

    def step_body(ev):
        ev[0].record()
        step()
        ev[1].record()
    step_body.n_events = 2

    def attn_body(ev):
        ev[0].record()
        attend()
        ev[1].record()
    attn_body.n_events = 2

    def e2e_body(ev):
        ev[0].record()
        e2e_inputs()
        step()
        out_host.copy_(out, non_blocking=True)
        ev[1].record()
    e2e_body.n_events = 2

    def timed(body, steps, eager=False):
        """Per-step device times (ms) of each event interval over `steps` steps:
        inside CUDA-graph replays, or around eager launches when `eager`."""
        intervals = [[] for _ in range(body.n_events - 1)]
        if in_graph_events and not eager:
            g, evs = capture(body)
            g.replay()  # one untimed replay after capture
            torch.cuda.synchronize()
            done = 0
            while done < steps:
                g.replay()
                torch.cuda.synchronize()
                take = min(S, steps - done)
                for i in range(take):
                    for k in range(body.n_events - 1):
                        intervals[k].append(evs[i][k].elapsed_time(evs[i][k + 1]))
                done += take
        else:
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(body.n_events)]
                   for _ in range(steps)]
            for i in range(steps):
                flush()
                body(evs[i])
            torch.cuda.synchronize()
            for i in range(steps):
                for k in range(body.n_events - 1):
                    intervals[k].append(evs[i][k].elapsed_time(evs[i][k + 1]))
        return intervals

    # untimed graph warm-up
    if in_graph_events:
        timed(step_body, min(S, max(1, args.warmup)))
        timed(attn_body, min(S, max(1, args.warmup)))

    sampler = ClockSampler(gpu_selector(torch, device))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    (step_ms_list,) = timed(step_body, args.steps)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    # the dominant kernel alone (paged_decode_attention), same flush discipline
    (attn_ms,) = timed(attn_body, args.steps)
    clocks = sampler.stop()

    if pkv.get_error(err) != 0:
        raise SystemExit("bench.py: the device flagged an index error")
    step_ms_rank = statistics.fmean(step_ms_list)
    attn_ms_mean = statistics.fmean(attn_ms)
    step_ms, value = aggregate(step_ms_rank, nbytes["step"] / 1e9, world, device)

    # one eager-launch figure for the same step (host launch gaps included)
    eager_steps = min(args.steps, 200)
    (eager_ms,) = timed(step_body, eager_steps, eager=True)

    e2e = None
    if not args.no_e2e:
        (e2e_ms_list,) = timed(e2e_body, args.steps)
        e2e_ms, e2e_val = aggregate(statistics.fmean(e2e_ms_list), nbytes["step"] / 1e9, world,
                                    device)
        e2e = {"value": round(e2e_val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": d2h_bytes, "ms_per_step": round(e2e_ms, 5)}

    layers = MODEL_LAYERS.get(args.workload, 1)
    peak, peak_src = load_peak()
    achieved = nbytes["attention"] / (attn_ms_mean * 1e-3) / 1e9
    # the committed summary covers the fp16 one-token kernel
    traffic = None if (fp8 or multi) else ncu_traffic(args.workload)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not fp8 and not multi:
        cpu = cpu_baseline(batch, args.cpu_seconds)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": wl.WORKLOADS[args.workload], "B": B, "n_q_heads": H, "n_kv_heads": Hk,
            "head_dim": D, "block_size": bs, "max_context_len": mcl,
            "sum_context_len": int(batch.context_lens.sum()), "num_blocks": batch.num_blocks,
            "partition_tokens": P, "step": "append + attention" if has_append else "attention",
            "bytes_per_step": nbytes["step"], "logical_bytes_per_step": nbytes["logical_step"],
            "accumulate": "f32", "l2": "flushed before every timed step (write 2xL2, read 2xL2)",
            "timing": "CUDA events inside CUDA-graph replays" if in_graph_events
                      else "CUDA events around eager launches",
            "parallelism": f"replicas x{world}",
            "decode_kernel": os.environ.get("PKV_DECODE_KERNEL",
                                            "auto (tensor-core kernel when block_size % 16 == 0)"),
            "prefix_shared": groups is not None,
            "kv_dtype": "e4m3 (per-tensor scales)" if fp8 else "f16",
            "q_len": nq,
        },
        "steps_per_sec": round(1e3 / step_ms, 1),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "attention_ms": round(attn_ms_mean, 5),
        "percentiles_ms": {"step": pcts(step_ms_list), "attention": pcts(attn_ms)},
        "eager_step_ms": round(statistics.fmean(eager_ms), 5),
        "model_context": {"layers": layers,
                          "model_steps_per_sec": round(1e3 / step_ms / layers, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "paged_decode_attention: decode_balanced_kernel (one launch, "
                               "in-kernel LSE merge)" if P == 0 else
                               "paged_decode_attention: partition kernel + LSE merge kernel",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_note": "per step: the append (when the step has one) and the attention "
                             "kernel(s) -- one balanced kernel, or partition + merge kernels, or "
                             "the shared-prefix pass + suffix pass; the attention-only timing "
                             f"pass adds {(launches_per_step - (1 if has_append else 0)) * args.steps}"
                             f" more, the eager pass {launches_per_step * eager_steps} more",
        "clocks": clocks,
        "wall_s_timed": round(wall1 - wall0, 3),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the reference arm: the CPU oracle as it stands
# ----------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_213_gb300 import workloads as wl
    oracle.load()
    batch = wl.workload(args.workload, poison=False)
    threads = oracle_threads()
    # one step = a bounded sample: a few whole sequences (all heads, with append)
    per_seq = 4
    rng = np.random.default_rng(0)
    for _ in range(max(0, args.warmup)):
        oracle_step_sample(batch, rng.choice(batch.num_seqs, per_seq, replace=False), threads)
    times, nb = [], []
    for _ in range(args.steps):
        dt, b = oracle_step_sample(batch, rng.choice(batch.num_seqs, per_seq, replace=False),
                                   threads)
        times.append(dt)
        nb.append(b)
    total_t = sum(times)
    value = sum(nb) / total_t / 1e9
    ms = 1e3 * total_t / len(times)
    sample = (f"each step: {per_seq} random whole sequences of {batch.num_seqs} (all "
              f"{batch.n_q_heads} heads, append + attention), double, {threads} OpenMP threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.WORKLOADS[args.workload], "B": batch.num_seqs,
                   "n_q_heads": batch.n_q_heads, "n_kv_heads": batch.n_kv_heads,
                   "head_dim": batch.head_dim, "block_size": batch.block_size},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
