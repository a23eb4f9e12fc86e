#!/usr/bin/env python3
"""Benchmark of the paged decode step on GB300: slot-mapped append of one
token per sequence, then paged decode attention, on the LLaMA-3-8B-shaped
layer (B=32, 32/8 heads, head_dim 128, block size 16, context lengths
uniform in [128, 2048], pool +10 %, random physical block order, fp16 values
from N(0, 1)).

Prints one JSON line.  `value` is the step's algorithmic bytes (unique K/V
rows read + Q + O + block tables + context lengths + the append's reads and
writes) divided by the mean device time of one step, in GB/s.  Steps run as
CUDA-graph replays with timing events inside the graph, back to back: the
steps cycle through four device copies of the workload's inputs, each larger
than L2, so that no step finds its inputs in L2.  The same calls are also
timed one at a time, each after an L2 flush (a 2x-L2 buffer is written, then
a second one is read so that L2 holds clean lines) and between its own two
events, so that each pays its own launch latency (the `_isolated` keys).

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
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the attention-only rows of workloads 3, 4 and 5")
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
    # the translation unit of the headline kernel and what it includes
    for name in ("decode_balanced.cu", "balanced_kernel.cuh", "mma_tile.cuh",
                 "mma_tile_multi.cuh", "pkv_ptx.cuh", "shared_prefix.cuh", "tile_cursor.cuh",
                 "pkv_internal.h"):
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


def oracle_step_sample(batch, seqs, threads, work=None):
    """Run the oracle's append + decode for the sequences `seqs` (all heads);
    returns (seconds, bytes of that sample).

    work: (k_cache, v_cache) working copies, made once outside the timed
    region; the append writes only the sampled sequences' slots into them, in
    place (rewriting a slot with the same token leaves the copies valid for
    the next sample)."""
    import oracle
    B, H = batch.num_seqs, batch.n_q_heads
    mask = np.zeros((B, H), dtype=bool)
    mask[list(seqs)] = True
    if work is None:
        work = (batch.k_cache.copy(), batch.v_cache.copy())
    kc, vc = work
    t0 = time.perf_counter()
    if batch.has_append:
        sel = [b for b in seqs if b < batch.slot_mapping.shape[0]]
        oracle.append_inplace(batch.k_new[sel], batch.v_new[sel], batch.slot_mapping[sel], kc, vc,
                              batch.block_size)
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
    work = (batch.k_cache.copy(), batch.v_cache.copy())
    while total_t < seconds or steps == 0:
        dt, nb = oracle_step_sample(batch, everything, threads, work)
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

# Back-to-back timing cycles through this many device copies of a workload's
# inputs: each copy is larger than L2, so a launch finds none of its inputs
# left in L2 by the launch before it.
ROTATE = 4


class Path:
    """Device inputs (ROTATE copies) and the library calls of one timed path:
    `step(i)` = one decode step on copy i (append + attention, or attention
    alone), `attend(i)` = the attention call alone."""

    def __init__(self, pkv, wl, torch, batch, device, *, fp8=False, q_len=1, prefix=False,
                 partition=0, copies=ROTATE, q_seed=20300):
        self.batch = batch
        self.fp8, self.nq = fp8, max(1, q_len)
        self.multi = self.nq > 1
        B, H, Hk, D, bs = batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, \
            batch.block_size
        MB, mcl = batch.max_blocks_per_seq, batch.max_context_len
        self.has_append = batch.has_append and not self.multi

        def t(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        if self.multi:
            rng_q = np.random.default_rng(q_seed)
            qh = rng_q.standard_normal((B * self.nq, H, D)).astype(np.float16)
        else:
            qh = batch.q
        first = {"q": t(qh), "kc": t(batch.k_cache), "vc": t(batch.v_cache),
                 "bt": t(batch.block_tables), "cl": t(batch.context_lens)}
        self.k_scale = self.v_scale = 1.0
        if fp8:
            # per-tensor scales max|x| / 448; the caches' E4M3 codes made by torch
            # (input preparation, outside the timed path)
            def amax(*xs):
                return max(float(np.max(np.abs(x.astype(np.float32)))) for x in xs)
            extra_k = [batch.k_new] if self.has_append else []
            extra_v = [batch.v_new] if self.has_append else []
            self.k_scale = np.float32(amax(batch.k_cache, *extra_k) / 448)
            self.v_scale = np.float32(amax(batch.v_cache, *extra_v) / 448)
            for key, sc in (("kc", self.k_scale), ("vc", self.v_scale)):
                first[key] = (first[key].float() / float(sc)).clamp(-448, 448) \
                    .to(torch.float8_e4m3fn).view(torch.uint8)
        if self.has_append:
            first.update(kn=t(batch.k_new), vn=t(batch.v_new), sm=t(batch.slot_mapping))
        if self.multi:
            first["qstart"] = t(np.arange(B + 1, dtype=np.int32) * self.nq)
        self.P, self.ws_bytes = pkv.decode_plan(B, H, Hk, D, bs, MB, mcl, partition)
        if fp8:
            self.P, self.ws_bytes = 0, pkv.decode_plan_fp8(B, H, Hk, D, bs, MB, mcl)
        if self.multi:
            self.P, self.ws_bytes = pkv.multi_plan(B, B * self.nq, self.nq, H, Hk, D, bs, MB,
                                                   mcl, partition)
        # the balanced split (P == 0) merges in-kernel; fixed partitions add a merge kernel
        self.attn_launches = 1 + (1 if self.ws_bytes > 0 and self.P > 0 else 0)
        self.groups = None
        if prefix and batch.meta.get("shared") and not self.multi:
            offs, pref, gmax, pmax = wl.prefix_groups(batch)
            first["offs"], first["pref"] = t(offs), t(pref)
            self.groups = (gmax, pmax, len(pref))
            plan = pkv.prefix_shared_plan_fp8 if fp8 else pkv.prefix_shared_plan
            self.ws_bytes = plan(B, H, Hk, D, bs, MB, mcl, len(pref), gmax, pmax)
            self.attn_launches = 2
        self.step_launches = self.attn_launches + (1 if self.has_append else 0)
        # launch flags of the attention call (PKV_TABLES_READY where the caller
        # knows that the kernel before writes no lengths or tables)
        self.attn_flags = 0
        # flags of the one-call step (paged_decode_step_ex); see set_step_flags
        self.step_flags = 0
        self._sizes = (B, H, Hk, D, bs, MB, mcl)
        self.copies = [first] + [{k: v.clone() for k, v in first.items()}
                                 for _ in range(copies - 1)]
        for c in self.copies:
            c["out"] = torch.empty_like(c["q"])
            c["work"] = torch.zeros(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
            c["err"] = torch.zeros(1, dtype=torch.int32, device=device)
        self.pkv = pkv

    def attend(self, i):
        pkv, bt, c = self.pkv, self.batch, self.copies[i]
        H, Hk, D, bs, mcl = bt.n_q_heads, bt.n_kv_heads, bt.head_dim, bt.block_size, \
            bt.max_context_len
        ws = c["work"] if self.ws_bytes > 0 else None
        if self.multi:
            pkv.paged_decode_attention_multi(c["q"], c["kc"], c["vc"], c["bt"], c["cl"],
                                             c["qstart"], bt.scale, H, Hk, D, bs, self.nq,
                                             max_context_len=mcl, partition_tokens=self.P,
                                             out=c["out"], workspace=ws, err_word=c["err"],
                                             flags=self.attn_flags)
        elif self.fp8 and self.groups is not None:
            gmax, pmax, _ = self.groups
            pkv.paged_decode_attention_prefix_shared_fp8(
                c["q"], c["kc"], c["vc"], c["bt"], c["cl"], bt.scale, self.k_scale, self.v_scale,
                H, Hk, D, bs, c["offs"], c["pref"], gmax, pmax, max_context_len=mcl,
                out=c["out"], workspace=ws, err_word=c["err"], flags=self.attn_flags)
        elif self.fp8:
            pkv.paged_decode_attention_fp8(c["q"], c["kc"], c["vc"], c["bt"], c["cl"], bt.scale,
                                           self.k_scale, self.v_scale, H, Hk, D, bs,
                                           max_context_len=mcl, out=c["out"], workspace=ws,
                                           err_word=c["err"], flags=self.attn_flags)
        elif self.groups is not None:
            gmax, pmax, _ = self.groups
            pkv.paged_decode_attention_prefix_shared(
                c["q"], c["kc"], c["vc"], c["bt"], c["cl"], bt.scale, H, Hk, D, bs, c["offs"],
                c["pref"], gmax, pmax, max_context_len=mcl, out=c["out"], workspace=ws,
                err_word=c["err"], flags=self.attn_flags)
        else:
            pkv.paged_decode_attention(c["q"], c["kc"], c["vc"], c["bt"], c["cl"], bt.scale, H,
                                       Hk, D, bs, max_context_len=mcl, partition_tokens=self.P,
                                       out=c["out"], workspace=ws, err_word=c["err"],
                                       flags=self.attn_flags)

    def fused_step(self):
        """The step is one paged_decode_step(_fp8) call (one query token, an
        append, no prefix groups), which takes step flags."""
        return self.has_append and self.groups is None

    def set_step_flags(self, flags):
        """Flags of the one-call step; the launch count follows the library's
        own answer for these sizes and flags."""
        if not self.fused_step():
            return
        self.step_flags = flags
        B, H, Hk, D, bs, MB, mcl = self._sizes
        if self.fp8:  # the E4M3 step: the append kernel, then the attention
            self.step_launches = 2
        else:
            self.step_launches = self.pkv.step_launches(B, H, Hk, D, bs, MB, mcl, self.P,
                                                        num_tokens=B, flags=flags)

    def flaggable(self):
        """The attention call takes launch flags (every entry point here has
        an _ex form)."""
        return True

    def step(self, i, out=None):
        """append + attention: one library call when the step has an append on
        the default (fp16, one query token) path: under PKV_APPEND_NEWEST one
        kernel that also appends, otherwise the append kernel with the
        attention's prologue overlapping it.  out (that path only): where the
        result goes instead of the copy's device buffer, e.g. pinned host
        memory."""
        pkv, bt, c = self.pkv, self.batch, self.copies[i]
        if not self.has_append:
            self.attend(i)
            return
        if self.fp8 and self.groups is None:
            pkv.paged_decode_step_fp8(c["kn"], c["vn"], c["sm"], c["q"], c["kc"], c["vc"],
                                      c["bt"], c["cl"], bt.scale, self.k_scale, self.v_scale,
                                      bt.n_q_heads, bt.n_kv_heads, bt.head_dim, bt.block_size,
                                      max_context_len=bt.max_context_len, out=c["out"],
                                      workspace=c["work"], err_word=c["err"],
                                      flags=self.step_flags)
            return
        if self.fp8:
            pkv.paged_kv_append_fp8(c["kn"], c["vn"], c["sm"], c["kc"], c["vc"], self.k_scale,
                                    self.v_scale, err_word=c["err"])
            self.attend(i)
            return
        if self.groups is not None:
            pkv.paged_kv_append(c["kn"], c["vn"], c["sm"], c["kc"], c["vc"], err_word=c["err"])
            self.attend(i)
            return
        pkv.paged_decode_step(c["kn"], c["vn"], c["sm"], c["q"], c["kc"], c["vc"], c["bt"],
                              c["cl"], bt.scale, bt.n_q_heads, bt.n_kv_heads, bt.head_dim,
                              bt.block_size, max_context_len=bt.max_context_len,
                              partition_tokens=self.P, out=c["out"] if out is None else out,
                              workspace=c["work"] if self.ws_bytes > 0 else None,
                              err_word=c["err"], flags=self.step_flags)

    def errors(self):
        return [self.pkv.get_error(c["err"]) for c in self.copies]


class Timer:
    """CUDA-event timing inside CUDA-graph replays (eager launches when this
    torch cannot record events inside a graph).

    isolated(): every call is its own timed region -- flush L2, event, call,
      event -- so each call starts cold and pays its own launch latency.
    back_to_back(): S calls in a row between two events, cycling through the
      input copies (each larger than L2, so no call finds its inputs in L2);
      a call's launch overlaps the call before it, as in a serving step where
      the attention follows other kernels.  One figure per graph replay: the
      interval divided by S.
    """

    def __init__(self, torch, device, graph_steps):
        self.torch, self.device, self.S = torch, device, max(1, graph_steps)
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.flush_w = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
        self.flush_r = torch.ones(2 * l2 // 4 + 1024, dtype=torch.float32, device=device)
        self.sink = torch.empty(1, dtype=torch.float32, device=device)
        try:
            torch.cuda.Event(enable_timing=True, external=True)
            self.in_graph = True
        except TypeError:
            self.in_graph = False
        self.side = torch.cuda.Stream(device)

    def flush(self):
        """L2 flush: write a 2xL2 buffer, then read another 2xL2 buffer so
        that L2 holds only clean lines."""
        self.flush_w.zero_()
        self.torch.sum(self.flush_r, dim=0, out=self.sink[0])

    def _ev(self):
        return self.torch.cuda.Event(enable_timing=True, external=self.in_graph)

    def _graph(self, record):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        self.side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.graph(g, stream=self.side):
            record()
        torch.cuda.synchronize()
        g.replay()  # one untimed replay after capture
        torch.cuda.synchronize()
        return g

    def isolated(self, body, steps, eager=False):
        """Per-call device times (ms) of `body(i)` (i = the call's index)."""
        torch, S = self.torch, min(self.S, steps)
        out = []
        if self.in_graph and not eager:
            evs = [(self._ev(), self._ev()) for _ in range(S)]

            def record():
                for i in range(S):
                    self.flush()
                    evs[i][0].record()
                    body(i)
                    evs[i][1].record()
            g = self._graph(record)
            while len(out) < steps:
                g.replay()
                torch.cuda.synchronize()
                out += [a.elapsed_time(b) for a, b in evs][:steps - len(out)]
            return out
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            self.flush()
            evs[i][0].record()
            body(i)
            evs[i][1].record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def back_to_back(self, body, steps):
        """Per-call device times (ms), one per replay of S back-to-back calls
        of `body(i)`, S the largest divisor of `steps` up to the graph size:
        exactly `steps` calls are timed."""
        torch = self.torch
        S = max(d for d in range(1, min(self.S, steps) + 1) if steps % d == 0)
        self.last_s = S
        out = []
        if self.in_graph:
            e0, e1 = self._ev(), self._ev()

            def record():
                self.flush()
                e0.record()
                for i in range(S):
                    body(i)
                e1.record()
            g = self._graph(record)
            for _ in range(max(1, -(-steps // S))):
                g.replay()
                torch.cuda.synchronize()
                out.append(e0.elapsed_time(e1) / S)
            return out
        for _ in range(max(1, -(-steps // S))):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            self.flush()
            e0.record()
            for i in range(S):
                body(i)
            e1.record()
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) / S)
        return out


# Rows besides the headline, timed like it: (key, workload, E4M3 caches,
# query tokens per sequence, prefix-aware entry).
PER_CONFIG = [
    ("w3_regular", 3, False, 1, False), ("w3_prefix_shared", 3, False, 1, True),
    ("w4_regular", 4, False, 1, False),
    ("w5_regular", 5, False, 1, False), ("w5_prefix_shared", 5, False, 1, True),
    ("w2_multi4", 2, False, 4, False),
    ("w2_fp8", 2, True, 1, False),
    ("w5_fp8_regular", 5, True, 1, False), ("w5_fp8_prefix_shared", 5, True, 1, True),
]


def kernel_label(path, torch, device):
    """The entry point and kernel(s) the attention call of `path` runs (the
    library's dispatch rule, restated for the label only)."""
    bt = path.batch
    if path.multi:
        return ("paged_decode_attention_multi_ex (PKV_TABLES_READY): decode_balanced_kernel "
                "with multi-token rows (one launch)" if path.P == 0 else
                "paged_decode_attention_multi: decode_multi_kernel + multi_merge_kernel")
    if path.groups is not None:
        return ("paged_decode_attention_prefix_shared" + ("_fp8" if path.fp8 else "") +
                "_ex (PKV_TABLES_READY): decode_shared_kernel (shared pass) + "
                "decode_balanced_kernel (suffix pass), or the regular call when the shared "
                "blocks fit in L2")
    if path.fp8:
        return ("paged_decode_attention_fp8_ex (PKV_TABLES_READY): decode_balanced_kernel on "
                "E4M3 tiles (one launch)")
    if path.P != 0:
        return "paged_decode_attention: partition kernel + LSE merge kernel"
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    if bt.num_seqs * bt.n_kv_heads > 2 * sms and not os.environ.get("PKV_DECODE_KERNEL"):
        return ("paged_decode_attention_ex (PKV_TABLES_READY): decode_pipeline_kernel "
                "(producer/consumer CTAs, one launch, in-kernel LSE merge)")
    return ("paged_decode_attention_ex (PKV_TABLES_READY): decode_balanced_kernel (one launch, "
            "in-kernel LSE merge)")


def per_config_rows(pkv, wl, torch, device, timer, peak, steps, rows_spec=PER_CONFIG):
    """Attention-only rows for the other standard workloads, the prefix-aware
    entry where a workload shares prefix blocks, 4 query tokens per sequence
    (the multi-token call) and E4M3 caches, each timed like the headline
    (both ways)."""
    rows = {}
    batches = {}
    for key, w, fp8, nq, prefix in rows_spec:
        if w not in batches:
            batch = wl.workload(w, poison=False)
            if batch.has_append:  # attention over the cache as generated
                batch.slot_mapping = batch.k_new = batch.v_new = None
            batches = {w: batch}  # one workload's arrays at a time
        batch = batches[w]
        nbytes = workload_bytes(batch, 1 if fp8 else 2)["attention"]
        if nq > 1:  # the extra query rows and output rows
            nbytes += 2 * (nq - 1) * batch.num_seqs * batch.n_q_heads * batch.head_dim * 2
        path = Path(pkv, wl, torch, batch, device, fp8=fp8, q_len=nq, prefix=prefix)
        for i in range(3):
            timer.flush()
            path.attend(i % ROTATE)
        torch.cuda.synchronize()
        plain = None
        if path.flaggable():  # as the headline: flagged back to back, plain too
            plain = timer.back_to_back(lambda i: path.attend(i % ROTATE), steps)
            path.attn_flags = pkv.PKV_TABLES_READY
        b2b = timer.back_to_back(lambda i: path.attend(i % ROTATE), steps)
        path.attn_flags = 0
        iso = timer.isolated(lambda i: path.attend(i % ROTATE), min(steps, 200))
        if any(path.errors()):
            raise SystemExit(f"bench.py: device error word on row {key}")
        ms, ms_iso = statistics.fmean(b2b), statistics.fmean(iso)
        entry = ("paged_decode_attention" + ("_multi" if nq > 1 else "") +
                 ("_prefix_shared" if prefix else "") + ("_fp8" if fp8 else "") +
                 ("_ex (PKV_TABLES_READY)" if plain is not None else ""))
        rows[key] = {
            "workload": wl.WORKLOADS[w], "entry": entry,
            "kv_dtype": "e4m3" if fp8 else "f16", "query_tokens_per_seq": nq,
            "attention_bytes": nbytes, "attention_ms": round(ms, 5),
            "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4),
            "attention_ms_isolated": round(ms_iso, 5),
            "frac_isolated": round(nbytes / (ms_iso * 1e-3) / 1e9 / peak, 4),
            "percentiles_ms": pcts(b2b), "percentiles_ms_isolated": pcts(iso),
            "launches_per_call": path.attn_launches,
            "flags": "PKV_TABLES_READY" if plain is not None else "none",
        }
        if plain is not None:
            mp = statistics.fmean(plain)
            rows[key]["attention_ms_plain_call"] = round(mp, 5)
            rows[key]["frac_plain_call"] = round(nbytes / (mp * 1e-3) / 1e9 / peak, 4)
        del path
        torch.cuda.empty_cache()
    rows.update(fp8_step_row(pkv, wl, torch, device, timer, peak, steps))
    return rows


def fp8_step_row(pkv, wl, torch, device, timer, peak, steps):
    """The decode step over E4M3 caches on the LLaMA-3-8B-shaped layer:
    paged_decode_step_fp8 (the quantizing append kernel, then the attention
    with its prologue under the append), timed like the headline step."""
    batch = wl.workload(2, poison=False)
    nbytes = workload_bytes(batch, 1)["step"]
    path = Path(pkv, wl, torch, batch, device, fp8=True)
    path.set_step_flags(0)
    for i in range(3):
        timer.flush()
        path.step(i % ROTATE)
    torch.cuda.synchronize()
    b2b = timer.back_to_back(lambda i: path.step(i % ROTATE), steps)
    iso = timer.isolated(lambda i: path.step(i % ROTATE), min(steps, 200))
    if any(path.errors()):
        raise SystemExit("bench.py: device error word on the E4M3 step row")
    ms, mi = statistics.fmean(b2b), statistics.fmean(iso)
    row = {
        "workload": wl.WORKLOADS[2], "entry": "paged_decode_step_fp8: append_f8_kernel, then "
        "decode_balanced_kernel on E4M3 tiles",
        "kv_dtype": "e4m3", "step_bytes": nbytes, "step_ms": round(ms, 5),
        "step_gbs": round(nbytes / (ms * 1e-3) / 1e9, 2),
        "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4),
        "step_ms_isolated": round(mi, 5), "launches_per_step": path.step_launches,
        "percentiles_ms": pcts(b2b),
    }
    del path
    torch.cuda.empty_cache()
    return {"w2_fp8_step": row}


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
    nbytes = workload_bytes(batch, 1 if fp8 else 2)
    if multi:
        extra = 2 * (nq - 1) * batch.num_seqs * batch.n_q_heads * batch.head_dim * 2
        for key in ("step", "attention", "logical_step"):
            nbytes[key] += extra
    path = Path(pkv, wl, torch, batch, device, fp8=fp8, q_len=nq, prefix=args.prefix_shared,
                partition=args.partition, q_seed=20300 + args.workload)
    has_append = path.has_append
    B, H, Hk, D, bs = batch.num_seqs, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, \
        batch.block_size
    # The step's promises, both true of a decode loop: token b is sequence b's
    # newest token (so the attention kernel appends it itself, in one launch),
    # and the kernel before the step (here the previous step) writes no
    # lengths, tables or slot mapping.  The same steps without the flags (the
    # append kernel, then the attention) are timed too (ms_per_step_plain_call).
    step_flags = pkv.PKV_APPEND_NEWEST | pkv.PKV_TABLES_READY
    path.set_step_flags(step_flags)
    timer = Timer(torch, device, args.graph_steps)

    # The end-to-end leg: each input copy's per-step inputs live as
    # 256-byte-aligned views of one device buffer, mirrored by one pinned host
    # buffer, so that one host-to-device copy per step moves them all.
    stages = []
    if not args.no_e2e:
        c0 = path.copies[0]
        names = ["q", "bt", "cl"] + (["kn", "vn", "sm"] if has_append else []) + \
            (["qstart"] if multi else []) + (["offs", "pref"] if path.groups else [])
        offs, total = [], 0
        for n in names:
            offs.append(total)
            total += (c0[n].numel() * c0[n].element_size() + 255) // 256 * 256
        for c in path.copies:
            stage_dev = torch.zeros(total, dtype=torch.uint8, device=device)
            stage_host = torch.zeros(total, dtype=torch.uint8).pin_memory()
            for n, off in zip(names, offs):
                a = c[n]
                nb = a.numel() * a.element_size()
                v = stage_dev[off:off + nb].view(a.dtype).view(a.shape)
                v.copy_(a)
                stage_host[off:off + nb].copy_(a.cpu().contiguous().view(-1).view(torch.uint8))
                c[n] = v
            out_host = torch.empty(c["out"].shape, dtype=c["out"].dtype).pin_memory()
            stages.append((stage_dev, stage_host, out_host))
        h2d_bytes = total
        d2h_bytes = stages[0][2].numel() * stages[0][2].element_size()

    # eager warm-up on every copy (also sets kernel attributes before any capture)
    with torch.cuda.stream(timer.side):
        for i in range(max(3, args.warmup) * ROTATE):
            timer.flush()
            path.step(i % ROTATE)
    torch.cuda.synchronize()
    if any(path.errors()):
        raise SystemExit(f"bench.py: device error word {path.errors()}")
    # untimed graph warm-up
    warm = max(1, min(args.warmup, args.graph_steps))
    timer.back_to_back(lambda i: path.step(i % ROTATE), warm)
    timer.isolated(lambda i: path.step(0), warm)

    sampler = ClockSampler(gpu_selector(torch, device))
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    step_ms_list = timer.back_to_back(lambda i: path.step(i % ROTATE), args.steps)
    torch.cuda.synchronize()
    wall1 = time.perf_counter()
    if world > 1:
        dist.barrier()
    # the dominant call alone, both ways.  Back to back, each call is made as
    # in a decode loop whose tables are copied in before the layers run: the
    # kernel before it (the previous call) writes no lengths or tables, so the
    # call takes PKV_TABLES_READY; the same calls without the flag are timed
    # too (attention_ms_plain_call).
    attn_plain = None
    if path.flaggable():
        attn_plain = timer.back_to_back(lambda i: path.attend(i % ROTATE), args.steps)
        path.attn_flags = pkv.PKV_TABLES_READY
    attn_ms = timer.back_to_back(lambda i: path.attend(i % ROTATE), args.steps)
    path.attn_flags = 0
    step_plain = None
    if path.fused_step():
        path.set_step_flags(0)
        step_plain = timer.back_to_back(lambda i: path.step(i % ROTATE), args.steps)
        path.set_step_flags(step_flags)
    step_iso = timer.isolated(lambda i: path.step(i % ROTATE), args.steps)
    attn_iso = timer.isolated(lambda i: path.attend(i % ROTATE), args.steps)
    clocks = sampler.stop()

    if any(path.errors()):
        raise SystemExit("bench.py: the device flagged an index error")
    n_calls = args.steps
    step_ms, value = aggregate(statistics.fmean(step_ms_list), nbytes["step"] / 1e9, world,
                               device)
    attn_ms_mean = statistics.fmean(attn_ms)
    attn_iso_mean = statistics.fmean(attn_iso)

    # one eager-launch figure for the same step (host launch gaps included)
    eager_steps = min(args.steps, 200)
    eager_ms = timer.isolated(lambda i: path.step(i % ROTATE), eager_steps, eager=True)

    e2e = None
    if not args.no_e2e:
        # The fp16 step's kernel writes its result straight into the pinned host
        # buffer (plain stores over the host link); other steps copy it after.
        zero_copy_out = path.fused_step() and not fp8

        def e2e_body(i, engine=False):
            stage_dev, stage_host, out_host = stages[i % ROTATE]
            if engine:  # the copy engine (cudaMemcpyAsync), for comparison
                stage_dev.copy_(stage_host, non_blocking=True)
            else:  # the library's copy kernel: one 16-byte piece per thread
                pkv.paged_copy_in(stage_dev, stage_host)
            if zero_copy_out:
                path.step(i % ROTATE, out=out_host)
            else:
                path.step(i % ROTATE)
                out_host.copy_(path.copies[i % ROTATE]["out"], non_blocking=True)
        e2e_ms_list = timer.back_to_back(e2e_body, args.steps)
        e2e_iso_list = timer.isolated(e2e_body, args.steps)
        e2e_engine_list = timer.back_to_back(lambda i: e2e_body(i, True), args.steps)
        # the host buffers hold what a device-memory step computes, bit for bit
        torch.cuda.synchronize()
        for k in range(ROTATE):
            path.step(k)
        torch.cuda.synchronize()
        for k in range(ROTATE):
            if not torch.equal(path.copies[k]["out"].cpu().view(torch.int16),
                               stages[k][2].view(torch.int16)):
                raise SystemExit("bench.py: the end-to-end output differs from the device step")
        e2e_ms, e2e_val = aggregate(statistics.fmean(e2e_ms_list), nbytes["step"] / 1e9, world,
                                    device)
        e2e_iso_ms, e2e_iso_val = aggregate(statistics.fmean(e2e_iso_list), nbytes["step"] / 1e9,
                                            world, device)
        e2e = {"value": round(e2e_val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": d2h_bytes, "ms_per_step": round(e2e_ms, 5),
               "value_isolated": round(e2e_iso_val, 2),
               "ms_per_step_copy_engine": round(statistics.fmean(e2e_engine_list), 5),
               "ms_per_step_isolated": round(e2e_iso_ms, 5),
               "timing": "every step: pinned-host -> device copy of the step's inputs by the "
                         "library's copy kernel (paged_copy_in; ms_per_step_copy_engine: the "
                         "same steps with cudaMemcpyAsync instead), the step (paged_decode_step "
                         "with the step flags), whose kernel writes out into pinned host memory "
                         "(no copy after it); steps back to "
                         "back over the four input copies (value), or each its own timed region "
                         "after an L2 flush (value_isolated)"}

    layers = MODEL_LAYERS.get(args.workload, 1)
    peak, peak_src = load_peak()
    achieved = nbytes["attention"] / (attn_ms_mean * 1e-3) / 1e9
    # the committed summary covers the fp16 one-token kernel
    traffic = None if (fp8 or multi) else ncu_traffic(args.workload)
    per_config = None
    if rank == 0 and args.per_config and not fp8 and not multi and args.workload == WORKLOAD:
        per_config = per_config_rows(pkv, wl, torch, device, timer, peak, args.steps)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not fp8 and not multi:
        cpu = cpu_baseline(batch, args.cpu_seconds)

    if rank != 0:
        return
    per_call = path.step_launches
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": n_calls, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": wl.WORKLOADS[args.workload], "B": B, "n_q_heads": H, "n_kv_heads": Hk,
            "head_dim": D, "block_size": bs, "max_context_len": batch.max_context_len,
            "sum_context_len": int(batch.context_lens.sum()), "num_blocks": batch.num_blocks,
            "partition_tokens": path.P,
            "step": "append + attention" if has_append else "attention",
            "bytes_per_step": nbytes["step"], "logical_bytes_per_step": nbytes["logical_step"],
            "accumulate": "f32",
            "l2": f"inputs larger than L2: back-to-back calls cycle through {ROTATE} device "
                  "copies of the workload's inputs (each larger than L2); the isolated "
                  "figures flush L2 before every call (write 2xL2, read 2xL2)",
            "timing": ("CUDA events inside CUDA-graph replays" if timer.in_graph
                       else "CUDA events around eager launches") +
                      f"; value, ms_per_step, attention_ms: {timer.last_s} back-to-back "
                      "calls between two events, divided by the calls",
            "parallelism": f"replicas x{world}",
            "decode_kernel": os.environ.get("PKV_DECODE_KERNEL",
                                            "auto (tensor-core kernel when block_size % 16 == 0)"),
            "prefix_shared": path.groups is not None,
            "kv_dtype": "e4m3 (per-tensor scales)" if fp8 else "f16",
            "q_len": nq,
        },
        "steps_per_sec": round(1e3 / step_ms, 1),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "attention_ms": round(attn_ms_mean, 5),
        "attention_flags": "PKV_TABLES_READY" if attn_plain is not None else "none",
        "attention_ms_plain_call": round(statistics.fmean(attn_plain), 5)
        if attn_plain is not None else None,
        "step_flags": "PKV_APPEND_NEWEST|PKV_TABLES_READY" if path.fused_step() else "none",
        "ms_per_step_plain_call": round(statistics.fmean(step_plain), 5)
        if step_plain is not None else None,
        "ms_per_step_isolated": round(statistics.fmean(step_iso), 5),
        "attention_ms_isolated": round(attn_iso_mean, 5),
        "percentiles_ms": {"step": pcts(step_ms_list), "attention": pcts(attn_ms),
                           "step_isolated": pcts(step_iso),
                           "attention_isolated": pcts(attn_iso)},
        "eager_step_ms": round(statistics.fmean(eager_ms), 5),
        "model_context": {"layers": layers,
                          "model_steps_per_sec": round(1e3 / step_ms / layers, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "frac_isolated": round(nbytes["attention"] / (attn_iso_mean * 1e-3) / 1e9
                                            / peak, 4),
                     "frac_plain_call": round(nbytes["attention"] /
                                              (statistics.fmean(attn_plain) * 1e-3) / 1e9 / peak,
                                              4) if attn_plain is not None else None,
                     "kernel": kernel_label(path, torch, device),
                     "timing": "achieved = attention bytes / attention_ms (back-to-back "
                               "calls, made with PKV_TABLES_READY); "
                               "frac_plain_call: the same calls without the flag; "
                               "frac_isolated uses attention_ms_isolated",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": per_call * n_calls,
        "gpu_launches_note": f"{per_call} launch(es) per step (the append when the step has "
                             "one and the attention does not do it under PKV_APPEND_NEWEST, "
                             "then the attention: one balanced kernel, or partition + "
                             "merge kernels, or the shared-prefix pass + suffix pass), times "
                             "the timed steps of `value`; the other timing passes (attention "
                             "alone, isolated calls, eager, e2e, per_config) launch more",
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
    work = (batch.k_cache.copy(), batch.v_cache.copy())
    for _ in range(max(0, args.warmup)):
        oracle_step_sample(batch, rng.choice(batch.num_seqs, per_seq, replace=False), threads,
                           work)
    times, nb = [], []
    for _ in range(args.steps):
        dt, b = oracle_step_sample(batch, rng.choice(batch.num_seqs, per_seq, replace=False),
                                   threads, work)
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
