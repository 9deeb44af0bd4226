#!/usr/bin/env python3
"""Benchmark of the gated-DeltaNet decode step (one JSON line on stdout).

A step is one dn_step call: one layer advances every sequence of its batch by
one token (in_proj GEMV, conv + SiLU with the ring, L2 norms, gated delta
rule, readout, gated RMSNorm, out_proj GEMV).  The headline workload is the
35B-shape layer (hidden 2048, 16 q/k heads and 32 value heads of 128, conv
kernel 4, int8 projections 2048 -> 12288 and 4096 -> 2048) at batch 64 with
random initial state; the batch-1 workload of the same layer is measured in
the same run and reported under "batch1".

Timed regions rotate over --layers independent layer objects (distinct
weights and states), so the working set of consecutive steps (about 300 MB
per layer-step at batch 64) is larger than the 129 MB L2: nothing of a step
is served from L2 by the previous step of the same layer.  The timed region
replays CUDA graphs of up to 512 consecutive dn_step calls (the same kernels
and work as eager calls, without the per-launch CPU cost; consecutive steps
overlap through programmatic dependent launch as eager calls do), so that
exactly --steps steps are timed; the region is repeated (at least five times
and 0.5 s) and the median reported with its spread; --no-graph times
eager dn_step calls.  The end-to-end figure ("e2e") always goes through
dn_step with pinned host buffers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank runs independent replicas of the same
workload (the sequences of a batch are independent; nothing is exchanged);
`value` counts the layer-steps of all ranks divided by the slowest rank's
time.  --impl reference times the CPU oracle (float64 numpy) on a bounded
sample of the same workload, on rank 0 only.

Other workloads (--workload): 35b_b1 and 35b_b8 (the same layer at batch 1
and 8), stack30_b1 and stack30_b16 (30 distinct layers per token through
dn_stack_step; the line adds tokens_per_s and ms_per_token).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gated_deltanet_hybrid_gb300.inputs import (SHAPE_35B, WORKLOADS, DNConfig,  # noqa: E402
                                                WorkloadStream, gates_from_ab, make_weights)

METRIC = "DeltaNet layer-steps/s and achieved HBM GB/s (% of roofline) at batch 1 and 64"
UNIT = "layer-steps/s"
# the library's projections take the tensor cores (and a packing kernel) from
# this many columns (sequences of a step, token columns of a prompt block)
TC_MIN_COLS = 2
# seconds the reference arm's --steps + --warmup steps may take
REFERENCE_BUDGET_S = 100.0
KERNELS = ("in_proj", "dn_state", "out_proj")
# stage -> (first, last) index of the five events dn_profile_next_step records
# (events 1 -> 2 bracket a separate preparation kernel, which this library
# does not launch: the state kernel builds its inputs itself)
STAGE_EVENTS = {"in_proj": (0, 1), "dn_state": (1, 3), "out_proj": (3, 4)}


# --------------------------------------------------------------------- bytes
def weight_bytes(cfg: DNConfig) -> int:
    """The two projections' weight bytes (int8, or int4 at half a byte)."""
    n = cfg.in_rows * cfg.hidden + cfg.hidden * cfg.v_dim
    return n // 2 if getattr(cfg, "int4", False) else n


def step_bytes(cfg: DNConfig, B: int) -> int:
    """Algorithmic HBM bytes of one layer-step: weights once, plus per
    sequence the state read and written, the ring's conv_k-1 slots read and
    one slot written, x, out and the two gates.  Scratch is not counted."""
    shared = (weight_bytes(cfg) + cfg.in_rows * 4 + cfg.hidden * 4
              + cfg.conv_ch * cfg.conv_k * 4 + cfg.dv * 4)
    per_seq = (2 * cfg.n_v_heads * cfg.dk * cfg.dv * 4 + (cfg.conv_k - 1) * cfg.conv_ch * 4
               + cfg.conv_ch * 4 + 2 * cfg.hidden * 4 + 2 * cfg.n_v_heads * 4)
    return shared + B * per_seq


def kernel_bytes(cfg: DNConfig, B: int) -> dict[str, int]:
    """Algorithmic bytes of each stage of the step (its unique inputs and
    outputs; an intermediate result counts once as the producer's output and
    once as the consumer's input, since both move it).

    in_proj: W_in, s_in, x in, the projection out.  dn_state: the projection
    in, the ring's conv_k-1 history slots in and the new slot out, the conv
    weights, the gates, the state read and written, the gated-norm output
    out, the norm weight.  out_proj: W_out, s_out, its input in, the layer
    output out."""
    half = 2 if getattr(cfg, "int4", False) else 1
    k1 = cfg.in_rows * cfg.hidden // half + cfg.in_rows * 4 + B * (cfg.hidden + cfg.in_rows) * 4
    ks = (B * (cfg.in_rows * 4 + (cfg.conv_k - 1) * cfg.conv_ch * 4 + cfg.conv_ch * 4
               + 2 * cfg.n_v_heads * 4 + 2 * cfg.n_v_heads * cfg.dk * cfg.dv * 4 + cfg.v_dim * 4)
          + cfg.conv_ch * cfg.conv_k * 4 + cfg.dv * 4)
    k3 = cfg.hidden * cfg.v_dim // half + cfg.hidden * 4 + B * (cfg.v_dim + cfg.hidden) * 4
    return {"in_proj": k1, "dn_state": ks, "out_proj": k3}


def load_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# the files each profiled kernel is built from: its translation unit, the
# library headers it includes and the public header they include
KERNEL_SOURCES = {
    "dn_state": ("gated_deltanet_hybrid_gb300/csrc/dn_core_stream.cu", "gated_deltanet_hybrid_gb300/csrc/dn_device.cuh",
                 "gated_deltanet_hybrid_gb300/csrc/dn_internal.cuh", "gated_deltanet_hybrid_gb300/csrc/dn_sched.cuh",
                 "include/dn.h"),
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """sha256 (first 16 hex digits) of a profiled kernel's source files
    (KERNEL_SOURCES), or of every .cu/.cuh file of the library."""
    if kernel is None:
        csrc = os.path.join("gated_deltanet_hybrid_gb300", "csrc")
        files = sorted(os.path.join(csrc, f) for f in os.listdir(os.path.join(ROOT, csrc)) if f.endswith((".cu", ".cuh")))
    else:
        files = sorted(KERNEL_SOURCES[kernel])
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload, if it was taken from the kernel's current sources (the
    summary's source_hash against kernel_source_hash(kernel))."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("- source_hash", "- dram_bytes_per_launch")):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if kernel not in KERNEL_SOURCES or vals.get("source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons; each sample is
    stamped on arrival so that only those inside the timed region count."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid: str | None):
        self.uuid = device_uuid
        self.proc = None
        self.rows: list[tuple[float, list[str]]] = []

    def _reader(self):
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def __enter__(self):
        import threading
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t_start: float, t_end: float) -> dict:
        inside = [r for t, r in self.rows if t_start <= t <= t_end + 0.05]
        where = "timed region"
        if not inside:  # region shorter than one sampling period: nearest samples
            inside = [r for t, r in sorted(self.rows, key=lambda tr: abs(tr[0] - t_end))[:3]]
            where = "nearest to the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in inside if num(r[1]) is not None]
        smax = [num(r[2]) for r in inside if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "samples_from": where,
                "power_w_max": max((num(r[3]) or 0.0) for r in inside)}


# --------------------------------------------------------------------- GPU arm
def setup_layers(cfg: DNConfig, B: int, n_layers: int, init_std: float, seed: int, torch, abi):
    """n_layers layer objects with seeded weights; the initial state is drawn
    on the device (normal, std init_std) and pushed through dn_set_state."""
    layers = []
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    for l in range(n_layers):
        w = make_weights(cfg, np.random.Generator(np.random.PCG64(seed * 1000 + l)))
        h = abi.dn_create(cfg, w, B)
        if init_std > 0:
            S = torch.randn((B, cfg.n_v_heads, cfg.dk, cfg.dv), generator=gen, device="cuda") * init_std
            ring = torch.randn((B, cfg.conv_k - 1, cfg.conv_ch), generator=gen, device="cuda") * init_std
            rp = torch.zeros(B, dtype=torch.int32, device="cuda")
            abi.dn_set_state(h, 0, S, ring, rp)
            del S, ring
        layers.append(h)
    return layers


def make_inputs(cfg: DNConfig, B: int, n: int, seed: int):
    """n sets of (x, g, beta) on the host, float32, drawn with the workload's
    recipe (x ~ N(0,1); a, b ~ N(0,1) -> g, beta)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sets = []
    for _ in range(n):
        x = rng.standard_normal((B, cfg.hidden)).astype(np.float32)
        g, beta = gates_from_ab(rng.standard_normal((B, cfg.n_v_heads)), rng.standard_normal((B, cfg.n_v_heads)))
        sets.append((x, g, beta))
    return sets


GRAPH_CHUNK = 512  # steps per captured graph


def capture_steps(n_steps, step, torch):
    """One CUDA graph holding steps 0 .. n_steps-1 (dn_step calls in stream
    order, so programmatic dependent launch overlaps consecutive steps inside
    it as it does for eager calls); None if capture is not possible."""
    stream = torch.cuda.current_stream()
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for i in range(n_steps):
                    step(i)
        torch.cuda.synchronize()
    except Exception as e:  # capture not possible: time eager launches
        print(f"[bench] graph capture failed ({e}); timing eager launches", file=sys.stderr)
        return None
    return g


def step_graphs(steps, n_layers, step, torch):
    """Graphs for a region of exactly `steps` steps: a graph of
    min(steps, GRAPH_CHUNK) steps (a multiple of n_layers when longer than
    that) replayed whole, then one graph of the remainder.  Returns a list of
    graphs to replay in order, or None."""
    chunk = min(steps, max(n_layers, GRAPH_CHUNK // n_layers * n_layers))
    reps, rem = divmod(steps, chunk)
    main = capture_steps(chunk, step, torch)
    if main is None:
        return None
    seq = [main] * reps
    if rem:
        tail = capture_steps(rem, step, torch)
        if tail is None:
            return None
        seq.append(tail)
    return seq


def timed_regions(run_region, steps, dist_ctx, torch, min_repeats=5, min_total_s=0.5, max_repeats=2000):
    """Times the region (exactly `steps` steps) with CUDA events on the
    launching stream, a barrier and a synchronize on both sides, the max over
    ranks; repeats it until it has run at least min_repeats times and for at
    least min_total_s in total.  Returns (per-repeat ms list, wall start, wall
    end).  Every rank takes the same decision (it uses the max over ranks)."""
    stream = torch.cuda.current_stream()
    ms_list = []
    t_first = None
    total = 0.0
    while True:
        dist_ctx.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        if t_first is None:
            t_first = t0
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        run_region()
        ev1.record(stream)
        torch.cuda.synchronize()
        dist_ctx.barrier()
        ms = dist_ctx.max(ev0.elapsed_time(ev1))
        ms_list.append(ms)
        total += ms / 1e3
        if (len(ms_list) >= min_repeats and total >= min_total_s) or len(ms_list) >= max_repeats:
            break
    return ms_list, t_first, time.time()


def region_stats(ms_list, steps):
    med = statistics.median(ms_list)
    return {"repeats": len(ms_list), "steps_per_repeat": steps,
            "ms_per_step_median": med / steps, "ms_per_step_min": min(ms_list) / steps,
            "ms_per_step_max": max(ms_list) / steps}


def bench_gpu(cfg, B, init_std, steps, warmup, n_layers, seed, use_graph, dist_ctx, torch, abi,
              profile=True, e2e=True):
    dev = torch.device("cuda")
    layers = setup_layers(cfg, B, n_layers, init_std, seed, torch, abi)
    host_inputs = make_inputs(cfg, B, n_layers, seed + 7)
    d_in = [(torch.from_numpy(x).to(dev), torch.from_numpy(g).to(dev), torch.from_numpy(b).to(dev))
            for x, g, b in host_inputs]
    d_out = [torch.empty((B, cfg.hidden), dtype=torch.float32, device=dev) for _ in range(n_layers)]
    stream = torch.cuda.current_stream()

    def step(i):
        l = i % n_layers
        x, g, b = d_in[l]
        abi.dn_step(layers[l], B, x, g, b, d_out[l])

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    graphs = step_graphs(steps, n_layers, step, torch) if use_graph else None
    launches_per_step = abi.dn_step_kernels(layers[0], B)

    # ---- timed region: exactly `steps` steps, rotating over the layers ----
    def run_region():
        if graphs is not None:
            for g in graphs:
                g.replay()
        else:
            for i in range(steps):
                step(i)

    ms_list, t0, t1 = timed_regions(run_region, steps, dist_ctx, torch)
    out = {"ms": statistics.median(ms_list), "region": region_stats(ms_list, steps), "t_wall": (t0, t1),
           "graph": graphs is not None, "launches": steps * launches_per_step * len(ms_list),
           "launches_per_region": steps * launches_per_step}

    # ---- per-kernel device times (CUDA events between the kernels) ----
    if profile:
        n_prof = min(steps, 2048)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_prof)]
        for es in evs:  # torch creates the CUDA event on first record
            for e in es:
                e.record(stream)
        torch.cuda.synchronize()
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(200_000_000)  # ~0.1 s: the CPU queues the steps meanwhile
        for i in range(n_prof):
            l = i % n_layers
            abi.dn_profile_next_step(layers[l], evs[i])
            x, g, b = d_in[l]
            abi.dn_step(layers[l], B, x, g, b, d_out[l])
        torch.cuda.synchronize()
        per_kernel = {k: 0.0 for k in KERNELS}
        for e in evs:
            for k in KERNELS:
                a, z = STAGE_EVENTS[k]
                per_kernel[k] += e[a].elapsed_time(e[z])
        out["per_kernel_ms"] = {k: v / n_prof for k, v in per_kernel.items()}

    # ---- end to end through the ABI with host buffers ----
    if e2e:
        n_e2e = min(steps, 2000)
        hx = [torch.from_numpy(x).pin_memory() for x, _, _ in host_inputs]
        hg = [torch.from_numpy(g).pin_memory() for _, g, _ in host_inputs]
        hb = [torch.from_numpy(b).pin_memory() for _, _, b in host_inputs]
        ho = [torch.empty((B, cfg.hidden), dtype=torch.float32).pin_memory() for _ in range(n_layers)]
        for i in range(min(warmup, 8)):
            l = i % n_layers
            abi.dn_step(layers[l], B, hx[l], hg[l], hb[l], ho[l], stream=stream.cuda_stream)
        dist_ctx.barrier()
        torch.cuda.synchronize()
        te0 = time.perf_counter()
        for i in range(n_e2e):
            l = i % n_layers
            abi.dn_step(layers[l], B, hx[l], hg[l], hb[l], ho[l], stream=stream.cuda_stream)
        torch.cuda.synchronize()
        out["e2e_s"] = dist_ctx.max(time.perf_counter() - te0)
        out["n_e2e"] = n_e2e
        out["h2d_bytes"] = B * (cfg.hidden + 2 * cfg.n_v_heads) * 4
        out["d2h_bytes"] = B * cfg.hidden * 4
        dist_ctx.barrier()

    del graphs
    for h in layers:
        abi.dn_destroy(h)
    return out


# --------------------------------------------------------------------- CPU oracle
BLAS_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _oracle_worker(q, barrier, cfg, n_seq, init_std, seconds, steps, warmup):
    """One spawned process of the CPU oracle: n_seq independent sequences of
    the workload's layer (float64 oracle, one BLAS thread), stepped either
    exactly `steps` times or until `seconds` have passed, timed from a barrier
    that every worker passes together.  Puts (sequence-steps, seconds)."""
    try:
        from oracle import OracleLayer
        from gated_deltanet_hybrid_gb300.inputs import random_state, zero_state
        rng = np.random.Generator(np.random.PCG64(99))
        w = make_weights(cfg, rng)
        st = random_state(cfg, n_seq, rng, init_std) if init_std > 0 else zero_state(cfg, n_seq)
        layer = OracleLayer(cfg, w, st)
        inputs = make_inputs(cfg, n_seq, 4, 123)
        for i in range(warmup):
            layer.step(*inputs[i % 4])
        barrier.wait()
        t0 = time.perf_counter()
        n = 0
        while (n < steps) if steps else (time.perf_counter() - t0 < seconds):
            layer.step(*inputs[n % 4])
            n += 1
        q.put((n * n_seq, time.perf_counter() - t0))
    except Exception as e:  # reported by the parent
        barrier.abort()
        q.put(("error", repr(e)))


def run_oracle_pool(cfg, B, init_std, workers, seconds=None, steps=None, warmup=1):
    """The float64 oracle on the host cores: the B sequences of one
    layer-step split over `workers` spawned processes (one BLAS thread each),
    all started together.  Returns (sequence-steps, seconds of the slowest
    worker, workers used)."""
    import multiprocessing as mp
    workers = max(1, min(workers, B))
    shares = [B // workers + (1 if i < B % workers else 0) for i in range(workers)]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    barrier = ctx.Barrier(workers)
    saved = {v: os.environ.get(v) for v in BLAS_ENV}
    procs = []
    try:
        for v in BLAS_ENV:
            os.environ[v] = "1"
        for n_seq in shares:
            pr = ctx.Process(target=_oracle_worker,
                             args=(q, barrier, cfg, n_seq, init_std, seconds, steps, warmup))
            pr.start()
            procs.append(pr)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    res = [q.get() for _ in procs]
    for pr in procs:
        pr.join()
    errs = [r[1] for r in res if r[0] == "error"]
    if errs:
        raise RuntimeError(f"oracle worker failed: {errs[0]}")
    return sum(r[0] for r in res), max(r[1] for r in res), workers


def cpu_baseline(cfg, B, init_std, seconds, workload):
    """The oracle as it stands on a bounded sample of the workload: every
    host core steps its share of the batch's sequences (two thirds of the
    budget), then one core steps min(B, 4) sequences (one third)."""
    cores = host_cores()
    n_all, t_all, used = run_oracle_pool(cfg, B, init_std, cores, seconds=2 * seconds / 3)
    n1, t1, _ = run_oracle_pool(cfg, min(B, 4), init_std, 1, seconds=seconds / 3)
    return {"value": n_all / t_all / B, "unit": UNIT, "cores": used, "kind": "oracle",
            "value_1core": n1 / t1 / B,
            "sample": f"{n_all} sequence-steps of the {workload} layer's {B} sequences spread over "
                      f"{used} host processes (one BLAS thread each, {t_all:.1f} s), and {n1} "
                      f"sequence-steps on one core ({t1:.1f} s); float64 numpy oracle, scaled to "
                      f"layer-steps of batch {B}"}


# --------------------------------------------------------------------- distributed
class DistCtx:
    def __init__(self, torch):
        self.torch = torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend=backend)
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            if self.torch.cuda.is_available():
                self.dist.barrier(device_ids=[self.local_rank])
            else:
                self.dist.barrier()

    def max(self, v: float) -> float:
        if self.dist is None:
            return v
        dev = "cuda" if self.torch.cuda.is_available() else "cpu"
        t = self.torch.tensor([float(v)], dtype=self.torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# --------------------------------------------------------------------- arms
WORKLOAD_SPECS = {
    "35b_b64": (SHAPE_35B, 64, 0.02),
    "35b_b1": (SHAPE_35B, 1, 0.0),
    "35b_b8": (SHAPE_35B, 8, 0.0),  # the batch of the 2048-token long-prompt parity case
    "35b_b1_int4": (dataclasses.replace(SHAPE_35B, int4=True), 1, 0.0),  # the page's per-row int4 model
}
# stacks of distinct layers driven through dn_stack_step (zero initial state)
STACK_SPECS = {
    "stack30_b1": (SHAPE_35B, 1, 30),
    "stack30_b16": (SHAPE_35B, 16, 30),
}


def bench_stack(cfg, batches, n_layers, steps, warmup, seed, use_graph, dist_ctx, torch, abi):
    """Tokens through a stack of n_layers layer objects (held once, for the
    largest batch): for each batch size, `warmup` tokens (the prompt, token
    by token), then timed regions of `steps` tokens, each token starting the
    residual stream from the same fresh input rows (as a new token's
    embedding would) and running dn_stack_step over every layer."""
    dev = torch.device("cuda")
    Bmax = max(batches)
    layers = setup_layers(cfg, Bmax, n_layers, 0.0, seed, torch, abi)
    stream = torch.cuda.current_stream()
    res = {}
    for B in batches:
        rng = np.random.Generator(np.random.PCG64(seed + 7 + B))
        h0 = torch.from_numpy(rng.standard_normal((B, cfg.hidden)).astype(np.float32)).to(dev)
        gb = [gates_from_ab(rng.standard_normal((B, cfg.n_v_heads)), rng.standard_normal((B, cfg.n_v_heads)))
              for _ in range(n_layers)]
        g = torch.from_numpy(np.stack([x[0] for x in gb]).astype(np.float32)).to(dev)
        beta = torch.from_numpy(np.stack([x[1] for x in gb]).astype(np.float32)).to(dev)
        h = torch.empty_like(h0)

        def token():
            h.copy_(h0)
            abi.dn_stack_step(layers, B, h, g, beta)

        for _ in range(warmup):
            token()
        torch.cuda.synchronize()
        graph = None
        if use_graph:
            try:
                graph = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream()
                cap.wait_stream(stream)
                with torch.cuda.stream(cap):
                    with torch.cuda.graph(graph, stream=cap):
                        token()
                torch.cuda.synchronize()
            except Exception as e:  # capture not possible: time eager launches
                print(f"[bench] graph capture failed ({e}); timing eager launches", file=sys.stderr)
                graph = None

        def run_region():
            for _ in range(steps):
                if graph is not None:
                    graph.replay()
                else:
                    token()

        ms_list, t0, t1 = timed_regions(run_region, steps, dist_ctx, torch, min_repeats=3, min_total_s=0.2)
        per_token = steps * (n_layers * abi.dn_step_kernels(layers[0], B) + n_layers + 1)
        res[B] = {"ms": statistics.median(ms_list), "region": region_stats(ms_list, steps),
                  "t_wall": (t0, t1), "graph": graph is not None, "launches": per_token * len(ms_list)}
        del graph
    for l in layers:
        abi.dn_destroy(l)
    return res


PREFILL_COLS = 512  # dn_prefill's block: token columns (sequences x tokens)


def prefill_blocks(B, S):
    """(sequences, token columns) of each block dn_prefill cuts a prompt into:
    up to PREFILL_COLS sequences at a time, PREFILL_COLS // sequences tokens
    per block."""
    for b0 in range(0, B, PREFILL_COLS):
        nb = min(PREFILL_COLS, B - b0)
        T = max(1, PREFILL_COLS // nb)
        for t0 in range(0, S, T):
            yield nb, nb * min(T, S - t0)


def prefill_block_kernels(cfg, nb, cols, torch):
    """Kernels dn_prefill launches for one block: gather, (pack +) in_proj,
    steps 2-4 (one kernel for 128-wide heads when (in_proj row tiles x
    sequences) covers the SMs, else row sums, conv/norms and ring), the
    recurrence, the gated norm, the out_proj and its reduction."""
    in_rows = 2 * cfg.n_qk_heads * cfg.dk + 2 * cfg.n_v_heads * cfg.dv
    proj_rows = in_rows + (cfg.n_v_heads * cfg.gate_width + cfg.n_v_heads if cfg.device_gates else 0)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    fused = cfg.dk == 128 and cfg.dv == 128 and cfg.conv_k <= 8 and -(-proj_rows // 128) * nb >= sms
    return 1 + (2 if cols >= TC_MIN_COLS else 1) + (1 if fused else 3) + 4


def bench_prefill(cfg, B, S, n_layers, seed, dist_ctx, torch, abi, init_std=0.0, repeats_min=3):
    """Prompts through dn_prefill: each timed region runs one prompt of S
    tokens for all B sequences on each of n_layers layer objects (distinct
    weights and states, so consecutive prompts do not find each other's data
    in L2), replayed from a CUDA graph.  Returns the median ms per prompt."""
    dev = torch.device("cuda")
    layers = setup_layers(cfg, B, n_layers, init_std, seed, torch, abi)
    rng = np.random.Generator(np.random.PCG64(seed + 11))
    x = torch.from_numpy(rng.standard_normal((B, S, cfg.hidden)).astype(np.float32)).to(dev)
    g, beta = gates_from_ab(rng.standard_normal((B, S, cfg.n_v_heads)), rng.standard_normal((B, S, cfg.n_v_heads)))
    g, beta = torch.from_numpy(g).to(dev), torch.from_numpy(beta).to(dev)
    out = torch.empty((B, S, cfg.hidden), dtype=torch.float32, device=dev)

    def run(i):
        abi.dn_prefill(layers[i % n_layers], B, S, x, g, beta, out)

    for i in range(n_layers):  # first calls allocate the prefill scratch
        run(i)
    torch.cuda.synchronize()
    graph = capture_steps(n_layers, run, torch)

    def region():
        if graph is not None:
            graph.replay()
        else:
            for i in range(n_layers):
                run(i)

    ms_list, t0, t1 = timed_regions(region, n_layers, dist_ctx, torch, min_repeats=repeats_min, min_total_s=0.3)
    launches = sum(prefill_block_kernels(cfg, nb, cols, torch) for nb, cols in prefill_blocks(B, S))
    del graph
    for h in layers:
        abi.dn_destroy(h)
    return {"ms": statistics.median(ms_list) / n_layers, "region": region_stats(ms_list, n_layers),
            "t_wall": (t0, t1), "launches": launches * n_layers * len(ms_list)}


def stack_summary(cfg, B, n_layers, steps, r, n, hbm_peak):
    s = r["ms"] / 1e3
    ms_layer = r["ms"] / (steps * n_layers)
    sb = step_bytes(cfg, B)
    return {"value": n * steps * n_layers / s, "unit": UNIT, "tokens_per_s": n * steps * B / s,
            "ms_per_token": r["ms"] / steps, "ms_per_step": ms_layer, "batch": B, "layers": n_layers,
            "hbm_gbs_step": sb / (ms_layer / 1e3) / 1e9,
            "step_roofline_frac": sb / (ms_layer / 1e3) / 1e9 / hbm_peak,
            "region": r["region"], "launch": "cuda graph of one token" if r["graph"] else "eager"}


def run_stack(args, torch, dist_ctx):
    from gated_deltanet_hybrid_gb300 import abi
    abi.load_library()
    hbm_peak, peak_kind = load_peaks()
    cfg, B, n_layers = STACK_SPECS[args.workload]
    with ClockSampler(gpu_uuid(torch)) as clk:
        r = bench_stack(cfg, [B], n_layers, args.steps, args.warmup, 3, args.graph, dist_ctx, torch, abi)[B]
    n = dist_ctx.world
    summ = stack_summary(cfg, B, n_layers, args.steps, r, n, hbm_peak)
    line = {
        "metric": METRIC, "value": summ["value"], "unit": UNIT, "n_gpus": n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": summ["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 (int8 weights)",
        "data": "synthetic (seeded random weights and inputs of the 35B-shape layer, zero initial state)",
        "config": {"workload": args.workload, "layers": n_layers, "batch": B, "hidden": cfg.hidden,
                   "l2": f"inputs larger than L2: {n_layers} distinct layers per token",
                   "launch": summ["launch"],
                   "parallelism": f"replicas x{n}" if n > 1 else "single GPU"},
        "clocks": clk.summary(*r["t_wall"]), "gpu_launches": r["launches"] * n, "peak_kind": peak_kind,
    }
    line.update({k: summ[k] for k in ("tokens_per_s", "ms_per_token", "hbm_gbs_step", "step_roofline_frac",
                                      "region")})
    return line


def gpu_uuid(torch):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        return None


def run_ours(args, torch, dist_ctx):
    from gated_deltanet_hybrid_gb300 import abi
    abi.load_library()
    hbm_peak, peak_kind = load_peaks()
    cfg, B, init_std = WORKLOAD_SPECS[args.workload]
    with ClockSampler(gpu_uuid(torch)) as clk:
        r = bench_gpu(cfg, B, init_std, args.steps, args.warmup, args.layers, 2, args.graph,
                      dist_ctx, torch, abi)
    clocks = clk.summary(*r["t_wall"])
    n = dist_ctx.world
    ms_per_step = r["ms"] / args.steps
    value = n * args.steps / (r["ms"] / 1e3)
    sb = step_bytes(cfg, B)
    kb = kernel_bytes(cfg, B)
    dom = max(KERNELS, key=lambda k: r["per_kernel_ms"][k])
    dom_ms = r["per_kernel_ms"][dom]
    achieved = kb[dom] / (dom_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (int8 weights)",
        "data": "synthetic (seeded random weights, state and inputs of the 35B-shape layer)",
        "config": {"workload": args.workload, "hidden": cfg.hidden, "qk_heads": cfg.n_qk_heads,
                   "v_heads": cfg.n_v_heads, "dk": cfg.dk, "dv": cfg.dv, "conv_k": cfg.conv_k,
                   "batch": B, "layers_rotated": args.layers,
                   "l2": f"inputs larger than L2: {args.layers} layer objects rotated, "
                         f"{sb / 1e6:.1f} MB per layer-step",
                   "launch": f"cuda graphs of up to {GRAPH_CHUNK} consecutive steps" if r["graph"] else "eager",
                   "parallelism": f"replicas x{n}" if n > 1 else "single GPU"},
        "region": r["region"],
        "hbm_gbs_step": sb / (ms_per_step / 1e3) / 1e9,
        "step_roofline_frac": sb / (ms_per_step / 1e3) / 1e9 / hbm_peak,
        "per_kernel_us": {k: v * 1e3 for k, v in r["per_kernel_ms"].items()},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "algorithmic_bytes_per_launch": kb[dom],
                     "traffic": ncu_traffic(dom, args.workload),
                     "timing": "CUDA events around each kernel, eager pass over min(K, 2048) steps"},
        "clocks": clocks,
        "gpu_launches": r["launches"] * n,
        "e2e": {"value": n * r["n_e2e"] / r["e2e_s"], "unit": UNIT,
                "h2d_bytes_per_step": r["h2d_bytes"], "d2h_bytes_per_step": r["d2h_bytes"],
                "steps": r["n_e2e"], "api": "dn_step with pinned host pointers (copies + sync inside)"},
    }
    if args.secondary and args.workload == "35b_b64":
        for key, wl in (("batch1", "35b_b1"), ("batch8", "35b_b8"), ("batch1_int4", "35b_b1_int4")):
            c2, B2, std2 = WORKLOAD_SPECS[wl]
            st2 = max(args.steps, 2000)
            r2 = bench_gpu(c2, B2, std2, st2, args.warmup, args.layers, 1, True, dist_ctx, torch, abi,
                           profile=key == "batch1", e2e=key == "batch1")
            ms2 = r2["ms"] / st2
            sb2 = step_bytes(c2, B2)
            sec = {"value": n / (ms2 / 1e3), "unit": UNIT, "ms_per_step": ms2, "batch": B2,
                   "hbm_gbs_step": sb2 / (ms2 / 1e3) / 1e9,
                   "step_roofline_frac": sb2 / (ms2 / 1e3) / 1e9 / hbm_peak, "region": r2["region"],
                   "launch": "cuda graph" if r2["graph"] else "eager"}
            if "per_kernel_ms" in r2:
                sec["per_kernel_us"] = {k: v * 1e3 for k, v in r2["per_kernel_ms"].items()}
            if "e2e_s" in r2:
                sec["e2e_value"] = n * r2["n_e2e"] / r2["e2e_s"]
            line[key] = sec
            line["gpu_launches"] += r2["launches"] * n
        # the 30-layer stack: 49 prompt tokens token by token, then 200 timed tokens
        cs, _, nl = STACK_SPECS["stack30_b1"]
        rs = bench_stack(cs, [1, 16], nl, 200, 49, 3, True, dist_ctx, torch, abi)
        for Bs, rr in rs.items():
            line[f"stack30_b{Bs}"] = stack_summary(cs, Bs, nl, 200, rr, n, hbm_peak)
            line["gpu_launches"] += rr["launches"] * n
        # the page's measured setup: 30 layers with per-row int4 weights, batch 1
        c4 = dataclasses.replace(cs, int4=True)
        rr = bench_stack(c4, [1], nl, 200, 49, 3, True, dist_ctx, torch, abi)[1]
        line["stack30_b1_int4"] = stack_summary(c4, 1, nl, 200, rr, n, hbm_peak)
        line["gpu_launches"] += rr["launches"] * n
        # prompts through dn_prefill: the stack's 49-token prompt at batch 1 and
        # the long-prompt workload's 2048 tokens at batch 8, one layer
        for key, (Bp, Sp, nl) in (("prefill_b1_s49", (1, 49, 8)), ("prefill_b8_s2048", (8, 2048, 4))):
            rp = bench_prefill(SHAPE_35B, Bp, Sp, nl, 5, dist_ctx, torch, abi)
            line[key] = {"tokens_per_s": n * Bp * Sp / (rp["ms"] / 1e3), "ms_per_prompt": rp["ms"],
                         "batch": Bp, "prompt_tokens": Sp, "layers_rotated": nl, "region": rp["region"],
                         "api": "dn_prefill (one call per prompt), cuda graph"}
            line["gpu_launches"] += rp["launches"] * n
    if dist_ctx.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, B, init_std, args.cpu_seconds, args.workload)
    return line


def run_reference(args, dist_ctx):
    """The oracle as the reference arm: each timed step is one whole
    layer-step (all B sequences of the workload advance one token), the
    sequences spread over the host cores; rank 0 only."""
    if dist_ctx.rank != 0:
        return None
    if args.workload in STACK_SPECS:
        cfg, B, _ = STACK_SPECS[args.workload]
        init_std = 0.0
    else:
        cfg, B, init_std = WORKLOAD_SPECS[args.workload]
    # each timed step advances n_seq of the B sequences: all of them when
    # --steps + --warmup whole layer-steps fit the time budget, else as many
    # as keep the run within it (at least one per host process)
    cores = host_cores()
    n_probe, t_probe, _ = run_oracle_pool(cfg, B, init_std, cores, steps=2, warmup=1)
    t_layer = t_probe / 2
    n_seq = B
    if (args.steps + args.warmup) * t_layer > REFERENCE_BUDGET_S:
        n_seq = max(min(cores, B), min(B, math.ceil(B * REFERENCE_BUDGET_S / ((args.steps + args.warmup) * t_layer))))
    seq_steps, dt, used = run_oracle_pool(cfg, n_seq, init_std, cores, steps=args.steps, warmup=args.warmup)
    value = seq_steps / dt / B
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist_ctx.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random weights and inputs of the workload's shape)",
            "config": {"workload": args.workload, "batch": B, "hidden": cfg.hidden,
                       "v_heads": cfg.n_v_heads, "dk": cfg.dk, "dv": cfg.dv},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": f"{args.steps} timed steps, each advancing {n_seq} of the batch-{B} "
                                       f"layer's {B} sequences by one token ({seq_steps} sequence-steps in "
                                       f"{dt:.1f} s), spread over {used} host processes (one BLAS thread "
                                       f"each), float64 numpy oracle, scaled to layer-steps of batch {B}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_prefill_only(args, torch, dist_ctx):
    """One prompt shape through dn_prefill (the secondary prompt keys of the
    default run, for any B and S)."""
    from gated_deltanet_hybrid_gb300 import abi
    B, S = (int(v) for v in args.prefill.split(","))
    r = bench_prefill(SHAPE_35B, B, S, args.layers, 5, dist_ctx, torch, abi)
    return {"metric": "prompt tokens/s", "value": B * S / (r["ms"] / 1e3), "unit": "tokens/s",
            "ms_per_prompt": r["ms"], "batch": B, "prompt_tokens": S, "layers_rotated": args.layers,
            "gpu_launches": r["launches"], "region": r["region"],
            "api": "dn_prefill (one call per prompt), cuda graph"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(WORKLOAD_SPECS) + tuple(STACK_SPECS), default="35b_b64")
    ap.add_argument("--layers", type=int, default=8, help="layer objects rotated in the timed region")
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=True,
                    help="replay a CUDA graph of one step per layer in the timed region "
                         "(--no-graph: eager dn_step calls)")
    ap.add_argument("--secondary", action=argparse.BooleanOptionalAction, default=True,
                    help="also measure the batch-1 workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", metavar="B,S",
                    help="only time prompts of S tokens for B sequences through dn_prefill "
                         "(35B-shape layer) and print their line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    import torch
    dist_ctx = DistCtx(torch)
    try:
        if args.impl == "reference":
            line = run_reference(args, dist_ctx)
        else:
            if not torch.cuda.is_available():
                raise SystemExit("bench.py --impl ours needs a CUDA device")
            torch.cuda.set_device(dist_ctx.local_rank)
            if args.prefill:
                line = run_prefill_only(args, torch, dist_ctx)
            else:
                line = (run_stack if args.workload in STACK_SPECS else run_ours)(args, torch, dist_ctx)
        if line is not None and dist_ctx.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist_ctx.close()


if __name__ == "__main__":
    main()
