"""Benchmark of the H2O decode / prefill path on one (or N) GPUs.

A step is one pass of the whole path over one batch of the OPT-6.7B
attention-layer workload (batch 8, 32 heads, head_dim 128, fp16 K/V, prompt
2048 + 256 decode steps, 205 heavy + 205 recent slots), for every one of the
model's 32 attention layers: the prefill of each layer (row statistics,
column sums, keep rule, output) followed by 256 decode steps, each visiting
the 32 layers in turn.  The 32 per-layer caches (1.8 GB) and inputs (14 GB)
are far larger than L2, so every layer's K/V comes from HBM.  The per-step
launches are captured once in two CUDA graphs (prefill, decode) and replayed.

value = decode tokens per attention layer per second over the whole step
        (batch * 256 tokens * 32 layers * N GPUs / step time).
Also reported: the decode kernel's roofline against the measured HBM
bandwidth, the end-to-end number through the public API with host buffers,
and the fp64 CPU oracle timed on the host's cores.

`--impl reference` times the CPU oracle alone on a bounded sample.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from kv_cache_eviction_03_gb300 import accounting as A  # noqa: E402
from kv_cache_eviction_03_gb300 import sharding  # noqa: E402
from kv_cache_eviction_03_gb300 import workload as W  # noqa: E402

METRIC = "H2O decode tokens/s per attention layer; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s/layer"
WORKLOAD = "opt-6.7b"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=None, help="override the layer rotation (default: model's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--decode-only", action="store_true", help="profiling aid: replay only the decode graph")
    return ap.parse_args()


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


# ------------------------------------------------------------------ CPU oracle leg
def _warm(_=None):
    from oracle import h2o_oracle  # noqa: F401

    return 0


def _oracle_pairs(args):
    """Worker: prefill + every decode step of a few pairs (one process)."""
    (q, k, v, dq, dk, dv, heavy, recent, scale) = args
    import time as _t

    from oracle import h2o_oracle as O

    t0 = _t.perf_counter()
    st, _, _ = O.prefill(q, k, v, heavy, recent, scale)
    t1 = _t.perf_counter()
    for t in range(dq.shape[0]):
        st, _, _, _ = O.decode_step(st, dq[t], dk[t], dv[t], heavy, recent, scale)
    t2 = _t.perf_counter()
    return t1 - t0, t2 - t1


def oracle_sample(w, seed, batch_rows=1, decode_steps=None):
    """Inputs for the CPU leg: `batch_rows` batch rows (all heads) of layer 0."""
    ws = w.with_(batch=batch_rows)
    q, k, v = W.prefill_inputs(ws, seed)
    T = w.decode if decode_steps is None else decode_steps
    dq, dk, dv = W.decode_sequence(ws, w.prompt, T, seed)
    return ws, (q, k, v, dq, dk, dv), T


def time_oracle(w, seed, workers=None, batch_rows=4):
    """fp64 oracle on the host cores over a sample of the workload; returns
    (tokens/s/layer scaled to the whole workload, cores, sample text, seconds)."""
    import multiprocessing as mp

    ws, (q, k, v, dq, dk, dv), T = oracle_sample(w, seed, batch_rows)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    workers = workers or min(cores, ws.pairs)
    # one task per (batch row, head) pair (pairs are independent);
    # single-threaded BLAS per worker
    tasks = [(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], dq[:, b:b + 1, h:h + 1],
              dk[:, b:b + 1, h:h + 1], dv[:, b:b + 1, h:h + 1], w.heavy, w.recent, w.scale)
             for b in range(ws.batch) for h in range(ws.heads)]
    env_keep = {x: os.environ.get(x) for x in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for x in env_keep:
        os.environ[x] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            pool.map(_warm, range(workers))  # imports done before the clock starts
            t0 = time.perf_counter()
            res = pool.map(_oracle_pairs, tasks)
            wall = time.perf_counter() - t0
    finally:
        for x, val in env_keep.items():
            if val is None:
                os.environ.pop(x, None)
            else:
                os.environ[x] = val
    sample_pairs = ws.pairs
    scale_up = w.pairs / sample_pairs  # the whole workload has this many more pairs
    full_layer_time = wall * scale_up
    value = w.batch * T / full_layer_time
    sample = (f"{batch_rows} of {w.batch} batch rows ({sample_pairs} of {w.pairs} (batch, head) pairs), "
              f"one layer, prefill {w.prompt} + {T} decode steps; wall time x {scale_up:g} pairs ratio")
    return value, workers, sample, wall


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.idx = gpu_index

    def start(self):
        try:
            listed = subprocess.run(["nvidia-smi", "-L"], capture_output=True, text=True, timeout=20).stdout
            sel = [] if len(listed.strip().splitlines()) <= 1 else [f"--id={self.idx}"]
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError, subprocess.SubprocessError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


DECODE_SOURCES = ("decode.cu", "ptx.cuh", "h2o_internal.cuh")


def decode_source_digest():
    """sha256 over the sources the decode kernel is compiled from."""
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "kv_cache_eviction_03_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic_record():
    """DRAM bytes per decode launch from the committed ncu summary, if the
    kernel's sources have not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("decode_sources_sha256") == decode_source_digest() and rec.get("workload") == WORKLOAD:
            return rec.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


# ------------------------------------------------------------------ GPU leg
def run_ours(args, rank, world, local_rank):
    import torch

    from kv_cache_eviction_03_gb300 import binding as B

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    B.lib()
    w = W.WORKLOADS[WORKLOAD]
    NL = args.layers or w.layers
    T, L = w.decode, w.prompt
    seed = W.seed_for(WORKLOAD) + 1000 * rank  # every rank runs its own batch
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    inp = W.device_inputs(w, seed, NL)
    caches = [B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, B.H2O_F16) for _ in range(NL)]
    pout = torch.empty((w.batch, w.heads, L, w.head_dim), dtype=torch.float32, device="cuda")
    dout = torch.empty((T, NL, w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
    dev_ev = torch.empty((T, NL, w.batch, w.heads), dtype=torch.int32, device="cuda")

    def prefill_all(inp, pout):
        for l in range(NL):
            q, k, v = inp["prefill"][l]
            B.h2o_prefill(caches[l], q, k, v, w.scale, out=pout, stream=stream)

    def decode_all(inp, dout, dev_ev):
        for t in range(T):
            for l in range(NL):
                qd, kd, vd = inp["decode"][l]
                B.h2o_decode_step(caches[l], qd[t], kd[t], vd[t], w.scale, dout[t, l], dev_ev[t, l], stream=stream)

    def capture(inp, pout, dout, dev_ev):
        """The step's launches as two CUDA graphs (prefill, decode) over these buffers."""
        g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre, stream=stream):
            prefill_all(inp, pout)
        with torch.cuda.graph(g_dec, stream=stream):
            decode_all(inp, dout, dev_ev)
        return g_pre, g_dec

    def capture_layers(inp, pout):
        """One prefill graph per layer, so each can wait for its own inputs."""
        gs = []
        for l in range(NL):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                q, k, v = inp["prefill"][l]
                B.h2o_prefill(caches[l], q, k, v, w.scale, out=pout, stream=stream)
            gs.append(g)
        return gs

    # eager pass: allocates the prefill workspaces, checks every call works
    prefill_all(inp, pout)
    decode_all(inp, dout, dev_ev)
    for c in caches:
        B.h2o_cache_check(c, stream=stream)
    g_pre, g_dec = capture(inp, pout, dout, dev_ev)
    # per layer: row statistics, attention output, column sums, keep rule; per decode step and layer: one
    launches_per_step = (0 if args.decode_only else 4 * NL) + T * NL

    def step(evs=None):
        if not args.decode_only:
            g_pre.replay()
        if evs is not None:
            evs.record(stream)
        g_dec.replay()

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    mid = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step(mid[i])
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    elapsed = t_begin.elapsed_time(t_end) / 1e3
    decode_s = sum(mid[i].elapsed_time(ends[i]) for i in range(args.steps)) / 1e3
    prefill_s = sum(starts[i].elapsed_time(mid[i]) for i in range(args.steps)) / 1e3
    elapsed, decode_s, prefill_s = sharding.max_over_ranks([elapsed, decode_s, prefill_s], dist, device="cuda")
    for c in caches:
        B.h2o_cache_check(c, stream=stream)

    tokens_per_layer = w.batch * T * world  # per step, every layer
    value = tokens_per_layer * NL * args.steps / elapsed
    step_bytes = A.decode_step_bytes(w.pairs, w.cache_slots, w.head_dim, 2)
    per_launch = decode_s / (args.steps * T * NL)
    achieved = step_bytes / per_launch / 1e9
    peak, peak_kind = measured_peak()
    info = B.h2o_cache_info(caches[0])
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded Zipf-keyed generator, drawn on the GPU)",
        "config": workload_config(w, NL, world, args.decode_only),
        "launch": {"decode_splits": info[6], "decode_stages": info[7]},
        "phases": {"prefill_ms_per_step": prefill_s / args.steps * 1e3,
                   "decode_ms_per_step": decode_s / args.steps * 1e3,
                   "decode_only_tokens_per_s_per_layer": tokens_per_layer * NL * args.steps / decode_s,
                   "prefill_tflops": A.prefill_flops(w.pairs, L, w.head_dim) * NL * args.steps / prefill_s / 1e12
                   if prefill_s > 0 else None},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (fused attention + score + evict + overwrite)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "traffic": decode_traffic_record(),
                     "algorithmic_bytes_per_launch": step_bytes,
                     "avg_launch_us": per_launch * 1e6},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    # ---- end to end through the public API with pinned host buffers
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, w, NL, stream, (inp, pout, dout, dev_ev, capture_layers(inp, pout), g_dec),
                                capture, capture_layers, world, dist)
    del inp
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result


def run_e2e(args, w, NL, stream, set_a, capture, capture_layers, world, dist):
    """The same step through the public API with pinned host buffers: every
    step copies all of its inputs host -> device and reads its decode outputs
    and evicted slots back.  Two device buffer sets (each with its own graphs:
    one prefill graph per layer and the decode graph) let step s+1's
    host -> device copy and step s-1's read-back run on copy streams while
    step s computes, and each layer's prefill waits only for its own inputs;
    every step's bytes still cross the link inside the timed region."""
    import torch

    def pinned(x):
        h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        h.copy_(x)
        return h

    inp_a = set_a[0]
    host_pre = [[pinned(x) for x in inp_a["prefill"][l]] for l in range(NL)]
    host_dec = [[pinned(x) for x in inp_a["decode"][l]] for l in range(NL)]
    inp_b = {k: [[torch.empty_like(x) for x in inp_a[k][l]] for l in range(NL)] for k in ("prefill", "decode")}
    pout_b, dout_b, ev_b = (torch.empty_like(x) for x in set_a[1:4])
    sets = [set_a, (inp_b, pout_b, dout_b, ev_b, capture_layers(inp_b, pout_b),
                    capture(inp_b, pout_b, dout_b, ev_b)[1])]
    host_out = [torch.empty(set_a[2].shape, dtype=set_a[2].dtype, pin_memory=True) for _ in range(2)]
    host_ev = [torch.empty(set_a[3].shape, dtype=set_a[3].dtype, pin_memory=True) for _ in range(2)]
    h2d_bytes = sum(x.numel() * x.element_size() for l in range(NL) for x in host_pre[l] + host_dec[l])
    d2h_bytes = host_out[0].numel() * 4 + host_ev[0].numel() * 4
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_layer = [[torch.cuda.Event() for _ in range(NL)] for _ in range(2)]  # set X, layer l's prompt is on the device
    ev_dec = [torch.cuda.Event() for _ in range(2)]   # set X's decode inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # the step on set X has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of set X are on the host

    copy_ev = []  # (start, end) events around each step's host -> device copies

    def h2d(x, first):
        inp = sets[x][0]
        if not first:
            up.wait_event(ev_done[x])  # the previous step on this set has read its inputs
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(up)
        copy_ev.append((c0, c1))
        with torch.cuda.stream(up):
            for l in range(NL):
                for dst, src in zip(inp["prefill"][l], host_pre[l]):
                    dst.copy_(src, non_blocking=True)
                ev_layer[x][l].record(up)
            for l in range(NL):
                for dst, src in zip(inp["decode"][l], host_dec[l]):
                    dst.copy_(src, non_blocking=True)
            ev_dec[x].record(up)
        c1.record(up)

    def compute(x, first):
        g_pre, g_dec = sets[x][4], sets[x][5]
        if not first:
            stream.wait_event(ev_out[x])  # the previous step's outputs on this set are read back
        for l in range(NL):
            stream.wait_event(ev_layer[x][l])
            if not args.decode_only:
                g_pre[l].replay()
        stream.wait_event(ev_dec[x])
        g_dec.replay()
        ev_done[x].record(stream)

    def d2h(x):
        down.wait_event(ev_done[x])
        with torch.cuda.stream(down):
            host_out[x].copy_(sets[x][2], non_blocking=True)
            host_ev[x].copy_(sets[x][3], non_blocking=True)
        ev_out[x].record(down)

    def run(nsteps, t0=None):
        h2d(0, True)
        for i in range(nsteps):
            x = i % 2
            compute(x, i < 2)
            if i + 1 < nsteps:
                h2d((i + 1) % 2, i + 1 < 2)
            d2h(x)
        stream.wait_event(ev_out[(nsteps - 1) % 2])
        if nsteps > 1:
            stream.wait_event(ev_out[nsteps % 2])

    run(max(2, min(args.warmup, 3)))
    torch.cuda.synchronize()
    copy_ev.clear()
    if dist:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(up)
    stream.wait_event(a)
    run(args.steps)
    b.record(stream)
    torch.cuda.synchronize()
    el = a.elapsed_time(b) / 1e3
    el = sharding.max_over_ranks([el], dist, device="cuda")[0]
    copy_s = sum(c0.elapsed_time(c1) for c0, c1 in copy_ev) / 1e3 / max(len(copy_ev), 1)
    return {"value": w.batch * w.decode * world * NL * args.steps / el, "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "h2d_gbps_measured": h2d_bytes / copy_s / 1e9 if copy_s > 0 else None,
            "pipelined": "step s+1 host->device copy and step s-1 read-back overlap step s"}


def workload_config(w, NL, world, decode_only):
    """The `config` object of the JSON line, identical for both arms."""
    return {"workload": f"{WORKLOAD}: batch {w.batch}, {w.heads} heads, head_dim {w.head_dim}, fp16 K/V, "
                        f"prompt {w.prompt} + {w.decode} decode steps, heavy {w.heavy} + recent {w.recent} slots",
            "layers": NL, "batch": w.batch, "decode_steps": w.decode, "prompt": w.prompt, "accumulate": "f32",
            "l2": f"inputs larger than L2: {NL} layer caches rotated every decode step",
            "parallelism": f"weak: each of {world} GPUs runs its own batch" if world > 1 else "1 GPU",
            "decode_only": bool(decode_only)}


def main():
    args = parse()
    rank, world, local_rank = dist_info()
    w = W.WORKLOADS[WORKLOAD]
    if args.impl == "reference":
        if rank != 0:
            return
        seed = W.seed_for(WORKLOAD)
        vals, walls = [], []
        cores = sample = None
        for i in range(args.warmup + args.steps):
            v, cores, sample, wall = time_oracle(w, seed)
            if i >= args.warmup:
                vals.append(v)
                walls.append(wall)
        value = statistics.median(vals)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(walls) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded Zipf-keyed generator)",
                "config": workload_config(w, args.layers or w.layers, world, args.decode_only),
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    # CPU oracle pool first (spawned before any GPU work)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, cores, sample, wall = time_oracle(w, W.seed_for(WORKLOAD))
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "sample_wall_s": wall}
    result = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if cpu is not None:
            result["cpu_baseline"] = cpu
        print(json.dumps(result))


if __name__ == "__main__":
    main()
