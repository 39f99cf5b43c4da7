"""Benchmark of the H2O decode / prefill path on one (or N) GPUs.

A step is one pass of the whole path over one batch of the chosen workload
(default: the OPT-6.7B attention-layer shape, batch 8, 32 heads, head_dim 128,
fp16 K/V, prompt 2048 + 256 decode steps, 205 heavy + 205 recent slots), for
every one of the model's attention layers: the prefill of each layer (row
statistics, column sums, keep rule, output) followed by the decode steps, each
visiting the layers in turn.  The per-layer caches and inputs are far larger
than L2, so every layer's K/V comes from HBM.  The per-step launches are
captured once in CUDA graphs (prefill, decode) and replayed.

value = decode tokens per attention layer per second over the whole step
        (batch * decode steps * layers * N GPUs / step time).
Also reported: the decode kernel's roofline against the measured HBM
bandwidth (back-to-back layers, and isolated launches with a plain kernel in
between), the end-to-end number through the public API with host buffers,
the fp64 CPU oracle timed on the host's cores, and `per_config`: the decode
launch of every measured workload shape (including the 1,000,000-step
streaming shape's steady state) with its roofline and the oracle's rate.

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
DEFAULT_WORKLOAD = "opt-6.7b"
MAIN_WORKLOADS = ("tiny-ref", "opt-6.7b", "opt-30b", "llama-7b-16k")  # shapes with a prompt
FALLBACK_HBM_GBS = 6800.0

# per_config decode timing: decode steps per graph replay (each visiting every
# layer), untimed and timed replays
PER_CONFIG_STEPS = {"tiny-ref": 64, "opt-6.7b": 64, "opt-30b": 32, "llama-7b-16k": 64}
PER_CONFIG_REPS = (2, 5)
# streaming steady state: the 2048-step fill, then this many decode steps in
# chunks whose inputs are drawn on the GPU between chunks (outside the timing)
STREAM_CHUNK = 1024
STREAM_WINDOW = 10 * 1024
# shapes whose decode launch is also timed with position rolling on (rotary
# embedding at in-cache ranks; base 10000), next to the plain launch
ROLLING = ("opt-6.7b", "llama-7b-16k", "streaming")
ROPE_BASE = 10000.0
# oracle samples per workload: (batch rows, heads or None for all, decode steps or None for all)
ORACLE_SAMPLE = {"tiny-ref": (1, None, None), "opt-6.7b": (4, None, None), "opt-30b": (8, None, None),
                 "llama-7b-16k": (1, 4, None)}
STREAM_ORACLE_PAIRS = 16      # of the streaming shape's 128 pairs
STREAM_ORACLE_WINDOW = 1000   # steady-state steps timed after the oracle's own fill


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_WORKLOAD, choices=MAIN_WORKLOADS,
                    help="workload of the main line (the streaming shape is measured under per_config)")
    ap.add_argument("--seed", type=int, default=None, help="generator seed (default: the workload's)")
    ap.add_argument("--layers", type=int, default=None, help="override the layer rotation (default: model's)")
    ap.add_argument("--check-every", type=int, default=0,
                    help="check every cache's device error flags after every K timed steps (0: at the end)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--per-config", default=",".join(W.WORKLOAD_ORDER),
                    help="comma-separated workloads measured under per_config")
    ap.add_argument("--only-per-config", default=None,
                    help="profiling aid: measure this one workload's decode launch and print it, nothing else")
    ap.add_argument("--stream-window", type=int, default=STREAM_WINDOW,
                    help="steady-state decode steps timed on the streaming shape (a multiple of 1024)")
    ap.add_argument("--decode-only", action="store_true", help="profiling aid: replay only the decode graph")
    return ap.parse_args()


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


# ------------------------------------------------------------------ CPU oracle leg
def _warm(_=None):
    from oracle import h2o_oracle  # noqa: F401

    return 0


def _oracle_pairs(args):
    """Worker: prefill + every decode step of one pair (one process).  With
    `untimed` > 0 the first that many decode steps (a fill) are not timed."""
    (q, k, v, dq, dk, dv, heavy, recent, scale, untimed) = args
    import time as _t

    from oracle import h2o_oracle as O

    t0 = _t.perf_counter()
    if q is not None:
        st, _, _ = O.prefill(q, k, v, heavy, recent, scale)
    else:
        st = O.empty_cache(1, heavy, recent, dq.shape[-1])
    t1 = _t.perf_counter()
    for t in range(untimed):
        st, _, _, _ = O.decode_step(st, dq[t], dk[t], dv[t], heavy, recent, scale)
    t2 = _t.perf_counter()
    for t in range(untimed, dq.shape[0]):
        st, _, _, _ = O.decode_step(st, dq[t], dk[t], dv[t], heavy, recent, scale)
    t3 = _t.perf_counter()
    return t1 - t0, t3 - t2


def _pool_map(tasks, workers):
    """Run oracle tasks on a spawn pool with single-threaded BLAS per worker;
    returns (results, wall seconds)."""
    import multiprocessing as mp

    env_keep = {x: os.environ.get(x) for x in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for x in env_keep:
        os.environ[x] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers) as pool:
            pool.map(_warm, range(workers))  # imports done before the clock starts
            t0 = time.perf_counter()
            res = pool.map(_oracle_pairs, tasks, chunksize=1)
            wall = time.perf_counter() - t0
    finally:
        for x, val in env_keep.items():
            if val is None:
                os.environ.pop(x, None)
            else:
                os.environ[x] = val
    return res, wall


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def time_oracle(w, seed, batch_rows=None, heads=None, decode_steps=None):
    """fp64 oracle on the host cores over a sample of the workload (prefill +
    decode steps of `batch_rows` batch rows and `heads` heads of layer 0).
    Returns a dict: whole-step and decode-only tokens/s/layer scaled to the
    whole workload, cores, sample text, wall seconds."""
    rows = batch_rows or w.batch
    nh = heads or w.heads
    ws = w.with_(batch=rows)
    T = w.decode if decode_steps is None else decode_steps
    q, k, v = W.prefill_inputs(ws, seed)
    dq, dk, dv = W.decode_sequence(ws, w.prompt, T, seed)
    tasks = [(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], dq[:, b:b + 1, h:h + 1],
              dk[:, b:b + 1, h:h + 1], dv[:, b:b + 1, h:h + 1], w.heavy, w.recent, w.scale, 0)
             for b in range(rows) for h in range(nh)]
    workers = min(host_cores(), len(tasks))
    res, wall = _pool_map(tasks, workers)
    sample_pairs = len(tasks)
    scale_up = w.pairs / sample_pairs
    decode_frac = sum(r[1] for r in res) / max(sum(r[0] + r[1] for r in res), 1e-12)
    full = wall * scale_up
    sample = (f"{rows} of {w.batch} batch rows x {nh} of {w.heads} heads ({sample_pairs} of {w.pairs} pairs), "
              f"one layer, prefill {w.prompt} + {T} decode steps; wall time x {scale_up:g} pairs ratio")
    return {"value": w.batch * T / full, "decode_only": w.batch * T / (full * decode_frac),
            "cores": workers, "sample": sample, "wall_s": wall}


def time_oracle_streaming(w, seed, pairs=STREAM_ORACLE_PAIRS, window=STREAM_ORACLE_WINDOW):
    """Streaming shape: each sampled pair fills its cache (untimed), then a
    steady-state window of `window` decode steps is timed."""
    fill = w.cache_slots
    steps = fill + window
    dq, dk, dv = W.decode_sequence(w, 0, steps, seed)  # [steps, B, H, D]
    dq, dk, dv = (a.reshape(steps, w.pairs, w.head_dim) for a in (dq, dk, dv))
    sel = np.linspace(0, w.pairs - 1, pairs).astype(int)
    tasks = [(None, None, None, dq[:, i][:, None, None], dk[:, i][:, None, None], dv[:, i][:, None, None],
              w.heavy, w.recent, w.scale, fill) for i in sel]
    workers = min(host_cores(), len(tasks))
    res, wall = _pool_map(tasks, workers)
    # per-pair window time summed over pairs / workers used = wall share of the window
    window_s = sum(r[1] for r in res) / workers
    scale_up = w.pairs / pairs
    sample = (f"{pairs} of {w.pairs} pairs, one layer, each filled to {fill} slots (untimed), then a "
              f"{window}-step steady-state window timed; time x {scale_up:g} pairs ratio")
    v = w.batch * window / (window_s * scale_up)
    return {"value": v, "decode_only": v, "cores": workers, "sample": sample, "wall_s": wall}


def oracle_baselines(names, seed_override=None):
    out = {}
    for name in names:
        w = W.WORKLOADS[name]
        seed = W.seed_for(name) if seed_override is None else seed_override
        if name == "streaming":
            out[name] = time_oracle_streaming(w, seed)
        else:
            rows, heads, steps = ORACLE_SAMPLE[name]
            out[name] = time_oracle(w, seed, rows, heads, steps)
    return out


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


def decode_traffic_record(workload):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload, if the kernel's sources have not changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("decode_sources_sha256") != decode_source_digest():
            return None
        entry = rec.get("workloads", {}).get(workload)
        return entry.get("dram_bytes_per_launch") if entry else None
    except (OSError, ValueError, AttributeError):
        return None


def elem_bytes(w):
    return 2 if w.dtype == "f16" else 4


def kv_code(w):
    from kv_cache_eviction_03_gb300 import binding as B

    return B.H2O_F16 if w.dtype == "f16" else B.H2O_F32


def timed_replays(fn, stream, reps):
    """Run fn() `reps` times between two CUDA events on `stream`; seconds."""
    import torch

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / 1e3


def decode_roofline(w, us_per_launch, peak):
    nbytes = A.decode_step_bytes(w.pairs, w.cache_slots, w.head_dim, elem_bytes(w))
    gbs = nbytes / us_per_launch / 1e3
    return {"us_per_launch": us_per_launch, "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs,
            "frac": gbs / peak, "tokens_per_s_per_layer": w.batch / us_per_launch * 1e6}


# ------------------------------------------------------------------ per-config decode launches
def measure_decode_shape(name, stream, peak, layers=None, seed=None):
    """Decode launch of one workload shape: `layers` caches (the model's
    attention layers) prefilled with the shape's prompt, then graphs of decode
    steps that visit the layers in turn (cold L2: the caches together are
    larger than L2, except the one-layer tiny shape, which is launch-bound).
    Timed back to back (consecutive layers overlap through programmatic
    dependent launch) and isolated (a plain one-thread kernel between
    launches, as a model's projection kernel would sit there; its own time,
    measured alone, is subtracted)."""
    import torch

    from kv_cache_eviction_03_gb300 import binding as B

    w = W.WORKLOADS[name]
    NL = layers or w.layers
    S = PER_CONFIG_STEPS[name]
    warm, reps = PER_CONFIG_REPS
    draws = W.DeviceDraws(w, W.seed_for(name) if seed is None else seed)
    caches = []
    for _ in range(NL):
        c = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, kv_code(w))
        q, k, v = draws.prefill()
        B.h2o_prefill(c, q, k, v, w.scale, stream=stream)
        caches.append(c)
        del q, k, v
    dq, dk, dv = draws.decode(S, NL)
    del draws
    out = torch.empty((S, NL, w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
    tiny = torch.zeros(1, device="cuda")

    def run(filler):
        for t in range(S):
            for l in range(NL):
                if filler:
                    tiny.add_(1.0)
                B.h2o_decode_step(caches[l], dq[t, l], dk[t, l], dv[t, l], w.scale, out[t, l], stream=stream)

    def run_filler():
        for _ in range(S * NL):
            tiny.add_(1.0)

    graphs = []
    with torch.cuda.stream(stream):
        run(False)  # eager pass: every call works
        for body in (lambda: run(False), lambda: run(True), run_filler):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                body()
            graphs.append(g)
        for g in graphs:
            for _ in range(warm):
                g.replay()
        stream.synchronize()
        t_b2b = timed_replays(graphs[0].replay, stream, reps)
        t_iso = timed_replays(graphs[1].replay, stream, reps)
        t_fill = timed_replays(graphs[2].replay, stream, reps)
    for c in caches:
        B.h2o_cache_check(c, stream=stream)
    launches = S * NL * reps
    info = B.h2o_cache_info(caches[0])
    rolling = None
    if name in ROLLING:  # same caches, rolling switched on after the prefill (ranks from positions)
        for c in caches:
            B.h2o_cache_set_position_rolling(c, ROPE_BASE)
        with torch.cuda.stream(stream):
            run(False)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run(False)
            for _ in range(warm):
                g.replay()
            t_rope = timed_replays(g.replay, stream, reps)
        for c in caches:
            B.h2o_cache_check(c, stream=stream)
        rinfo = B.h2o_cache_info(caches[0])
        rolling = decode_roofline(w, t_rope / launches * 1e6, peak)
        rolling = {"us_per_launch": rolling["us_per_launch"], "frac": rolling["frac"],
                   "vs_plain": t_rope / t_b2b, "launch": {"decode_splits": rinfo[6], "decode_stages": rinfo[7]},
                   "rope_base": ROPE_BASE}
        del g
    res = decode_roofline(w, t_b2b / launches * 1e6, peak)
    if rolling:
        res["rolling"] = rolling
    iso = decode_roofline(w, max(t_iso - t_fill, 1e-9) / launches * 1e6, peak)
    res["isolated"] = {k: iso[k] for k in ("us_per_launch", "achieved_gbs", "frac", "tokens_per_s_per_layer")}
    res["isolated"]["filler_us"] = t_fill / launches * 1e6
    res.update({"layers": NL, "decode_steps_timed": S * reps, "launches_timed": launches,
                "launch": {"decode_splits": info[6], "decode_stages": info[7]},
                "l2": "L2-resident (one 0.1 MB layer; launch-bound)" if name == "tiny-ref"
                else f"cold: {NL} layer caches rotated, larger than L2"})
    for g in graphs:
        del g
    for c in caches:
        B.h2o_cache_destroy(c)
    del dq, dk, dv, out
    torch.cuda.empty_cache()
    return res


def measure_streaming(stream, peak, layers=None, seed=None, window=STREAM_WINDOW, chunk=STREAM_CHUNK):
    """The streaming shape (no prompt, 1024 + 1024 slots, 32 layers): every
    layer's cache fills for 2048 steps, then a steady-state window of
    `window` steps in which every step evicts.  Decode inputs are drawn on
    the GPU, `chunk` steps at a time, into one of two buffers, each with its
    own captured graph of chunk x layers decode launches; the draws run
    between chunks and are timed separately from the decode launches."""
    import torch

    from kv_cache_eviction_03_gb300 import binding as B

    w = W.WORKLOADS["streaming"]
    NL = layers or w.layers
    fill = w.cache_slots
    assert fill % chunk == 0 and window % chunk == 0
    draws = W.DeviceDraws(w, W.seed_for("streaming") if seed is None else seed)
    caches = [B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, B.H2O_F16) for _ in range(NL)]
    for c in caches:
        B.h2o_cache_reset(c, stream=stream)
    shp = (chunk, NL, w.batch, w.heads, w.head_dim)
    bufs = [tuple(torch.empty(shp, dtype=torch.float16, device="cuda") for _ in range(3)) for _ in range(2)]
    out = torch.empty(shp, dtype=torch.float32, device="cuda")

    def run(buf):
        q, k, v = buf
        for t in range(chunk):
            for l in range(NL):
                B.h2o_decode_step(caches[l], q[t, l], k[t, l], v[t, l], w.scale, out[t, l], stream=stream)

    gen_s = 0.0

    def draw_into(buf):
        nonlocal gen_s
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            for dst, src in zip(buf, draws.decode(chunk, NL)):
                dst.copy_(src)
        b.record(stream)
        b.synchronize()
        gen_s += a.elapsed_time(b) / 1e3

    graphs = []
    with torch.cuda.stream(stream):
        for x in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run(bufs[x])
            graphs.append(g)
        # capture issued nothing to the device: the caches are still empty
        n_chunks = 0
        for _ in range(fill // chunk):  # fill phase (untimed)
            draw_into(bufs[n_chunks % 2])
            graphs[n_chunks % 2].replay()
            n_chunks += 1
        stream.synchronize()
        for c in caches:
            B.h2o_cache_check(c, stream=stream)
        gen_s = 0.0
        dec_s = 0.0
        for _ in range(window // chunk):
            draw_into(bufs[n_chunks % 2])
            dec_s += timed_replays(graphs[n_chunks % 2].replay, stream, 1)
            n_chunks += 1
    for c in caches:
        B.h2o_cache_check(c, stream=stream)
    g0 = B.unpack_state(caches[0], B.h2o_cache_export_state(caches[0], stream=stream))
    launches = window * NL
    # position rolling on the same full caches: one chunk, twice
    for c in caches:
        B.h2o_cache_set_position_rolling(c, ROPE_BASE)
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run(bufs[0])
        g.replay()
        t_rope = timed_replays(g.replay, stream, 2)
    for c in caches:
        B.h2o_cache_check(c, stream=stream)
    rinfo = B.h2o_cache_info(caches[0])
    del g
    res = decode_roofline(w, dec_s / launches * 1e6, peak)
    r_us = t_rope / (2 * chunk * NL) * 1e6
    res["rolling"] = {"us_per_launch": r_us, "frac": decode_roofline(w, r_us, peak)["frac"],
                      "vs_plain": r_us / res["us_per_launch"], "decode_steps_timed": 2 * chunk,
                      "launch": {"decode_splits": rinfo[6], "decode_stages": rinfo[7]}, "rope_base": ROPE_BASE}
    info = B.h2o_cache_info(caches[0])
    res.update({"layers": NL, "fill_steps": fill, "decode_steps_timed": window, "launches_timed": launches,
                "position_after": int(g0["p"][0]), "full_after": bool(np.all(g0["count"] == w.cache_slots)),
                "input_draw_ms_per_chunk": gen_s / (window // chunk) * 1e3, "chunk_steps": chunk,
                "input_draw": "torch generator kernels between chunks, not in the decode timing",
                "launch": {"decode_splits": info[6], "decode_stages": info[7]},
                "l2": f"cold: {NL} layer caches of 134 MB rotated"})
    for g in graphs:
        del g
    for c in caches:
        B.h2o_cache_destroy(c)
    del bufs, out
    torch.cuda.empty_cache()
    return res


def run_per_config(names, stream, peak, oracle=None, layers=None, seed=None, stream_window=STREAM_WINDOW):
    res = {}
    for name in names:
        w = W.WORKLOADS[name]
        if name == "streaming":
            r = measure_streaming(stream, peak, layers=layers, seed=seed, window=stream_window)
        else:
            r = measure_decode_shape(name, stream, peak, layers=layers, seed=seed)
        r["workload"] = describe(w)
        r["traffic"] = decode_traffic_record(name)
        if oracle and name in oracle:
            o = oracle[name]
            r["oracle"] = {"decode_tokens_per_s_per_layer": o["decode_only"], "cores": o["cores"],
                           "sample": o["sample"]}
        res[name] = r
    return res


# ------------------------------------------------------------------ GPU leg
def describe(w):
    return (f"{w.name}: batch {w.batch}, {w.heads} heads, head_dim {w.head_dim}, {w.dtype} K/V, "
            f"prompt {w.prompt} + {w.decode} decode steps, heavy {w.heavy} + recent {w.recent} slots")


def run_ours(args, rank, world, local_rank):
    import torch

    from kv_cache_eviction_03_gb300 import binding as B

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    B.lib()
    w = W.WORKLOADS[args.config]
    NL = args.layers or w.layers
    T, L = w.decode, w.prompt
    base_seed = W.seed_for(args.config) if args.seed is None else args.seed
    seed = base_seed + 1000 * rank  # every rank runs its own batch
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    inp = W.device_inputs(w, seed, NL)
    caches = [B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, kv_code(w)) for _ in range(NL)]
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
    # per layer: row statistics, attention output, column sums (fp16: the
    # output pass's partials reduced), keep rule; per decode step and layer: one
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
    checks = 0
    for i in range(args.steps):
        starts[i].record(stream)
        step(mid[i])
        ends[i].record(stream)
        if args.check_every and (i + 1) % args.check_every == 0:
            for c in caches:  # synchronises: the step time below excludes it
                B.h2o_cache_check(c, stream=stream)
            checks += 1
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    if checks:
        elapsed = sum(starts[i].elapsed_time(ends[i]) for i in range(args.steps)) / 1e3
    else:
        elapsed = t_begin.elapsed_time(t_end) / 1e3
    decode_s = sum(mid[i].elapsed_time(ends[i]) for i in range(args.steps)) / 1e3
    prefill_s = sum(starts[i].elapsed_time(mid[i]) for i in range(args.steps)) / 1e3
    elapsed, decode_s, prefill_s = sharding.max_over_ranks([elapsed, decode_s, prefill_s], dist, device="cuda")
    for c in caches:
        B.h2o_cache_check(c, stream=stream)

    tokens_per_layer = w.batch * T * world  # per step, every layer
    value = tokens_per_layer * NL * args.steps / elapsed
    step_bytes = A.decode_step_bytes(w.pairs, w.cache_slots, w.head_dim, elem_bytes(w))
    per_launch = decode_s / (args.steps * T * NL)
    achieved = step_bytes / per_launch / 1e9
    peak, peak_kind = measured_peak()
    info = B.h2o_cache_info(caches[0])
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded Zipf-keyed generator, drawn on the GPU)",
        "config": workload_config(w, NL, world, args.decode_only, args.check_every),
        "launch": {"decode_splits": info[6], "decode_stages": info[7]},
        "phases": {"prefill_ms_per_step": prefill_s / args.steps * 1e3,
                   "decode_ms_per_step": decode_s / args.steps * 1e3,
                   "decode_only_tokens_per_s_per_layer": tokens_per_layer * NL * args.steps / decode_s,
                   "prefill_tflops": A.prefill_flops(w.pairs, L, w.head_dim) * NL * args.steps / prefill_s / 1e12
                   if prefill_s > 0 else None},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (fused attention + score + evict + overwrite)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "traffic": decode_traffic_record(args.config),
                     "algorithmic_bytes_per_launch": step_bytes,
                     "avg_launch_us": per_launch * 1e6,
                     "timing": "decode launches back to back over the layer caches inside the step "
                               "(consecutive layers overlap through programmatic dependent launch)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    # ---- end to end through the public API with pinned host buffers
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, w, NL, stream, (inp, pout, dout, dev_ev, capture_layers(inp, pout), g_dec),
                                capture, capture_layers, world, dist, elapsed / args.steps)
    del inp, g_pre, g_dec
    for c in caches:
        B.h2o_cache_destroy(c)
    torch.cuda.empty_cache()
    # ---- the decode launch in isolation, and every other workload shape
    if rank == 0 and world == 1 and not args.no_per_config:
        names = [n for n in args.per_config.split(",") if n]
        pc = run_per_config(names, stream, peak, oracle=args.oracle_per_config, seed=args.seed,
                            stream_window=args.stream_window)
        result["per_config"] = pc
        if args.config in pc:
            result["roofline"]["isolated"] = dict(pc[args.config]["isolated"],
                                                  timing="a plain one-thread kernel between decode launches, "
                                                         "its own time subtracted (per_config)")
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result


def run_e2e(args, w, NL, stream, set_a, capture, capture_layers, world, dist, device_step_s):
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
    h2d_gbps = h2d_bytes / copy_s / 1e9 if copy_s > 0 else None
    return {"value": w.batch * w.decode * world * NL * args.steps / el, "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "h2d_gbps_measured": h2d_gbps, "h2d_s_per_step": copy_s, "device_s_per_step": device_step_s,
            "link_bound": bool(copy_s > device_step_s),
            "pipelined": "step s+1 host->device copy and step s-1 read-back overlap step s"}


def workload_config(w, NL, world, decode_only, check_every=0):
    """The `config` object of the JSON line, identical for both arms."""
    return {"workload": describe(w),
            "layers": NL, "batch": w.batch, "decode_steps": w.decode, "prompt": w.prompt, "accumulate": "f32",
            "l2": f"inputs larger than L2: {NL} layer caches rotated every decode step",
            "parallelism": f"weak: each of {world} GPUs runs its own batch" if world > 1 else "1 GPU",
            "decode_only": bool(decode_only), "check_every": check_every}


def main():
    args = parse()
    rank, world, local_rank = dist_info()
    w = W.WORKLOADS[args.config]
    seed0 = W.seed_for(args.config) if args.seed is None else args.seed
    args.oracle_per_config = None
    if args.only_per_config:
        import torch

        torch.cuda.set_device(local_rank)
        stream = torch.cuda.Stream()
        peak, _ = measured_peak()
        pc = run_per_config([args.only_per_config], stream, peak, layers=args.layers, seed=args.seed,
                            stream_window=args.stream_window)
        print(json.dumps({"per_config": pc}))
        return
    if args.impl == "reference":
        if rank != 0:
            return
        rows, heads, steps = ORACLE_SAMPLE[args.config]
        vals, walls = [], []
        o = None
        for i in range(args.warmup + args.steps):
            o = time_oracle(w, seed0, rows, heads, steps)
            if i >= args.warmup:
                vals.append(o["value"])
                walls.append(o["wall_s"])
        value = statistics.median(vals)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(walls) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded Zipf-keyed generator)",
                "config": workload_config(w, args.layers or w.layers, world, args.decode_only, args.check_every),
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": o["cores"], "kind": "oracle",
                                 "sample": o["sample"]},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    # CPU oracle pools first (spawned before any GPU work)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        rows, heads, steps = ORACLE_SAMPLE[args.config]
        o = time_oracle(w, seed0, rows, heads, steps)
        cpu = {"value": o["value"], "unit": UNIT, "cores": o["cores"], "kind": "oracle", "sample": o["sample"],
               "sample_wall_s": o["wall_s"]}
        if not args.no_per_config:
            names = [n for n in args.per_config.split(",") if n]
            args.oracle_per_config = oracle_baselines(names, args.seed)
    result = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if cpu is not None:
            result["cpu_baseline"] = cpu
        print(json.dumps(result))


if __name__ == "__main__":
    main()
