"""Per-phase timeline of the cluster decode kernel, from a profiling build.

    python -m kv_cache_eviction_03_gb300.timeline --workload llama-7b-16k

Builds a copy of the library compiled with H2O_DECODE_TIMELINE next to the
product library (libh2o_gb300_timeline.so; the product build is not
touched), in which thread 0 of every decode CTA records %globaltimer at
eleven points: entry, grid dependency released, step inputs loaded, first
stage landed, every consumer past its loop, the pair's softmax normaliser
known, the CTA's scores stored, its block minimum found, its candidate
pushed to the cluster peers, the victim known, exit.  It then runs the workload's decode rotation
(one cache per attention layer, every decode step visiting the layers in
turn, from a CUDA graph, as the benchmark does) and prints, for the last
launches, each phase's time in microseconds relative to the end of the
previous launch (its last CTA's exit): median and latest over the launch's
CTAs.  The stamps cost a few global stores per CTA; the kernel is otherwise
the product kernel.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import statistics

import numpy as np

from . import _build
from . import workload as W

# (name, stamp index) in the order a CTA passes them
STAMPS = [("entry", 0), ("dependency released", 1), ("inputs loaded", 2), ("first stage landed", 3),
          ("loop done", 4), ("normaliser known", 5), ("scores stored", 8), ("block minimum", 9),
          ("candidate pushed", 10), ("victim known", 6), ("exit", 7)]
SLOTS, MAX_CTAS, NSTAMP, EXIT = 4, 4096, 11, 7


def load_timeline_build():
    from . import binding as B

    path = _build.build(extra=["-DH2O_DECODE_TIMELINE"], variant="timeline")
    if B._lib is not None and _build.LIB != path:
        raise RuntimeError("the product library is already loaded in this process")
    _build.LIB = path
    lib = B.lib(build_if_missing=False)
    fn = lib.h2o_debug_decode_timeline
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int)]
    return B, fn


def run(workload: str, layers: int | None, steps: int, splits: int = 0, stages: int = 0, isolated: bool = False,
        rolling: float = 0.0):
    import torch

    B, read = load_timeline_build()
    w = W.WORKLOADS[workload]
    NL = layers or w.layers
    stream = torch.cuda.Stream()
    draws = W.DeviceDraws(w, W.seed_for(workload))
    code = B.H2O_F16 if w.dtype == "f16" else B.H2O_F32
    caches = []
    for _ in range(NL):
        c = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, code)
        if splits or stages:
            B.h2o_cache_set_decode_shape(c, splits, stages)
        if w.prompt:
            q, k, v = draws.prefill()
            B.h2o_prefill(c, q, k, v, w.scale, stream=stream)
        else:  # streaming shape: fill the cache first (eager), then time evicting steps
            B.h2o_cache_reset(c, stream=stream)
        caches.append(c)
    if rolling > 0:  # position rolling, switched on after the prefill (ranks from positions)
        for c in caches:
            B.h2o_cache_set_position_rolling(c, rolling)
            if splits or stages:
                B.h2o_cache_set_decode_shape(c, splits, stages)
    info = B.h2o_cache_info(caches[0])
    if info[6] < 1:
        raise SystemExit("the timeline covers the cluster kernel only; this shape runs warp per pair")
    S = info[6]
    grid = S * w.pairs
    if grid > MAX_CTAS:
        raise SystemExit(f"{grid} CTAs per launch: more than the {MAX_CTAS} the timeline records")
    if not w.prompt:
        fq, fk, fv = draws.decode(w.cache_slots, NL)
        out = torch.empty((NL, w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
        for t in range(w.cache_slots):
            for l in range(NL):
                B.h2o_decode_step(caches[l], fq[t, l], fk[t, l], fv[t, l], w.scale, out[l], stream=stream)
        del fq, fk, fv
    dq, dk, dv = draws.decode(steps, NL)
    out = torch.empty((steps, NL, w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")

    tiny = torch.zeros(1, device="cuda")

    def body():
        for t in range(steps):
            for l in range(NL):
                if isolated:  # a plain kernel between launches, as a model's projection would be
                    tiny.add_(1.0)
                B.h2o_decode_step(caches[l], dq[t, l], dk[t, l], dv[t, l], w.scale, out[t, l], stream=stream)

    with torch.cuda.stream(stream):
        body()
        buf = np.zeros((SLOTS, MAX_CTAS, NSTAMP), dtype=np.uint64)
        nxt = ctypes.c_int(0)
        B._check(read(buf.ctypes.data, buf.nbytes, ctypes.byref(nxt)))
        first = nxt.value  # slot of the graph's first launch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        for _ in range(3):
            g.replay()
        stream.synchronize()
    B._check(read(buf.ctypes.data, buf.nbytes, ctypes.byref(nxt)))
    for c in caches:
        B.h2o_cache_check(c, stream=stream)
    n = steps * NL
    order = [(first + i) % SLOTS for i in range(n - SLOTS, n)]  # the graph's last launches, oldest first
    stamps = [buf[s, :grid, :].astype(np.int64) for s in order]
    return w, NL, info, grid, stamps


def phase_table(stamps):
    """Rows: launches after the first; columns: each stamp relative to the
    previous launch's last exit (us), median and latest over CTAs."""
    rows = []
    for prev, cur in zip(stamps[:-1], stamps[1:]):
        prev_end = int(prev[:, EXIT].max())
        rel = (cur - prev_end) / 1e3
        rows.append({name: (float(statistics.median(rel[:, i])), float(rel[:, i].max())) if cur[:, i].any() else None
                     for name, i in STAMPS})  # None: a stamp this kernel shape never passes
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama-7b-16k", choices=[n for n in W.WORKLOAD_ORDER if n != "tiny-ref"])
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--steps", type=int, default=16)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--isolated", action="store_true", help="a plain kernel between decode launches")
    ap.add_argument("--rolling", type=float, default=0.0, help="position rolling with this rotary base (0: off)")
    a = ap.parse_args()
    w, NL, info, grid, stamps = run(a.workload, a.layers, a.steps, a.splits, a.stages, a.isolated, a.rolling)
    print(f"workload {w.name}: {NL} layer caches, {w.pairs} pairs x {info[6]} CTAs = {grid} CTAs per launch, "
          f"{info[7]} stages, {info[8]} threads{', isolated launches' if a.isolated else ''}"
          f"{f', position rolling (base {a.rolling:g})' if a.rolling else ''}")
    print("times in us after the previous launch's last CTA exit: median over CTAs / latest CTA")
    rows = phase_table(stamps)
    print("| stamp | " + " | ".join(f"launch {i + 1}" for i in range(len(rows))) + " |")
    print("|---|" + "---|" * len(rows))
    for name, _ in STAMPS:
        print(f"| {name} | " + " | ".join(f"{r[name][0]:.2f} / {r[name][1]:.2f}" if r[name] else "-" for r in rows)
              + " |")
    spans = [r["exit"][1] for r in rows]
    print(f"launch-to-launch (last exit to last exit): {', '.join(f'{x:.2f}' for x in spans)} us")


if __name__ == "__main__":
    main()
