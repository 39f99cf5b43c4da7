"""GPU parity of the fused decode step against the fp64 oracle.

Step-wise protocol: before each checked step the oracle's own state is
imported into the CUDA cache, both sides run one step on the same inputs, and
outputs, evicted slots, scores, positions, ring and counters are compared
(out within 2e-3 for fp16 K/V, 1e-5 for fp32; scores within 1e-5 relative;
slots and positions bit-exact unless the oracle's two lowest candidate scores
are within 1e-6).  Free-run protocol: both sides run a whole prefill + decode
trajectory on their own and are compared step by step.
"""
import numpy as np
import pytest

from harness import StepReport, check_other_victim, compare_decode_step, oracle_image, out_tol
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dtype_code(w):
    return B.H2O_F16 if w.dtype == "f16" else B.H2O_F32


def flat(a):
    a = np.asarray(a, dtype=np.float64)
    return a.reshape((-1,) + a.shape[2:])


def oracle_start(w, seed, pattern=None):
    if w.prompt:
        q, k, v = W.prefill_inputs(w, seed)
        st, _, _ = O.prefill(q, k, v, w.heavy, w.recent, w.scale, pattern)
        return st
    return O.empty_cache(w.pairs, w.heavy, w.recent, w.head_dim)


def run_stepwise(w, seed, check=None, splits=None, stages=0, pattern=None):
    """Every checked step starts both sides from the oracle's state.
    pattern: an oracle StaticPattern, also set on the cache."""
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, dtype_code(w))
    if splits or stages:
        B.h2o_cache_set_decode_shape(cache, splits or 0, stages)
    if pattern is not None:
        B.h2o_cache_set_static_pattern(cache, pattern.offset, pattern.stride, pattern.count)
    st = oracle_start(w, seed, pattern)
    out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
    ev = torch.empty((w.batch, w.heads), dtype=torch.int32, device="cuda")
    rep = StepReport()
    P, D = w.pairs, w.head_dim
    for t in range(w.decode):
        qd, kd, vd = W.decode_inputs(w, w.prompt + t, seed)
        nxt, r_out, r_ev, gap = O.decode_step(st, qd, kd, vd, w.heavy, w.recent, w.scale, pattern=pattern)
        if check is None or t in check:
            B.h2o_cache_import_state(cache, oracle_image(cache, st))
            B.h2o_decode_step(cache, torch.from_numpy(qd).cuda(), torch.from_numpy(kd).cuda(),
                              torch.from_numpy(vd).cuda(), w.scale, out, ev)
            B.h2o_cache_check(cache)
            after = B.unpack_state(cache, B.h2o_cache_export_state(cache))
            compare_decode_step(cache, after, out.cpu().numpy().reshape(P, D), ev.cpu().numpy().reshape(P),
                                st, nxt, r_out, r_ev, gap, rep, inputs=(flat(qd), flat(kd), flat(vd)),
                                scale=w.scale, pattern=pattern)
        st = nxt
    B.h2o_cache_destroy(cache)
    return rep


def run_free(w, seed, splits=None, pattern=None):
    """Both sides run prefill + every decode step on their own.  A different
    victim is accepted only for an equally good candidate (near tie); the
    pair's trajectories then part and it is no longer compared."""
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, dtype_code(w))
    if pattern is not None:
        B.h2o_cache_set_static_pattern(cache, pattern.offset, pattern.stride, pattern.count)
    if splits:
        B.h2o_cache_set_decode_shape(cache, splits)
    P, D = w.pairs, w.head_dim
    st = oracle_start(w, seed, pattern)
    if w.prompt:
        q, k, v = W.prefill_inputs(w, seed)
        B.h2o_prefill(cache, torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                      w.scale)
        g0 = B.unpack_state(cache, B.h2o_cache_export_state(cache))
        alive = np.array([np.array_equal(g0["pos"][i], st.pos[i]) for i in range(P)])
    else:
        B.h2o_cache_reset(cache)
        alive = np.ones(P, dtype=bool)
    tol = out_tol(cache.kv_dtype)
    out = torch.empty((w.batch, w.heads, D), dtype=torch.float32, device="cuda")
    ev = torch.empty((w.batch, w.heads), dtype=torch.int32, device="cuda")
    worst = 0.0
    for t in range(w.decode):
        qd, kd, vd = W.decode_inputs(w, w.prompt + t, seed)
        B.h2o_decode_step(cache, torch.from_numpy(qd).cuda(), torch.from_numpy(kd).cuda(),
                          torch.from_numpy(vd).cuda(), w.scale, out, ev)
        before = st
        st, r_out, r_ev, gap = O.decode_step(st, qd, kd, vd, w.heavy, w.recent, w.scale, pattern=pattern)
        g_out = out.cpu().numpy().reshape(P, D)
        g_ev = ev.cpu().numpy().reshape(P)
        for i in np.nonzero(alive)[0]:
            err = float(np.max(np.abs(g_out[i] - r_out[i])))
            worst = max(worst, err)
            assert err <= tol, f"step {t} pair {i}: out err {err}"
            if g_ev[i] != r_ev[i]:
                f64 = lambda a: flat(a)[i]
                check_other_victim(before.pair(i), f64(qd), f64(kd), f64(vd), w.scale, w.heavy, w.recent, g_ev[i],
                                   r_ev[i], gap[i], pattern=pattern, where=f"step {t} pair {i}")
                alive[i] = False  # trajectories legitimately part at a near tie
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    for i in np.nonzero(alive)[0]:
        assert np.array_equal(g["pos"][i], st.pos[i])
        used = st.pos[i] >= 0
        rel = np.abs(g["score"][i][used] - st.score[i][used]) / st.score[i][used]
        assert rel.max() <= 1e-5
    B.h2o_cache_destroy(cache)
    return worst, int(alive.sum())


TINY = W.WORKLOADS["tiny-ref"]


def test_tiny_reference_workload_every_step():
    """The 4-head fp32 workload (prompt 256 + 64 steps, 26+26 slots), all steps."""
    rep = run_stepwise(TINY, W.seed_for("tiny-ref"))
    assert rep.pairs == TINY.pairs * TINY.decode
    assert rep.max_out_err <= 1e-5


def test_tiny_reference_free_run():
    worst, alive = run_free(TINY, W.seed_for("tiny-ref"))
    assert alive >= TINY.pairs - 1


SMALL = [
    # name, batch, heads, D, dtype, prompt, decode, heavy, recent
    ("f16-d128-ragged", 2, 3, 128, "f16", 100, 40, 20, 17),
    ("f16-d64", 1, 5, 64, "f16", 90, 30, 13, 11),
    ("f32-d128", 2, 2, 128, "f32", 70, 30, 9, 14),
    ("fill-then-evict", 1, 4, 128, "f16", 10, 60, 25, 12),
    ("no-prompt", 2, 2, 128, "f16", 0, 50, 20, 10),
    ("no-heavy", 1, 3, 128, "f16", 60, 30, 0, 9),
    ("recent-1", 1, 3, 64, "f32", 40, 30, 7, 1),
    ("prompt-equals-cache", 1, 2, 128, "f16", 29, 20, 17, 12),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_shapes_every_step(case):
    name, b, h, d, dt, L, T, hv, rc = case
    w = W.Workload(name, b, h, d, dt, L, T, hv, rc, 1.1)
    rep = run_stepwise(w, 7)
    assert rep.pairs == w.pairs * T


@pytest.mark.parametrize("splits", [1, 2, 4, 8, 16, B.H2O_DECODE_WARP_PER_PAIR])
def test_splits_agree(splits):
    """Every cluster size (CTAs per pair) and the warp-per-pair kernel give
    the oracle's result, including ragged last CTAs (301 slots) and CTAs
    whose slot range is still empty while filling."""
    w = W.Workload("splits", 1, 4, 128, "f16", 280, 40, 150, 151, 1.1)
    rep = run_stepwise(w, 11, check=set(range(0, 40, 3)) | {21, 22}, splits=splits)
    assert rep.pairs > 0


@pytest.mark.parametrize("splits,stages", [(1, 6), (1, 12), (1, 18), (2, 4), (2, 8), (4, 16)])
def test_ring_depths_agree(splits, stages):
    """Every legal ring depth (a multiple of the consumer warps: six for one
    CTA per pair, four in a cluster) gives the oracle's result, with more
    tiles than stages so stages are reused."""
    w = W.Workload("ring", 1, 3, 128, "f16", 600, 12, 300, 200, 1.1)
    cache_check = set(range(12))
    rep = run_stepwise(w, 23, check=cache_check, splits=splits, stages=stages)
    assert rep.pairs == w.pairs * 12


def test_ring_depth_must_be_a_multiple_of_the_consumer_warps():
    cache = B.h2o_cache_create(1, 2, 128, 40, 40, B.H2O_F16)
    for bad in (1, 3, 4, 8, 16, 24):  # one CTA per pair: six consumer warps
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_decode_shape(cache, 1, bad)
    for bad in (1, 3, 6, 10, 18, 20):  # a cluster: four consumer warps
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_decode_shape(cache, 2, bad)
    B.h2o_cache_set_decode_shape(cache, 1, 12)
    assert B.h2o_cache_info(cache)[6:9] == [1, 12, 224]
    B.h2o_cache_set_decode_shape(cache, 2, 8)
    assert B.h2o_cache_info(cache)[6:9] == [2, 8, 160]
    B.h2o_cache_destroy(cache)


@pytest.mark.parametrize("stages", [2, 3, 5, 6])
def test_warp_per_pair_ring_depths_and_pair_hand_over(stages):
    """Warp per pair with more pairs than warps in the grid, so each warp's
    ring runs on from one pair into the next (tiles of consecutive pairs
    share stages), for several ring depths; ragged tiles (C = 61) and a
    fill phase right after a short prompt."""
    w = W.Workload("warp", 32, 100, 128, "f16", 50, 14, 31, 30, 1.1)
    rep = run_stepwise(w, 31, check={0, 5, 10, 11, 12, 13}, splits=B.H2O_DECODE_WARP_PER_PAIR, stages=stages)
    assert rep.pairs == w.pairs * 6


def test_warp_per_pair_shape_limits():
    cache = B.h2o_cache_create(1, 2, 128, 40, 40, B.H2O_F16)
    for bad in (1, 9):
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_decode_shape(cache, B.H2O_DECODE_WARP_PER_PAIR, bad)
    B.h2o_cache_set_decode_shape(cache, B.H2O_DECODE_WARP_PER_PAIR, 5)
    assert B.h2o_cache_info(cache)[6:8] == [-1, 5]
    B.h2o_cache_set_decode_shape(cache, 0, 0)
    assert B.h2o_cache_info(cache)[6] != -1  # two pairs: the automatic shape is a cluster per pair
    B.h2o_cache_destroy(cache)
    big = B.h2o_cache_create(1, 1, 64, 600, 500, B.H2O_F16)  # 1100 slots: beyond warp per pair
    with pytest.raises(B.H2OError):
        B.h2o_cache_set_decode_shape(big, B.H2O_DECODE_WARP_PER_PAIR, 0)
    B.h2o_cache_destroy(big)


@pytest.mark.parametrize("ratio", [0.04, 0.10, 0.20, 0.60])
def test_budget_ratios_every_step(ratio):
    """Cache budgets of 4, 10, 20 and 60% of a 1000-token prompt (heavy =
    recent), every decode step checked from identical states."""
    half = int(round(ratio * 1000 / 2))
    w = W.Workload(f"budget{ratio}", 1, 4, 128, "f16", 1000, 16, half, half, 1.1)
    rep = run_stepwise(w, 61)
    assert rep.pairs == w.pairs * 16


@pytest.mark.parametrize("splits", [1, 4, 16, B.H2O_DECODE_WARP_PER_PAIR])
def test_free_run_fp16(splits):
    w = W.Workload("free", 2, 4, 128, "f16", 300, 80, 40, 30, 1.1)
    worst, alive = run_free(w, 5, splits=splits)
    assert alive >= w.pairs - 2


def test_decode_rejects_wrong_shapes_and_devices():
    w = W.Workload("x", 1, 2, 64, "f16", 0, 1, 4, 4, 1.1)
    cache = B.h2o_cache_create(1, 2, 64, 4, 4, B.H2O_F16)
    q = torch.zeros((1, 2, 64), dtype=torch.float16, device="cuda")
    out = torch.empty((1, 2, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        B.h2o_decode_step(cache, q.float(), q, q, 0.1, out)
    with pytest.raises(ValueError):
        B.h2o_decode_step(cache, q.cpu(), q, q, 0.1, out)
    with pytest.raises(B.H2OError):
        B._check(B.lib().h2o_decode_step(cache.handle, q.data_ptr(), q.data_ptr(), q.data_ptr(), -1.0,
                                         out.data_ptr(), None, None))
    with pytest.raises(B.H2OError):
        B.h2o_cache_set_decode_shape(cache, 3)
    B.h2o_cache_destroy(cache)


def test_import_rejects_bad_counters():
    cache = B.h2o_cache_create(1, 2, 64, 4, 4, B.H2O_F16)
    img = B.h2o_cache_export_state(cache)
    st = B.unpack_state(cache, img)
    st["count"][0] = 99
    with pytest.raises(B.H2OError):
        B.h2o_cache_import_state(cache, img)
    B.h2o_cache_destroy(cache)


WARP_TYPES = [
    # name, D, dtype: the warp-per-pair kernel's other instantiations
    ("f16-d64", 64, "f16"),
    ("f32-d128", 128, "f32"),
    ("f32-d64", 64, "f32"),
]


@pytest.mark.parametrize("case", WARP_TYPES, ids=[c[0] for c in WARP_TYPES])
def test_warp_per_pair_dtypes_and_head_dims(case):
    """Every K/V type and head width of the warp-per-pair kernel, with more
    pairs than warps (ragged C = 45, fill phase then evictions)."""
    name, D, dt = case
    w = W.Workload("warp-" + name, 24, 100, D, dt, 30, 24, 23, 22, 1.1)
    rep = run_stepwise(w, 37, check={0, 7, 14, 15, 16, 23}, splits=B.H2O_DECODE_WARP_PER_PAIR, stages=3)
    assert rep.pairs == w.pairs * 6


@pytest.mark.parametrize("splits", [0, B.H2O_DECODE_WARP_PER_PAIR])
def test_graph_replay_matches_eager(splits):
    """Counters live on the device, so a captured step replays correctly
    (automatic cluster shape, and the warp-per-pair kernel)."""
    w = W.Workload("graph", 2, 4, 128, "f16", 64, 24, 16, 16, 1.1)
    q, k, v = (torch.from_numpy(a).cuda() for a in W.prefill_inputs(w, 3))
    seq = [tuple(torch.from_numpy(a).cuda() for a in W.decode_inputs(w, w.prompt + t, 3)) for t in range(w.decode)]
    res = []
    for use_graph in (False, True):
        cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, B.H2O_F16)
        if splits:
            B.h2o_cache_set_decode_shape(cache, splits)
        B.h2o_prefill(cache, q, k, v, w.scale)
        xq, xk, xv = (torch.empty_like(seq[0][0]) for _ in range(3))
        out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
        outs = []
        if use_graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                B.h2o_decode_step(cache, xq, xk, xv, w.scale, out, stream=s)
            torch.cuda.current_stream().wait_stream(s)
        for t in range(w.decode):
            xq.copy_(seq[t][0]); xk.copy_(seq[t][1]); xv.copy_(seq[t][2])
            if use_graph:
                g.replay()
            else:
                B.h2o_decode_step(cache, xq, xk, xv, w.scale, out)
            outs.append(out.clone())
        torch.cuda.synchronize()
        res.append((torch.stack(outs).cpu(), B.h2o_cache_export_state(cache)))
        B.h2o_cache_destroy(cache)
    assert torch.equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][1], res[1][1])


def test_maximum_cache_size_every_step():
    """The largest cache a pair may have (65,536 slots: 16 CTAs of 4,096), full,
    from a seeded synthetic state deep into a stream, every step checked."""
    Hh = Rr = 32768
    C, D, P, p0 = Hh + Rr, 128, 2, 1_000_000
    rng = np.random.default_rng(123)
    cache = B.h2o_cache_create(1, P, D, Hh, Rr, B.H2O_F16)
    heavy_pos = np.sort(rng.choice(p0 - Rr, size=Hh, replace=False))
    pos = np.concatenate([heavy_pos, np.arange(p0 - Rr, p0)])
    K = rng.standard_normal((P, C, D)).astype(np.float16).astype(np.float64)
    V = rng.standard_normal((P, C, D)).astype(np.float16).astype(np.float64)
    score = O.to_f32(rng.pareto(1.5, size=(P, C)) * 0.05 + 1e-4)
    ring = np.tile(np.arange(Hh, C), (P, 1))
    st = O.CacheState(K, V, score, np.tile(pos, (P, 1)), ring, np.zeros(P, dtype=np.int64), np.full(P, C),
                      np.full(P, p0))
    out = torch.empty((1, P, D), dtype=torch.float32, device="cuda")
    ev = torch.empty((1, P), dtype=torch.int32, device="cuda")
    rep = StepReport()
    scale = 1 / np.sqrt(D)
    for t in range(4):
        qd, kd, vd = (rng.standard_normal((1, P, D)).astype(np.float16) for _ in range(3))
        nxt, r_out, r_ev, gap = O.decode_step(st, qd, kd, vd, Hh, Rr, scale)
        B.h2o_cache_import_state(cache, oracle_image(cache, st))
        B.h2o_decode_step(cache, torch.from_numpy(qd).cuda(), torch.from_numpy(kd).cuda(),
                          torch.from_numpy(vd).cuda(), scale, out, ev)
        B.h2o_cache_check(cache)
        after = B.unpack_state(cache, B.h2o_cache_export_state(cache))
        compare_decode_step(cache, after, out.cpu().numpy().reshape(P, D), ev.cpu().numpy().reshape(P), st, nxt,
                            r_out, r_ev, gap, rep, inputs=(flat(qd), flat(kd), flat(vd)), scale=scale)
        st = nxt
    assert rep.pairs == 4 * P
    assert B.h2o_cache_info(cache)[6] == 16  # 16 CTAs of 4,096 slots
    B.h2o_cache_destroy(cache)
