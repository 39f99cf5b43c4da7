"""Position rolling: rotary embedding at positions counted inside the cache.

Each case starts from an empty cache with rolling on, runs decode steps
through the fill phase into evictions and compares every step with the
oracle's decode_step(..., rope_base).  The kept tokens' ranks change as
tokens are evicted, so a wrong rank update shows up as a wrong output.  A
second test imports a mid-stream oracle state, whose ranks the library
derives from the positions, and checks the next steps.
"""
import numpy as np
import pytest

from harness import StepReport, check_other_victim, compare_decode_step, oracle_image, out_tol
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BASE = 10000.0

CASES = [
    # name, batch, heads, D, dtype, heavy, recent, steps, CTAs per pair (0: automatic)
    ("r-f16-d128-auto", 1, 3, 128, "f16", 20, 12, 70, 0),
    ("r-f16-d128-s2", 1, 3, 128, "f16", 20, 12, 70, 2),
    ("r-f32-d64-s4", 2, 2, 64, "f32", 24, 16, 60, 4),
    ("r-f16-d64-s8", 1, 2, 64, "f16", 60, 36, 120, 8),
]


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rolling_decode_matches_oracle(case):
    name, Bn, H, D, dt, heavy, recent, steps, splits = case
    w = W.Workload(name, Bn, H, D, dt, 0, steps, heavy, recent, 1.1)
    code = B.H2O_F16 if dt == "f16" else B.H2O_F32
    cache = B.h2o_cache_create(Bn, H, D, heavy, recent, code)
    B.h2o_cache_set_position_rolling(cache, BASE)
    if splits:
        B.h2o_cache_set_decode_shape(cache, splits)
    assert B.h2o_cache_info(cache)[6] != B.H2O_DECODE_WARP_PER_PAIR
    ref = O.empty_cache(w.pairs, heavy, recent, D)
    tol = out_tol(code)
    o_dev = torch.empty((Bn, H, D), dtype=torch.float32, device="cuda")
    e_dev = torch.empty((Bn, H), dtype=torch.int32, device="cuda")
    alive = np.ones(w.pairs, dtype=bool)
    evictions = 0
    for t in range(steps):
        qd, kd, vd = W.decode_inputs(w, t, 29)
        B.h2o_decode_step(cache, dev(qd), dev(kd), dev(vd), w.scale, o_dev, e_dev)
        before = ref
        ref, r_out, r_ev, gap = O.decode_step(ref, qd, kd, vd, heavy, recent, w.scale, rope_base=BASE)
        g_o = o_dev.cpu().numpy().reshape(w.pairs, D)
        g_e = e_dev.cpu().numpy().reshape(w.pairs)
        for i in np.nonzero(alive)[0]:
            err = np.max(np.abs(g_o[i] - r_out[i]))
            assert err <= tol, f"step {t} pair {i}: out err {err}"
            if g_e[i] != r_ev[i]:
                f64 = lambda a: a.reshape(w.pairs, D)[i].astype(np.float64)
                check_other_victim(before.pair(i), f64(qd), f64(kd), f64(vd), w.scale, heavy, recent, g_e[i],
                                   r_ev[i], gap[i], rope_base=BASE, where=f"step {t} pair {i}")
                alive[i] = False
        evictions += int(np.sum(r_ev >= 0))
    B.h2o_cache_check(cache)
    assert evictions > 0 and alive.sum() >= w.pairs - 1
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    for i in np.nonzero(alive)[0]:
        assert np.array_equal(g["pos"][i], ref.pos[i])
        used = ref.pos[i] >= 0
        assert np.max(np.abs(g["score"][i][used] - ref.score[i][used]) / ref.score[i][used]) <= 1e-5
    B.h2o_cache_destroy(cache)


def test_rolling_after_import_mid_stream():
    """An oracle state with gaps in its positions (after evictions) goes into
    a rolling cache; the library ranks the kept tokens from the imported
    positions, and the next steps match the oracle's."""
    Bn, H, D, heavy, recent, warm, steps = 1, 4, 128, 16, 8, 50, 6
    w = W.Workload("r-import", Bn, H, D, "f16", 0, warm + steps, heavy, recent, 1.1)
    ref = O.empty_cache(w.pairs, heavy, recent, D)
    for t in range(warm):
        qd, kd, vd = W.decode_inputs(w, t, 31)
        ref, _, _, _ = O.decode_step(ref, qd, kd, vd, heavy, recent, w.scale, rope_base=BASE)
    assert np.all(ref.count == heavy + recent) and np.all(ref.p == warm)
    cache = B.h2o_cache_create(Bn, H, D, heavy, recent, B.H2O_F16)
    B.h2o_cache_set_position_rolling(cache, BASE)
    B.h2o_cache_import_state(cache, oracle_image(cache, ref))
    o_dev = torch.empty((Bn, H, D), dtype=torch.float32, device="cuda")
    e_dev = torch.empty((Bn, H), dtype=torch.int32, device="cuda")
    for t in range(warm, warm + steps):
        qd, kd, vd = W.decode_inputs(w, t, 31)
        B.h2o_decode_step(cache, dev(qd), dev(kd), dev(vd), w.scale, o_dev, e_dev)
        before = ref
        ref, r_out, r_ev, gap = O.decode_step(ref, qd, kd, vd, heavy, recent, w.scale, rope_base=BASE)
        assert np.max(np.abs(o_dev.cpu().numpy().reshape(w.pairs, D) - r_out)) <= 2e-3, f"step {t}"
        g_e = e_dev.cpu().numpy().reshape(w.pairs)
        for i in np.nonzero(g_e != r_ev)[0]:
            f64 = lambda a: a.reshape(w.pairs, D)[i].astype(np.float64)
            check_other_victim(before.pair(i), f64(qd), f64(kd), f64(vd), w.scale, heavy, recent, g_e[i], r_ev[i],
                               gap[i], rope_base=BASE, where=f"step {t} pair {i}")
        if np.any(g_e != r_ev):
            break  # the two caches have parted at a near tie
    B.h2o_cache_check(cache)
    B.h2o_cache_destroy(cache)


STEPWISE = [
    # name, batch, heads, D, dtype, heavy, recent, steps, CTAs per pair (0: automatic)
    ("sw-f16-d128-auto", 1, 3, 128, "f16", 20, 12, 64, 0),
    ("sw-f32-d64-s2", 2, 2, 64, "f32", 24, 16, 60, 2),
    ("sw-f16-d128-s8", 1, 2, 128, "f16", 70, 30, 130, 8),
    # ranks 0..C in two digits with a 5-bit lowest one (C in 256..511), and in
    # a single 5-bit digit (C in 16..31): the tables' other layouts
    ("sw-f16-d128-low5", 1, 2, 128, "f16", 180, 120, 330, 0),
    ("sw-f32-d128-low5-s2", 1, 2, 128, "f32", 260, 200, 480, 2),
    ("sw-f16-d64-one-level", 1, 3, 64, "f16", 12, 8, 45, 0),
]


@pytest.mark.parametrize("case", STEPWISE, ids=[c[0] for c in STEPWISE])
def test_rolling_stepwise_from_oracle_states(case):
    """Every step from the oracle's own state (imported; the library ranks the
    kept tokens from the imported positions), through the fill and well past
    it, so ranks and positions differ: outputs, victims (a different one only
    at a near tie, and only an equally low candidate), scores, slots, ring and
    counters through the step-wise comparison."""
    name, Bn, H, D, dt, heavy, recent, steps, splits = case
    w = W.Workload(name, Bn, H, D, dt, 0, steps, heavy, recent, 1.1)
    code = B.H2O_F16 if dt == "f16" else B.H2O_F32
    cache = B.h2o_cache_create(Bn, H, D, heavy, recent, code)
    B.h2o_cache_set_position_rolling(cache, BASE)
    if splits:
        B.h2o_cache_set_decode_shape(cache, splits)
    st = O.empty_cache(w.pairs, heavy, recent, D)
    o_dev = torch.empty((Bn, H, D), dtype=torch.float32, device="cuda")
    e_dev = torch.empty((Bn, H), dtype=torch.int32, device="cuda")
    rep = StepReport()
    flat = lambda a: a.reshape(w.pairs, D).astype(np.float64)
    for t in range(steps):
        qd, kd, vd = W.decode_inputs(w, t, 43)
        nxt, r_out, r_ev, gap = O.decode_step(st, qd, kd, vd, heavy, recent, w.scale, rope_base=BASE)
        B.h2o_cache_import_state(cache, oracle_image(cache, st))
        B.h2o_decode_step(cache, dev(qd), dev(kd), dev(vd), w.scale, o_dev, e_dev)
        B.h2o_cache_check(cache)
        after = B.unpack_state(cache, B.h2o_cache_export_state(cache))
        compare_decode_step(cache, after, o_dev.cpu().numpy().reshape(w.pairs, D), e_dev.cpu().numpy().reshape(-1),
                            st, nxt, r_out, r_ev, gap, rep, inputs=(flat(qd), flat(kd), flat(vd)), scale=w.scale,
                            rope_base=BASE)
        st = nxt
    assert rep.pairs == w.pairs * steps
    assert np.all(st.p - st.count > 10)  # far past the fill: ranks differ from positions
    B.h2o_cache_destroy(cache)


def test_rolling_refuses_prefill_and_warp_per_pair():
    cache = B.h2o_cache_create(1, 2, 64, 8, 8, B.H2O_F16)
    x = torch.zeros((1, 2, 16, 64), dtype=torch.float16, device="cuda")
    B.h2o_cache_set_position_rolling(cache, BASE)
    with pytest.raises(B.H2OError):
        B.h2o_prefill(cache, x, x, x, 0.125)
    with pytest.raises(B.H2OError):
        B.h2o_cache_set_decode_shape(cache, B.H2O_DECODE_WARP_PER_PAIR)
    with pytest.raises(B.H2OError):
        B.h2o_cache_set_position_rolling(cache, -1.0)
    B.h2o_cache_set_position_rolling(cache, 0.0)  # off again: the prefill is accepted
    B.h2o_prefill(cache, x, x, x, 0.125)
    B.h2o_cache_check(cache)
    B.h2o_cache_destroy(cache)


def test_rolling_launch_shape_rules():
    """Rolling runs eight consumer warps (one stage each of the ring) and two
    producer warps (K rows, V rows): ring
    depths are multiples of eight while it is on, and the plain kernel's
    rules come back when it is switched off."""
    cache = B.h2o_cache_create(1, 2, 128, 40, 24, B.H2O_F16)
    info = B.h2o_cache_info(cache)
    assert info[8] in (5 * 32, 7 * 32)  # plain: four or six consumer warps + the producer
    B.h2o_cache_set_decode_shape(cache, 1, 12)
    B.h2o_cache_set_position_rolling(cache, BASE)
    info = B.h2o_cache_info(cache)
    assert info[8] == 10 * 32 and info[7] % 8 == 0  # the explicit shape went back to the automatic one
    for splits in (1, 2):
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_decode_shape(cache, splits, 12)
        B.h2o_cache_set_decode_shape(cache, splits, 8)
        assert B.h2o_cache_info(cache)[6:9] == [splits, 8, 10 * 32]
    B.h2o_cache_set_decode_shape(cache, 1, 8)
    B.h2o_cache_set_position_rolling(cache, 0.0)  # off: the rolling shape does not carry over
    info = B.h2o_cache_info(cache)
    assert info[8] in (5 * 32, 7 * 32) and info[7] % (info[8] // 32 - 1) == 0
    B.h2o_cache_set_decode_shape(cache, 1, 12)
    assert B.h2o_cache_info(cache)[7:9] == [12, 7 * 32]
    B.h2o_cache_destroy(cache)
