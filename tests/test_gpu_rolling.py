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
    # name, batch, heads, D, dtype, heavy, recent, steps, CTAs per pair (0: automatic),
    # digit widths (low, hi) of the ranks (None: automatic)
    ("sw-f16-d128-auto", 1, 3, 128, "f16", 20, 12, 64, 0, None),
    ("sw-f32-d64-s2", 2, 2, 64, "f32", 24, 16, 60, 2, None),
    ("sw-f16-d128-s8", 1, 2, 128, "f16", 70, 30, 130, 8, None),
    # ranks 0..C (C = 300, 460) in two digits (automatic: 4 + 5 bits), three
    # (4 + 4 + 4 bits: two key-side rotations) and two with a wide lowest
    # digit (6 + 4); and in a single digit (C = 20)
    ("sw-f16-d128-two-levels", 1, 2, 128, "f16", 180, 120, 330, 0, None),
    ("sw-f16-d128-three-levels", 1, 2, 128, "f16", 180, 120, 330, 0, (4, 4)),
    ("sw-f32-d128-three-levels-s2", 1, 2, 128, "f32", 260, 200, 480, 2, (4, 4)),
    ("sw-f16-d64-wide-low-s4", 1, 2, 64, "f16", 260, 200, 480, 4, (6, 4)),
    ("sw-f16-d64-one-level", 1, 3, 64, "f16", 12, 8, 45, 0, None),
    # a 16-CTA cluster (600 slots, 40 per CTA) through the fill into evictions
    ("sw-f16-d128-s16", 1, 1, 128, "f16", 380, 220, 640, 16, None),
]


@pytest.mark.parametrize("case", STEPWISE, ids=[c[0] for c in STEPWISE])
def test_rolling_stepwise_from_oracle_states(case):
    """Every step from the oracle's own state (imported; the library ranks the
    kept tokens from the imported positions), through the fill and well past
    it, so ranks and positions differ: outputs, victims (a different one only
    at a near tie, and only an equally low candidate), scores, slots, ring and
    counters through the step-wise comparison."""
    name, Bn, H, D, dt, heavy, recent, steps, splits, digits = case
    w = W.Workload(name, Bn, H, D, dt, 0, steps, heavy, recent, 1.1)
    code = B.H2O_F16 if dt == "f16" else B.H2O_F32
    cache = B.h2o_cache_create(Bn, H, D, heavy, recent, code)
    B.h2o_cache_set_position_rolling(cache, BASE)
    if digits:
        B.h2o_cache_set_rolling_digits(cache, *digits)
        low, hi, levels, entries = B.h2o_cache_rolling_digits(cache)
        C = heavy + recent
        assert (low, hi) == digits and (1 << (low + hi * (levels - 2))) <= C < (1 << (low + hi * (levels - 1)))
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


def test_rolling_digit_choice():
    """The automatic digit widths: one level when every rank fits the lowest
    digit, two where those tables still fit beside the ring (the OPT-6.7B
    cache shape, 1000 slots of 128-wide heads), three where two levels'
    tables would cost resident CTAs (the LLaMA-7B 16K shape, 1640 slots, whose
    two-level tables miss two CTAs per SM by a few entries; 2048 slots).
    Explicit widths are checked and reported; the automatic ones come back
    with (0, 0)."""
    def digits(Bn, H, D, heavy, recent):
        cache = B.h2o_cache_create(Bn, H, D, heavy, recent, B.H2O_F16)
        assert B.h2o_cache_rolling_digits(cache) == [0, 0, 0, 0]
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_rolling_digits(cache, 4, 4)  # rolling is off
        B.h2o_cache_set_position_rolling(cache, BASE)
        d = B.h2o_cache_rolling_digits(cache)
        B.h2o_cache_destroy(cache)
        return d
    assert digits(1, 2, 64, 12, 8)[2] == 1
    assert digits(8, 32, 128, 205, 205)[2] == 2
    assert digits(1, 32, 128, 500, 500)[2] == 2
    assert digits(1, 32, 128, 820, 820)[2] == 3
    assert digits(4, 32, 128, 1024, 1024)[2] == 3
    cache = B.h2o_cache_create(1, 2, 64, 100, 60, B.H2O_F16)
    B.h2o_cache_set_position_rolling(cache, BASE)
    auto = B.h2o_cache_rolling_digits(cache)
    for bad in ((3, 4), (4, 7), (0, 4)):
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_rolling_digits(cache, *bad)
    B.h2o_cache_set_rolling_digits(cache, 4, 4)
    assert B.h2o_cache_rolling_digits(cache) == [4, 4, 2, 16 + (160 >> 4) + 1]
    B.h2o_cache_set_rolling_digits(cache, 0, 0)
    assert B.h2o_cache_rolling_digits(cache) == auto
    B.h2o_cache_destroy(cache)
