"""Static sparse pattern + heavy hitters ("H2O ... 深度解读报告", section 4.5,
Table 2): pattern positions are kept first at prefill and never evicted.
GPU prefill and decode against the oracle with the same StaticPattern, on
both decode kernels and several cluster sizes, with and without position
rolling."""
import numpy as np
import pytest

from harness import StepReport, compare_decode_step, oracle_image
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

import test_gpu_decode as TD
import test_gpu_prefill as TP

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PREFILL = [
    # name, batch, heads, D, dtype, L, heavy, recent, (offset, stride, count)
    ("strided-f16-d128", 1, 3, 128, "f16", 400, 40, 30, (0, 8, 25)),
    ("fixed-f16-d64", 2, 2, 64, "f16", 300, 30, 20, (15, 16, 12)),
    ("first-f32-d128", 1, 2, 128, "f32", 200, 20, 20, (0, 1, 6)),
    ("full-heavy-f16", 1, 2, 128, "f16", 500, 16, 40, (3, 25, 16)),  # heavy == count: no heavy hitters
    ("beyond-prompt-f16", 1, 2, 64, "f16", 90, 20, 10, (0, 9, 20)),  # lattice reaches past L - recent
]


@pytest.mark.parametrize("case", PREFILL, ids=[c[0] for c in PREFILL])
def test_prefill_keeps_pattern_then_heavy_hitters(case):
    name, b, h, d, dt, L, hv, rc, pat = case
    w = W.Workload(name, b, h, d, dt, L, 0, hv, rc, 1.1)
    TP.check_prefill(w, 71, with_out=False, pattern=O.StaticPattern(*pat))


DECODE = [
    # name, batch, heads, D, dtype, prompt, decode, heavy, recent, pattern, splits
    ("strided-auto", 1, 4, 128, "f16", 300, 40, 40, 30, (0, 7, 20), 0),
    ("fixed-s2", 2, 2, 128, "f16", 260, 40, 30, 20, (9, 10, 15), 2),
    ("first-s4-f32", 1, 3, 64, "f32", 150, 30, 24, 16, (0, 1, 4), 4),
    ("full-heavy-s1", 1, 2, 128, "f16", 200, 30, 12, 10, (1, 13, 12), 1),
    ("warp", 16, 40, 128, "f16", 80, 14, 20, 16, (0, 5, 10), B.H2O_DECODE_WARP_PER_PAIR),
    ("no-prompt-arrivals", 1, 3, 128, "f16", 0, 90, 16, 12, (2, 6, 10), 0),  # pattern tokens arrive in decode
]


@pytest.mark.parametrize("case", DECODE, ids=[c[0] for c in DECODE])
def test_decode_never_evicts_pattern_every_step(case):
    name, b, h, d, dt, L, T, hv, rc, pat, splits = case
    w = W.Workload(name, b, h, d, dt, L, T, hv, rc, 1.1)
    rep = TD.run_stepwise(w, 73, splits=splits, pattern=O.StaticPattern(*pat))
    assert rep.pairs == w.pairs * T


@pytest.mark.parametrize("splits", [0, 4])
def test_free_run_with_pattern(splits):
    sp = O.StaticPattern(0, 11, 18)
    w = W.Workload("free-static", 2, 4, 128, "f16", 400, 60, 30, 25, 1.1)
    worst, alive = TD.run_free(w, 79, splits=splits, pattern=sp)
    assert alive >= w.pairs - 2


def test_pattern_with_position_rolling_every_step():
    """Both extensions at once on the cluster kernel: rotary embedding at
    in-cache ranks and protected pattern positions."""
    Bn, H, D, heavy, recent, steps = 1, 3, 128, 20, 12, 80
    sp = O.StaticPattern(1, 4, 8)
    base = 10000.0
    w = W.Workload("static-rope", Bn, H, D, "f16", 0, steps, heavy, recent, 1.1)
    cache = B.h2o_cache_create(Bn, H, D, heavy, recent, B.H2O_F16)
    B.h2o_cache_set_position_rolling(cache, base)
    B.h2o_cache_set_static_pattern(cache, sp.offset, sp.stride, sp.count)
    st = O.empty_cache(w.pairs, heavy, recent, D)
    o_dev = torch.empty((Bn, H, D), dtype=torch.float32, device="cuda")
    e_dev = torch.empty((Bn, H), dtype=torch.int32, device="cuda")
    rep = StepReport()
    flat = lambda a: a.reshape(w.pairs, D).astype(np.float64)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for t in range(steps):
        qd, kd, vd = W.decode_inputs(w, t, 83)
        nxt, r_out, r_ev, gap = O.decode_step(st, qd, kd, vd, heavy, recent, w.scale, rope_base=base, pattern=sp)
        B.h2o_cache_import_state(cache, oracle_image(cache, st))
        B.h2o_decode_step(cache, dev(qd), dev(kd), dev(vd), w.scale, o_dev, e_dev)
        B.h2o_cache_check(cache)
        after = B.unpack_state(cache, B.h2o_cache_export_state(cache))
        compare_decode_step(cache, after, o_dev.cpu().numpy().reshape(w.pairs, D), e_dev.cpu().numpy().reshape(-1),
                            st, nxt, r_out, r_ev, gap, rep, inputs=(flat(qd), flat(kd), flat(vd)), scale=w.scale,
                            rope_base=base, pattern=sp)
        st = nxt
    kept = set(st.pos[0][st.pos[0] >= 0].tolist())
    assert set(np.nonzero(sp.protects(np.arange(steps)))[0].tolist()) <= kept
    B.h2o_cache_destroy(cache)


def test_pattern_arguments_are_checked():
    cache = B.h2o_cache_create(1, 2, 64, 8, 4, B.H2O_F16)
    for bad in ((-1, 2, 3), (0, 0, 3), (0, 2, -1), (0, 2, 9), (2_000_000_000, 1_000_000_000, 3)):
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_static_pattern(cache, *bad)
    B.h2o_cache_set_static_pattern(cache, 0, 2, 8)  # count == heavy is allowed
    B.h2o_cache_set_static_pattern(cache, 0, 1, 0)  # off
    B.h2o_cache_destroy(cache)
