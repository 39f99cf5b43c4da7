"""Allocation failures injected on the host (h2o_debug_fail_alloc): every
device allocation a call makes can fail, the call then returns H2O_ENOMEM,
frees what it had already allocated, and leaves the cache usable."""
import numpy as np
import pytest

from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CREATE_ALLOCS = 7  # K, V, scores, positions, ring, counters, error word


def free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


@pytest.fixture(autouse=True)
def disarm():
    yield
    B.h2o_debug_fail_alloc(-1)


def test_every_create_allocation_can_fail_without_leaking():
    # a large cache (2 x 268 MB of K/V) so that a leaked buffer shows
    shape = (8, 32, 128, 2048, 2048, B.H2O_F16)
    before = free_bytes()
    for k in range(CREATE_ALLOCS):
        B.h2o_debug_fail_alloc(k)
        with pytest.raises(B.H2OError) as ei:
            B.h2o_cache_create(*shape)
        assert ei.value.code == -2, f"allocation {k}: {ei.value}"
    assert abs(free_bytes() - before) < 64 << 20
    B.h2o_debug_fail_alloc(CREATE_ALLOCS)  # one more than create needs: it succeeds
    c = B.h2o_cache_create(*shape)
    B.h2o_cache_destroy(c)


def test_prefill_workspace_failure_leaves_the_cache_usable():
    w = W.Workload("ws", 1, 2, 128, "f16", 300, 0, 20, 20, 1.1)
    q, k, v = (torch.from_numpy(a).cuda() for a in W.prefill_inputs(w, 5))
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, B.H2O_F16)
    B.h2o_debug_fail_alloc(0)
    with pytest.raises(B.H2OError) as ei:
        B.h2o_prefill(cache, q, k, v, w.scale)
    assert ei.value.code == -2
    B.h2o_prefill(cache, q, k, v, w.scale)  # the hook has disarmed: now it allocates and runs
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    assert np.all(g["count"] == w.cache_slots) and np.all(g["p"] == w.prompt)
    B.h2o_cache_destroy(cache)


def test_position_rolling_failure_leaves_rolling_off():
    cache = B.h2o_cache_create(1, 2, 64, 8, 8, B.H2O_F16)
    x = torch.zeros((1, 2, 16, 64), dtype=torch.float16, device="cuda")
    for k in (0, 1):  # the rank array, then the (cos, sin) table
        B.h2o_debug_fail_alloc(k)
        with pytest.raises(B.H2OError):
            B.h2o_cache_set_position_rolling(cache, 10000.0)
        B.h2o_prefill(cache, x, x, x, 0.125)  # still accepted: rolling stayed off
    B.h2o_cache_check(cache)
    B.h2o_cache_destroy(cache)
