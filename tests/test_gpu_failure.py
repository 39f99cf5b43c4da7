"""Failure detection without a GPU fault: every wait in the library's kernels
is bounded and, when it gives up, sets an error flag instead of hanging.  The
self-test entry point makes a wait run out on purpose (an mbarrier that
nothing completes) with both wait forms the kernels use, and the device must
stay usable afterwards."""
import numpy as np
import pytest

from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("polls", [1, 2000])
def test_bounded_waits_give_up(polls):
    gave_up, ns = B.h2o_selftest_wait_timeout(polls)
    assert gave_up == [1, 1]
    # each poll suspends for at most about 1 us: both waits end well within this
    assert 0 < ns < 2 * polls * 20_000 + 5_000_000


def test_device_is_usable_after_a_wait_gave_up():
    assert B.h2o_selftest_wait_timeout(5000)[0] == [1, 1]
    w = W.Workload("after-timeout", 1, 2, 64, "f16", 40, 3, 8, 8, 1.1)
    q, k, v = W.prefill_inputs(w, 5)
    dev = lambda a: torch.from_numpy(a).cuda()
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, B.H2O_F16)
    B.h2o_prefill(cache, dev(q), dev(k), dev(v), w.scale)
    st, _, _ = O.prefill(q, k, v, w.heavy, w.recent, w.scale)
    out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
    qd, kd, vd = W.decode_inputs(w, w.prompt, 5)
    B.h2o_decode_step(cache, dev(qd), dev(kd), dev(vd), w.scale, out)
    _, r_out, _, _ = O.decode_step(st, qd, kd, vd, w.heavy, w.recent, w.scale)
    B.h2o_cache_check(cache)  # no flag left over from the self-test (it has its own buffer)
    assert np.abs(out.cpu().numpy().reshape(r_out.shape) - r_out).max() <= 2e-3
    B.h2o_cache_destroy(cache)
