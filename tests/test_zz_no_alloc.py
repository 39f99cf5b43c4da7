"""The allocation-free column-sum entry point, checked against the regular one.

h2o_prefill_colsum_static is meant for programs that may not call cudaMalloc
(engines that own all device memory through their own pools, or loops that
cannot take the device-wide synchronisation an allocation implies).  It must
return the same column sums as h2o_prefill_ex, whose scratch the library
allocates, and it must keep doing so on consecutive calls that reuse its one
fixed scratch array.  This file is collected last on purpose.
"""
import math

import numpy as np
import pytest

from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def regular_colsum(w, q, k, v):
    dt = B.H2O_F16 if w.dtype == "f16" else B.H2O_F32
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, dt)
    cs = torch.empty((w.batch, w.heads, w.prompt), dtype=torch.float32, device="cuda")
    B.h2o_prefill_ex(cache, q, k, v, w.scale, colsum=cs)
    torch.cuda.synchronize()
    B.h2o_cache_destroy(cache)
    return cs


def static_colsum(w, q, k):
    cs = torch.full((w.batch, w.heads, w.prompt), float("nan"), dtype=torch.float32, device="cuda")
    lib = B.lib()
    code = lib.h2o_prefill_colsum_static(q.data_ptr(), k.data_ptr(), w.batch, w.heads, w.head_dim, w.prompt,
                                         B.H2O_F16 if w.dtype == "f16" else B.H2O_F32, w.scale, cs.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert code == 0, lib.h2o_last_error().decode()
    # no bounded wait of the call's kernels gave up (synchronises the stream)
    B.h2o_prefill_colsum_static_check()
    return cs


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_static_scratch_matches_allocating_path_twice(dtype):
    # two different shapes back to back: the second call runs on the scratch
    # the first one left behind
    shapes = [W.Workload("a", 2, 8, 128, dtype, 700, 0, 40, 40, 1.1),
              W.Workload("b", 1, 4, 64 if dtype == "f16" else 128, dtype, 333, 0, 20, 20, 1.1)]
    for i, w in enumerate(shapes):
        q, k, v = (torch.from_numpy(a).cuda() for a in W.prefill_inputs(w, 40 + i))
        want = regular_colsum(w, q, k, v)
        got = static_colsum(w, q, k)
        assert torch.isfinite(got).all()
        rel = ((got - want).abs() / want.abs()).max().item()
        assert rel <= 1e-5, f"call {i}: relative difference {rel}"
        # and the column sums still carry the whole attention mass
        assert abs(got.double().sum(-1) - w.prompt).max().item() <= 1e-5 * w.prompt
        # against the fp64 oracle on a few pairs (exact definition of the sums)
        qf = q.double().cpu().numpy().reshape(w.pairs, w.prompt, w.head_dim)
        kf = k.double().cpu().numpy().reshape(w.pairs, w.prompt, w.head_dim)
        g = got.cpu().numpy().reshape(w.pairs, w.prompt).astype(np.float64)
        for p in (0, w.pairs // 2, w.pairs - 1):
            _, ref, _ = O.causal_attention_stats(qf[p], kf[p], np.zeros((w.prompt, 1)), w.scale)
            assert np.max(np.abs(g[p] - ref) / ref) <= 1e-5, f"call {i} pair {p}: against the oracle"


def test_static_scratch_rejects_oversize():
    lib = B.lib()
    q = torch.zeros(16, dtype=torch.float16, device="cuda")
    cs = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 64 x 64 pairs x 1024 tokens = 4,194,304 row statistics > 2,097,152
    code = lib.h2o_prefill_colsum_static(q.data_ptr(), q.data_ptr(), 64, 64, 128, 1024, B.H2O_F16,
                                         1 / math.sqrt(128), cs.data_ptr(), None)
    assert code == -1
    assert "exceeds the fixed scratch" in lib.h2o_last_error().decode()
