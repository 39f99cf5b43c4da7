"""Sharding by heads needs no exchange ("H2O ... 深度解读报告", section 3.4:
eviction is decided per head): two caches of H/2 heads each, run on the two
halves of the inputs, must give exactly what one H-head cache gives.  The
comparison is bit-exact (attention outputs, evicted slots, the whole exported
cache state), so every library kernel must index its pairs the same way
whatever the cache's pair count.  All caches use one fixed decode launch
shape, since a different cluster size sums the softmax in another order."""
import numpy as np
import pytest

from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CASES = [
    # name, batch, heads, D, dtype, prompt, decode, heavy, recent, (splits, stages)
    ("f16-d128-cluster", 2, 8, 128, "f16", 600, 60, 60, 50, (2, 8)),
    ("f16-d128-one-cta", 1, 6, 128, "f16", 300, 55, 40, 30, (1, 12)),
    ("f32-d64-warp", 4, 4, 64, "f32", 200, 50, 20, 20, (B.H2O_DECODE_WARP_PER_PAIR, 3)),
]


def states_by_head(cache, Bn, H):
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    return {k: v.reshape((Bn, H) + v.shape[1:]) for k, v in g.items()}


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_two_half_head_caches_equal_the_full_cache(case):
    name, Bn, H, D, dt, L, T, heavy, recent, shape = case
    w = W.Workload(name, Bn, H, D, dt, L, T, heavy, recent, 1.1)
    code = B.H2O_F16 if dt == "f16" else B.H2O_F32
    q, k, v = (torch.from_numpy(a).cuda() for a in W.prefill_inputs(w, 97))
    dec = [tuple(torch.from_numpy(a).cuda() for a in W.decode_inputs(w, L + t, 97)) for t in range(T)]
    half = H // 2
    parts = [(0, H), (0, half), (half, H)]
    caches = [B.h2o_cache_create(Bn, hi - lo, D, heavy, recent, code) for lo, hi in parts]
    for c in caches:
        B.h2o_cache_set_decode_shape(c, *shape)
    outs = [[] for _ in parts]
    evs = [[] for _ in parts]
    pre = []
    for c, (lo, hi) in zip(caches, parts):
        sl = lambda x: x[:, lo:hi].contiguous()
        o = torch.empty((Bn, hi - lo, L, D), dtype=torch.float32, device="cuda")
        cs = torch.empty((Bn, hi - lo, L), dtype=torch.float32, device="cuda")
        B.h2o_prefill_ex(c, sl(q), sl(k), sl(v), w.scale, out=o, colsum=cs)
        pre.append((o, cs))
    for t in range(T):
        for i, (c, (lo, hi)) in enumerate(zip(caches, parts)):
            qd, kd, vd = (x[:, lo:hi].contiguous() for x in dec[t])
            o = torch.empty((Bn, hi - lo, D), dtype=torch.float32, device="cuda")
            e = torch.empty((Bn, hi - lo), dtype=torch.int32, device="cuda")
            B.h2o_decode_step(c, qd, kd, vd, w.scale, o, e)
            outs[i].append(o)
            evs[i].append(e)
    for c in caches:
        B.h2o_cache_check(c)
    cat = lambda a, b: torch.cat([a, b], dim=1)
    assert torch.equal(pre[0][0], cat(pre[1][0], pre[2][0])), "prefill output"
    assert torch.equal(pre[0][1], cat(pre[1][1], pre[2][1])), "prefill column sums"
    for t in range(T):
        assert torch.equal(outs[0][t], cat(outs[1][t], outs[2][t])), f"step {t}: out"
        assert torch.equal(evs[0][t], cat(evs[1][t], evs[2][t])), f"step {t}: evicted"
    full = states_by_head(caches[0], Bn, H)
    lo_s = states_by_head(caches[1], Bn, half)
    hi_s = states_by_head(caches[2], Bn, H - half)
    for key in full:
        assert np.array_equal(full[key], np.concatenate([lo_s[key], hi_s[key]], axis=1)), f"state {key}"
    assert int(np.sum(torch.stack(evs[0]).cpu().numpy() >= 0)) > 0  # evictions happened
    for c in caches:
        B.h2o_cache_destroy(c)
