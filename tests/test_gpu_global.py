"""Global (offline) heavy hitters and the drift of the online rule from them.

The global selector keeps, out of a whole sequence of N tokens, the last
`recent` positions plus the `heavy` positions before them that receive the
most attention from all N rows (the report's section 2.3 and its Figure 2(d)
comparison of local and global H2O).  That is the prefill keep rule applied
to the whole sequence's column sums, so on the GPU it is h2o_prefill over all
N tokens into a cache with the same budgets.  These tests check it against
the oracle's global_select_pair and compare, pair by pair, the positions an
online run (prefill L tokens, then T decode steps) keeps with the global set.
"""
import numpy as np
import pytest

from harness import NEAR_TIE
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def kept_positions(cache):
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    return [sorted(int(x) for x in row if x >= 0) for row in g["pos"]]


def full_sequence(w, seed):
    """q, k, v for positions 0..L+T-1: [B, H, L+T, D] in the K/V dtype."""
    q, k, v = W.prefill_inputs(w, seed)
    qd, kd, vd = W.decode_sequence(w, w.prompt, w.decode, seed)
    cat = lambda a, d: np.concatenate([a, np.moveaxis(d, 0, 2)], axis=2)
    return cat(q, qd), cat(k, kd), cat(v, vd)


def local_and_global(w, seed):
    """Kept positions per pair: after the online run, and globally."""
    code = B.H2O_F16 if w.dtype == "f16" else B.H2O_F32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    qN, kN, vN = full_sequence(w, seed)
    L, N = w.prompt, w.prompt + w.decode
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, code)
    B.h2o_prefill(cache, dev(qN[:, :, :L]), dev(kN[:, :, :L]), dev(vN[:, :, :L]), w.scale)
    out = torch.empty((w.batch, w.heads, w.head_dim), dtype=torch.float32, device="cuda")
    for p in range(L, N):
        B.h2o_decode_step(cache, dev(qN[:, :, p]), dev(kN[:, :, p]), dev(vN[:, :, p]), w.scale, out)
    B.h2o_cache_check(cache)
    local = kept_positions(cache)
    B.h2o_cache_destroy(cache)
    gcache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, code)
    cs = torch.empty((w.batch, w.heads, N), dtype=torch.float32, device="cuda")
    B.h2o_prefill_ex(gcache, dev(qN), dev(kN), dev(vN), w.scale, colsum=cs)
    B.h2o_cache_check(gcache)
    glob = kept_positions(gcache)
    B.h2o_cache_destroy(gcache)
    return local, glob, cs.cpu().numpy().reshape(w.pairs, N), (qN, kN)


CASES = [
    # name, batch, heads, D, dtype, prompt, steps, heavy, recent
    ("g-f16-d128", 1, 4, 128, "f16", 500, 120, 60, 50),
    ("g-f32-d64", 2, 2, 64, "f32", 260, 90, 30, 30),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_global_selection_matches_oracle(case):
    name, Bn, H, D, dt, L, T, heavy, recent = case
    w = W.Workload(name, Bn, H, D, dt, L, T, heavy, recent, 1.1)
    local, glob, cs, (qN, kN) = local_and_global(w, 61)
    N = L + T
    qf = qN.reshape(w.pairs, N, D).astype(np.float64)
    kf = kN.reshape(w.pairs, N, D).astype(np.float64)
    mismatched = 0
    for i in range(w.pairs):
        kept, score = O.global_select_pair(qf[i], kf[i], heavy, recent, w.scale)
        assert np.max(np.abs(cs[i] - score) / score) <= 1e-5, f"pair {i}: global scores"
        if glob[i] != kept:
            # only positions at the heavy boundary may differ: each one kept by
            # one side and not the other scores within NEAR_TIE of the boundary
            s32 = O.to_f32(score)
            boundary = np.sort(s32[:N - recent])[::-1][heavy - 1]
            for j in set(glob[i]) ^ set(kept):
                assert j < N - recent and abs(s32[j] - boundary) <= NEAR_TIE, f"pair {i}: position {j}"
            mismatched += 1
        # both sets hold exactly the recent window plus `heavy` earlier positions
        for s in (local[i], glob[i]):
            assert len(s) == heavy + recent and s[-recent:] == list(range(N - recent, N))
        shared, of = O.heavy_overlap(local[i], glob[i], N, recent)
        assert of == heavy and 0 <= shared <= heavy
    assert mismatched <= 1


def test_drift_on_the_opt_layer_shape():
    """One layer of the OPT-6.7B decode shape (8 x 32 pairs, prompt 2048,
    256 decode steps, 205 + 205 slots): share of the global heavy hitters the
    online rule still holds at the end, printed for the design notes."""
    w = W.WORKLOADS["opt-6.7b"]
    local, glob, _, _ = local_and_global(w, W.seed_for(w.name))
    N = w.prompt + w.decode
    shares = [O.heavy_overlap(local[i], glob[i], N, w.recent) for i in range(w.pairs)]
    frac = np.array([s / o for s, o in shares])
    print(f"\nglobal heavy hitters kept by the online rule (opt-6.7b layer, {w.pairs} pairs): "
          f"mean {frac.mean():.4f}, min {frac.min():.4f}, max {frac.max():.4f}")
    assert all(o == w.heavy for _, o in shares)
    assert 0.0 < frac.mean() <= 1.0
