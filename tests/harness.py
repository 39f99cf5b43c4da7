"""Shared helpers of the GPU parity tests: run the oracle, move its states into
the CUDA cache, and compare the CUDA results with the oracle's.

The oracle never receives anything the CUDA path produced: its inputs come
from the workload generator, and the states imported into the CUDA cache come
from the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from kv_cache_eviction_03_gb300 import binding as B
from oracle import h2o_oracle as O

NEAR_TIE = 1e-6  # candidate score gap below which either choice is accepted
SCORE_RTOL = 1e-5


def out_tol(kv_dtype: int) -> float:
    return 2e-3 if kv_dtype == B.H2O_F16 else 1e-5


def torch_dev(a, dtype=None):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def oracle_image(cache: B.Cache, st: O.CacheState) -> np.ndarray:
    """Import image of an oracle state (values are exact in the K/V dtype and
    the float32 score buffer, so nothing is rounded here)."""
    kd = cache.np_dtype()
    K = st.K.astype(kd)
    assert np.array_equal(K.astype(np.float64), st.K)
    V = st.V.astype(kd)
    score = st.score.astype(np.float32)
    assert np.array_equal(score.astype(np.float64), st.score)
    return B.pack_state(cache, K, V, score, st.pos.astype(np.int32), st.ring.astype(np.int32),
                        st.p.astype(np.int32), st.count.astype(np.int32), st.head.astype(np.int32))


@dataclass
class StepReport:
    pairs: int = 0
    near_ties: int = 0
    tie_mismatch: int = 0
    max_out_err: float = 0.0
    max_score_rel: float = 0.0
    notes: list = field(default_factory=list)


def candidate_near_ties(before: O.PairState, prob, recent, pattern=None) -> set:
    """Slots whose updated score is within NEAR_TIE of the lowest candidate
    (candidates: kept positions <= p - recent outside the static pattern)."""
    n = before.count
    new = O.to_f32(before.score[:n] + prob[:n])
    prot = pattern.protects(before.pos[:n]) if pattern is not None else np.zeros(n, dtype=bool)
    cand = [j for j in range(n) if before.pos[j] <= before.p - recent and not prot[j]]
    lo = min(new[j] for j in cand)
    return {j for j in cand if new[j] - lo <= NEAR_TIE}


def check_other_victim(before: O.PairState, q, k_new, v_new, scale, heavy, recent, gpu_victim, ref_victim, gap,
                       rope_base=None, pattern=None, where=""):
    """A GPU victim that differs from the oracle's is accepted only at a near
    tie (the oracle's two lowest candidates within NEAR_TIE) and only if the
    GPU's victim is itself one of the candidates within NEAR_TIE of the
    lowest updated score (any of them is a correct choice)."""
    assert gap <= NEAR_TIE, f"{where}: evicted slot {gpu_victim} != oracle {ref_victim} (gap {gap})"
    r = O.decode_step_pair(before.copy(), q, k_new, v_new, scale, heavy, recent, rope_base, pattern)
    assert int(gpu_victim) in candidate_near_ties(before, r.prob, recent, pattern), \
        f"{where}: GPU victim {gpu_victim} is not a near tie"


def compare_decode_step(cache: B.Cache, gpu_after: dict, gpu_out, gpu_ev, ref_before: O.CacheState,
                        ref_after: O.CacheState, ref_out, ref_ev, ref_gap, rep: StepReport, inputs, scale,
                        pairs=None, rope_base=None, pattern=None):
    """Compare one decode step (identical pre-step state) pair by pair.

    inputs = (q, k_new, v_new) as float64 [P, D] arrays of this step;
    rope_base / pattern: position rolling and static pattern of the step."""
    tol = out_tol(cache.kv_dtype)
    R = cache.recent
    pairs = range(ref_out.shape[0]) if pairs is None else pairs
    for i in pairs:
        rep.pairs += 1
        err = float(np.max(np.abs(gpu_out[i].astype(np.float64) - ref_out[i])))
        rep.max_out_err = max(rep.max_out_err, err)
        assert err <= tol, f"pair {i}: out max abs err {err} > {tol}"
        ge, re_ = int(gpu_ev[i]), int(ref_ev[i])
        if ref_gap[i] <= NEAR_TIE:
            rep.near_ties += 1
        if ge != re_:
            # accepted only at a near tie, and only for an equally good victim
            check_other_victim(ref_before.pair(i), inputs[0][i], inputs[1][i], inputs[2][i], scale, cache.heavy,
                               R, ge, re_, ref_gap[i], rope_base, pattern, where=f"pair {i}")
            rep.tie_mismatch += 1
            rep.notes.append((i, ge, re_))
            continue
        C = cache.slots
        used = ref_after.pos[i] >= 0
        assert np.array_equal(gpu_after["pos"][i], ref_after.pos[i].astype(np.int32)), f"pair {i}: positions"
        assert np.array_equal(gpu_after["ring"][i], ref_after.ring[i].astype(np.int32)), f"pair {i}: ring"
        assert (int(gpu_after["p"][i]), int(gpu_after["count"][i]), int(gpu_after["head"][i])) == \
            (int(ref_after.p[i]), int(ref_after.count[i]), int(ref_after.head[i])), f"pair {i}: counters"
        gs = gpu_after["score"][i][used].astype(np.float64)
        rs = ref_after.score[i][used]
        rel = float(np.max(np.abs(gs - rs) / np.maximum(np.abs(rs), 1e-30))) if used.any() else 0.0
        rep.max_score_rel = max(rep.max_score_rel, rel)
        assert rel <= SCORE_RTOL, f"pair {i}: score rel err {rel}"
        kd = cache.np_dtype()
        assert np.array_equal(gpu_after["K"][i][used], ref_after.K[i][used].astype(kd)), f"pair {i}: K slots"
        assert np.array_equal(gpu_after["V"][i][used], ref_after.V[i][used].astype(kd)), f"pair {i}: V slots"


def heavy_boundary_gap(colsum_f32: np.ndarray, L: int, heavy: int, recent: int, pattern=None) -> float:
    """Gap between the last kept and the first dropped candidate score at the
    heavy boundary (candidates: positions < L - recent outside the pattern)."""
    if L <= heavy + recent:
        return np.inf
    n = L - recent
    prot = pattern.protects(np.arange(n)) if pattern is not None else np.zeros(n, dtype=bool)
    take = heavy - int(prot.sum())
    c = np.sort(colsum_f32[:n][~prot])[::-1]
    if take == 0 or take >= c.size:
        return np.inf
    return float(c[take - 1] - c[take])


def check_prefill_pair(g: dict, i: int, st: O.PairState, colsum_ref, k_pair, v_pair, L: int, heavy: int,
                       recent: int, kv_np_dtype, pattern=None) -> bool:
    """Pair i of an exported GPU state after the prefill, against the oracle.

    Equal kept sets: slots, K/V, scores (1e-5 relative to the oracle's column
    sums), ring and counters are compared.  Different kept sets are accepted
    only at the heavy boundary: every position kept by one side and not the
    other must be a non-pattern candidate whose float32 column sum lies within
    NEAR_TIE of the boundary score, and the GPU's own set must still be laid
    out correctly (heavy hitters ascending below L - recent with every pattern
    position among them, the recent window after them, each slot's K/V row,
    score, the ring and the counters).  Returns True when the sets are equal.
    """
    C = heavy + recent
    gp = g["pos"][i].astype(np.int64)
    count = int(g["count"][i])
    assert (int(g["p"][i]), count, int(g["head"][i])) == (st.p, st.count, st.head), f"pair {i}: counters"
    assert np.array_equal(g["ring"][i], st.ring.astype(np.int32)), f"pair {i}: ring"
    same = np.array_equal(gp, st.pos)
    if not same:
        assert L > C, f"pair {i}: a prompt within the budget keeps every position"
        cs32 = O.to_f32(colsum_ref)
        n = L - recent
        gh, rh = gp[:heavy], st.pos[:heavy]
        assert np.all(np.diff(gh) > 0) and gh.max() < n, f"pair {i}: heavy slots not ascending below L-recent"
        assert np.array_equal(gp[heavy:C], np.arange(n, L)), f"pair {i}: recent window"
        prot = pattern.protects(np.arange(n)) if pattern is not None else np.zeros(n, dtype=bool)
        assert set(np.nonzero(prot)[0].tolist()) <= set(gh.tolist()), f"pair {i}: pattern position dropped"
        free = np.nonzero(~prot)[0]
        take = heavy - int(prot.sum())
        boundary = np.sort(cs32[free])[::-1][take - 1]
        for j in set(gh.tolist()) ^ set(rh.tolist()):
            assert not prot[j] and abs(cs32[j] - boundary) <= NEAR_TIE, \
                f"pair {i}: position {j} (score {cs32[j]}) differs away from the heavy boundary {boundary}"
    used = gp[:count]
    gs = g["score"][i][:count].astype(np.float64)
    rs = colsum_ref[used]
    assert count == 0 or np.max(np.abs(gs - rs) / rs) <= SCORE_RTOL, f"pair {i}: slot scores"
    assert np.array_equal(g["K"][i][:count], k_pair[used].astype(kv_np_dtype)), f"pair {i}: K slots"
    assert np.array_equal(g["V"][i][:count], v_pair[used].astype(kv_np_dtype)), f"pair {i}: V slots"
    assert np.all(g["pos"][i][count:] == -1)
    return same
