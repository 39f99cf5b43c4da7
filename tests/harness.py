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


def candidate_near_ties(before: O.PairState, prob, recent) -> set:
    """Slots whose updated score is within NEAR_TIE of the lowest candidate."""
    n = before.count
    new = O.to_f32(before.score[:n] + prob[:n])
    cand = [j for j in range(n) if before.pos[j] <= before.p - recent]
    lo = min(new[j] for j in cand)
    return {j for j in cand if new[j] - lo <= NEAR_TIE}


def compare_decode_step(cache: B.Cache, gpu_after: dict, gpu_out, gpu_ev, ref_before: O.CacheState,
                        ref_after: O.CacheState, ref_out, ref_ev, ref_gap, rep: StepReport, inputs, scale,
                        pairs=None):
    """Compare one decode step (identical pre-step state) pair by pair.

    inputs = (q, k_new, v_new) as float64 [P, D] arrays of this step."""
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
            assert ref_gap[i] <= NEAR_TIE, f"pair {i}: evicted slot {ge} != oracle {re_} (gap {ref_gap[i]})"
            before = ref_before.pair(i)
            r = O.decode_step_pair(before.copy(), inputs[0][i], inputs[1][i], inputs[2][i], scale,
                                   cache.heavy, cache.recent)
            assert ge in candidate_near_ties(before, r.prob, R), f"pair {i}: GPU victim {ge} is not a near tie"
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


def heavy_boundary_gap(colsum_f32: np.ndarray, L: int, heavy: int, recent: int) -> float:
    """Gap between the heavy-th and (heavy+1)-th largest candidate scores."""
    if L <= heavy + recent or heavy == 0:
        return np.inf
    c = np.sort(colsum_f32[:L - recent])[::-1]
    return float(c[heavy - 1] - c[heavy]) if heavy < c.size else np.inf
