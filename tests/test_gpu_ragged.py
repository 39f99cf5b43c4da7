"""Ragged batches: every batch row's prompt has its own length.  The GPU
prefill (h2o_prefill_ragged) is compared pair by pair with the oracle's
prefill of the unpadded prompt, then both sides run free decode steps from
there (each pair at its own position)."""
import numpy as np
import pytest

from harness import check_other_victim, check_prefill_pair, out_tol
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CASES = [
    # name, heads, D, dtype, max_len, lengths, heavy, recent
    ("f16-d128", 3, 128, "f16", 700, [700, 257, 0, 37, 129], 60, 50),
    ("f16-d64", 2, 64, "f16", 300, [1, 300, 111], 20, 17),
    ("f32-d128", 2, 128, "f32", 200, [200, 60, 150], 30, 30),
]


def run_case(name, H, D, dt, Lmax, lengths, heavy, recent, steps=12, seed=41):
    Bn = len(lengths)
    w = W.Workload(name, Bn, H, D, dt, Lmax, steps, heavy, recent, 1.1)
    code = B.H2O_F16 if dt == "f16" else B.H2O_F32
    cache = B.h2o_cache_create(Bn, H, D, heavy, recent, code)
    q, k, v = W.prefill_inputs(w, seed)  # padded positions keep their (finite) draws
    dev = lambda a: torch.from_numpy(a).cuda()
    lens = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = torch.empty((Bn, H, Lmax, D), dtype=torch.float32, device="cuda")
    cs = torch.empty((Bn, H, Lmax), dtype=torch.float32, device="cuda")
    B.h2o_prefill_ragged(cache, dev(q), dev(k), dev(v), lens, w.scale, out=out, colsum=cs)
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    P, C = w.pairs, heavy + recent
    qf, kf, vf = (a.reshape(P, Lmax, D).astype(np.float64) for a in (q, k, v))
    g_cs = cs.cpu().numpy().reshape(P, Lmax).astype(np.float64)
    g_out = out.cpu().numpy().reshape(P, Lmax, D)
    tol = out_tol(code)
    states, alive = [], np.ones(P, dtype=bool)
    for i in range(P):
        Lb = lengths[i // H]
        if Lb == 0:
            st = O.empty_pair(C, recent, D)
            assert (g["p"][i], g["count"][i], g["head"][i]) == (0, 0, 0)
            assert np.all(g["pos"][i] == -1) and np.all(g["ring"][i] == -1)
            states.append(st)
            continue
        st, c, o = O.prefill_pair(qf[i, :Lb], kf[i, :Lb], vf[i, :Lb], heavy, recent, w.scale)
        rel = np.max(np.abs(g_cs[i, :Lb] - c) / c)
        assert rel <= 1e-5, f"pair {i}: colsum rel err {rel}"
        err = np.max(np.abs(g_out[i, :Lb] - o))
        assert err <= tol, f"pair {i}: out err {err}"
        kd = np.float16 if dt == "f16" else np.float32
        if not check_prefill_pair(g, i, st, c, kf[i, :Lb], vf[i, :Lb], Lb, heavy, recent, kd):
            alive[i] = False
        states.append(st)
    ref = O.CacheState.stack(states)
    # free decode from the prefilled state: every pair at its own position
    o_dev = torch.empty((Bn, H, D), dtype=torch.float32, device="cuda")
    e_dev = torch.empty((Bn, H), dtype=torch.int32, device="cuda")
    for t in range(steps):
        qd, kd, vd = W.decode_inputs(w, Lmax + t, seed)
        B.h2o_decode_step(cache, dev(qd), dev(kd), dev(vd), w.scale, o_dev, e_dev)
        before = ref
        ref, r_out, r_ev, gap = O.decode_step(ref, qd, kd, vd, heavy, recent, w.scale)
        g_o = o_dev.cpu().numpy().reshape(P, D)
        g_e = e_dev.cpu().numpy().reshape(P)
        for i in np.nonzero(alive)[0]:
            assert np.max(np.abs(g_o[i] - r_out[i])) <= tol, f"step {t} pair {i}"
            if g_e[i] != r_ev[i]:
                f64 = lambda a: a.reshape(P, D)[i].astype(np.float64)
                check_other_victim(before.pair(i), f64(qd), f64(kd), f64(vd), w.scale, heavy, recent, g_e[i],
                                   r_ev[i], gap[i], where=f"step {t} pair {i}")
                alive[i] = False
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    for i in np.nonzero(alive)[0]:
        assert np.array_equal(g["pos"][i], ref.pos[i]), f"pair {i}: positions after decode"
        assert g["p"][i] == ref.p[i]
    B.h2o_cache_destroy(cache)
    return int(alive.sum()), P


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_ragged_prefill_then_decode(case):
    alive, P = run_case(*case)
    assert alive >= P - 1


def test_ragged_lengths_are_clamped_and_checked():
    cache = B.h2o_cache_create(2, 1, 64, 4, 4, B.H2O_F16)
    x = torch.zeros((2, 1, 16, 64), dtype=torch.float16, device="cuda")
    lens = torch.tensor([-5, 99], dtype=torch.int32, device="cuda")  # clamped to 0 and 16
    B.h2o_prefill_ragged(cache, x, x, x, lens, 0.125)
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    assert list(g["p"]) == [0, 16] and list(g["count"]) == [0, 8]
    with pytest.raises(B.H2OError):
        B._check(B.lib().h2o_prefill_ragged(cache.handle, x.data_ptr(), x.data_ptr(), x.data_ptr(), 16, None,
                                            0.125, None, None, None, None))
    B.h2o_cache_destroy(cache)
