"""Parity on the five measured workload shapes at their full sizes.

The CUDA path runs every pair in the launch configuration the benchmark
times (the cache's automatic cluster size); the oracle recomputes a sample of
pairs, which is exact because pairs never interact.  Checks: prefill column
sums / output / kept slots on sampled pairs; a free-running decode trajectory
on sampled pairs; and step-wise checks from identical states, where every
pair of the CUDA cache is loaded with one of the sampled pairs' oracle
states so that all pairs' results are checked.
"""
import numpy as np
import pytest

from harness import StepReport, check_other_victim, check_prefill_pair, compare_decode_step, oracle_image, out_tol
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def subset_state(st_list):
    return O.CacheState.stack(st_list)


def replicate(st: O.CacheState, P: int) -> O.CacheState:
    idx = np.arange(P) % st.K.shape[0]
    return O.CacheState(st.K[idx], st.V[idx], st.score[idx], st.pos[idx], st.ring[idx], st.head[idx],
                        st.count[idx], st.p[idx])


def run_workload(w, seed, sample, decode_steps, stepwise_at):
    dt = B.H2O_F16 if w.dtype == "f16" else B.H2O_F32
    P, D, L = w.pairs, w.head_dim, w.prompt
    cache = B.h2o_cache_create(w.batch, w.heads, D, w.heavy, w.recent, dt)
    tol = out_tol(dt)
    ns = len(sample)
    # ---- prefill: GPU on every pair, oracle on the sample
    if L:
        q, k, v = W.prefill_inputs(w, seed)
        out = torch.empty((w.batch, w.heads, L, D), dtype=torch.float32, device="cuda")
        cs = torch.empty((w.batch, w.heads, L), dtype=torch.float32, device="cuda")
        B.h2o_prefill_ex(cache, torch.from_numpy(q).cuda(), torch.from_numpy(k).cuda(),
                         torch.from_numpy(v).cuda(), w.scale, out=out, colsum=cs)
        B.h2o_cache_check(cache)
        g0 = B.unpack_state(cache, B.h2o_cache_export_state(cache))
        qf, kf, vf = (a.reshape(P, L, D) for a in (q, k, v))
        states, alive = [], []
        for i in sample:
            st, c, o = O.prefill_pair(qf[i].astype(np.float64), kf[i].astype(np.float64),
                                      vf[i].astype(np.float64), w.heavy, w.recent, w.scale)
            gc = cs[i // w.heads, i % w.heads].cpu().numpy().astype(np.float64)
            assert np.max(np.abs(gc - c) / c) <= 1e-5
            go = out[i // w.heads, i % w.heads].cpu().numpy()
            assert np.max(np.abs(go - o)) <= tol
            same = check_prefill_pair(g0, i, st, c, kf[i].astype(np.float64), vf[i].astype(np.float64), L, w.heavy,
                                      w.recent, w.np_dtype)
            states.append(st)
            alive.append(same)
        del out, cs
    else:
        B.h2o_cache_reset(cache)
        states = [O.empty_pair(w.heavy + w.recent, w.recent, D) for _ in sample]
        alive = [True] * ns
    ref = subset_state(states)
    alive = np.array(alive)
    # ---- free-running decode
    o_dev = torch.empty((w.batch, w.heads, D), dtype=torch.float32, device="cuda")
    e_dev = torch.empty((w.batch, w.heads), dtype=torch.int32, device="cuda")
    saved = {}
    sidx = np.array(sample)
    for t in range(decode_steps):
        qd, kd, vd = W.decode_inputs(w, L + t, seed)
        B.h2o_decode_step(cache, torch.from_numpy(qd).cuda(), torch.from_numpy(kd).cuda(),
                          torch.from_numpy(vd).cuda(), w.scale, o_dev, e_dev)
        sub = lambda a: a.reshape(P, D)[sidx][:, None, :]
        if t in stepwise_at:
            saved[t] = (ref.copy(), (qd, kd, vd))
        before = ref
        ref, r_out, r_ev, gap = O.decode_step(ref, sub(qd), sub(kd), sub(vd), w.heavy, w.recent, w.scale)
        g_out = o_dev.cpu().numpy().reshape(P, D)[sidx]
        g_ev = e_dev.cpu().numpy().reshape(P)[sidx]
        for j in np.nonzero(alive)[0]:
            assert np.max(np.abs(g_out[j] - r_out[j])) <= tol, f"step {t} pair {sample[j]}"
            if g_ev[j] != r_ev[j]:
                f64 = lambda a: sub(a)[j, 0].astype(np.float64)
                check_other_victim(before.pair(j), f64(qd), f64(kd), f64(vd), w.scale, w.heavy, w.recent, g_ev[j],
                                   r_ev[j], gap[j], where=f"step {t} pair {sample[j]}")
                alive[j] = False
    B.h2o_cache_check(cache)
    # ---- step-wise from identical states (every pair holds a sampled state)
    rep = StepReport()
    for t, (st, (qd, kd, vd)) in sorted(saved.items()):
        big = replicate(st, P)
        idx = np.arange(P) % ns
        rq, rk, rv = (a.reshape(P, D)[sidx][idx] for a in (qd, kd, vd))
        B.h2o_cache_import_state(cache, oracle_image(cache, big))
        shape = (w.batch, w.heads, D)
        B.h2o_decode_step(cache, torch.from_numpy(np.ascontiguousarray(rq.reshape(shape))).cuda(),
                          torch.from_numpy(np.ascontiguousarray(rk.reshape(shape))).cuda(),
                          torch.from_numpy(np.ascontiguousarray(rv.reshape(shape))).cuda(), w.scale, o_dev, e_dev)
        B.h2o_cache_check(cache)
        after = B.unpack_state(cache, B.h2o_cache_export_state(cache))
        f64 = lambda a: a.astype(np.float64)
        nxt, r_out, r_ev, gap = O.decode_step(st, f64(qd.reshape(P, D)[sidx][:, None]),
                                              f64(kd.reshape(P, D)[sidx][:, None]),
                                              f64(vd.reshape(P, D)[sidx][:, None]), w.heavy, w.recent, w.scale)
        R = replicate
        compare_decode_step(cache, after, o_dev.cpu().numpy().reshape(P, D), e_dev.cpu().numpy().reshape(P),
                            R(st, P), R(nxt, P), r_out[idx], r_ev[idx], gap[idx], rep,
                            inputs=(f64(rq), f64(rk), f64(rv)), scale=w.scale)
    B.h2o_cache_destroy(cache)
    return rep, int(alive.sum())


def test_opt_6_7b_shape():
    w = W.WORKLOADS["opt-6.7b"]
    rep, alive = run_workload(w, W.seed_for(w.name), sample=[0, 1, 37, 100, 129, 200, 254, 255],
                              decode_steps=w.decode, stepwise_at={0, 1, 127, 255})
    assert rep.pairs == 4 * w.pairs and alive >= 6


def test_opt_30b_shape():
    w = W.WORKLOADS["opt-30b"]
    rep, alive = run_workload(w, W.seed_for(w.name), sample=[0, 5, 777, 1800, 2999, 3583],
                              decode_steps=w.decode, stepwise_at={0, 31})
    assert rep.pairs == 2 * w.pairs and alive >= 5


def test_llama_16k_shape():
    w = W.WORKLOADS["llama-7b-16k"]
    rep, alive = run_workload(w, W.seed_for(w.name), sample=[0, 17, 31], decode_steps=w.decode,
                              stepwise_at={0, 511, 1023})
    assert rep.pairs == 3 * w.pairs and alive >= 2


def test_streaming_shape_fill_and_first_evictions():
    """No prompt: 2048 fill steps then eviction every step (checked to 2100)."""
    w = W.WORKLOADS["streaming"]
    rep, alive = run_workload(w, W.seed_for(w.name), sample=[0, 63, 127], decode_steps=2100,
                              stepwise_at={0, 1, 2047, 2048, 2049, 2099})
    assert rep.pairs == 6 * w.pairs and alive >= 2


def test_streaming_steady_state_far_positions():
    """A full cache deep into a 1,000,000-token stream: recent window just
    below the position, heavy hitters scattered over the past, scores drawn
    from a heavy-tailed law (a seeded synthetic state, not a CUDA result)."""
    w = W.WORKLOADS["streaming"]
    P, D, C, R, Hh = w.pairs, w.head_dim, w.cache_slots, w.recent, w.heavy
    rng = np.random.default_rng(99)
    cache = B.h2o_cache_create(w.batch, w.heads, D, Hh, R, B.H2O_F16)
    for p0 in (100_000, 999_000):
        heavy_pos = np.sort(rng.choice(p0 - R, size=Hh, replace=False))
        pos = np.concatenate([heavy_pos, np.arange(p0 - R, p0)])
        ks, vs = [], []
        for t in pos:
            _, k, v = W.decode_inputs(w, int(t), W.seed_for(w.name))
            ks.append(k.reshape(P, D))
            vs.append(v.reshape(P, D))
        K = np.stack(ks, 1).astype(np.float64)
        V = np.stack(vs, 1).astype(np.float64)
        score = O.to_f32(rng.pareto(1.5, size=(P, C)) * 0.05 + 1e-4)
        ring = np.tile(np.arange(Hh, C), (P, 1))
        st = O.CacheState(K, V, score, np.tile(pos, (P, 1)), ring, np.zeros(P, dtype=np.int64),
                          np.full(P, C), np.full(P, p0))
        o_dev = torch.empty((w.batch, w.heads, D), dtype=torch.float32, device="cuda")
        e_dev = torch.empty((w.batch, w.heads), dtype=torch.int32, device="cuda")
        rep = StepReport()
        for t in range(16):
            qd, kd, vd = W.decode_inputs(w, p0 + t, W.seed_for(w.name))
            nxt, r_out, r_ev, gap = O.decode_step(st, qd, kd, vd, Hh, R, w.scale)
            B.h2o_cache_import_state(cache, oracle_image(cache, st))
            B.h2o_decode_step(cache, torch.from_numpy(qd).cuda(), torch.from_numpy(kd).cuda(),
                              torch.from_numpy(vd).cuda(), w.scale, o_dev, e_dev)
            B.h2o_cache_check(cache)
            after = B.unpack_state(cache, B.h2o_cache_export_state(cache))
            f = lambda a: a.reshape(P, D).astype(np.float64)
            compare_decode_step(cache, after, o_dev.cpu().numpy().reshape(P, D), e_dev.cpu().numpy().reshape(P),
                                st, nxt, r_out, r_ev, gap, rep, inputs=(f(qd), f(kd), f(vd)), scale=w.scale)
            st = nxt
        assert rep.pairs == 16 * P
    B.h2o_cache_destroy(cache)
