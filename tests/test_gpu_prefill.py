"""GPU parity of the prefill (row statistics, column sums, keep rule, slot
layout) against the fp64 oracle."""
import math

import numpy as np
import pytest

from harness import check_prefill_pair, out_tol
from kv_cache_eviction_03_gb300 import binding as B
from kv_cache_eviction_03_gb300 import workload as W
from oracle import h2o_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def check_prefill(w, seed, pairs=None, with_out=True, pattern=None):
    """Run the GPU prefill on the full shape, compare `pairs` (default all).
    pattern: an oracle StaticPattern, also set on the cache."""
    dt = B.H2O_F16 if w.dtype == "f16" else B.H2O_F32
    cache = B.h2o_cache_create(w.batch, w.heads, w.head_dim, w.heavy, w.recent, dt)
    if pattern is not None:
        B.h2o_cache_set_static_pattern(cache, pattern.offset, pattern.stride, pattern.count)
    q, k, v = W.prefill_inputs(w, seed)
    L, P, D = w.prompt, w.pairs, w.head_dim
    dev = lambda a: torch.from_numpy(a).cuda()
    out = torch.empty((w.batch, w.heads, L, D), dtype=torch.float32, device="cuda") if with_out else None
    colsum = torch.empty((w.batch, w.heads, L), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.batch, w.heads, L), dtype=torch.float32, device="cuda")
    B.h2o_prefill_ex(cache, dev(q), dev(k), dev(v), w.scale, out=out, colsum=colsum, lse=lse)
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    g_cs = colsum.cpu().numpy().reshape(P, L).astype(np.float64)
    g_lse = lse.cpu().numpy().reshape(P, L).astype(np.float64)
    g_out = out.cpu().numpy().reshape(P, L, D) if with_out else None
    qf, kf, vf = (a.reshape(P, L, D).astype(np.float64) for a in (q, k, v))
    tol = out_tol(dt)
    stats = {"colsum_rel": 0.0, "out_err": 0.0, "lse_err": 0.0, "ties": 0}
    for i in (range(P) if pairs is None else pairs):
        st, cs, o = O.prefill_pair(qf[i], kf[i], vf[i], w.heavy, w.recent, w.scale, pattern)
        lse_ref, _, _ = O.causal_attention_stats(qf[i], kf[i], vf[i], w.scale) if L <= 4096 else (None, 0, 0)
        rel = float(np.max(np.abs(g_cs[i] - cs) / cs))
        stats["colsum_rel"] = max(stats["colsum_rel"], rel)
        assert rel <= 1e-5, f"pair {i}: colsum rel err {rel}"
        assert abs(g_cs[i].sum() - L) <= 1e-5 * L
        if lse_ref is not None:
            e = float(np.max(np.abs(g_lse[i] - lse_ref)))
            stats["lse_err"] = max(stats["lse_err"], e)
            assert e <= 5e-5, f"pair {i}: lse err {e}"
        if with_out:
            e = float(np.max(np.abs(g_out[i] - o)))
            stats["out_err"] = max(stats["out_err"], e)
            assert e <= tol, f"pair {i}: out err {e}"
        kd = np.float16 if w.dtype == "f16" else np.float32
        if not check_prefill_pair(g, i, st, cs, kf[i], vf[i], L, w.heavy, w.recent, kd, pattern):
            stats["ties"] += 1
    B.h2o_cache_destroy(cache)
    return stats


CASES = [
    # name, batch, heads, D, dtype, L, heavy, recent
    ("f16-d128-L200", 1, 3, 128, "f16", 200, 30, 20),
    ("f16-d128-L64", 2, 2, 128, "f16", 64, 10, 10),
    ("f16-d128-L65", 2, 2, 128, "f16", 65, 10, 10),
    ("f16-d128-L1", 1, 2, 128, "f16", 1, 4, 3),
    ("f16-d64-L257", 1, 3, 64, "f16", 257, 40, 33),
    ("f16-keep-all", 1, 2, 128, "f16", 50, 40, 30),
    ("f16-keep-all-short", 1, 2, 128, "f16", 7, 40, 30),
    ("f16-no-heavy", 1, 2, 128, "f16", 130, 0, 17),
    ("f16-L-eq-C", 1, 2, 64, "f16", 48, 24, 24),
    ("f16-L-eq-C+1", 1, 2, 64, "f16", 49, 24, 24),
    ("f32-d64-L300", 1, 2, 64, "f32", 300, 30, 30),
    ("f32-d128-L97", 2, 1, 128, "f32", 97, 11, 9),
    ("f16-large-heavy", 1, 1, 128, "f16", 1500, 700, 100),
    # 128-row tensor-core blocks: exact multiples, one past, several + ragged tail
    ("f16-d128-L128", 1, 2, 128, "f16", 128, 20, 20),
    ("f16-d64-L129", 1, 2, 64, "f16", 129, 20, 20),
    ("f16-d128-L256", 1, 1, 128, "f16", 256, 40, 40),
    ("f16-d128-L643", 2, 2, 128, "f16", 643, 60, 50),
]
F16_CASES = [c for c in CASES if c[4] == "f16"]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_parity(case):
    name, b, h, d, dt, L, hv, rc = case
    w = W.Workload(name, b, h, d, dt, L, 0, hv, rc, 1.1)
    check_prefill(w, 13)


@pytest.mark.parametrize("case", F16_CASES, ids=[c[0] for c in F16_CASES])
def test_prefill_parity_lse_only(case):
    """Without the attention output the fp16 row pass runs on tcgen05."""
    name, b, h, d, dt, L, hv, rc = case
    w = W.Workload(name, b, h, d, dt, L, 0, hv, rc, 1.1)
    check_prefill(w, 29, with_out=False)


def test_prefill_without_output():
    w = W.Workload("noout", 1, 2, 128, "f16", 180, 0, 20, 20, 1.1)
    check_prefill(w, 17, with_out=False)


def test_tiny_reference_prefill():
    w = W.WORKLOADS["tiny-ref"]
    s = check_prefill(w, W.seed_for("tiny-ref"))
    assert s["out_err"] <= 1e-5


def test_constant_keys_harmonic_colsum_on_gpu():
    """Equal keys: colsum_j = H_L - H_j exactly in real arithmetic."""
    L, D = 300, 128
    cache = B.h2o_cache_create(1, 1, D, 20, 20, B.H2O_F16)
    rng = np.random.default_rng(0)
    q = torch.from_numpy(rng.standard_normal((1, 1, L, D)).astype(np.float16)).cuda()
    k = torch.from_numpy(np.tile(rng.standard_normal(D).astype(np.float16), (1, 1, L, 1))).cuda()
    v = torch.from_numpy(rng.standard_normal((1, 1, L, D)).astype(np.float16)).cuda()
    cs = torch.empty((1, 1, L), dtype=torch.float32, device="cuda")
    B.h2o_prefill_ex(cache, q, k, v, 1 / math.sqrt(D), colsum=cs)
    Hn = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, L + 1))])
    np.testing.assert_allclose(cs.cpu().numpy()[0, 0], Hn[L] - Hn[:L], rtol=1e-5)
    B.h2o_cache_destroy(cache)


def test_prefill_zero_length_empties_cache():
    cache = B.h2o_cache_create(1, 2, 64, 4, 4, B.H2O_F16)
    B.h2o_prefill(cache, torch.zeros((1, 2, 0, 64), dtype=torch.float16, device="cuda"),
                  torch.zeros((1, 2, 0, 64), dtype=torch.float16, device="cuda"),
                  torch.zeros((1, 2, 0, 64), dtype=torch.float16, device="cuda"), 0.125)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    assert (g["pos"] == -1).all() and (g["count"] == 0).all() and (g["p"] == 0).all()
    B.h2o_cache_destroy(cache)


BUDGETS = [0.04, 0.10, 0.20, 0.60]  # total cache budget as a fraction of the prompt, heavy = recent


@pytest.mark.parametrize("ratio", BUDGETS, ids=[f"{int(r * 100)}pct" for r in BUDGETS])
def test_prefill_budget_ratios(ratio):
    L = 1000
    half = int(round(ratio * L / 2))
    w = W.Workload(f"budget{ratio}", 1, 4, 128, "f16", L, 0, half, half, 1.1)
    check_prefill(w, 53, with_out=False)


def test_long_prompt_output_with_separate_column_pass():
    """4096 pairs x 4096 tokens: the output pass's column-sum partials would
    take ~4.4 GB, past the 2 GB cap, so the separate column pass runs next to
    the output pass; sampled pairs against the oracle."""
    Bn, H, L, D, hv, rc = 64, 64, 4096, 64, 100, 60
    g = torch.Generator(device="cuda").manual_seed(5)
    q, k, v = (torch.randn((Bn, H, L, D), generator=g, device="cuda").half() for _ in range(3))
    cache = B.h2o_cache_create(Bn, H, D, hv, rc, B.H2O_F16)
    out = torch.empty((Bn, H, L, D), dtype=torch.float32, device="cuda")
    cs = torch.empty((Bn, H, L), dtype=torch.float32, device="cuda")
    scale = 1 / math.sqrt(D)
    B.h2o_prefill_ex(cache, q, k, v, scale, out=out, colsum=cs)
    B.h2o_cache_check(cache)
    g = B.unpack_state(cache, B.h2o_cache_export_state(cache))
    for i in (0, 1, 2047, Bn * H - 1):
        b, h = divmod(i, H)
        qf, kf, vf = (x[b, h].double().cpu().numpy() for x in (q, k, v))
        st, c, o = O.prefill_pair(qf, kf, vf, hv, rc, scale)
        assert np.max(np.abs(cs[b, h].cpu().numpy() - c) / c) <= 1e-5
        assert np.max(np.abs(out[b, h].cpu().numpy() - o)) <= 2e-3
        check_prefill_pair(g, i, st, c, kf, vf, L, hv, rc, np.float16)
    B.h2o_cache_destroy(cache)
