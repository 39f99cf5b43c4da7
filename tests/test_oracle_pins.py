"""Pins of the fp64 oracle to facts fixed outside the oracle itself.

Each test checks the oracle against a library routine, a closed form, an
invariant the method guarantees, or an independent brute-force restatement on
tiny inputs, chosen so that a plausible slip (a dropped self term, a wrong
softmax axis, an off-by-one recent window, argmax for argmin, a wrong tie
rule) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import h2o_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_seq(rng, L, D, key_mean=None):
    q = rng.standard_normal((L, D))
    k = rng.standard_normal((L, D)) * 1.3
    v = rng.standard_normal((L, D))
    if key_mean is not None:
        k += key_mean
    return q, k, v


def run_pair(q_all, k_all, v_all, L, heavy, recent, scale, rope_base=None, pattern=None):
    """Prefill positions < L, then decode the rest; returns per-step results."""
    st, colsum, out_prefill = O.prefill_pair(q_all[:L], k_all[:L], v_all[:L], heavy, recent, scale, pattern)
    steps = []
    for p in range(L, q_all.shape[0]):
        before = st.copy()
        r = O.decode_step_pair(st, q_all[p], k_all[p], v_all[p], scale, heavy, recent, rope_base, pattern)
        steps.append((before, r, st.copy()))
    return st, colsum, out_prefill, steps


def sdpa_causal(q, k, v, scale):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=scale)
    return o[0, 0].numpy()


def sdpa_masked(q, k, v, scale, allowed):
    """torch fp64 attention where query row i sees key j only if allowed[i, j]."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    mask = torch.from_numpy(np.ascontiguousarray(allowed))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask, scale=scale)
    return o[0, 0].numpy()


def rotary_at(x, positions, base):
    """Rotary embedding computed as complex rotations in torch (independent of
    the oracle's rope_rotate): pair (2i, 2i+1) as one complex number, times
    exp(i * position * base^(-2i/D))."""
    n, D = x.shape
    xc = torch.from_numpy(x[:, 0::2] + 1j * x[:, 1::2])
    theta = base ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    ang = torch.as_tensor(positions, dtype=torch.float64)[:, None] * theta[None, :]
    r = xc * torch.exp(1j * ang)
    return torch.stack([r.real, r.imag], dim=-1).reshape(n, D).numpy()


# ------------------------------------------------------------------ library routine
@pytest.mark.parametrize("L,T,heavy,recent", [(12, 6, 10, 8), (5, 9, 7, 7), (0, 10, 4, 6), (16, 1, 9, 8)])
def test_full_budget_equals_causal_attention(L, T, heavy, recent):
    """Budget >= L+T: nothing is ever evicted, so every output is plain causal
    attention (the report's "local H2O ~ Full" at full budget), checked against
    torch's fp64 scaled_dot_product_attention."""
    rng = np.random.default_rng(1)
    D = 8
    scale = 1 / math.sqrt(D)
    q, k, v = rand_seq(rng, L + T, D)
    st, colsum, out_prefill, steps = run_pair(q, k, v, L, heavy, recent, scale)
    ref = sdpa_causal(q, k, v, scale)
    if L:
        np.testing.assert_allclose(out_prefill, ref[:L], rtol=0, atol=1e-12)
    for t, (_, r, _) in enumerate(steps):
        assert r.evicted == -1
        np.testing.assert_allclose(r.out, ref[L + t], rtol=0, atol=1e-12)
    assert st.count == L + T


@pytest.mark.parametrize("L,recent", [(20, 5), (3, 4), (0, 1), (9, 1)])
def test_no_heavy_budget_is_sliding_window(L, recent):
    """heavy = 0 reduces H2O to the Local baseline: the token at p attends to
    positions p-recent..p exactly (closed form), here via torch SDPA on the
    sliced window."""
    rng = np.random.default_rng(2)
    D, T = 4, 15
    scale = 0.7
    q, k, v = rand_seq(rng, L + T, D)
    _, _, _, steps = run_pair(q, k, v, L, 0, recent, scale)
    for t, (_, r, after) in enumerate(steps):
        p = L + t
        lo = max(0, p - recent)
        qt = torch.from_numpy(q[p:p + 1])[None, None]
        kt = torch.from_numpy(k[lo:p + 1])[None, None]
        vt = torch.from_numpy(v[lo:p + 1])[None, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, 0, 0].numpy()
        np.testing.assert_allclose(r.out, ref, rtol=0, atol=1e-12)
        assert sorted(after.pos[after.pos >= 0].tolist()) == list(range(max(0, p + 1 - recent), p + 1))


# ------------------------------------------------------------------ closed forms
def test_colsum_mass_is_prompt_length():
    """Every causal softmax row sums to one, so the column sums add up to L."""
    rng = np.random.default_rng(3)
    for L in (1, 2, 7, 64):
        q, k, v = rand_seq(rng, L, 16)
        _, colsum, _ = O.causal_attention_stats(q, k, v, 0.25)
        assert abs(colsum.sum() - L) < 1e-10 * L
        assert np.all(colsum > 0)


def test_colsum_constant_keys_harmonic():
    """Equal keys give uniform rows p_ij = 1/(i+1), so
    colsum_j = sum_{i=j}^{L-1} 1/(i+1) = H_L - H_j (harmonic numbers)."""
    rng = np.random.default_rng(4)
    L, D = 50, 6
    q = rng.standard_normal((L, D))
    k = np.tile(rng.standard_normal(D), (L, 1))
    v = rng.standard_normal((L, D))
    _, colsum, out = O.causal_attention_stats(q, k, v, 0.9)
    Hn = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, L + 1))])
    np.testing.assert_allclose(colsum, Hn[L] - Hn[:L], rtol=1e-13, atol=0)
    # and the output is the running mean of v
    np.testing.assert_allclose(out, np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None], atol=1e-12)


def test_golden_uniform_three_tokens():
    """Hand-worked example stored as a fixture (uniform attention, L = 3)."""
    vals = {}
    with open(os.path.join(GOLDEN, "uniform_colsum_L3.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, val = line.split("=")
                vals[key.strip()] = [float(eval(x, {})) for x in val.split(",")]
    q = np.zeros((3, 2))
    k = np.ones((3, 2))
    v = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    _, colsum, out = O.causal_attention_stats(q, k, v, 1.0)
    np.testing.assert_allclose(colsum, vals["colsum"], rtol=1e-15)
    np.testing.assert_allclose(out[:, 0], vals["out0"], rtol=1e-15)
    np.testing.assert_allclose(out[:, 1], vals["out1"], rtol=1e-15)


def test_constant_values_give_that_value():
    """Probabilities sum to one, so with every V row equal to c, out = c."""
    rng = np.random.default_rng(5)
    L, T, D = 30, 40, 8
    q, k, _ = rand_seq(rng, L + T, D)
    c = rng.standard_normal(D)
    v = np.tile(c, (L + T, 1))
    _, _, out_prefill, steps = run_pair(q, k, v, L, 6, 5, 0.5)
    np.testing.assert_allclose(out_prefill, np.tile(c, (L, 1)), atol=1e-13)
    for _, r, _ in steps:
        np.testing.assert_allclose(r.out, c, atol=1e-13)


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("L,heavy,recent", [(40, 6, 5), (8, 6, 5), (0, 3, 2), (11, 0, 3), (25, 4, 1)])
def test_budget_window_and_single_eviction(L, heavy, recent):
    """Section 3.1/3.4 invariants after every step: |S| <= heavy+recent, the last
    `recent` positions are always kept, at most one entry leaves per step, the
    ring lists the recent window oldest-first, and probabilities sum to one."""
    rng = np.random.default_rng(6)
    T, D = 60, 4
    q, k, v = rand_seq(rng, L + T, D, key_mean=rng.standard_normal(D))
    C = heavy + recent
    _, _, _, steps = run_pair(q, k, v, L, heavy, recent, 0.8)
    for t, (before, r, after) in enumerate(steps):
        p = L + t
        kept_before = set(before.pos[before.pos >= 0].tolist())
        kept_after = set(after.pos[after.pos >= 0].tolist())
        assert len(kept_after) == after.count <= C
        assert set(range(max(0, p + 1 - recent), p + 1)) <= kept_after
        assert len(kept_before - kept_after) <= 1
        assert kept_after - kept_before == {p}
        assert abs(r.prob.sum() - 1) < 1e-12
        ring_pos = [after.pos[s] for s in np.roll(after.ring, -after.head) if s >= 0]
        assert ring_pos == list(range(max(0, p + 1 - recent), p + 1))
        if r.evicted >= 0:
            assert before.pos[r.evicted] <= p - recent
            assert before.count == C


def test_score_mass_conservation():
    """Each query row hands out probability mass exactly 1, so after t decode
    steps: sum of kept scores + scores of evicted tokens at eviction time
    + prompt mass of tokens dropped at prefill = L + t (up to the float32
    rounding of the score buffer)."""
    rng = np.random.default_rng(7)
    L, T, D, heavy, recent = 48, 80, 8, 7, 6
    q, k, v = rand_seq(rng, L + T, D, key_mean=rng.standard_normal(D))
    st, colsum, _, steps = run_pair(q, k, v, L, heavy, recent, 0.6)
    kept0 = steps[0][0]
    dropped_prefill = colsum.sum() - colsum[kept0.pos[kept0.pos >= 0]].sum()
    evicted_mass = 0.0
    for before, r, _ in steps:
        if r.evicted >= 0:
            n = before.count
            evicted_mass += before.score[r.evicted] + r.prob[r.evicted]
    total = st.score[st.pos >= 0].sum() + evicted_mass + dropped_prefill
    assert abs(total - (L + T)) < 1e-5


# ------------------------------------------------------------------ brute force
def brute_force_run(q, k, v, L, heavy, recent, scale, protected=frozenset(), rope_base=None):
    """Independent restatement on position sets with pure-Python arithmetic.

    Prefill: colsum by explicit double sums; the heavy set is found by evicting
    the lowest (score, position) candidate one at a time.  Decode: Algorithm 1
    taken literally, u = argmax_v F(S + {p} - {v}) with F the sum of scores,
    enumerated over every candidate v outside the recent window (ties: lowest
    position evicted).  `protected`: positions of a static pattern, never
    candidates (kept first at prefill).  `rope_base`: position rolling, every
    key rotated by its rank in the cache (counted here as the number of kept
    positions below it) and the query by the number of kept tokens, element
    pair (2i, 2i+1) by the angle rank * base^(-2i/D).
    """
    C = heavy + recent
    D = len(q[0])
    f32 = lambda x: float(np.float32(x))
    dot = lambda a, b: sum(a[d] * b[d] for d in range(D))

    def rot(x, r):
        if rope_base is None:
            return x
        y = list(x)
        for i in range(D // 2):
            a = r * rope_base ** (-2.0 * i / D)
            y[2 * i] = x[2 * i] * math.cos(a) - x[2 * i + 1] * math.sin(a)
            y[2 * i + 1] = x[2 * i] * math.sin(a) + x[2 * i + 1] * math.cos(a)
        return y

    score = {}
    if L:
        colsum = [0.0] * L
        for i in range(L):
            s = [scale * dot(q[i], k[j]) for j in range(i + 1)]
            mx = max(s)
            z = sum(math.exp(x - mx) for x in s)
            for j in range(i + 1):
                colsum[j] += math.exp(s[j] - mx) / z
        if L <= C:
            kept = set(range(L))
        else:
            cand = set(range(L - recent))
            while len(cand) > heavy:
                cand.remove(min(cand - set(protected), key=lambda j: (f32(colsum[j]), j)))
            kept = cand | set(range(L - recent, L))
        score = {j: f32(colsum[j]) for j in kept}
    outs, kept_sets, evictions = [], [], []
    for p in range(L, len(q)):
        S = sorted(score) + [p]
        n = len(S) - 1
        qr = rot(q[p], n)
        s = [scale * dot(qr, rot(k[j], sum(1 for i in S[:-1] if i < j) if j != p else n)) for j in S]
        mx = max(s)
        z = sum(math.exp(x - mx) for x in s)
        pr = [math.exp(x - mx) / z for x in s]
        outs.append([sum(pr[a] * v[j][d] for a, j in enumerate(S)) for d in range(D)])
        for a, j in enumerate(S[:-1]):
            score[j] = f32(score[j] + pr[a])
        ev = None
        if len(S) - 1 == C:
            cand = [j for j in S[:-1] if j <= p - recent and j not in protected]
            total = sum(score.values())
            best = max(total - score[j] for j in cand)
            ev = min(j for j in cand if total - score[j] == best)
            del score[ev]
        score[p] = f32(pr[-1])
        evictions.append(ev)
        kept_sets.append(set(score))
    return outs, kept_sets, evictions


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("L,heavy,recent", [(12, 3, 2), (5, 2, 3), (0, 2, 2), (9, 0, 2), (7, 4, 1)])
def test_against_position_set_brute_force(seed, L, heavy, recent):
    rng = np.random.default_rng(100 + seed)
    T, D = 40, 3
    mean = rng.standard_normal(D)
    q, k, v = rand_seq(rng, L + T, D, key_mean=mean)
    # a few repeated keys make heavy hitters and near ties likely
    k[rng.integers(0, L + T, 6)] = k[0]
    _, _, _, steps = run_pair(q, k, v, L, heavy, recent, 0.9)
    outs, kept_sets, evictions = brute_force_run(q.tolist(), k.tolist(), v.tolist(), L, heavy, recent, 0.9)
    for t, (before, r, after) in enumerate(steps):
        assert set(after.pos[after.pos >= 0].tolist()) == kept_sets[t]
        ev_pos = None if r.evicted < 0 else int(before.pos[r.evicted])
        assert ev_pos == evictions[t]
        np.testing.assert_allclose(r.out, outs[t], atol=1e-12)


def test_prefill_selection_brute_force():
    """Heavy set = top-Hh of the key (score, position) by a full lexicographic
    sort, which also equals Hh iterated lowest-key evictions."""
    rng = np.random.default_rng(8)
    for trial in range(20):
        L = int(rng.integers(10, 200))
        heavy = int(rng.integers(0, 12))
        recent = int(rng.integers(1, 12))
        colsum = rng.integers(0, 5, size=L).astype(np.float64) / 4  # many exact ties
        keep = O.select_prefill(colsum, L, heavy, recent)
        if L <= heavy + recent:
            assert keep == list(range(L))
            continue
        n = L - recent
        order = np.lexsort((np.arange(n), colsum[:n]))  # ascending (score, pos)
        top = sorted(order[n - heavy:].tolist()) if heavy else []
        assert keep == top + list(range(n, L))
        cand = list(range(n))
        while len(cand) > heavy:
            cand.remove(min(cand, key=lambda j: (colsum[j], j)))
        assert keep[:heavy] == cand


def test_tie_evicts_lowest_position():
    """Equal scores: the candidate with the lowest position is evicted."""
    D = 2
    C_heavy, recent = 3, 1
    st = O.empty_pair(C_heavy + recent, recent, D)
    st.count = 4
    st.p = 10
    st.pos[:] = [7, 2, 5, 9]
    st.score[:] = [0.5, 0.5, 0.5, 0.1]
    st.ring[:] = [3]
    st.head = 0
    q = np.zeros(D)  # uniform attention: every kept score rises by the same amount
    r = O.decode_step_pair(st, q, np.zeros(D), np.zeros(D), 1.0, C_heavy, recent)
    # candidates: pos <= 9 -> all four; slot 3 (pos 9, score 0.1 + 0.2) is lowest
    assert r.evicted == 3
    st2 = O.empty_pair(4, 1, D)
    st2.count, st2.p, st2.head = 4, 10, 0
    st2.pos[:] = [7, 2, 5, 9]
    st2.score[:] = [0.5, 0.5, 0.5, 0.9]
    st2.ring[:] = [3]
    r2 = O.decode_step_pair(st2, q, np.zeros(D), np.zeros(D), 1.0, C_heavy, recent)
    assert r2.evicted == 1  # equal lowest scores at pos 7, 2, 5 -> pos 2
    assert st2.pos[1] == 10 and st2.ring[0] == 1


def test_kv_cache_size_worked_example():
    """The report's sizing example (section 1.1): a 30B model (OPT-30B: 48
    layers, hidden 7168) at batch 128 and sequence 1024 holds ~180 GB of fp16
    K and V.  Pins the byte accounting used by the benchmark."""
    from kv_cache_eviction_03_gb300.accounting import kv_cache_bytes

    with open(os.path.join(GOLDEN, "kv_size_opt30b.txt")) as f:
        fields = {a.strip(): b.strip() for a, b in
                  (l.split("=") for l in (x.split("#")[0].strip() for x in f) if l)}
    b = kv_cache_bytes(int(fields["layers"]), int(fields["hidden"]), int(fields["batch"]),
                       int(fields["seq"]), int(fields["bytes_per_elem"]))
    assert round(b / 1e9) == int(fields["approx_gb"])


# ------------------------------------------------------------------ global selector
def _brute_force_global(q, k, heavy, recent, scale):
    """Global kept set by explicit loops: each row's softmax over its causal
    prefix, scores as sums down each column, and a candidate kept when fewer
    than `heavy` other candidates have a larger (score, position) key."""
    N = len(q)
    score = [0.0] * N
    for i in range(N):
        s = [scale * sum(a * b for a, b in zip(q[i], k[j])) for j in range(i + 1)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = sum(e)
        for j in range(i + 1):
            score[j] += e[j] / z
    if N <= heavy + recent:
        return list(range(N)), score
    n = N - recent
    f32 = [float(np.float32(x)) for x in score]
    kept = [j for j in range(n) if sum(1 for o in range(n) if (f32[o], o) > (f32[j], j)) < heavy]
    return kept + list(range(n, N)), score


@pytest.mark.parametrize("seed", range(8))
def test_global_select_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    N = int(rng.integers(1, 14))
    heavy, recent = int(rng.integers(0, 5)), int(rng.integers(1, 4))
    D = 3
    q, k, _ = rand_seq(rng, N, D, key_mean=rng.standard_normal(D))
    k[rng.integers(0, N, 3)] = k[0]  # repeated keys: heavy hitters and near ties
    kept, score = O.global_select_pair(q, k, heavy, recent, 0.8)
    bf_kept, bf_score = _brute_force_global(q.tolist(), k.tolist(), heavy, recent, 0.8)
    np.testing.assert_allclose(score, bf_score, rtol=1e-12)
    assert kept == bf_kept


def test_global_select_uniform_attention_keeps_the_earliest():
    """Equal keys: row i gives 1/(i+1) to every j <= i, so the scores are
    H_N - H_j (harmonic numbers), decreasing in j, and the global heavy
    hitters are the first `heavy` positions."""
    N, D, heavy, recent = 40, 4, 6, 5
    rng = np.random.default_rng(2)
    q = rng.standard_normal((N, D))
    k = np.tile(rng.standard_normal(D), (N, 1))
    kept, score = O.global_select_pair(q, k, heavy, recent, 0.5)
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, N + 1))])
    np.testing.assert_allclose(score, H[N] - H[np.arange(N)], rtol=1e-12)
    assert kept == list(range(heavy)) + list(range(N - recent, N))


@pytest.mark.parametrize("N,heavy,recent", [(0, 2, 2), (7, 4, 3), (5, 4, 3), (9, 0, 9)])
def test_global_select_within_budget_keeps_all(N, heavy, recent):
    rng = np.random.default_rng(N)
    q, k, _ = rand_seq(rng, N, 3)
    kept, _ = O.global_select_pair(q, k, heavy, recent, 0.7)
    assert kept == list(range(N))


def test_local_run_matches_global_under_uniform_attention():
    """Equal keys make every kept token receive the same probability each
    step, so the local rule never reorders the prompt's heavy hitters
    (scores H_L - H_j) and ends with the global set: full overlap."""
    L, T, D, heavy, recent = 30, 25, 4, 5, 4
    rng = np.random.default_rng(5)
    q = rng.standard_normal((L + T, D))
    k = np.tile(rng.standard_normal(D), (L + T, 1))
    v = rng.standard_normal((L + T, D))
    st, _, _, _ = run_pair(q, k, v, L, heavy, recent, 0.6)
    kept, _ = O.global_select_pair(q, k, heavy, recent, 0.6)
    local = sorted(int(x) for x in st.pos if x >= 0)
    assert local == kept == list(range(heavy)) + list(range(L + T - recent, L + T))
    assert O.heavy_overlap(local, kept, L + T, recent) == (heavy, heavy)


def test_heavy_overlap_counts_only_heavy_positions():
    assert O.heavy_overlap([0, 3, 5, 8, 9], [0, 4, 5, 8, 9], 10, 2) == (2, 3)
    assert O.heavy_overlap([8, 9], [8, 9], 10, 2) == (0, 0)


# ------------------------------------------------------------------ position rolling
def test_rope_rotation_closed_form_and_relative_property():
    """D = 2: the pair is rotated by exactly `position` radians (theta_0 = 1).
    Any D: rotations keep norms, and <R(m) q, R(n) k> = <q, R(n - m) k>."""
    x = np.array([[1.0, 0.0], [0.6, -0.8]])
    got = O.rope_rotate(x, [0.5, 2.0], 10000.0)
    want = np.array([[math.cos(0.5), math.sin(0.5)],
                     [0.6 * math.cos(2.0) + 0.8 * math.sin(2.0), 0.6 * math.sin(2.0) - 0.8 * math.cos(2.0)]])
    np.testing.assert_allclose(got, want, atol=1e-15)
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal((2, 16))
    for m, n in [(0, 0), (3, 11), (40, 7), (1000, 1003)]:
        a = float(O.rope_rotate(q[None], [m], 500.0)[0] @ O.rope_rotate(k[None], [n], 500.0)[0])
        b = float(q @ O.rope_rotate(k[None], [n - m], 500.0)[0])
        assert abs(a - b) < 1e-12
    np.testing.assert_allclose(np.linalg.norm(O.rope_rotate(q[None], [123], 500.0)), np.linalg.norm(q), rtol=1e-14)


def test_cache_ranks_count_smaller_positions():
    rng = np.random.default_rng(9)
    for _ in range(30):
        C = int(rng.integers(1, 20))
        pos = rng.permutation(100)[:C].astype(np.int64)
        pos[rng.random(C) < 0.3] = -1
        ranks = O.cache_ranks(pos)
        for j in range(C):
            want = -1 if pos[j] < 0 else int(np.sum((pos >= 0) & (pos < pos[j])))
            assert ranks[j] == want


def test_rolling_without_eviction_is_rotary_attention():
    """From an empty cache that never fills, every kept token's rank is its
    position, so each step is causal attention over rotary-embedded q and k
    at their text positions: checked against torch's fp64 attention on vectors
    rotated here as complex numbers."""
    T, D, heavy, recent, base = 14, 8, 10, 8, 100.0
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((3, T, D))
    st = O.empty_pair(heavy + recent, recent, D)
    outs = [O.decode_step_pair(st, q[t], k[t], v[t], 0.7, heavy, recent, rope_base=base).out for t in range(T)]

    ref = sdpa_causal(rotary_at(q, np.arange(T), base), rotary_at(k, np.arange(T), base), v, 0.7)
    np.testing.assert_allclose(np.stack(outs), ref, atol=1e-12)


@pytest.mark.parametrize("recent", [1, 5, 9])
def test_rolling_without_heavy_is_rotary_sliding_window(recent):
    """heavy = 0 with rolling on: past the fill the cache holds exactly the
    window p-recent..p-1 at ranks 0..recent-1 and the query sits at rank
    `recent`.  Rotary logits depend only on rank differences, which then equal
    text-position differences, so every step must be sliding-window attention
    over q and k rotated at their text positions (torch fp64, masked).  A
    query placed at its text position p, or keys at theirs, fails this once
    p > recent."""
    T, D, base = 40, 8, 50.0
    rng = np.random.default_rng(12)
    q, k, v = rng.standard_normal((3, T, D))
    st = O.empty_pair(recent, recent, D)
    outs = [O.decode_step_pair(st, q[t], k[t], v[t], 0.8, 0, recent, rope_base=base).out for t in range(T)]
    i, j = np.arange(T)[:, None], np.arange(T)[None, :]
    allowed = (j <= i) & (j >= i - recent)
    ref = sdpa_masked(rotary_at(q, np.arange(T), base), rotary_at(k, np.arange(T), base), v, 0.8, allowed)
    np.testing.assert_allclose(np.stack(outs), ref, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
@pytest.mark.parametrize("heavy,recent", [(3, 2), (4, 1), (2, 4)])
def test_rolling_after_evictions_brute_force(seed, heavy, recent):
    """heavy > 0 with rolling on, far past the fill (ranks and positions
    differ): outputs, kept sets and victims against the position-set brute
    force, which ranks every kept key by counting the kept positions below it
    and rotates with its own cos / sin loops."""
    rng = np.random.default_rng(300 + seed)
    T, D, base = 45, 4, 30.0
    q, k, v = rand_seq(rng, T, D, key_mean=rng.standard_normal(D))
    k[rng.integers(0, T, 5)] = k[1]
    _, _, _, steps = run_pair(q, k, v, 0, heavy, recent, 0.9, rope_base=base)
    outs, kept_sets, evictions = brute_force_run(q.tolist(), k.tolist(), v.tolist(), 0, heavy, recent, 0.9,
                                                 rope_base=base)
    moved = 0
    for t, (before, r, after) in enumerate(steps):
        assert set(after.pos[after.pos >= 0].tolist()) == kept_sets[t]
        ev_pos = None if r.evicted < 0 else int(before.pos[r.evicted])
        assert ev_pos == evictions[t]
        np.testing.assert_allclose(r.out, outs[t], atol=1e-12)
        moved += int(before.count < t)  # the query's rank n differs from its position t
    assert moved > 20


# ------------------------------------------------------------------ static pattern + heavy hitters
def test_static_pattern_positions():
    """Closed form of the three pattern families."""
    pos = np.arange(40)
    strided = O.StaticPattern(0, 4, 5)
    assert np.nonzero(strided.protects(pos))[0].tolist() == [0, 4, 8, 12, 16]
    fixed = O.StaticPattern(7, 8, 3)  # last position of each block of 8
    assert np.nonzero(fixed.protects(pos))[0].tolist() == [7, 15, 23]
    first = O.StaticPattern(0, 1, 4)
    assert np.nonzero(first.protects(pos))[0].tolist() == [0, 1, 2, 3]
    assert not O.StaticPattern(3, 2, 0).protects(pos).any()
    assert not strided.protects([-1]).any()
    with pytest.raises(ValueError):
        O.StaticPattern(0, 0, 3)


@pytest.mark.parametrize("pattern,L,recent", [((0, 5, 6), 40, 6), ((4, 5, 4), 33, 4), ((0, 1, 3), 20, 2)])
def test_static_pattern_filling_the_heavy_budget_is_sparse_attention(pattern, L, recent):
    """heavy == count with every pattern position inside the prompt's
    candidate region: the heavy budget holds only the pattern, so the cache is
    exactly the pattern plus the recent window at every step (the Sparse
    Transformer baseline of section 4.5 without heavy hitters), and each decode
    output equals torch fp64 attention over that key set plus the token
    itself."""
    sp = O.StaticPattern(*pattern)
    heavy = sp.count
    T, D = 30, 6
    rng = np.random.default_rng(21)
    q, k, v = rand_seq(rng, L + T, D, key_mean=rng.standard_normal(D))
    lattice = set(np.nonzero(sp.protects(np.arange(L + T)))[0].tolist())
    assert max(lattice) < L - recent
    st, _, _, steps = run_pair(q, k, v, L, heavy, recent, 0.7, pattern=sp)
    i, j = np.arange(L + T)[:, None], np.arange(L + T)[None, :]
    allowed = (j <= i) & ((j >= i - recent) | sp.protects(np.arange(L + T))[None, :])
    ref = sdpa_masked(q, k, v, 0.7, allowed)
    for t, (before, r, after) in enumerate(steps):
        p = L + t
        assert set(before.pos[before.pos >= 0].tolist()) == lattice | set(range(p - recent, p))
        np.testing.assert_allclose(r.out, ref[p], atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("pattern,L,heavy,recent", [((0, 3, 2), 12, 3, 2), ((2, 3, 3), 9, 4, 2),
                                                    ((0, 1, 2), 0, 3, 2), ((1, 4, 4), 14, 4, 1)])
def test_static_pattern_against_position_set_brute_force(seed, pattern, L, heavy, recent):
    """Static pattern + heavy hitters against the brute force with protected
    positions (never candidates, kept first at prefill); pattern positions
    also arrive during decode and become protected once they leave the
    recent window."""
    sp = O.StaticPattern(*pattern)
    rng = np.random.default_rng(200 + seed)
    T, D = 40, 3
    q, k, v = rand_seq(rng, L + T, D, key_mean=rng.standard_normal(D))
    k[rng.integers(0, L + T, 6)] = k[0]
    _, _, _, steps = run_pair(q, k, v, L, heavy, recent, 0.9, pattern=sp)
    prot = frozenset(np.nonzero(sp.protects(np.arange(L + T)))[0].tolist())
    outs, kept_sets, evictions = brute_force_run(q.tolist(), k.tolist(), v.tolist(), L, heavy, recent, 0.9,
                                                 protected=prot)
    for t, (before, r, after) in enumerate(steps):
        assert set(after.pos[after.pos >= 0].tolist()) == kept_sets[t]
        assert prot & set(range(L + t + 1)) <= kept_sets[t]  # a pattern position is never evicted
        ev_pos = None if r.evicted < 0 else int(before.pos[r.evicted])
        assert ev_pos == evictions[t]
        np.testing.assert_allclose(r.out, outs[t], atol=1e-12)


def test_static_pattern_prefill_selection_brute_force():
    """Pattern positions below L-recent are all kept; the rest of the heavy
    budget goes to the top keys (score, position) of the other positions,
    which also equals iterated lowest-key evictions among non-pattern ones."""
    rng = np.random.default_rng(18)
    for trial in range(30):
        L = int(rng.integers(10, 150))
        heavy = int(rng.integers(0, 12))
        recent = int(rng.integers(1, 12))
        sp = O.StaticPattern(int(rng.integers(0, 6)), int(rng.integers(1, 9)), int(rng.integers(0, heavy + 1)))
        colsum = rng.integers(0, 5, size=L).astype(np.float64) / 4  # many exact ties
        keep = O.select_prefill(colsum, L, heavy, recent, sp)
        if L <= heavy + recent:
            assert keep == list(range(L))
            continue
        n = L - recent
        prot = set(np.nonzero(sp.protects(np.arange(n)))[0].tolist())
        cand = list(range(n))
        while len(cand) > heavy:
            cand.remove(min((j for j in cand if j not in prot), key=lambda j: (colsum[j], j)))
        assert keep[:heavy] == cand and prot <= set(cand)
        assert keep[heavy:] == list(range(n, L))


def test_empty_static_pattern_is_plain_h2o():
    rng = np.random.default_rng(4)
    L, T, D, heavy, recent = 30, 25, 4, 5, 4
    q, k, v = rand_seq(rng, L + T, D, key_mean=rng.standard_normal(D))
    a = run_pair(q, k, v, L, heavy, recent, 0.8)[3]
    b = run_pair(q, k, v, L, heavy, recent, 0.8, pattern=O.StaticPattern(0, 3, 0))[3]
    for (_, ra, sa), (_, rb, sb) in zip(a, b):
        assert ra.evicted == rb.evicted and np.array_equal(ra.out, rb.out) and np.array_equal(sa.pos, sb.pos)
