"""Plain fp64 CPU oracle for H2O (Heavy-Hitter Oracle) KV-cache eviction.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the timed CPU
baseline of the benchmark do.  It shares no code with the CUDA library.

Everything is computed per (batch, head) pair, in float64, step by step in the
order the method states it.  Sources (page title, then section):

* "H2O ... 深度解读报告" (zako-mio knowledge base), section 3.1: budgeted
  generation; at most one eviction per step; evicted entries leave the softmax
  normaliser.
* same page, section 3.3 (Definition 4.3 / Algorithm 1): S_i = (S_{i-1} + {i})
  minus {u}, u = argmax_v F_score(S_{i-1} + {i} - {v}); only grow while i <= k;
  F_score is the accumulated attention a token has received.
* same page, section 3.4: preallocated cache overwritten in place; cache =
  heavy-hitter region + recent region kept as a circular queue; prefill keeps
  heavy + recent when the prompt is longer than the cache, else keeps all;
  each decode step the oldest recent entry leaves the recent region and one
  heavy-hitter per head is evicted to make room for the newest token.
* same page, section 2.3, and "H2O" (phantomic12 inference-research notes):
  the score is the running sum of the attention probability each token
  receives, lowest-scoring entry evicted when full, recent window kept.
* same page, section 2.3 (its Figure 2(d) comparison): the online ("local")
  rule set against a global one that may use the whole sequence's attention,
  future rows included (global_select_pair, heavy_overlap).
* same page, section 4.4 (Q1, infinite streaming "with position rolling"):
  rotary position embedding applied with positions counted inside the cache
  rather than in the text (rope_rotate, cache_ranks, decode_step_pair with
  rope_base).
* same page, section 4.5 (Table 2: Sparse Transformer strided / fixed
  patterns combined with heavy hitters): positions chosen by a fixed pattern
  are kept for good, the heavy hitters fill the rest of the heavy budget
  (StaticPattern, the `pattern` argument of select_prefill, prefill_pair and
  decode_step_pair).

Readings taken where the pages are loose (each also listed in the design
notes): the score is the column sum of attention probabilities (the report's
"row sum" cannot rank tokens, every softmax row sums to 1); the new token
attends to itself, scores are updated with this step's probabilities and only
then is the victim chosen; the victim is the minimum of the key
(score, position) over kept tokens at position <= p - R, i.e. lowest position
on equal scores; the newcomer's score starts at its own probability; the
score buffer is float32 (values are rounded to float32 when stored); slot ids
are canonical: prefill lays heavy hitters in ascending position into slots
0..Hh-1 and the recent tokens into slots Hh..C-1, and every decode step writes
the newcomer into the slot it frees.

Parity pins for each function live in tests/test_oracle_pins.py; no function
here is parity unpinned.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def to_f32(x):
    """Round float64 values to the float32 score buffer, back as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- prefill
def causal_attention_stats(q, k, v, scale):
    """Full causal attention over one pair's prompt (section 3.1, 3.3).

    q, k, v: float64 [L, D].  Returns (lse [L], colsum [L], O [L, D]) with
    s_ij = scale * q_i . k_j for j <= i, p_ij = softmax_j(s_ij),
    lse_i = log sum_j exp(s_ij), colsum_j = sum_{i >= j} p_ij (the accumulated
    attention token j has received after the prompt), O_i = sum_j p_ij v_j.
    """
    L = q.shape[0]
    s = q @ k.T
    s *= scale
    s[np.triu_indices(L, k=1)] = -np.inf  # token i sees positions j <= i only
    m = s.max(axis=1, keepdims=True)
    s -= m
    p = np.exp(s, out=s)  # in place: the [L, L] matrix is the large one
    z = p.sum(axis=1, keepdims=True)
    p /= z
    lse = (m + np.log(z))[:, 0]
    colsum = p.sum(axis=0)
    out = p @ v
    return lse, colsum, out


# --------------------------------------------------------------------------- static pattern
@dataclass(frozen=True)
class StaticPattern:
    """Positions a fixed sparse pattern keeps for good (section 4.5, Table 2:
    Sparse Transformer strided / fixed patterns plus heavy hitters).

    Reading (the pages give the combination's accuracy only, not how the two
    share a budget): the protected positions are offset, offset + stride, ...,
    offset + (count - 1) * stride.  They occupy heavy-budget slots (count <=
    heavy) and are never eviction candidates; the heavy hitters take the
    remaining heavy slots.  offset 0 gives the strided lattice, offset
    stride - 1 the fixed pattern's block-summary positions (the last position
    of each block of `stride`), stride 1 the first `count` tokens.
    """

    offset: int
    stride: int
    count: int

    def __post_init__(self):
        if self.offset < 0 or self.stride < 1 or self.count < 0:
            raise ValueError("static pattern needs offset >= 0, stride >= 1, count >= 0")

    def protects(self, pos):
        """Boolean array: which of the positions `pos` are protected."""
        pos = np.asarray(pos, dtype=np.int64)
        d = pos - self.offset
        return (self.count > 0) & (d >= 0) & (d % self.stride == 0) & (d // self.stride < self.count)


def _protected(pattern, pos):
    pos = np.asarray(pos, dtype=np.int64)
    return np.zeros(pos.shape, dtype=bool) if pattern is None else pattern.protects(pos)


def select_prefill(colsum, L, heavy, recent, pattern=None):
    """Positions kept after a prompt of length L, in slot order (section 3.4).

    L <= heavy + recent: every position, slot j holds position j.
    Otherwise: the recent window is positions L-recent..L-1; the heavy hitters
    are the `heavy` largest keys (score, position) among positions < L-recent,
    where score is colsum as stored in the float32 buffer.  Slots 0..heavy-1
    hold the heavy hitters in ascending position, then the recent window.
    With a static pattern (section 4.5) its positions below L-recent are kept
    first and the heavy hitters fill the remaining heavy slots.
    """
    C = heavy + recent
    if L <= C:
        return list(range(L))
    n = L - recent
    score = to_f32(colsum[:n])
    prot = _protected(pattern, np.arange(n))
    free = np.nonzero(~prot)[0]
    take = heavy - int(prot.sum())
    assert take >= 0, "a static pattern holds at most `heavy` positions"
    ascending = free[np.lexsort((free, score[free]))]  # by score, then position
    heavy_pos = sorted(np.nonzero(prot)[0].tolist() + (ascending[free.size - take:].tolist() if take else []))
    return heavy_pos + list(range(n, L))


@dataclass
class PairState:
    """One pair's preallocated cache (section 3.4): C slots + recent ring."""

    K: np.ndarray  # [C, D] float64 (values exact in the K/V dtype)
    V: np.ndarray  # [C, D]
    score: np.ndarray  # [C] float64 holding float32 values
    pos: np.ndarray  # [C] int64, -1 = empty
    ring: np.ndarray  # [R] int64 slot ids of the recent window, -1 = empty
    head: int  # ring index the next token goes to (its entry is the oldest)
    count: int  # occupied slots (slots 0..count-1)
    p: int  # absolute position of the next token

    def copy(self) -> "PairState":
        return PairState(self.K.copy(), self.V.copy(), self.score.copy(), self.pos.copy(),
                         self.ring.copy(), self.head, self.count, self.p)


def empty_pair(C, R, D) -> PairState:
    return PairState(np.zeros((C, D)), np.zeros((C, D)), np.zeros(C),
                     np.full(C, -1, dtype=np.int64), np.full(R, -1, dtype=np.int64), 0, 0, 0)


def prefill_pair(q, k, v, heavy, recent, scale, pattern=None):
    """Prefill one pair: attention stats, keep rule, cache laid out in slots."""
    L, D = k.shape
    C = heavy + recent
    st = empty_pair(C, recent, D)
    if L == 0:
        return st, np.zeros((0,)), np.zeros((0, D))
    lse, colsum, out = causal_attention_stats(q, k, v, scale)
    keep = select_prefill(colsum, L, heavy, recent, pattern)
    n = len(keep)
    st.K[:n] = k[keep]
    st.V[:n] = v[keep]
    st.score[:n] = to_f32(colsum[keep])
    st.pos[:n] = keep
    st.count = n
    st.p = L
    # recent ring: oldest recent token first; the next token goes to `head`
    if L >= recent:
        for r in range(recent):
            st.ring[r] = keep.index(L - recent + r)
        st.head = 0
    else:
        for r in range(L):
            st.ring[r] = keep.index(r)
        st.head = L
    return st, colsum, out


# --------------------------------------------------------------------------- global selector
def global_select_pair(q, k, heavy, recent, scale):
    """Global (offline) heavy hitters of one pair's whole sequence.

    Section 2.3 compares the online rule, which only ever sums the attention
    each token has received so far, with a global rule that may look at the
    whole sequence.  Reading: token j's global score is the attention it
    receives from every row of the sequence, sum_{i >= j} softmax_i(s_ij)
    over all N rows (the prefill column sum taken over the whole sequence),
    and the global kept set is the prefill keep rule applied to those
    scores: the last `recent` positions plus the `heavy` largest keys
    (score, position) before them.  q, k: float64 [N, D].
    Returns (kept positions in ascending order, scores [N]).
    """
    N = q.shape[0]
    if N == 0:
        return [], np.zeros((0,))
    _, colsum, _ = causal_attention_stats(q, k, np.zeros((N, 1)), scale)
    return sorted(select_prefill(colsum, N, heavy, recent)), colsum


def heavy_overlap(local_pos, global_pos, n, recent):
    """Share of the global heavy hitters that a local run also kept.

    Both sets hold the same recent window (positions n-recent..n-1); the heavy
    hitters are the kept positions before it.  Returns (shared, of): `of` is
    the number of global heavy hitters, `shared` how many of them the local
    set holds too (1.0 drift-free when shared == of).
    """
    lh = {int(x) for x in local_pos if 0 <= x < n - recent}
    gh = {int(x) for x in global_pos if 0 <= x < n - recent}
    return len(lh & gh), len(gh)


# --------------------------------------------------------------------------- position rolling
def rope_rotate(x, positions, base):
    """Rotary position embedding (Su et al., RoFormer, 2021): the element pair
    (2i, 2i+1) of each row is rotated by the angle position * base^(-2i/D).
    x: [n, D] float64, positions: [n]."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[:, 0::2] = x[:, 0::2] * c - x[:, 1::2] * s
    out[:, 1::2] = x[:, 0::2] * s + x[:, 1::2] * c
    return out


def cache_ranks(pos):
    """Position inside the cache of every kept slot: its rank among the kept
    tokens ordered by their position in the text (-1 for an empty slot).
    Reading of "position rolling" (section 4.4): the kept tokens are numbered
    0..n-1 in text order, the token being generated gets n."""
    pos = np.asarray(pos)
    ranks = np.full(pos.shape, -1, dtype=np.int64)
    kept = np.nonzero(pos >= 0)[0]
    ranks[kept[np.argsort(pos[kept], kind="stable")]] = np.arange(kept.size)
    return ranks


# --------------------------------------------------------------------------- decode
@dataclass
class StepResult:
    out: np.ndarray  # [D] attention output of the new token
    evicted: int  # slot freed this step, -1 while the cache is filling
    gap: float  # difference of the two lowest candidate scores (inf if < 2)
    prob: np.ndarray  # [count + 1] probabilities (kept slots, then self)


def decode_step_pair(st: PairState, q, k_new, v_new, scale, heavy, recent, rope_base=None,
                     pattern=None) -> StepResult:
    """One decode step of one pair, in place on `st` (sections 3.1, 3.3, 3.4).

    With rope_base (position rolling, section 4.4) the logits are taken
    between rotary-embedded vectors, each kept key at its rank inside the
    cache (cache_ranks) and the query and the new key at n, the number of
    kept tokens; the cache stores the keys as given (not rotated).
    With a static pattern (section 4.5) its positions are never candidates.

    1. attend over the kept slots and the new token itself; the softmax
       normaliser covers only those entries;
    2. add each kept slot's probability to its accumulated score;
    3. if the cache is full, evict the kept slot with the lowest
       (score, position) among positions <= p - recent (the heavy hitters and
       the token that just left the recent window); otherwise take the next
       free slot;
    4. write the new token's K/V, score (its own probability) and position into
       that slot and append the slot to the recent ring.
    """
    C = heavy + recent
    n = st.count
    p = st.p
    logits = np.empty(n + 1)
    if rope_base is None:
        logits[:n] = scale * (st.K[:n] @ q)
        logits[n] = scale * float(k_new @ q)
    else:
        qr = rope_rotate(np.asarray(q)[None, :], [n], rope_base)[0]
        kr = rope_rotate(st.K[:n], cache_ranks(st.pos[:n]), rope_base)
        logits[:n] = scale * (kr @ qr)
        logits[n] = scale * float(rope_rotate(np.asarray(k_new)[None, :], [n], rope_base)[0] @ qr)
    m = logits.max()
    e = np.exp(logits - m)
    prob = e / e.sum()
    out = prob[:n] @ st.V[:n] + prob[n] * v_new

    st.score[:n] = to_f32(st.score[:n] + prob[:n])

    gap = np.inf
    if n < C:
        u = n
        evicted = -1
        st.count = n + 1
    else:
        cand = np.nonzero((st.pos[:C] <= p - recent) & ~_protected(pattern, st.pos[:C]))[0]
        ranked = cand[np.lexsort((st.pos[cand], st.score[cand]))]  # by score, then position
        u = int(ranked[0])
        evicted = u
        if ranked.size > 1:
            gap = st.score[ranked[1]] - st.score[ranked[0]]

    st.K[u] = k_new
    st.V[u] = v_new
    st.score[u] = to_f32(prob[n])
    st.pos[u] = p
    st.ring[st.head] = u
    st.head = (st.head + 1) % recent
    st.p = p + 1
    return StepResult(out, evicted, gap, prob)


# --------------------------------------------------------------------------- batched drivers
@dataclass
class CacheState:
    """All pairs of a cache; arrays carry a leading pair axis P = B*H."""

    K: np.ndarray  # [P, C, D]
    V: np.ndarray
    score: np.ndarray  # [P, C]
    pos: np.ndarray  # [P, C]
    ring: np.ndarray  # [P, R]
    head: np.ndarray  # [P]
    count: np.ndarray  # [P]
    p: np.ndarray  # [P]

    def pair(self, i) -> PairState:
        return PairState(self.K[i].copy(), self.V[i].copy(), self.score[i].copy(),
                         self.pos[i].copy(), self.ring[i].copy(), int(self.head[i]),
                         int(self.count[i]), int(self.p[i]))

    def copy(self) -> "CacheState":
        return CacheState(*(a.copy() for a in (self.K, self.V, self.score, self.pos,
                                                self.ring, self.head, self.count, self.p)))

    @staticmethod
    def stack(pairs) -> "CacheState":
        return CacheState(np.stack([s.K for s in pairs]), np.stack([s.V for s in pairs]),
                          np.stack([s.score for s in pairs]), np.stack([s.pos for s in pairs]),
                          np.stack([s.ring for s in pairs]),
                          np.array([s.head for s in pairs]), np.array([s.count for s in pairs]),
                          np.array([s.p for s in pairs]))


def _pairs(x):
    x = np.asarray(x, dtype=np.float64)
    return x.reshape((-1,) + x.shape[2:])


def empty_cache(pairs, heavy, recent, head_dim) -> CacheState:
    return CacheState.stack([empty_pair(heavy + recent, recent, head_dim) for _ in range(pairs)])


def prefill(q, k, v, heavy, recent, scale, pattern=None):
    """Prefill every pair.  q, k, v: [B, H, L, D].  Returns (state, colsum, O)."""
    q, k, v = _pairs(q), _pairs(k), _pairs(v)
    states, colsums, outs = [], [], []
    for i in range(q.shape[0]):
        st, cs, o = prefill_pair(q[i], k[i], v[i], heavy, recent, scale, pattern)
        states.append(st)
        colsums.append(cs)
        outs.append(o)
    return CacheState.stack(states), np.stack(colsums), np.stack(outs)


def decode_step(state: CacheState, q, k_new, v_new, heavy, recent, scale, rope_base=None, pattern=None):
    """One decode step for every pair.  q, k_new, v_new: [B, H, D].

    Returns (new_state, out [P, D], evicted [P], gap [P]); `state` is untouched.
    rope_base: position rolling (see decode_step_pair), None for none.
    pattern: a StaticPattern (see decode_step_pair), None for none.
    """
    q, k_new, v_new = _pairs(q), _pairs(k_new), _pairs(v_new)
    new_pairs, outs, ev, gaps = [], [], [], []
    for i in range(q.shape[0]):
        st = state.pair(i)
        r = decode_step_pair(st, q[i], k_new[i], v_new[i], scale, heavy, recent, rope_base, pattern)
        new_pairs.append(st)
        outs.append(r.out)
        ev.append(r.evicted)
        gaps.append(r.gap)
    return CacheState.stack(new_pairs), np.stack(outs), np.array(ev), np.array(gaps)
