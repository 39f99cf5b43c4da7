"""Seeded synthetic inputs for the H2O decode / prefill path.

This module only draws random inputs; it holds none of the method's
arithmetic (no attention, no scores, no eviction).  Both the CUDA path and the
CPU oracle consume what it returns, so it is the one place they share.

Recipe (the pages describe padded synthetic prompts, XSUM and PG-19 streaming;
none of those datasets is used, these draws stand in for them):

* token ids: rank r ~ Zipf(s) on {1..50272} (P(r) proportional to r^-s), drawn by
  inverse CDF; id = r - 1.  One id per (batch row, position), shared by all
  heads.  Repeated ids share a key mean, which imitates the word
  co-occurrence effect behind heavy hitters (H2O report, section 2.2).
* E: per-head embedding table, E[h][id][d] ~ N(0,1), produced by a
  counter-based generator (SplitMix64 of (seed, h, id, d), Box-Muller), so any
  row can be drawn on its own without materialising the 50272-row table.
* k_t = 0.5 * E[h][id_t] + N(0,1); v_t ~ N(0,1); q_t ~ N(0,1).
* every value is drawn in float64, rounded to float32, then to the K/V dtype
  (round to nearest even each time).
* decode step t of a stream draws from a generator keyed by the absolute
  position, i.e. the seed is advanced per step.

`device_*` helpers draw the same recipe with torch's CUDA generator; they are
used for the large timed workloads, where the exact values do not matter and
only the distribution and shapes do.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

VOCAB = 50272
KEY_MEAN_WEIGHT = 0.5
BASE_SEED = 20230614

_KIND = {"q": 1, "k": 2, "v": 3, "ids": 4, "qd": 5, "kd": 6, "vd": 7}


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    head_dim: int
    dtype: str  # "f16" or "f32"
    prompt: int
    decode: int
    heavy: int
    recent: int
    zipf_s: float
    layers: int = 1  # attention layers of the model shape (cold-L2 rotation)

    @property
    def cache_slots(self) -> int:
        return self.heavy + self.recent

    @property
    def pairs(self) -> int:
        return self.batch * self.heads

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))

    @property
    def np_dtype(self):
        return np.float16 if self.dtype == "f16" else np.float32

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the method is measured on (sizes fixed by the task):
WORKLOADS = {
    "tiny-ref": Workload("tiny-ref", 1, 4, 64, "f32", 256, 64, 26, 26, 1.1, 1),
    "opt-6.7b": Workload("opt-6.7b", 8, 32, 128, "f16", 2048, 256, 205, 205, 1.1, 32),
    "opt-30b": Workload("opt-30b", 64, 56, 128, "f16", 512, 32, 51, 51, 1.2, 48),
    "llama-7b-16k": Workload("llama-7b-16k", 1, 32, 128, "f16", 16384, 1024, 820, 820, 1.1, 32),
    "streaming": Workload("streaming", 4, 32, 128, "f16", 0, 1_000_000, 1024, 1024, 1.1, 32),
}
WORKLOAD_ORDER = ["tiny-ref", "opt-6.7b", "opt-30b", "llama-7b-16k", "streaming"]


def seed_for(name: str) -> int:
    return BASE_SEED + WORKLOAD_ORDER.index(name) if name in WORKLOAD_ORDER else BASE_SEED


# ---------------------------------------------------------------- SplitMix64
_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014) on uint64."""
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def _uniform01(bits: np.ndarray) -> np.ndarray:
    # top 53 bits, shifted by half an ulp so the value is in (0, 1)
    return ((bits >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def embedding_rows(seed: int, head: int, ids: np.ndarray, dim: int) -> np.ndarray:
    """E[head][ids] as float64 [..., dim], counter-based (random access)."""
    ids = np.asarray(ids, dtype=np.uint64)
    d = np.arange(dim, dtype=np.uint64)
    with np.errstate(over="ignore"):
        key = _splitmix64(np.uint64(seed) * np.uint64(0x100000001B3) + np.uint64(head + 1))
        ctr = (ids[..., None] * np.uint64(dim) + d) * np.uint64(2)
        u1 = _uniform01(_splitmix64(key ^ ctr))
        u2 = _uniform01(_splitmix64(key ^ (ctr + np.uint64(1))))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


# ---------------------------------------------------------------- Zipf ids
_ZIPF_CDF: dict = {}


def _zipf_cdf(s: float) -> np.ndarray:
    if s not in _ZIPF_CDF:
        r = np.arange(1, VOCAB + 1, dtype=np.float64)
        w = r ** (-s)
        c = np.cumsum(w)
        _ZIPF_CDF[s] = c / c[-1]
    return _ZIPF_CDF[s]


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def token_ids(w: Workload, seed: int, layer: int, positions: np.ndarray) -> np.ndarray:
    """Zipf token ids, int64 [batch, len(positions)]; one stream per position."""
    positions = np.asarray(positions, dtype=np.int64)
    out = np.empty((w.batch, positions.size), dtype=np.int64)
    cdf = _zipf_cdf(w.zipf_s)
    # one generator per 4096-position block keeps long streams cheap and any
    # position reproducible on its own
    blocks = positions // 4096
    for blk in np.unique(blocks):
        sel = np.nonzero(blocks == blk)[0]
        u = _rng(seed, _KIND["ids"], layer, int(blk)).random((w.batch, 4096))
        ranks = np.searchsorted(cdf, u[:, positions[sel] - blk * 4096], side="left")
        out[:, sel] = np.minimum(ranks, VOCAB - 1)
    return out


def _round(x: np.ndarray, dtype) -> np.ndarray:
    return x.astype(np.float32).astype(dtype)


def _key_means(w: Workload, seed: int, ids: np.ndarray) -> np.ndarray:
    """0.5 * E[h][id] for every head: float64 [H, *ids.shape, D]."""
    uniq, inv = np.unique(ids, return_inverse=True)
    out = np.empty((w.heads,) + ids.shape + (w.head_dim,))
    for h in range(w.heads):
        rows = KEY_MEAN_WEIGHT * embedding_rows(seed, h, uniq, w.head_dim)
        out[h] = rows[inv.reshape(ids.shape)]
    return out


def prefill_inputs(w: Workload, seed: int | None = None, layer: int = 0):
    """q, k, v for the prompt: arrays [B, H, L, D] in the K/V dtype."""
    seed = seed_for(w.name) if seed is None else seed
    B, H, L, D = w.batch, w.heads, w.prompt, w.head_dim
    t = w.np_dtype
    ids = token_ids(w, seed, layer, np.arange(L))
    q, k, v = (np.empty((B, H, L, D), dtype=t) for _ in range(3))
    gq, gk, gv = (_rng(seed, _KIND[x], layer) for x in ("q", "k", "v"))
    # drawn one batch row at a time (same stream order as one [B,H,L,D] draw)
    for b in range(B):
        q[b] = _round(gq.standard_normal((H, L, D)), t)
        mean = _key_means(w, seed, ids[b])  # [H, L, D]
        k[b] = _round(gk.standard_normal((H, L, D)) + mean, t)
        v[b] = _round(gv.standard_normal((H, L, D)), t)
    return q, k, v


def decode_inputs(w: Workload, position: int, seed: int | None = None, layer: int = 0):
    """q, k_new, v_new for the token at absolute `position`: arrays [B, H, D]."""
    seed = seed_for(w.name) if seed is None else seed
    B, H, D = w.batch, w.heads, w.head_dim
    ids = token_ids(w, seed, layer, np.array([position]))[:, 0]  # [B]
    q = _rng(seed, _KIND["qd"], layer, position).standard_normal((B, H, D))
    k = _rng(seed, _KIND["kd"], layer, position).standard_normal((B, H, D))
    k += np.moveaxis(_key_means(w, seed, ids), 0, 1)  # [B, H, D]
    v = _rng(seed, _KIND["vd"], layer, position).standard_normal((B, H, D))
    t = w.np_dtype
    return _round(q, t), _round(k, t), _round(v, t)


def decode_sequence(w: Workload, start: int, steps: int, seed: int | None = None, layer: int = 0):
    """Stacked decode inputs for positions start..start+steps-1: [T, B, H, D] each."""
    qs, ks, vs = [], [], []
    for t in range(steps):
        q, k, v = decode_inputs(w, start + t, seed, layer)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    return np.stack(qs), np.stack(ks), np.stack(vs)


# ---------------------------------------------------------------- device draws
class DeviceDraws:
    """The same recipe drawn on the GPU with torch's generator, one layer's
    prompt or one chunk of decode steps at a time (timed workloads).  The
    per-head key-mean table E is drawn once per object."""

    def __init__(self, w: Workload, seed: int, device="cuda"):
        import torch

        self.w, self.device = w, device
        self.g = torch.Generator(device=device)
        self.g.manual_seed(seed)
        self.tdt = torch.float16 if w.dtype == "f16" else torch.float32
        self.cdf = torch.from_numpy(_zipf_cdf(w.zipf_s)).to(device)
        self.table = torch.randn((w.heads, VOCAB, w.head_dim), generator=self.g, device=device, dtype=torch.float32)
        self.hidx = torch.arange(w.heads, device=device)

    def _normal(self, shape):
        import torch

        return torch.randn(shape, generator=self.g, device=self.device)

    def _keys(self, n_pos, rows):
        """k = 0.5 * E[h][id] + N(0,1) for `rows` x n_pos Zipf ids: [rows, H, n, D] float32."""
        import torch

        u = torch.rand((rows, n_pos), generator=self.g, device=self.device, dtype=torch.float64)
        ids = torch.searchsorted(self.cdf, u).clamp_(max=VOCAB - 1)
        mean = self.table[self.hidx[None, :, None], ids[:, None, :]]
        return KEY_MEAN_WEIGHT * mean + self._normal((rows, self.w.heads, n_pos, self.w.head_dim))

    def prefill(self):
        """q, k, v [B, H, L, D] in the K/V dtype."""
        w = self.w
        shp = (w.batch, w.heads, w.prompt, w.head_dim)
        q = self._normal(shp).to(self.tdt)
        k = self._keys(w.prompt, w.batch).to(self.tdt)
        v = self._normal(shp).to(self.tdt)
        return q, k, v

    def decode(self, steps, layers=1):
        """q, k_new, v_new [steps, layers, B, H, D] in the K/V dtype."""
        w = self.w
        shp = (steps, layers, w.batch, w.heads, w.head_dim)
        q = self._normal(shp).to(self.tdt)
        k = self._keys(steps * layers, w.batch).reshape(w.batch, w.heads, steps, layers, w.head_dim)
        k = k.permute(2, 3, 0, 1, 4).contiguous().to(self.tdt)
        v = self._normal(shp).to(self.tdt)
        return q, k, v


def device_inputs(w: Workload, seed: int, layers: int, device="cuda"):
    """Same recipe drawn on the GPU with torch's generator (timed workloads).

    Returns dict with 'prefill' -> list of (q, k, v) [B, H, L, D] and
    'decode' -> list of (q, k, v) [T, B, H, D], one entry per layer, all in the
    K/V dtype and resident on `device`.
    """
    d = DeviceDraws(w, seed, device)
    out = {"prefill": [], "decode": []}
    for _ in range(layers):
        if w.prompt > 0:
            out["prefill"].append(d.prefill())
        q, k, v = d.decode(w.decode, 1)
        out["decode"].append((q[:, 0], k[:, 0], v[:, 0]))
    del d
    return out
