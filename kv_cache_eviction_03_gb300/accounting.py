"""Byte and FLOP accounting for the H2O decode / prefill path.

Algorithmic bytes count only what the method has to move: the kept K/V rows
(not the full-length cache the budget avoids), the per-slot score (read and
written) and position (read), the new token's q / k / v (read), the new K/V
row written into the freed slot, and the float32 output.
"""
from __future__ import annotations


def kv_cache_bytes(layers: int, hidden: int, batch: int, seq: int, elem_bytes: int) -> int:
    """Full (unevicted) KV cache size: K and V, every layer, every token."""
    return 2 * layers * hidden * batch * seq * elem_bytes


def decode_step_bytes(pairs: int, slots: int, head_dim: int, elem_bytes: int) -> int:
    """Algorithmic HBM bytes of one decode step of one attention layer.

    Per (batch, head) pair with a full cache of `slots` entries:
      K and V rows read            2 * slots * head_dim * e
      score read + write           8 * slots
      position read                4 * slots
      q, k_new, v_new read         3 * head_dim * e
      new K/V row written          2 * head_dim * e
      output written (float32)     4 * head_dim
    """
    per_pair = (2 * slots * head_dim * elem_bytes + 12 * slots
                + 5 * head_dim * elem_bytes + 4 * head_dim)
    return pairs * per_pair


def prefill_flops(pairs: int, prompt: int, head_dim: int, with_output: bool = True) -> float:
    """Tensor-core FLOPs of the prefill: causal q.k twice (row statistics and
    column sums) plus p.v once when the attention output is produced."""
    causal = prompt * (prompt + 1) / 2
    passes = 3 if with_output else 2
    return 2.0 * pairs * causal * head_dim * passes
