"""Speed-of-light byte accounting for one decode step.

The pages' model ("The delay is between operations" on the One-Kernel Server
page; the numbers paragraph of "Inside the Megakernel Serving Engine"; the
byte paragraph of "Cohere fuses an entire decode step into one GPU program"):
a batch-1 decode step must stream the active weights once plus the KV cache,
so tok/s <= HBM bandwidth / (active weight bytes + KV bytes).

``step_bytes`` counts what this decode step must move at its shapes: every
attention/router/norm weight, each selected expert once per layer even when
several requests picked it (the union), the LM head, the embedding rows
actually read, the K/V read for every cached token plus the new one, the
new token's K/V written back, and the logits when they are requested.
"""
from __future__ import annotations

from typing import Optional, Sequence


def step_bytes(dims, ctx: Sequence[int], union_per_layer: Optional[Sequence[int]] = None,
               logits: bool = False) -> dict:
    L, H = dims.n_layers, dims.hidden
    nq, nkv, d = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    E, F, V = dims.n_experts, dims.expert_ffn, dims.vocab
    B = len(ctx)
    if union_per_layer is None:
        union_per_layer = [min(E, B * dims.top_k)] * L
    assert len(union_per_layer) == L
    dense = 2 * (H * (nq + 2 * nkv) * d + nq * d * H + H * E + 2 * H)
    weights = L * dense + sum(2 * u * 3 * H * F for u in union_per_layer)
    weights += 2 * (V * H + H) + 2 * B * H
    per_tok = L * 2 * nkv * d * 2
    kv_read = sum((c + 1) * per_tok for c in ctx)
    kv_append = B * per_tok
    lg = 4 * B * V if logits else 0
    return {"weights": weights, "kv_read": kv_read, "kv_append": kv_append, "logits": lg,
            "total": weights + kv_read + kv_append + lg}


def sol_tokens_per_s(bytes_per_step: float, batch: int, bandwidth_bytes_per_s: float) -> float:
    """Tokens/s if the step did nothing but move its bytes at the given bandwidth."""
    return batch * bandwidth_bytes_per_s / bytes_per_step
