"""KV-cache memory footprint: naive per-request reservation against paged
blocks.

The naive scheme reserves the model's whole context for every request in
one contiguous region (Qualiteg, "About PagedAttention for LLM serving",
"In a Nutshell ... Problem 1" and the ChatStream capacity formula: total
memory = model + users x max context x KV bytes per token); the paged
scheme holds only the blocks a sequence has filled ("1-1 ... reserves only
as much as needed"), and shares the blocks of a common prompt prefix.
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elem_bytes: int, layers: int = 1) -> int:
    """K and V of one token, all KV heads, `layers` layers."""
    return 2 * num_kv_heads * head_dim * elem_bytes * layers


def naive_slots(num_seqs: int, max_context: int) -> int:
    """Token slots reserved up front: the full context per request."""
    return num_seqs * max_context


def paged_slots(context_lens, block_size: int, shared_prefix_blocks: int = 0,
                group_size: int = 1) -> int:
    """Token slots in the blocks the sequences occupy; a group of
    `group_size` sequences stores its `shared_prefix_blocks` once."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    blocks = int(((ctx + block_size - 1) // block_size).sum())
    if group_size > 1 and shared_prefix_blocks:
        blocks -= (group_size - 1) * (ctx.size // group_size) * shared_prefix_blocks
    return blocks * block_size


def report(w, max_context: int | None = None) -> dict:
    """Naive vs paged footprint of a Workload (one layer)."""
    cap = max_context if max_context is not None else w.max_blocks_per_seq * w.block_size
    per_tok = kv_bytes_per_token(w.num_kv_heads, w.head_dim, w.elem_bytes)
    used = int(np.asarray(w.context_lens, dtype=np.int64).sum())
    naive = naive_slots(w.num_seqs, cap)
    paged = paged_slots(w.context_lens, w.block_size,
                        w.prefix_len // w.block_size if w.group_size > 1 else 0, w.group_size)
    return {"max_context": cap, "tokens": used,
            "naive_bytes": naive * per_tok, "paged_bytes": paged * per_tok,
            "naive_waste_frac": 1 - used / naive if naive else 0.0,
            "paged_waste_frac": 1 - min(used, paged) / paged if paged else 0.0,
            "ratio": naive / paged if paged else float("inf")}
