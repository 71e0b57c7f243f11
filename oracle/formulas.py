"""The pages' KV-cache byte and bandwidth arithmetic (test infrastructure).

Sources (page titles; sections in quotes):
* "KV Cache Engineering: PagedAttention, Continuous Batching, Attention
  Variants, and the Bandwidth Wall": "Cache size calculation" (bytes per
  token = 2 x layers x KV heads x head_dim x dtype bytes), "Two Costs:
  Capacity and Bandwidth" (decode reads the whole cache each step, so the KV
  part of a step takes KV bytes / HBM bandwidth), "PagedAttention" (only the
  last block of a sequence is partly filled), "The Fragmentation Problem"
  (utilisation of reserved memory), "Memory Layout: Everything Together"
  (tokens that fit a memory budget).
* "KV-Cache Engineering: The Memory Wall of LLM Serving": "Why the cache
  explodes" (the same formula times sequence length and batch).
* "KV-Cache Engineering: Paged Attention, Prefix Cache, Disaggregation
  (2026)", cross-layer KV sharing Q&A: layers in groups share one KV, so the
  layer factor becomes the number of groups.
"""
from __future__ import annotations

import math


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: float) -> float:
    """2 (K and V) x layers x KV heads x head_dim x bytes per element."""
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes


def kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: float,
             seq_len: int, batch: int = 1) -> float:
    """Bytes per token x sequence length x batch."""
    return kv_bytes_per_token(n_layers, n_kv_heads, head_dim, dtype_bytes) * seq_len * batch


def kv_bytes_per_token_grouped(n_layers: int, layers_per_group: int, n_kv_heads: int,
                               head_dim: int, dtype_bytes: float) -> float:
    """Cross-layer sharing: one KV per group of consecutive layers."""
    if n_layers % layers_per_group:
        raise ValueError("layers must divide into whole groups")
    return kv_bytes_per_token(n_layers // layers_per_group, n_kv_heads, head_dim, dtype_bytes)


def decode_kv_read_seconds(kv_bytes_total: float, hbm_bytes_per_s: float) -> float:
    """KV term of a bandwidth-bound decode step: the whole cache is read once."""
    return kv_bytes_total / hbm_bytes_per_s


def blocks_for_tokens(n_tokens: int, block_size: int) -> int:
    """Physical blocks a sequence of n tokens occupies."""
    return -(-n_tokens // block_size)


def last_block_waste_tokens(n_tokens: int, block_size: int) -> int:
    """Unused token slots in the (only) partly filled last block."""
    return blocks_for_tokens(n_tokens, block_size) * block_size - n_tokens


def tokens_that_fit(budget_bytes: float, bytes_per_token: float) -> float:
    return budget_bytes / bytes_per_token


def naive_utilisation(used_tokens, reserved_tokens) -> float:
    """Fraction of reserved token slots actually used."""
    return sum(used_tokens) / sum(reserved_tokens)


__all__ = [n for n in dir() if not n.startswith("_") and n != "math"]
