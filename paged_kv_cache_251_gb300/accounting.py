"""Byte accounting for the roofline: the bytes a decode step must move at
minimum (each attended K/V row read once per (sequence, kv head)), never the
bytes of a padded contiguous cache.

KV bytes per token per layer = 2 (K and V) * num_kv_heads * head_dim * bytes
per element ("PagedAttention — 把 KV cache 当虚拟内存页来管理", 实践案例 案例 1:
2 * layers * hidden * bytes, about 800 KB per token for OPT-13B).
"""
from __future__ import annotations

import torch


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, elt_bytes: int, layers: int = 1) -> int:
    return 2 * layers * num_kv_heads * head_dim * elt_bytes


def attended_tokens(context_lens: torch.Tensor, window: int = 0) -> torch.Tensor:
    lens = context_lens.to(torch.int64).clamp_min(0)
    return lens.clamp_max(window) if window > 0 else lens


def decode_bytes(context_lens: torch.Tensor, num_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, elt_bytes: int, out_elt_bytes: int = 4, window: int = 0,
                 q_elt_bytes: int | None = None, row_scale_bytes: int = 0) -> dict:
    """Algorithmic bytes of one pa_decode call.

    kv:    attended tokens x 2 x H_kv x (d x elt + row_scale_bytes) (read once;
           an 8-bit cache has elt 1 and one fp32 scale per row)
    q:     N x H x d x q_elt (read; q_elt = elt unless given)
    out:   N x H x d x out_elt (written)
    table: one int32 entry per attended block, plus the context lengths
    """
    toks = attended_tokens(context_lens, window)
    n = int(context_lens.numel())
    kv = int(toks.sum()) * (kv_bytes_per_token(num_kv_heads, head_dim, elt_bytes)
                            + 2 * num_kv_heads * row_scale_bytes)
    if q_elt_bytes is None:
        q_elt_bytes = elt_bytes
    lens = context_lens.to(torch.int64).clamp_min(0)
    start = (lens - toks)
    blocks = torch.where(lens > 0, (lens - 1) // block_size - start // block_size + 1, torch.zeros_like(lens))
    q = n * num_heads * head_dim * q_elt_bytes
    out = n * num_heads * head_dim * out_elt_bytes
    table = int(blocks.sum()) * 4 + n * 4
    return {"kv": kv, "q": q, "out": out, "table": table, "total": kv + q + out + table,
            "attended_tokens": int(toks.sum())}


def append_quant_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, in_elt_bytes: int) -> int:
    """Quantise-on-append: read the new rows, write their 8-bit codes and one
    fp32 scale per row, read the slot mapping."""
    rows = 2 * num_tokens * num_kv_heads
    return rows * head_dim * in_elt_bytes + rows * (head_dim + 4) + 8 * num_tokens


def append_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, elt_bytes: int) -> int:
    """Read the new rows, write them into the cache, read the slot mapping."""
    rows = 2 * num_tokens * num_kv_heads * head_dim * elt_bytes
    return 2 * rows + 8 * num_tokens


def copy_bytes(num_pairs: int, num_kv_heads: int, block_size: int, head_dim: int, elt_bytes: int) -> int:
    """Read and write both caches' blocks for every pair."""
    return 2 * 2 * num_pairs * num_kv_heads * block_size * head_dim * elt_bytes + 16 * num_pairs
