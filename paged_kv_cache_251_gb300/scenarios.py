"""Decode-step states that need the block manager: a sliding window realised
by a ring of physical blocks, and prefix sharing with copy-on-write.

The random draws (pool values, block hand-out order, divergent-token counts)
come from ``workloads``; the block tables, slot mappings and copy pairs come
from the native block manager (``blocks.BlockManager``).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import workloads as wl
from .blocks import BlockManager


@dataclass
class WindowState:
    shape: wl.Shape
    context: int            # logical tokens per sequence
    ring_blocks: int        # physical blocks per sequence
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor   # int32 [N, M]; recycled entries are -1
    context_lens: torch.Tensor   # int32 [N]
    num_blocks: int
    manager: BlockManager
    k_new: torch.Tensor
    v_new: torch.Tensor


def window_state(device="cpu", context: int = 131072, window: int | None = None,
                 shape: wl.Shape | None = None, slack_blocks: int = 8) -> WindowState:
    """N sequences of `context` logical tokens whose K/V lives in rings of
    ceil(window / block) + 1 physical blocks (the window's tokens stay
    resident); table rows hold `context / block + slack_blocks` entries."""
    s = shape or wl.SHAPES["window"]
    W = window if window is not None else s.window
    bs = s.block_size
    R = -(-W // bs) + 1
    nb = s.num_seqs * R
    M = -(-context // bs) + slack_blocks
    order = wl.permutation(s.seed, 2, nb)
    bm = BlockManager(nb, bs, s.num_seqs, M, free_order=order)
    for i in range(s.num_seqs):
        bm.add_sequence(i, ring_blocks=R)
        bm.extend(i, context)
    tables, lens = bm.tables()
    kv_shape = (nb, s.num_kv_heads, bs, s.head_dim)
    return WindowState(
        shape=s, context=context, ring_blocks=R,
        q=wl.normal_tensor(s.seed, 3, (s.num_seqs, s.num_heads, s.head_dim), device, s.dtype),
        k_cache=wl.normal_tensor(s.seed, 4, kv_shape, device, s.dtype),
        v_cache=wl.normal_tensor(s.seed, 5, kv_shape, device, s.dtype),
        block_tables=tables, context_lens=lens, num_blocks=nb, manager=bm,
        k_new=wl.normal_tensor(s.seed, 6, (s.num_seqs, s.num_kv_heads, s.head_dim), device, s.dtype),
        v_new=wl.normal_tensor(s.seed, 7, (s.num_seqs, s.num_kv_heads, s.head_dim), device, s.dtype))


@dataclass
class PrefixState:
    shape: wl.Shape
    prompts: int
    samples: int
    prompt_len: int
    new_tokens: torch.Tensor     # int64 [prompts * samples] divergent tokens per sample
    q: torch.Tensor
    k_cache: torch.Tensor        # pool before the step (prompt K/V in place)
    v_cache: torch.Tensor
    free_order: torch.Tensor     # block hand-out order
    num_blocks: int
    max_blocks_per_seq: int
    # produced by the block manager for the step:
    pairs: torch.Tensor          # int64 [P, 2] copy-on-write (src, dst)
    slots: torch.Tensor          # int64 [T] slot of every new token, sample by sample
    token_seq: torch.Tensor      # int32 [T] sample of every new token
    block_tables: torch.Tensor   # int32 [prompts * samples, M] after the step
    context_lens: torch.Tensor   # int32 [prompts * samples] after the step
    k_new: torch.Tensor          # [T, H_kv, d]
    v_new: torch.Tensor


def prefix_state(block_size: int, device="cpu", prompts: int = 32, samples: int = 8, prompt_len: int = 2000,
                 max_new: int = 256, shape: wl.Shape | None = None) -> PrefixState:
    """`prompts` prompts of `prompt_len` tokens, each shared by `samples`
    samples (reference count `samples` per prompt block); every sample then
    appends U{1..max_new} tokens.  The block manager decides the slots and
    the copy-on-write pairs of that step."""
    base = shape or wl.SHAPES["prefix"]
    s = wl.Shape(base.name, prompts * samples, base.num_heads, base.num_kv_heads, base.head_dim, block_size,
                 base.dtype, seed=base.seed + block_size)
    bs = block_size
    n_new = wl.prefix_draws(base.seed, prompts * samples, 1, max_new)   # same samples at every block size
    per_prompt = -(-prompt_len // bs)
    M = -(-(prompt_len + max_new) // bs) + 1
    nb = prompts * per_prompt + prompts * samples * (-(-max_new // bs) + 1)
    order = wl.permutation(s.seed, 2, nb)
    bm = BlockManager(nb, bs, prompts * samples, M, free_order=order)
    for p in range(prompts):
        first = p * samples
        bm.add_sequence(first)
        bm.extend(first, prompt_len)
        for j in range(1, samples):
            bm.fork(first, first + j)
    token_seq = torch.repeat_interleave(torch.arange(prompts * samples, dtype=torch.int32), n_new)
    slots, pairs = bm.append(token_seq)
    tables, lens = bm.tables()
    T = int(n_new.sum())
    kv_shape = (nb, s.num_kv_heads, bs, s.head_dim)
    return PrefixState(
        shape=s, prompts=prompts, samples=samples, prompt_len=prompt_len, new_tokens=n_new,
        q=wl.normal_tensor(s.seed, 3, (s.num_seqs, s.num_heads, s.head_dim), device, s.dtype),
        k_cache=wl.normal_tensor(s.seed, 4, kv_shape, device, s.dtype),
        v_cache=wl.normal_tensor(s.seed, 5, kv_shape, device, s.dtype),
        free_order=order, num_blocks=nb, max_blocks_per_seq=M, pairs=pairs, slots=slots, token_seq=token_seq,
        block_tables=tables, context_lens=lens,
        k_new=wl.normal_tensor(s.seed, 6, (T, s.num_kv_heads, s.head_dim), device, s.dtype),
        v_new=wl.normal_tensor(s.seed, 7, (T, s.num_kv_heads, s.head_dim), device, s.dtype))
