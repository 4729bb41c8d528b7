"""Shared helpers for the parity tests: build inputs, run the CUDA path through
the C ABI binding, run the oracle, compare.

Tolerances (attention outputs):
  - fp32 K/V with fp32 out: max-abs <= 1e-5;
  - fp16 / bf16 K/V: max-abs <= 5e-3 and relative L2 <= 1e-3, checked on fp32
    out against the fp64 oracle;
  - fp16 / bf16 out: the oracle's result rounded to that type (round to
    nearest even), with the same bounds, except that an element may differ by
    one unit in the last place of the output type where the two sides' values
    straddle a rounding boundary.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from paged_kv_cache_251_gb300 import workloads as wl

MAXABS_F32 = 1e-5
MAXABS_LOW = 5e-3
RELL2_LOW = 1e-3


def shape(name="case", n=2, h=4, hkv=4, d=64, bs=16, dtype=torch.float16, window=0, seed=5):
    return wl.Shape(name, n, h, hkv, d, bs, dtype, window=window, seed=seed)


def make_inputs(sh: wl.Shape, lens, device="cpu", room_for_append=False, with_append=False, fill=1.0):
    lens_t = torch.as_tensor(lens, dtype=torch.int32)
    return wl.decode_inputs(sh, device=device, lens=lens_t, room_for_append=room_for_append,
                            fill=fill, with_append=with_append)


def to_cuda(inp: wl.DecodeInputs):
    out = {}
    for name in ("q", "k_cache", "v_cache", "block_tables", "context_lens", "k_new", "v_new"):
        t = getattr(inp, name)
        out[name] = None if t is None else t.to("cuda").contiguous()
    return out


def run_decode(inp: wl.DecodeInputs, dev: dict | None = None, out_dtype=torch.float32, window=None,
               partition_size=0, block_tables=None, context_lens=None):
    from paged_kv_cache_251_gb300 import pa
    dev = dev or to_cuda(inp)
    s = inp.shape
    q = dev["q"]
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = dev["block_tables"] if block_tables is None else block_tables.to("cuda").contiguous()
    cl = dev["context_lens"] if context_lens is None else context_lens.to("cuda").contiguous()
    pa.pa_decode(out, q, dev["k_cache"], dev["v_cache"], bt, cl, num_kv_heads=s.num_kv_heads,
                 scale=1.0 / math.sqrt(s.head_dim), window=s.window if window is None else window,
                 partition_size=partition_size, err_word=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


def oracle_decode(inp: wl.DecodeInputs, window=None, pairs=None, block_tables=None, context_lens=None,
                  invalid_policy=0, threads=8):
    s = inp.shape
    return oracle.paged_attention(inp.q, inp.k_cache, inp.v_cache,
                                  inp.block_tables if block_tables is None else block_tables,
                                  inp.context_lens if context_lens is None else context_lens,
                                  num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim),
                                  window=s.window if window is None else window, pairs=pairs,
                                  invalid_policy=invalid_policy, threads=threads)


def compare(got: torch.Tensor, ref: np.ndarray, kv_dtype: torch.dtype):
    """Assert the tolerance; return (max_abs, rel_l2)."""
    ref_t = torch.from_numpy(np.ascontiguousarray(ref))
    out_dtype = got.dtype
    g = got.double()
    assert torch.isfinite(g).all(), "non-finite output"
    if out_dtype == torch.float32:
        r = ref_t
        diff = (g - r).abs()
        slack = torch.zeros_like(diff)
    else:
        r = ref_t.to(out_dtype).double()
        diff = (g - r).abs()
        # one ulp of the output type where the rounding went the other way
        ulp = (r.abs().clamp_min(torch.finfo(out_dtype).tiny) * torch.finfo(out_dtype).eps).double()
        slack = torch.where(diff <= ulp * 1.0001, diff, torch.zeros_like(diff))
    max_abs = float((diff - slack).max()) if diff.numel() else 0.0
    rel = float(torch.linalg.vector_norm(g - r) / max(float(torch.linalg.vector_norm(r)), 1e-30))
    if kv_dtype == torch.float32 and out_dtype == torch.float32:
        assert max_abs <= MAXABS_F32, f"max-abs {max_abs:.3e} > {MAXABS_F32}"
    else:
        assert max_abs <= MAXABS_LOW, f"max-abs {max_abs:.3e} > {MAXABS_LOW}"
        assert rel <= RELL2_LOW, f"rel-L2 {rel:.3e} > {RELL2_LOW}"
    return max_abs, rel


def make_groups(prompts, samples, prompt_lens, extra, bs, hkv, d, dtype, seed):
    """Groups of sequences sharing a prompt, built by the block manager (a
    prompt, then forks that each append their own tokens), so that members'
    tables agree on the prompt's whole blocks: (tables, lens, k, v)."""
    from paged_kv_cache_251_gb300.blocks import BlockManager
    N = prompts * samples
    M = max(prompt_lens) // bs + max(extra) // bs + 4
    nb = N * M + 8
    bm = BlockManager(nb, bs, N, M, free_order=wl.permutation(seed, 2, nb))
    for p in range(prompts):
        first = p * samples
        bm.add_sequence(first)
        bm.extend(first, prompt_lens[p])
        for j in range(1, samples):
            bm.fork(first, first + j)
    seqs = [s for s in range(N) for _ in range(extra[s])]
    slots, pairs = bm.append(seqs)
    tables, lens = bm.tables()
    k = wl.normal_tensor(seed, 4, (nb, hkv, bs, d), dtype=dtype)
    v = wl.normal_tensor(seed, 5, (nb, hkv, bs, d), dtype=dtype)
    return tables, lens, k, v
