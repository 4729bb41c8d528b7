"""Seeded synthetic inputs shaped like the PagedAttention workloads.

This module holds random-number generation and input shapes only: it computes
no attention, no address translation and no copy-on-write.  Both the CUDA
path and the CPU oracle read what it produces, so it is the one module the two
sides share.

Generator: a counter-based SplitMix64 stream (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014; the finaliser
constants are that paper's ``mix64`` variant 13), evaluated with torch int64
ops so the same integers come out on CPU and GPU.  Normals come from the
Box-Muller transform of two 32-bit uniforms taken from one 64-bit draw.

Shapes (from the pages' examples and the OPT-13B sizing note):
  tiny     4 seqs, 4 MHA heads, d 64, block 16, fp32, L ~ U[1, 100], 64-block pool
  opt13b   64 seqs, 40 MHA heads, d 128, block 16, fp16, L ~ U[512, 2048],
           pool = exact need (the appended token included)
  gqa      256 seqs, 32 q / 8 kv heads, d 128, block 16, bf16,
           L = clip(round(exp(ln 1024 + N(0,1))), 16, 8192), pool 95% full
  window   4 seqs x 131072 tokens, 32 q / 8 kv heads, d 128, bf16, block 16,
           window 32768 over a ring of 2049 blocks per sequence
  prefix   32 prompts x 2000 tokens shared by 8 samples each, samples append
           U{1..256} tokens, 40 MHA heads, d 128, fp16, block 8/16/32
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

_M1 = -4658895280553007687      # 0xBF58476D1CE4E5B9 as int64
_M2 = -7723592293110705685      # 0x94D049BB133111EB as int64
_GOLDEN = -7046029254386353131  # 0x9E3779B97F4A7C15 as int64
_CHUNK = 1 << 26


def _srl(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix64(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _M1
    z = (z ^ _srl(z, 27)) * _M2
    return z ^ _srl(z, 31)


def _key(seed: int, stream: int) -> int:
    k = _mix64(torch.tensor([(seed * 1000003 + stream) & 0x7FFFFFFFFFFFFFFF], dtype=torch.int64))
    return int(k.item())


def bits64(seed: int, stream: int, n: int, device="cpu", offset: int = 0) -> torch.Tensor:
    """n raw 64-bit draws (int64 bit patterns) of stream ``stream``."""
    key = _key(seed, stream)
    idx = torch.arange(offset + 1, offset + n + 1, dtype=torch.int64, device=device)
    return _mix64(idx * _GOLDEN + key)


def uniform01(seed: int, stream: int, n: int) -> torch.Tensor:
    """n doubles in [0, 1) with 53 random bits each (CPU)."""
    return _srl(bits64(seed, stream, n), 11).to(torch.float64) * (2.0 ** -53)


def randint(seed: int, stream: int, n: int, lo: int, hi: int) -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive), int64 on CPU."""
    u = uniform01(seed, stream, n)
    return (lo + torch.floor(u * (hi - lo + 1))).to(torch.int64)


def normal(seed: int, stream: int, n: int, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """n N(0, 1) values (Box-Muller in fp32, fp64 on request), cast to dtype."""
    out = torch.empty(n, dtype=dtype, device=device)
    work = torch.float64 if dtype == torch.float64 else torch.float32
    pairs = (n + 1) // 2
    done = 0
    for start in range(0, pairs, _CHUNK):
        cnt = min(_CHUNK, pairs - start)
        z = bits64(seed, stream, cnt, device=device, offset=start)
        hi = _srl(z, 32).to(work)
        lo = (z & 0xFFFFFFFF).to(work)
        u1 = (hi + 1.0) * (2.0 ** -32)          # (0, 1]
        u2 = lo * (2.0 ** -32)                  # [0, 1)
        r = torch.sqrt(-2.0 * torch.log(u1))
        ang = (2.0 * torch.pi) * u2
        vals = torch.stack((r * torch.cos(ang), r * torch.sin(ang)), dim=1).reshape(-1)
        take = min(2 * cnt, n - done)
        out[done:done + take] = vals[:take].to(dtype)
        done += take
    return out


def normal_tensor(seed: int, stream: int, shape, device="cpu", dtype=torch.float32) -> torch.Tensor:
    n = 1
    for s in shape:
        n *= int(s)
    return normal(seed, stream, n, device=device, dtype=dtype).reshape(tuple(shape))


def permutation(seed: int, stream: int, n: int) -> torch.Tensor:
    """A seeded shuffle of 0..n-1 (sort by random 64-bit keys), int64 on CPU."""
    keys = bits64(seed, stream, n)
    return torch.argsort(keys, stable=True)


# ---------------------------------------------------------------------------
# Workload shapes


@dataclass
class Shape:
    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    window: int = 0
    partition_size: int = 0
    seed: int = 0


SHAPES = {
    "tiny": Shape("tiny", 4, 4, 4, 64, 16, torch.float32, seed=251001),
    "opt13b": Shape("opt13b", 64, 40, 40, 128, 16, torch.float16, seed=251002),
    "gqa": Shape("gqa", 256, 32, 8, 128, 16, torch.bfloat16, seed=251003),
    "window": Shape("window", 4, 32, 8, 128, 16, torch.bfloat16, window=32768,
                    partition_size=512, seed=251004),
    "prefix": Shape("prefix", 256, 40, 40, 128, 16, torch.float16, seed=251005),
    # the tiny shape scaled up so that it is not launch-bound: 4096 sequences
    "tiny_scaled": Shape("tiny_scaled", 4096, 4, 4, 64, 16, torch.float32, seed=251006),
}

# streams
_S_LENS, _S_PERM, _S_Q, _S_K, _S_V, _S_KNEW, _S_VNEW, _S_NEW = 1, 2, 3, 4, 5, 6, 7, 8


def context_lengths(shape: Shape) -> torch.Tensor:
    """Seeded context lengths (int32, CPU) for the named workload."""
    s = shape
    if s.name == "tiny":
        return randint(s.seed, _S_LENS, s.num_seqs, 1, 100).to(torch.int32)
    if s.name == "opt13b":
        return randint(s.seed, _S_LENS, s.num_seqs, 512, 2048).to(torch.int32)
    if s.name == "tiny_scaled":
        return randint(s.seed, _S_LENS, s.num_seqs, 1, 2048).to(torch.int32)
    if s.name == "gqa":
        g = normal(s.seed, _S_LENS, s.num_seqs, dtype=torch.float64)
        lens = torch.round(torch.exp(torch.log(torch.tensor(1024.0, dtype=torch.float64)) + g))
        return lens.clamp(16, 8192).to(torch.int32)
    raise ValueError(f"no length recipe for {s.name}")


@dataclass
class DecodeInputs:
    """A paged KV pool, block tables and queries.

    k_cache / v_cache: [num_blocks, H_kv, bs, d]; q: [N, H, d];
    block_tables: int32 [N, M] (unused entries hold -1); context_lens int32 [N];
    blocks_held: int32 [N] = table entries filled per sequence;
    k_new / v_new: [N, H_kv, d] rows for one appended token per sequence.
    """
    shape: Shape
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    blocks_held: torch.Tensor
    num_blocks: int
    k_new: torch.Tensor | None = None
    v_new: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)


def _ceil_div(a, b):
    return (a + b - 1) // b


def pool_and_tables(shape: Shape, lens: torch.Tensor, room_for_append: bool,
                    num_blocks: int | None = None, fill: float = 1.0, shuffle: bool = True):
    """Hand out a seeded shuffle of the pool's block ids (or, with
    shuffle=False, the ids in order, so each sequence's blocks are adjacent in
    memory), sequence by sequence, each sequence taking the blocks its tokens
    occupy.

    Returns (block_tables int32 [N, M], blocks_held int32 [N], num_blocks).
    """
    bs = shape.block_size
    toks = lens.to(torch.int64) + (1 if room_for_append else 0)
    held = _ceil_div(toks, bs)
    need = int(held.sum())
    if num_blocks is None:   # a pool that the sequences fill to the given fraction
        num_blocks = need if fill >= 1.0 else int(_ceil_div(need * 100, int(round(fill * 100))))
    if need > num_blocks:
        raise ValueError("pool too small for the requested lengths")
    perm = (permutation(shape.seed, _S_PERM, num_blocks) if shuffle
            else torch.arange(num_blocks)).to(torch.int32)
    width = max(1, int(held.max()))
    tables = torch.full((shape.num_seqs, width), -1, dtype=torch.int32)
    at = 0
    for s in range(shape.num_seqs):
        n = int(held[s])
        tables[s, :n] = perm[at:at + n]
        at += n
    return tables, held.to(torch.int32), num_blocks


def decode_inputs(shape: Shape, device="cpu", lens: torch.Tensor | None = None,
                  room_for_append: bool = True, num_blocks: int | None = None,
                  fill: float = 1.0, with_append: bool = True, shuffle: bool = True) -> DecodeInputs:
    """Pool, tables, queries and K/V values for a decode (+ append) step."""
    s = shape
    if lens is None:
        lens = context_lengths(s)
    tables, held, nb = pool_and_tables(s, lens, room_for_append, num_blocks, fill, shuffle)
    kv_shape = (nb, s.num_kv_heads, s.block_size, s.head_dim)
    q = normal_tensor(s.seed, _S_Q, (s.num_seqs, s.num_heads, s.head_dim), device, s.dtype)
    k = normal_tensor(s.seed, _S_K, kv_shape, device, s.dtype)
    v = normal_tensor(s.seed, _S_V, kv_shape, device, s.dtype)
    kn = vn = None
    if with_append:
        kn = normal_tensor(s.seed, _S_KNEW, (s.num_seqs, s.num_kv_heads, s.head_dim), device, s.dtype)
        vn = normal_tensor(s.seed, _S_VNEW, (s.num_seqs, s.num_kv_heads, s.head_dim), device, s.dtype)
    return DecodeInputs(s, q, k, v, tables, lens, held, nb, kn, vn)


def tiny(device="cpu") -> DecodeInputs:
    return decode_inputs(SHAPES["tiny"], device, num_blocks=64)


def opt13b(device="cpu") -> DecodeInputs:
    return decode_inputs(SHAPES["opt13b"], device)


def gqa(device="cpu") -> DecodeInputs:
    return decode_inputs(SHAPES["gqa"], device, room_for_append=False, fill=0.95,
                         with_append=False)


# 8-bit caches: random code and scale pools (raw draws, no quantisation)
_S_KCODE, _S_VCODE, _S_KSCALE, _S_VSCALE = 9, 10, 11, 12
CODE_DTYPES = {"int8": torch.int8, "e4m3": torch.float8_e4m3fn}


def code_pool(seed: int, stream: int, shape, fmt: str, device="cpu") -> torch.Tensor:
    """Random 8-bit cache codes of ``shape`` as int8 / float8_e4m3fn.

    INT8: uniform in [-127, 127].  E4M3: random sign and mantissa bits, the
    exponent field uniform in [2, 10], and one code in 16 with exponent field
    0 (a subnormal or zero); never the NaN pattern.
    """
    n = 1
    for d in shape:
        n *= int(d)
    out = torch.empty(n, dtype=torch.uint8, device=device)
    for start in range(0, n, _CHUNK):
        cnt = min(_CHUNK, n - start)
        z = bits64(seed, stream, cnt, device=device, offset=start)
        if fmt == "int8":
            c = (_srl(z, 33) % 255) - 127
            out[start:start + cnt] = (c & 0xFF).to(torch.uint8)
        else:
            e = 2 + _srl(z, 40) % 9
            e = torch.where((_srl(z, 36) & 15) == 0, torch.zeros_like(e), e)
            byte = ((_srl(z, 63) & 1) << 7) | (e << 3) | (_srl(z, 20) & 7)
            out[start:start + cnt] = byte.to(torch.uint8)
    return out.view(CODE_DTYPES[fmt]).reshape(tuple(shape))


def scale_pool(seed: int, stream: int, shape, fmt: str, device="cpu") -> torch.Tensor:
    """Random row scales (float32 of ``shape``): uniform in [0.5, 1.5) times
    1/64 for INT8 codes or 1/5 for E4M3 codes, so code * scale is of order one."""
    n = 1
    for d in shape:
        n *= int(d)
    u = _srl(bits64(seed, stream, n, device=device), 40).to(torch.float32) * (2.0 ** -24)
    base = 1.0 / 64 if fmt == "int8" else 0.2
    return ((0.5 + u) * base).reshape(tuple(shape))


def page_pool(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """An 8-bit page pool [nb, H_kv, bs + scale_rows, d] holding `codes`
    [nb, H_kv, bs, d] and the bytes of `scales` float32 [nb, H_kv, bs] in
    each page's trailing rows (zero padding after them)."""
    nb, hkv, bs, d = codes.shape
    sr = (4 * bs + d - 1) // d
    pool = torch.zeros((nb, hkv, bs + sr, d), dtype=torch.uint8, device=codes.device)
    pool[:, :, :bs] = codes.view(torch.uint8)
    tail = pool[:, :, bs:].reshape(nb, hkv, sr * d)
    tail[:, :, :4 * bs] = scales.contiguous().view(torch.uint8).reshape(nb, hkv, 4 * bs)
    pool[:, :, bs:] = tail.reshape(nb, hkv, sr, d)
    return pool.view(codes.dtype)


def quant_pools(inp: DecodeInputs, fmt: str, device="cpu"):
    """Random 8-bit page pools (codes and row scales from code_pool /
    scale_pool) with the block layout of ``inp``'s caches: (k_pages, v_pages)."""
    s = inp.shape
    shp = (inp.num_blocks, s.num_kv_heads, s.block_size, s.head_dim)
    kp = page_pool(code_pool(s.seed, _S_KCODE, shp, fmt, device), scale_pool(s.seed, _S_KSCALE, shp[:3], fmt, device))
    vp = page_pool(code_pool(s.seed, _S_VCODE, shp, fmt, device), scale_pool(s.seed, _S_VSCALE, shp[:3], fmt, device))
    return kp, vp


def prefix_draws(seed: int, num_samples: int, lo: int = 1, hi: int = 256) -> torch.Tensor:
    """Divergent-token counts per sample, uniform in [lo, hi]."""
    return randint(seed, _S_NEW, num_samples, lo, hi)
