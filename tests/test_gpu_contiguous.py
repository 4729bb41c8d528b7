"""GPU parity of pa_decode_contiguous: decode attention over contiguous
(non-paged) caches [N, H_kv, L, d], the baseline for the cost of the block
table ("PagedAttention — 把 KV cache 当虚拟内存页来管理", 踩过的坑).

Each case writes the same K/V into a contiguous cache and into a paged pool
whose block tables list every sequence's blocks in order (block b of sequence
s is block s * (L / 16) + b).  The contiguous decode must match the oracle
over the paged pool within the attention tolerances, and equal pa_decode over
the paged pool bit for bit (the same kernels read the same values in the same
order; only the addressing differs)."""
import math

import pytest
import torch

from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare, oracle_decode, run_decode, shape

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32

# name, N, H, H_kv, d, dtype, lens, window, partition
CASES = [
    ("mha_f16", 4, 4, 4, 128, F16, [1, 700, 2049, 16], 0, 0),
    ("mha_f32_d64", 3, 4, 4, 64, F32, [33, 1000, 0], 0, 64),
    ("mha_bf16_window", 3, 8, 8, 128, BF16, [3000, 77, 1500], 700, 0),
    ("tc_g2_f16", 3, 4, 2, 128, F16, [129, 1025, 2048], 0, 0),
    ("tc_g4_bf16", 4, 8, 2, 128, BF16, [5000, 127, 128, 1], 0, 0),
    ("tc_g4_parts", 3, 16, 4, 128, BF16, [3000, 640, 2049], 0, 512),
    ("tc_g8_window", 2, 16, 2, 128, F16, [4000, 300], 1000, 0),
    ("tc_g4_empty", 3, 8, 2, 128, BF16, [0, 256, 0], 0, 0),
]


def _inputs(name, n, h, hkv, d, dt, lens, window):
    """A paged pool with in-order tables, and the same values as contiguous caches."""
    L = max(16, -(-max(lens) // 16) * 16)
    mb = L // 16
    sh = shape(name, n, h, hkv, d, 16, dt, window=window, seed=60 + n + h + d)
    q = wl.normal_tensor(sh.seed, 3, (n, h, d), dtype=dt)
    kc = wl.normal_tensor(sh.seed, 4, (n, hkv, L, d), dtype=dt)
    vc = wl.normal_tensor(sh.seed, 5, (n, hkv, L, d), dtype=dt)
    paged = [c.reshape(n, hkv, mb, 16, d).permute(0, 2, 1, 3, 4).reshape(n * mb, hkv, 16, d).contiguous()
             for c in (kc, vc)]
    tables = (torch.arange(n, dtype=torch.int32)[:, None] * mb + torch.arange(mb, dtype=torch.int32)[None]).contiguous()
    inp = wl.DecodeInputs(sh, q, paged[0], paged[1], tables, torch.tensor(lens, dtype=torch.int32),
                          torch.full((n,), mb, dtype=torch.int32), n * mb)
    return inp, kc, vc


def _contiguous(inp, kc, vc, partition, window, context_lens=None):
    from paged_kv_cache_251_gb300 import pa
    s = inp.shape
    out = torch.full(inp.q.shape, float("nan"), dtype=F32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cl = inp.context_lens if context_lens is None else context_lens
    pa.pa_decode_contiguous(out, inp.q.cuda(), kc.cuda(), vc.cuda(), cl.cuda(), num_kv_heads=s.num_kv_heads,
                            scale=1.0 / math.sqrt(s.head_dim), window=window, partition_size=partition, err_word=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_contiguous_matches_oracle_and_paged_decode(case):
    name, n, h, hkv, d, dt, lens, window, part = case
    inp, kc, vc = _inputs(name, n, h, hkv, d, dt, lens, window)
    got, err = _contiguous(inp, kc, vc, part, window)
    assert err == 0
    compare(got, oracle_decode(inp), dt)
    paged, perr = run_decode(inp, partition_size=part)
    assert perr == 0
    assert torch.equal(got, paged)


def test_contiguous_context_beyond_the_cache_is_clamped_and_flagged():
    inp, kc, vc = _inputs("clamp", 2, 8, 2, 128, BF16, [300, 40], 0)
    L = kc.shape[2]
    got, err = _contiguous(inp, kc, vc, 0, 0, context_lens=torch.tensor([L + 50, 40], dtype=torch.int32))
    assert err & 16
    compare(got, oracle_decode(inp, context_lens=torch.tensor([L, 40], dtype=torch.int32)), BF16)


def _random_case(i):
    import random
    rng = random.Random(5100 + i)
    g = rng.choice([1, 2, 4, 8])
    hkv = rng.choice([1, 2, 4])
    d = 128 if g > 1 else rng.choice([64, 128])
    dt = rng.choice([F16, BF16]) if g > 1 else rng.choice([F16, BF16, F32])
    n = rng.randint(1, 6)
    max_len = rng.choice([40, 300, 1500, 4000])
    lens = [rng.choice([0, 1, 15, 16, 17, 127, 128, 129, rng.randint(1, max_len)]) for _ in range(n)]
    window = rng.choice([0, 0, rng.randint(1, max_len)])
    part = rng.choice([0, 0, 16 * rng.randint(1, 16), 16 * rng.randint(32, 128)])
    return f"rand{i}", n, hkv * g, hkv, d, dt, lens, window, part


@pytest.mark.parametrize("i", range(30))
def test_contiguous_random_configs_equal_paged_decode(i):
    """Seeded random shapes, lengths, windows and partitions: the contiguous
    decode equals pa_decode over the same values in a paged pool, bit for
    bit, and matches the oracle."""
    name, n, h, hkv, d, dt, lens, window, part = _random_case(i)
    inp, kc, vc = _inputs(name, n, h, hkv, d, dt, lens, window)
    got, err = _contiguous(inp, kc, vc, part, window)
    assert err == 0
    paged, perr = run_decode(inp, partition_size=part)
    assert perr == 0
    assert torch.equal(got, paged)
    compare(got, oracle_decode(inp), dt)
