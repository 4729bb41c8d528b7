"""Seeded random decode configurations against the oracle: dtypes, group sizes,
head dims, block sizes, partitions, windows and length mixes (empty and
one-token sequences, block and partition edges) drawn together, so that the
combinations the hand-picked cases do not list reach every kernel family
(MHA, tensor-core grouped heads, the general kernel, the 8-bit kernels)."""
import math
import random

import pytest
import torch

from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare, make_inputs, oracle_decode, run_decode, shape

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _lens(rng, n, bs, max_len):
    edges = [0, 1, bs - 1, bs, bs + 1, 2 * bs, 511, 512, 513]
    out = []
    for _ in range(n):
        if rng.random() < 0.35:
            out.append(min(rng.choice(edges), max_len))
        else:
            out.append(rng.randint(1, max_len))
    return out


def _config(i):
    rng = random.Random(9100 + i)
    d = rng.choice([64, 128])
    bs = rng.choice([8, 16, 32])
    hkv = rng.choice([1, 2, 4, 8])
    g = rng.choice([1, 2, 4, 8])
    n = rng.randint(1, 10)
    max_len = rng.choice([40, 300, 1200, 2600])
    window = rng.choice([0, 0, 0, rng.randint(1, max_len)])
    part = rng.choice([0, 0, bs * rng.randint(1, 8), bs * rng.randint(16, 64)])
    return d, bs, hkv, g, n, _lens(rng, n, bs, max_len), window, part, rng.choice(list(DT))


@pytest.mark.parametrize("i", range(120))
def test_random_decode_configs(i):
    d, bs, hkv, g, n, lens, window, part, dt = _config(i)
    sh = shape(f"fuzz{i}", n, hkv * g, hkv, d, bs, DT[dt], window=window, seed=700 + i)
    inp = make_inputs(sh, lens)
    got, err = run_decode(inp, partition_size=part)
    assert err == 0
    compare(got, oracle_decode(inp), DT[dt])


def _quant_config(i):
    rng = random.Random(9300 + i)
    d = rng.choice([64, 128, 128])
    bs = rng.choice([8, 16, 32])
    hkv = rng.choice([1, 2, 4, 4, 8])
    g = rng.choice([1, 2, 4, 8]) if d == 64 else rng.choice([1, 2, 4])
    n = rng.randint(1, 8)
    max_len = rng.choice([40, 300, 1500])
    window = rng.choice([0, 0, rng.randint(1, max_len)])
    part = rng.choice([0, 0, bs * rng.randint(1, 8), bs * rng.randint(16, 64)])
    return (d, bs, hkv, g, n, _lens(rng, n, bs, max_len), window, part, rng.choice(["f16", "bf16", "f32"]),
            rng.choice(["int8", "e4m3"]))


@pytest.mark.parametrize("i", range(60))
def test_random_quant_decode_configs(i):
    from paged_kv_cache_251_gb300 import pa
    import oracle
    d, bs, hkv, g, n, lens, window, part, qdt, fmt = _quant_config(i)
    sh = shape(f"qfuzz{i}", n, hkv * g, hkv, d, bs, DT[qdt], window=window, seed=900 + i)
    inp = wl.decode_inputs(sh, lens=torch.as_tensor(lens, dtype=torch.int32), room_for_append=False,
                           with_append=False)
    kp, vp = wl.quant_pools(inp, fmt)
    s = inp.shape
    out = torch.full(inp.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_quant(out, inp.q.cuda(), kp.cuda(), vp.cuda(), inp.block_tables.cuda(), inp.context_lens.cuda(),
                       num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim), window=window,
                       partition_size=part, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_attention(inp.q, kp, vp, inp.block_tables, inp.context_lens, num_kv_heads=s.num_kv_heads,
                                 scale=1.0 / math.sqrt(s.head_dim), window=window, threads=8)
    compare(out.cpu(), ref, torch.float16)
