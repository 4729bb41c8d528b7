"""Pins of the CPU oracle against facts that do not come from the oracle itself.

- the worked example printed on the study-notes page (block_size 16, table
  [7, 1, 3], token 34 -> physical block 3, offset 2);
- identity tables, where the paged cache is a plain contiguous tensor after a
  reshape, against torch's fp64 scaled_dot_product_attention (a library
  routine for softmax(Q K^T / sqrt(d)) V);
- invariance under a random permutation of the physical blocks;
- closed forms (identical keys or q = 0 give the mean of V, one token gives
  V_0, two tokens give the sigmoid-weighted pair, a dominant score selects
  one row);
- torch's own float16 / bfloat16 -> float64 conversion for every bit pattern.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_251_gb300 import workloads as wl

GOLDEN = Path(__file__).parent / "golden"
DTYPES = [torch.float32, torch.float16, torch.bfloat16]


def _identity_case(n_seqs, n_heads, n_kv, d, bs, dtype, lens, seed):
    """Cache whose tables are the identity: seq s owns blocks s*M .. s*M+M-1."""
    M = max(1, max((int(L) + bs - 1) // bs for L in lens))
    nb = n_seqs * M
    k = wl.normal_tensor(seed, 11, (nb, n_kv, bs, d), dtype=dtype)
    v = wl.normal_tensor(seed, 12, (nb, n_kv, bs, d), dtype=dtype)
    q = wl.normal_tensor(seed, 13, (n_seqs, n_heads, d), dtype=dtype)
    tables = torch.arange(nb, dtype=torch.int32).reshape(n_seqs, M)
    cl = torch.tensor(lens, dtype=torch.int32)
    return q, k, v, tables, cl, M


def _sdpa_reference(q, k, v, cl, M, bs, n_kv, window=0, scale=None):
    """torch fp64 SDPA on the contiguous view of an identity-table cache."""
    N, H, d = q.shape
    G = H // n_kv
    kc = k.double().reshape(N, M, n_kv, bs, d).permute(0, 2, 1, 3, 4).reshape(N, n_kv, M * bs, d)
    vc = v.double().reshape(N, M, n_kv, bs, d).permute(0, 2, 1, 3, 4).reshape(N, n_kv, M * bs, d)
    out = torch.zeros(N, H, d, dtype=torch.float64)
    for s in range(N):
        L = int(cl[s])
        lo = max(0, L - window) if window > 0 else 0
        if L == 0:
            continue
        kk = kc[s, :, lo:L].repeat_interleave(G, dim=0)          # [H, n, d]
        vv = vc[s, :, lo:L].repeat_interleave(G, dim=0)
        qq = q[s].double().unsqueeze(1)                          # [H, 1, d]
        out[s] = F.scaled_dot_product_attention(qq, kk, vv, scale=scale).squeeze(1)
    return out.numpy()


def test_locate_worked_example():
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    assert oracle.locate(g["block_table"], g["block_size"], g["token"]) == (g["physical"], g["offset"])


def test_locate_every_token_of_the_example_table():
    # every token of the 3-block table lands in its logical block's physical block
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    seen = []
    for t in range(3 * g["block_size"]):
        seen.append(oracle.locate(g["block_table"], g["block_size"], t))
    assert len(set(seen)) == len(seen)
    assert sorted({p for p, _ in seen}) == sorted(g["block_table"])
    with pytest.raises(IndexError):
        oracle.locate(g["block_table"], g["block_size"], 3 * g["block_size"])


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_element_conversion_matches_torch_for_every_bit_pattern(dtype):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = bits.view(dtype)
    ref = vals.double().numpy()
    got = oracle.to_double(vals)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


CASES = [
    # n_seqs, H, H_kv, d, bs, lens, window
    (3, 4, 4, 64, 16, [1, 17, 40], 0),
    (2, 8, 2, 128, 8, [33, 9], 0),
    (2, 4, 1, 64, 32, [70, 31], 0),
    (3, 8, 8, 128, 16, [50, 16, 15], 20),
    (2, 4, 2, 64, 16, [100, 7], 33),
]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("case", CASES)
def test_identity_table_equals_library_sdpa(case, dtype):
    n, H, hkv, d, bs, lens, window = case
    q, k, v, tables, cl, M = _identity_case(n, H, hkv, d, bs, dtype, lens, seed=7 + H + d)
    scale = 1.0 / math.sqrt(d)
    got = oracle.paged_attention(q, k, v, tables, cl, num_kv_heads=hkv, scale=scale, window=window)
    ref = _sdpa_reference(q, k, v, cl, M, bs, hkv, window=window, scale=scale)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", DTYPES)
def test_random_block_permutation_is_bit_identical(dtype):
    n, H, hkv, d, bs, lens = 3, 8, 2, 64, 16, [45, 80, 3]
    q, k, v, tables, cl, M = _identity_case(n, H, hkv, d, bs, dtype, lens, seed=99)
    nb = k.shape[0]
    spare = 5  # a bigger pool with unused blocks between the used ones
    perm = wl.permutation(1234, 1, nb + spare)[:nb]
    k2 = torch.zeros((nb + spare,) + tuple(k.shape[1:]), dtype=dtype)
    v2 = torch.zeros_like(k2)
    k2[perm] = k
    v2[perm] = v
    t2 = perm[tables.long()].to(torch.int32)
    a = oracle.paged_attention(q, k, v, tables, cl, num_kv_heads=hkv, scale=0.125)
    b = oracle.paged_attention(q, k2, v2, t2, cl, num_kv_heads=hkv, scale=0.125)
    assert np.array_equal(a, b)


def test_closed_forms():
    d, bs = 64, 16
    # identical keys -> uniform weights -> mean of V, whatever q is
    L = 37
    nb = 3
    k = torch.zeros(nb, 1, bs, d, dtype=torch.float32)
    k[:] = wl.normal_tensor(5, 1, (d,))
    v = wl.normal_tensor(5, 2, (nb, 1, bs, d))
    q = wl.normal_tensor(5, 3, (1, 1, d))
    tables = torch.tensor([[2, 0, 1]], dtype=torch.int32)
    got = oracle.paged_attention(q, k, v, tables, torch.tensor([L], dtype=torch.int32),
                                 num_kv_heads=1, scale=0.3)[0, 0]
    rows = [v[tables[0, t // bs], 0, t % bs].double() for t in range(L)]
    mean = torch.stack(rows).mean(0).numpy()
    assert np.allclose(got, mean, rtol=1e-13, atol=1e-15)
    # q = 0 -> mean of V for arbitrary keys
    k2 = wl.normal_tensor(5, 4, (nb, 1, bs, d))
    got0 = oracle.paged_attention(torch.zeros(1, 1, d), k2, v, tables,
                                  torch.tensor([L], dtype=torch.int32), num_kv_heads=1, scale=0.3)[0, 0]
    assert np.allclose(got0, mean, rtol=1e-13, atol=1e-15)
    # one token -> exactly V_0 (read through the table: block 2, offset 0)
    one = oracle.paged_attention(q, k2, v, tables, torch.tensor([1], dtype=torch.int32),
                                 num_kv_heads=1, scale=0.3)[0, 0]
    assert np.array_equal(one, v[2, 0, 0].double().numpy())
    # two tokens -> sigmoid(x0 - x1) v0 + sigmoid(x1 - x0) v1
    two = oracle.paged_attention(q, k2, v, tables, torch.tensor([2], dtype=torch.int32),
                                 num_kv_heads=1, scale=0.3)[0, 0]
    qd = q[0, 0].double()
    x0 = 0.3 * float(qd @ k2[2, 0, 0].double())
    x1 = 0.3 * float(qd @ k2[2, 0, 1].double())
    s0 = 1.0 / (1.0 + math.exp(x1 - x0))
    s1 = 1.0 / (1.0 + math.exp(x0 - x1))
    ref2 = s0 * v[2, 0, 0].double().numpy() + s1 * v[2, 0, 1].double().numpy()
    assert np.allclose(two, ref2, rtol=1e-12, atol=1e-14)
    # empty context -> zeros
    z = oracle.paged_attention(q, k2, v, tables, torch.tensor([0], dtype=torch.int32),
                               num_kv_heads=1, scale=0.3)
    assert np.array_equal(z, np.zeros_like(z))


def test_worked_example_inside_attention():
    """Token 34 of the page's table [7, 1, 3] is read at block 3, offset 2:
    give it the only large score and the output is that row of V."""
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    bs, d = g["block_size"], 64
    nb = 8
    k = torch.zeros(nb, 1, bs, d)
    v = wl.normal_tensor(3, 1, (nb, 1, bs, d))
    q = torch.zeros(1, 1, d)
    q[0, 0, 0] = 1.0
    k[g["physical"], 0, g["offset"], 0] = 60.0     # score 60 vs 0 elsewhere
    tables = torch.tensor([g["block_table"]], dtype=torch.int32)
    out = oracle.paged_attention(q, k, v, tables, torch.tensor([g["token"] + 1], dtype=torch.int32),
                                 num_kv_heads=1, scale=1.0)[0, 0]
    assert np.allclose(out, v[g["physical"], 0, g["offset"]].double().numpy(), rtol=0, atol=1e-20)


def test_dominant_score_is_one_hot_within_1e12():
    d, bs = 128, 16
    k = wl.normal_tensor(9, 1, (4, 2, bs, d)) * 0.01
    v = wl.normal_tensor(9, 2, (4, 2, bs, d))
    q = torch.zeros(1, 4, d)
    q[0, :, 0] = 1.0
    k[1, 1, 5, 0] = 60.0                               # token 21 of a 2-block table [3, 1]
    tables = torch.tensor([[3, 1]], dtype=torch.int32)
    out = oracle.paged_attention(q, k, v, tables, torch.tensor([30], dtype=torch.int32),
                                 num_kv_heads=2, scale=1.0)
    for h in (2, 3):                                   # heads of kv head 1
        assert np.allclose(out[0, h], v[1, 1, 5].double().numpy(), rtol=0, atol=1e-12)


def test_invalid_block_ids():
    d, bs = 64, 16
    q, k, v, tables, cl, M = _identity_case(1, 2, 2, d, bs, torch.float32, [40], seed=4)
    bad = tables.clone()
    bad[0, 1] = 10_000
    with pytest.raises(ValueError):
        oracle.paged_attention(q, k, v, bad, cl, num_kv_heads=2, scale=0.125)
    out, skipped = oracle.paged_attention(q, k, v, bad, cl, num_kv_heads=2, scale=0.125,
                                          invalid_policy=1, return_skipped=True)
    assert skipped == 2 * bs  # 16 tokens, for each of the 2 heads
    # tokens 16..31 left out == attention over tokens 0..15 and 32..39 (library SDPA)
    kc = k.reshape(M, 2, bs, d).permute(1, 0, 2, 3).reshape(2, M * bs, d).double()
    vc = v.reshape(M, 2, bs, d).permute(1, 0, 2, 3).reshape(2, M * bs, d).double()
    keep = torch.cat([torch.arange(0, 16), torch.arange(32, 40)])
    ref = F.scaled_dot_product_attention(q[0].double().unsqueeze(1), kc[:, keep], vc[:, keep],
                                         scale=0.125).squeeze(1).numpy()
    assert np.allclose(out[0], ref, rtol=1e-12, atol=1e-14)


def test_pairs_subset_matches_full():
    q, k, v, tables, cl, M = _identity_case(3, 4, 2, 64, 8, torch.float16, [20, 5, 64], seed=21)
    full = oracle.paged_attention(q, k, v, tables, cl, num_kv_heads=2, scale=0.125, threads=3)
    pairs = [[2, 3], [0, 1], [1, 0]]
    sub = oracle.paged_attention(q, k, v, tables, cl, num_kv_heads=2, scale=0.125, pairs=pairs)
    for i, (s, h) in enumerate(pairs):
        assert np.array_equal(sub[i], full[s, h])
