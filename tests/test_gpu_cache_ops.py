"""GPU parity of pa_append_kv and pa_copy_blocks: bit-exact against the oracle,
whole pools compared byte for byte (untouched blocks included)."""
import json
from pathlib import Path

import pytest
import torch

import oracle
from paged_kv_cache_251_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
GOLDEN = Path(__file__).parent / "golden"


def _bits(t):
    return t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)


def _pool(nb, hkv, bs, d, dtype, seed):
    return (wl.normal_tensor(seed, 1, (nb, hkv, bs, d), dtype=dtype),
            wl.normal_tensor(seed, 2, (nb, hkv, bs, d), dtype=dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("bs,d,hkv", [(16, 128, 8), (8, 64, 4), (32, 128, 40)])
def test_append_bit_exact(dtype, bs, d, hkv):
    from paged_kv_cache_251_gb300 import pa
    nb, T = 24, 37
    k, v = _pool(nb, hkv, bs, d, dtype, seed=bs + d)
    kn = wl.normal_tensor(5, 1, (T, hkv, d), dtype=dtype)
    vn = wl.normal_tensor(5, 2, (T, hkv, d), dtype=dtype)
    slots = wl.permutation(6, 1, nb * bs)[:T].clone()
    slots[3] = -1                                   # padding
    slots[10] = -1
    kg, vg = k.cuda(), v.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_append_kv(kn.cuda(), vn.cuda(), slots.cuda(), kg, vg, err_word=err)
    oracle.append_kv(k, v, kn, vn, slots)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(_bits(kg.cpu()), _bits(k)) and torch.equal(_bits(vg.cpu()), _bits(v))


def test_append_worked_example_slot():
    """Token 34 through the page's table [7, 1, 3] (block size 16) lands at
    physical block 3, offset 2."""
    from paged_kv_cache_251_gb300 import pa
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    bs, hkv, d = g["block_size"], 2, 128
    k, v = _pool(8, hkv, bs, d, torch.float16, seed=1)
    kg, vg = k.cuda(), v.cuda()
    kn = torch.full((1, hkv, d), 7.0, dtype=torch.float16)
    slot = g["physical"] * bs + g["offset"]
    pa.pa_append_kv(kn.cuda(), kn.cuda(), torch.tensor([slot], dtype=torch.int64).cuda(), kg, vg)
    torch.cuda.synchronize()
    kc = kg.cpu()
    assert torch.all(kc[3, :, 2] == 7.0)
    kc[3, :, 2] = k[3, :, 2]
    assert torch.equal(_bits(kc), _bits(k))


def test_append_out_of_range_slot_flagged_and_skipped():
    from paged_kv_cache_251_gb300 import pa
    nb, hkv, bs, d = 4, 2, 16, 64
    k, v = _pool(nb, hkv, bs, d, torch.float32, seed=3)
    kg, vg = k.cuda(), v.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kn = torch.ones(2, hkv, d)
    pa.pa_append_kv(kn.cuda(), kn.cuda(), torch.tensor([nb * bs, 1 << 40]).cuda(), kg, vg, err_word=err)
    torch.cuda.synchronize()
    assert err.item() & 2
    assert torch.equal(kg.cpu(), k) and torch.equal(vg.cpu(), v)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_copy_blocks_bit_exact(dtype, bs):
    from paged_kv_cache_251_gb300 import pa
    nb, hkv, d = 64, 8, 128
    k, v = _pool(nb, hkv, bs, d, dtype, seed=bs)
    perm = wl.permutation(9, 1, nb)
    pairs = torch.stack([perm[:20], perm[20:40]], dim=1).contiguous()
    kg, vg = k.cuda(), v.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(pairs.cuda(), kg, vg, err_word=err)
    oracle.copy_blocks(k, v, pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(_bits(kg.cpu()), _bits(k)) and torch.equal(_bits(vg.cpu()), _bits(v))


def test_copy_blocks_bad_pair_flagged_and_empty_list():
    from paged_kv_cache_251_gb300 import pa
    nb, hkv, bs, d = 8, 2, 16, 64
    k, v = _pool(nb, hkv, bs, d, torch.float16, seed=4)
    kg, vg = k.cuda(), v.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(torch.zeros((0, 2), dtype=torch.int64).cuda(), kg, vg, err_word=err)
    pa.pa_copy_blocks(torch.tensor([[1, nb], [-1, 2], [3, 5]]).cuda(), kg, vg, err_word=err)
    torch.cuda.synchronize()
    assert err.item() & 4
    k[5], v[5] = k[3], v[3]
    assert torch.equal(_bits(kg.cpu()), _bits(k)) and torch.equal(_bits(vg.cpu()), _bits(v))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_swap_out_to_pinned_host_and_back_bit_exact(dtype):
    """Swap blocks GPU -> pinned host -> GPU (other slots); pools compared byte
    for byte with the oracle after each direction."""
    from paged_kv_cache_251_gb300 import pa
    nb, hb, hkv, bs, d = 40, 24, 8, 16, 128
    k, v = _pool(nb, hkv, bs, d, dtype, seed=11)
    kg, vg = k.cuda(), v.cuda()
    hk = torch.zeros((hb, hkv, bs, d), dtype=dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    ok_, ov_ = torch.zeros_like(hk), torch.zeros_like(hv)
    perm = wl.permutation(12, 1, nb)
    out_pairs = torch.stack([perm[:20], wl.permutation(13, 1, hb)[:20]], 1).contiguous()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_swap_blocks(out_pairs.cuda(), kg, vg, hk, hv, err_word=err)
    oracle.swap_blocks(k, v, ok_, ov_, out_pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(_bits(hk), _bits(ok_)) and torch.equal(_bits(hv), _bits(ov_))
    # swap back in to other device blocks; the pairs live in pinned host memory
    in_pairs = torch.stack([out_pairs[:, 1], perm[20:40]], 1).contiguous().pin_memory()
    pa.pa_swap_blocks(in_pairs, hk, hv, kg, vg, err_word=err)
    oracle.swap_blocks(ok_, ov_, k, v, in_pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(_bits(kg.cpu()), _bits(k)) and torch.equal(_bits(vg.cpu()), _bits(v))
    # a pair outside a pool is skipped and flagged
    pa.pa_swap_blocks(torch.tensor([[0, hb]], dtype=torch.int64).cuda(), kg, vg, hk, hv, err_word=err)
    torch.cuda.synchronize()
    assert err.item() & 4
    assert torch.equal(_bits(hk), _bits(ok_))
