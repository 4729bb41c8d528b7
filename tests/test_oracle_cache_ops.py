"""Pins of the oracle's append, block copy, copy-on-write and window-ring models.

Facts used: the study-notes page's worked examples (token 34 of table
[7, 1, 3] lives at physical block 3 offset 2; a block shared by 4 candidates
is copied for the first writer and its count drops to 3; the copy unit is one
block) and the sliding-window page's claim that recycling a page only rewrites
the table (no K/V bytes move).
"""
import json
from pathlib import Path

import pytest
import torch

import oracle
from oracle import CowModel, RingModel
from paged_kv_cache_251_gb300 import workloads as wl

GOLDEN = Path(__file__).parent / "golden"


def _pool(nb, hkv, bs, d, dtype=torch.float16, seed=1):
    k = wl.normal_tensor(seed, 1, (nb, hkv, bs, d), dtype=dtype)
    v = wl.normal_tensor(seed, 2, (nb, hkv, bs, d), dtype=dtype)
    return k, v


def test_append_worked_example_lands_at_block3_offset2():
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    bs, hkv, d = g["block_size"], 2, 64
    k, v = _pool(8, hkv, bs, d)
    k0, v0 = k.clone(), v.clone()
    kn = wl.normal_tensor(9, 1, (1, hkv, d), dtype=torch.float16)
    vn = wl.normal_tensor(9, 2, (1, hkv, d), dtype=torch.float16)
    phys, off = oracle.locate(g["block_table"], bs, g["token"])
    slot = phys * bs + off
    assert oracle.append_kv(k, v, kn, vn, [slot]) == 0
    # written exactly at (3, h, 2); every other byte unchanged
    assert torch.equal(k[3, :, 2], kn[0]) and torch.equal(v[3, :, 2], vn[0])
    k0[3, :, 2] = kn[0]
    v0[3, :, 2] = vn[0]
    assert torch.equal(k.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(v.view(torch.int16), v0.view(torch.int16))


def test_append_skips_padding_counts_out_of_range_refuses_duplicates():
    bs, hkv, d = 8, 1, 64
    k, v = _pool(4, hkv, bs, d, torch.float32)
    before = k.clone()
    kn = torch.ones(3, hkv, d)
    assert oracle.append_kv(k, v, kn, kn, [-1, 4 * bs, 4 * bs + 100]) == 2
    assert torch.equal(k, before)
    with pytest.raises(ValueError):
        oracle.append_kv(k, v, kn[:2], kn[:2], [5, 5])


def test_copy_blocks_copies_whole_blocks_only():
    bs, hkv, d = 16, 4, 128
    k, v = _pool(10, hkv, bs, d, torch.bfloat16)
    k0, v0 = k.clone(), v.clone()
    pairs = [[2, 7], [5, 0]]
    assert oracle.copy_blocks(k, v, pairs) == 0
    k0[7], v0[7], k0[0], v0[0] = k0[2], v0[2], k0[5], v0[5]
    assert torch.equal(k.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(v.view(torch.int16), v0.view(torch.int16))
    assert oracle.copy_blocks(k, v, [[3, 99]]) == 1
    with pytest.raises(ValueError):
        oracle.copy_blocks(k, v, [[1, 2], [2, 3]])        # a destination is also a source
    with pytest.raises(ValueError):
        oracle.copy_blocks(k, v, [[1, 4], [2, 4]])        # repeated destination


def test_cow_worked_example():
    g = json.loads((GOLDEN / "cow_example.json").read_text())
    bs = 16
    m = CowModel(bs, range(100))
    m.add_sequence(0)
    for t in range(bs // 2):                              # a half-full prompt block
        m.write(0, t)
    for c in range(1, g["sharers"]):
        m.fork(0, c)
    shared = m.tables[0][0]
    assert m.ref[shared] == g["sharers"]
    slot, copy = m.write(0, bs // 2)                      # the first candidate writes
    assert (copy is not None) == g["after_first_write"]["writer_copied"]
    assert copy[0] == shared and m.ref[shared] == g["after_first_write"]["shared_ref_count"]
    assert m.ref[copy[1]] == g["after_first_write"]["copy_ref_count"]
    assert slot // bs == copy[1]
    # the unit is one block: the sharer's other (full) blocks are untouched
    assert g["copy_unit"] == "block"


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_cow_counts_for_prefix_sharing(bs):
    """Each shared partial block is copied sharers-1 times; the last sharer
    writes in place; no write ever lands in a block that is still shared;
    full prompt blocks are never copied."""
    prompt, sharers = 2000, 8
    m = CowModel(bs, range(10_000))
    m.add_sequence(0)
    for t in range(prompt):
        m.write(0, t)
    for c in range(1, sharers):
        m.fork(0, c)
    copies = []
    for c in range(sharers):
        for t in range(prompt, prompt + 3):
            slot, cp = m.write(c, t)
            assert m.ref[slot // bs] == 1
            if cp:
                copies.append(cp)
    expect = (sharers - 1) if prompt % bs else 0
    assert len(copies) == expect
    # every sharer still reads the same prompt blocks except the partial one
    full = prompt // bs
    for c in range(sharers):
        assert m.tables[c][:full] == m.tables[0][:full]


def test_ring_window_moves_no_data_and_keeps_the_window():
    bs, W = 16, 64
    R = W // bs + 1
    ring = [11, 3, 7, 2, 9]
    assert len(ring) == R
    m = RingModel(bs, ring, table_len=40, stale=-1)
    slots = [m.write(t) for t in range(300)]
    assert m.data_moves == 0
    # every token of the last W tokens is still at the slot it was written to
    L = 300
    seen = {}
    for t in range(L - W, L):
        phys, off = oracle.locate(m.table, bs, t)
        assert phys * bs + off == slots[t]
        seen[slots[t]] = t
    assert len(seen) == W                       # no two window tokens share a slot
    # stale entries are the logical blocks the ring has recycled
    last = (L - 1) // bs
    assert all(m.table[lb] == -1 for lb in range(0, last - R + 1))


def test_swap_round_trip_restores_the_blocks_and_touches_nothing_else():
    bs, hkv, d = 16, 4, 64
    dk, dv = _pool(12, hkv, bs, d, torch.bfloat16, seed=5)
    hk = torch.zeros((5,) + tuple(dk.shape[1:]), dtype=torch.bfloat16)
    hv = torch.zeros_like(hk)
    d0k, d0v = dk.clone(), dv.clone()
    out = [[3, 0], [7, 4], [11, 2]]
    assert oracle.swap_blocks(dk, dv, hk, hv, out) == 0
    for src, dst in out:
        assert torch.equal(hk[dst].view(torch.int16), dk[src].view(torch.int16))
        assert torch.equal(hv[dst].view(torch.int16), dv[src].view(torch.int16))
    assert torch.count_nonzero(hk[[1, 3]].view(torch.int16)) == 0      # untouched host blocks
    dk[3].zero_(), dv[3].zero_(), dk[7].zero_()
    assert oracle.swap_blocks(hk, hv, dk, dv, [[0, 3], [4, 7], [2, 11]]) == 0
    assert torch.equal(dk[[3, 11]].view(torch.int16), d0k[[3, 11]].view(torch.int16))
    assert torch.equal(dv[3].view(torch.int16), d0v[3].view(torch.int16))
    assert torch.equal(dk[7].view(torch.int16), d0k[7].view(torch.int16))
    assert oracle.swap_blocks(dk, dv, hk, hv, [[12, 0], [0, 5], [-1, 1]]) == 3
    with pytest.raises(ValueError):
        oracle.swap_blocks(dk, dv, hk, hv, [[1, 2], [3, 2]])
