"""The native block manager against the oracle's own block-table models
(CowModel / RingModel, written separately in plain Python) and the pages'
worked examples.  CPU only."""
import json
from pathlib import Path

import pytest
import torch

from oracle import CowModel, RingModel
import oracle

GOLDEN = Path(__file__).parent / "golden"


@pytest.fixture(scope="module")
def BM():
    from paged_kv_cache_251_gb300 import build
    build.build()
    from paged_kv_cache_251_gb300.blocks import BlockManager
    return BlockManager


def test_worked_example_slot(BM):
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    bs = g["block_size"]
    order = g["block_table"] + [b for b in range(16) if b not in g["block_table"]]
    bm = BM(16, bs, 1, 8, free_order=order)
    bm.add_sequence(0)
    slots, pairs = bm.extend(0, g["token"] + 1)
    assert slots[g["token"]].item() == g["physical"] * bs + g["offset"]
    t, lens = bm.tables()
    assert t[0, :3].tolist() == g["block_table"] and lens[0] == g["token"] + 1
    assert pairs.numel() == 0


def test_cow_worked_example(BM):
    g = json.loads((GOLDEN / "cow_example.json").read_text())
    bm = BM(32, 16, g["sharers"], 4)
    bm.add_sequence(0)
    bm.extend(0, 8)                          # a half-full prompt block
    for c in range(1, g["sharers"]):
        bm.fork(0, c)
    shared = bm.tables()[0][0, 0].item()
    assert bm.refcount(shared) == g["sharers"]
    slots, pairs = bm.append([0])
    assert pairs.shape[0] == 1 and pairs[0, 0].item() == shared
    assert bm.refcount(shared) == g["after_first_write"]["shared_ref_count"]
    assert bm.refcount(pairs[0, 1].item()) == g["after_first_write"]["copy_ref_count"]
    assert slots[0].item() // 16 == pairs[0, 1].item()


def _random_ops(seed, n_ops=400):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 1 << 30, (n_ops, 3), generator=g).tolist()


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_random_ops_match_the_oracle_model(BM, seed, bs):
    nb, S, M = 400, 12, 64
    order = torch.randperm(nb, generator=torch.Generator().manual_seed(seed)).tolist()
    bm = BM(nb, bs, S, M, free_order=order)
    model = CowModel(bs, order)
    lens = {}                                                 # tokens per live sequence
    for op, a, b in _random_ops(seed):
        kind = op % 10
        free_ids = sorted(set(range(S)) - set(lens))
        if kind == 0 and free_ids:                            # new sequence
            sid = free_ids[0]
            bm.add_sequence(sid)
            model.add_sequence(sid)
            lens[sid] = 0
        elif kind == 1 and lens and free_ids:                 # fork
            parent = sorted(lens)[a % len(lens)]
            child = free_ids[0]
            bm.fork(parent, child)
            model.fork(parent, child)
            lens[child] = lens[parent]
        elif kind == 2 and len(lens) > 1:                     # free
            sid = sorted(lens)[a % len(lens)]
            bm.free_sequence(sid)
            model.free_sequence(sid)
            del lens[sid]
        elif lens:                                            # a batch of appends
            ids = sorted(lens)
            batch = [ids[(a + i * 7) % len(ids)] for i in range(1 + b % 9)]
            budget = dict(lens)
            ok = []
            for sid in batch:                                 # keep within the table row
                if budget[sid] < (M - 1) * bs:
                    ok.append(sid)
                    budget[sid] += 1
            if not ok:
                continue
            slots, pairs = bm.append(ok)
            exp_slots, exp_pairs = [], []
            for sid in ok:
                slot, cp = model.write(sid, lens[sid])
                lens[sid] += 1
                exp_slots.append(slot)
                if cp:
                    exp_pairs.append(list(cp))
            assert slots.tolist() == exp_slots
            assert pairs.tolist() == exp_pairs
    t, tl = bm.tables()
    for sid, n in lens.items():
        row = model.tables[sid]
        assert t[sid, :len(row)].tolist() == row
        assert all(x == -1 for x in t[sid, len(row):].tolist())
        assert tl[sid] == n
    for blk in range(nb):
        assert bm.refcount(blk) == model.ref.get(blk, 0)
    assert bm.num_free() == len(model.free)


def test_prefix_sharing_cow_counts(BM):
    """32 prompts x 2000 tokens, 8 samples each: block 32 copies the partial
    last prompt block 7 times per prompt (224); blocks 8 and 16 end the prompt
    on a block boundary and copy nothing."""
    for bs, expect in ((8, 0), (16, 0), (32, 224)):
        prompts, samples, plen = 32, 8, 2000
        nb = prompts * ((plen + bs - 1) // bs) + prompts * samples * (256 // bs + 2)
        bm = BM(nb, bs, prompts * samples, (plen + 256) // bs + 2)
        for p in range(prompts):
            base = p * samples
            bm.add_sequence(base)
            bm.extend(base, plen)
            for j in range(1, samples):
                bm.fork(base, base + j)
        slots, pairs = bm.append(list(range(prompts * samples)))   # first divergent token each
        assert pairs.shape[0] == expect
        # no slot is written twice, and no written block is still shared
        assert len(set(slots.tolist())) == slots.numel()
        for s in slots.tolist():
            assert bm.refcount(s // bs) == 1


def test_window_ring_matches_the_oracle_model_and_moves_nothing(BM):
    bs, W = 16, 80
    R = -(-W // bs) + 1
    M = 64
    bm = BM(50, bs, 2, M, free_order=list(range(49, -1, -1)))
    bm.add_sequence(0, ring_blocks=R)
    slots, pairs = bm.extend(0, 700)
    assert pairs.numel() == 0                     # a window never copies
    ring = [49 - i for i in range(R)]
    model = RingModel(bs, ring, table_len=M, stale=-1)
    assert slots.tolist() == [model.write(t) for t in range(700)]
    t, lens = bm.tables()
    assert t[0].tolist() == model.table and lens[0] == 700
    assert bm.num_free() == 50 - R
    # the last W tokens are all still addressable through the table
    for tok in range(700 - W, 700):
        phys, off = oracle.locate(t[0].tolist(), bs, tok)
        assert phys * bs + off == slots[tok].item()


def test_exhaustion_and_bad_arguments(BM):
    from paged_kv_cache_251_gb300.pa import PagedAttentionError
    bm = BM(2, 16, 2, 8)
    bm.add_sequence(0)
    bm.extend(0, 32)
    with pytest.raises(PagedAttentionError) as e:
        bm.append([0])
    assert e.value.status == 5
    with pytest.raises(PagedAttentionError):
        bm.add_sequence(0)                        # already live
    with pytest.raises(ValueError):
        BM(4, 16, 1, 4, free_order=[0, 0, 1, 2])  # not a permutation
