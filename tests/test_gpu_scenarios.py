"""Full-size GPU parity of the two block-manager workloads:

- sliding window: 4 sequences of 131072 logical tokens, 32 q / 8 kv heads,
  d 128, bf16, block 16, window 32768 over rings of 2049 physical blocks,
  512-token partitions with the log-sum-exp reduce; then one more token per
  sequence (a table rewrite, no K/V movement) and decode again;
- prefix sharing: 32 prompts x 2000 tokens shared by 8 samples each, every
  sample appends U{1..256} tokens (copy-on-write of the partly filled last
  prompt block), then decode over all 256 samples; block 8, 16 and 32.

The oracle side rebuilds the tables with its own models (RingModel /
CowModel) and applies its own append and block copy; the pools must match
byte for byte and the attention outputs within the tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import CowModel, RingModel
from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _decode(q, k, v, bt, cl, hkv, window=0, partition=0):
    from paged_kv_cache_251_gb300 import pa
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(out, q, k, v, bt.cuda(), cl.cuda(), num_kv_heads=hkv, window=window, partition_size=partition,
                 err_word=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


def test_window_ring_full_size():
    from paged_kv_cache_251_gb300 import pa, scenarios
    st = scenarios.window_state(device="cuda")
    s = st.shape
    W, L, R = s.window, st.context, st.ring_blocks
    # the oracle's own ring model gives the same tables
    order = wl.permutation(s.seed, 2, st.num_blocks).tolist()
    models = []
    for i in range(s.num_seqs):
        m = RingModel(s.block_size, order[i * R:(i + 1) * R], table_len=st.block_tables.shape[1], stale=-1)
        for t in range(L):
            m.write(t)
        models.append(m)
        assert m.table == st.block_tables[i].tolist()
    scale = 1.0 / math.sqrt(s.head_dim)
    got, err = _decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, s.num_kv_heads, W, 512)
    assert err == 0
    kc, vc, q = st.k_cache.cpu(), st.v_cache.cpu(), st.q.cpu()
    ref = oracle.paged_attention(q, kc, vc, st.block_tables, st.context_lens, num_kv_heads=s.num_kv_heads,
                                 scale=scale, window=W, threads=16)
    compare(got, ref, s.dtype)

    # one more token per sequence: the ring recycles a page by a table rewrite
    slots, pairs = st.manager.append(list(range(s.num_seqs)))
    assert pairs.numel() == 0
    assert slots.tolist() == [models[i].write(L) for i in range(s.num_seqs)]
    tables, lens = st.manager.tables()
    assert [m.table for m in models] == tables.tolist()
    pa.pa_append_kv(st.k_new, st.v_new, slots.cuda(), st.k_cache, st.v_cache)
    oracle.append_kv(kc, vc, st.k_new.cpu(), st.v_new.cpu(), slots)
    torch.cuda.synchronize()
    # only the appended rows changed: no K/V data moved
    assert torch.equal(_bits(st.k_cache.cpu()), _bits(kc)) and torch.equal(_bits(st.v_cache.cpu()), _bits(vc))
    got1, err = _decode(st.q, st.k_cache, st.v_cache, tables, lens, s.num_kv_heads, W, 512)
    assert err == 0
    ref1 = oracle.paged_attention(q, kc, vc, tables, lens, num_kv_heads=s.num_kv_heads, scale=scale, window=W,
                                  threads=16)
    compare(got1, ref1, s.dtype)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefix_sharing_full_size(bs):
    from paged_kv_cache_251_gb300 import pa, scenarios
    st = scenarios.prefix_state(bs, device="cuda")
    s = st.shape
    # the oracle's own copy-on-write model gives the same pairs, slots and tables
    model = CowModel(bs, st.free_order.tolist())
    for p in range(st.prompts):
        first = p * st.samples
        model.add_sequence(first)
        for t in range(st.prompt_len):
            model.write(first, t)
        for j in range(1, st.samples):
            model.fork(first, first + j)
    pos = {i: st.prompt_len for i in range(s.num_seqs)}
    exp_slots, exp_pairs = [], []
    for sid in st.token_seq.tolist():
        slot, cp = model.write(sid, pos[sid])
        pos[sid] += 1
        exp_slots.append(slot)
        if cp:
            exp_pairs.append(list(cp))
    assert st.slots.tolist() == exp_slots and st.pairs.tolist() == exp_pairs
    assert len(exp_pairs) == (st.prompts * (st.samples - 1) if st.prompt_len % bs else 0)
    M = st.block_tables.shape[1]
    for sid in range(s.num_seqs):
        row = model.tables[sid]
        assert st.block_tables[sid, :len(row)].tolist() == row

    kc, vc = st.k_cache.cpu(), st.v_cache.cpu()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(st.pairs.cuda(), st.k_cache, st.v_cache, err_word=err)
    pa.pa_append_kv(st.k_new, st.v_new, st.slots.cuda(), st.k_cache, st.v_cache, err_word=err)
    oracle.copy_blocks(kc, vc, st.pairs)
    oracle.append_kv(kc, vc, st.k_new.cpu(), st.v_new.cpu(), st.slots)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(_bits(st.k_cache.cpu()), _bits(kc)) and torch.equal(_bits(st.v_cache.cpu()), _bits(vc))

    got, err2 = _decode(st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens, s.num_kv_heads)
    assert err2 == 0
    idx = wl.permutation(99, 1, s.num_seqs * s.num_heads)[:160]
    pairs = torch.stack([idx // s.num_heads, idx % s.num_heads], 1).to(torch.int32)
    ref = oracle.paged_attention(st.q.cpu(), kc, vc, st.block_tables, st.context_lens,
                                 num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim), pairs=pairs,
                                 threads=16)
    compare(got[pairs[:, 0].long(), pairs[:, 1].long()], ref, s.dtype)
