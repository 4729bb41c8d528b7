"""CPU checks of the benchmark's host logic: byte accounting against the
pages' printed KV sizes, and the max-over-ranks timing with two gloo ranks."""
import json
import os
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

import bench
from paged_kv_cache_251_gb300 import accounting as acc

GOLDEN = Path(__file__).parent / "golden"


def test_kv_bytes_match_the_pages_examples():
    g = json.loads((GOLDEN / "kv_bytes_per_token.json").read_text())
    o = g["opt13b"]
    per_tok = acc.kv_bytes_per_token(o["num_heads"], o["head_dim"], o["elt_bytes"], layers=o["layers"])
    assert per_tok == o["bytes_per_token"] and per_tok / 1024 == o["kib_per_token"]
    assert per_tok * o["tokens"] / 1024 ** 3 == o["gib_for_tokens"]
    l70 = g["llama2_70b"]
    per_tok = acc.kv_bytes_per_token(l70["num_heads"], l70["head_dim"], l70["elt_bytes"], layers=l70["layers"])
    assert per_tok == l70["bytes_per_token"] and per_tok / 2 ** 20 == l70["mib_per_token"]


def test_decode_bytes_counts_attended_tokens_and_blocks():
    lens = torch.tensor([0, 1, 16, 17, 100], dtype=torch.int32)
    b = acc.decode_bytes(lens, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16, elt_bytes=2)
    assert b["attended_tokens"] == 134
    assert b["kv"] == 134 * 2 * 2 * 64 * 2
    assert b["table"] == (0 + 1 + 1 + 2 + 7) * 4 + 5 * 4
    w = acc.decode_bytes(lens, num_heads=8, num_kv_heads=2, head_dim=64, block_size=16, elt_bytes=2, window=10)
    assert w["attended_tokens"] == 0 + 1 + 10 + 10 + 10
    # window 10 over L = 100 touches tokens 90..99: blocks 5 and 6
    assert w["table"] == (0 + 1 + 1 + 2 + 2) * 4 + 5 * 4


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    v = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    q.put((rank, v))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_bench_defaults_and_peak_file():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.steps >= 1 and a.warmup >= 3 and a.impl == "native"
    peak, kind = bench.hbm_peak()
    assert peak > 1000 and kind in ("measured", "fallback")
