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


def test_reference_arm_loads_no_product_code():
    """bench.py --impl reference runs the oracle on inputs from the seeded
    generator and the oracle's own block-table models: the CUDA library and
    its host block manager are never loaded."""
    import subprocess
    import sys
    root = Path(__file__).resolve().parent.parent
    code = (
        "import json, sys, io, contextlib, bench\n"
        "buf = io.StringIO()\n"
        "with contextlib.redirect_stdout(buf):\n"
        "    bench.main(['--impl', 'reference', '--workload', 'tiny', '--steps', '1', '--warmup', '1'])\n"
        "line = json.loads(buf.getvalue().strip().splitlines()[-1])\n"
        "maps = open('/proc/self/maps').read()\n"
        "print(json.dumps({'impl': line['impl'], 'value': line['value'],\n"
        "                  'libpa': 'libpa.so' in maps, 'liboracle': 'liboracle.so' in maps,\n"
        "                  'mods': [m for m in sys.modules if m.startswith('paged_kv_cache_251_gb300.')]}))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got["impl"] == "reference" and got["value"] > 0
    assert got["liboracle"] and not got["libpa"]
    assert set(got["mods"]) <= {"paged_kv_cache_251_gb300.workloads"}


def test_oracle_step_tables_match_the_block_manager():
    """The reference arm's tables, slots and copy-on-write pairs (oracle
    models) equal the native arm's (the C++ block manager) on small versions
    of the window and prefix-sharing workloads, and its append slots equal
    the block tables' translation of position L."""
    from paged_kv_cache_251_gb300 import scenarios
    ws = scenarios.window_state(context=4096, window=1024)
    slots, _ = ws.manager.append(list(range(ws.shape.num_seqs)))
    ost = bench.OracleStep.__new__(bench.OracleStep)
    import oracle
    ost.oracle = oracle
    ost._window(context=4096, window=1024)
    assert torch.equal(ost.tables[:, :ws.block_tables.shape[1]], ws.block_tables)
    assert torch.equal(ost.lens, ws.context_lens) and torch.equal(ost.slots, slots)
    for bs in (8, 32):
        ps = scenarios.prefix_state(bs, prompts=4, samples=3, prompt_len=100, max_new=40)
        ost = bench.OracleStep.__new__(bench.OracleStep)
        ost.oracle = oracle
        ost._prefix(bs, False, prompts=4, samples=3, prompt_len=100, max_new=40)
        assert torch.equal(ost.tables, ps.block_tables) and torch.equal(ost.lens, ps.context_lens)
        assert torch.equal(ost.slots, ps.slots) and torch.equal(ost.pairs, ps.pairs)
        assert (ost.pairs.shape[0] > 0) == (100 % bs != 0)


def test_kernel_source_hash_ignores_comments_and_layout_but_not_code(tmp_path):
    """The hash that keys the ncu traffic figures in profiles/ to the kernel
    sources changes with the code only."""
    import bench
    src = tmp_path / "a"
    src.mkdir()
    (src / "pa_decode_x.cuh").write_text("// a comment\nint f(int x) {\n    return x + 1;  // add one\n}\n/* block\n comment */\n")
    (src / "other.cu").write_text("int unrelated;\n")
    h0 = bench.kernel_source_hash(str(src))
    (src / "pa_decode_x.cuh").write_text("// another comment\nint f(int x) { return x + 1; }\n")
    assert bench.kernel_source_hash(str(src)) == h0
    (src / "other.cu").write_text("int changed_but_not_hashed;\n")
    assert bench.kernel_source_hash(str(src)) == h0
    (src / "pa_decode_x.cuh").write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_source_hash(str(src)) != h0
