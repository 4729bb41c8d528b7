"""GPU parity of pa_decode against the fp64 oracle (through the C ABI)."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare, make_inputs, oracle_decode, run_decode, shape, to_cuda

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# (N, H, H_kv, d, bs, lens, window, partition)  — each spans several tiles and a ragged tail
EDGE_CASES = [
    ("ctx_edges_bs16", 6, 4, 4, 64, 16, [1, 15, 16, 17, 512, 513], 0, 0),
    ("ctx_edges_bs8", 6, 8, 2, 128, 8, [1, 7, 8, 9, 512, 513], 0, 0),
    ("ctx_edges_bs32", 5, 8, 8, 128, 32, [31, 32, 33, 1000, 1025], 0, 0),
    ("one_seq_long", 1, 4, 1, 128, 16, [3001], 0, 0),
    ("many_parts", 3, 8, 2, 64, 16, [700, 129, 64], 0, 32),
    ("window_unaligned", 4, 8, 2, 128, 16, [100, 37, 500, 1200], 37, 0),
    ("window_ge_ctx", 3, 4, 4, 64, 16, [20, 50, 9], 64, 0),
    ("window_parts", 3, 8, 1, 128, 16, [2000, 777, 40], 300, 64),
    ("gqa8", 3, 16, 2, 128, 16, [90, 400, 1], 0, 0),
    ("gqa2_d64", 4, 8, 4, 64, 32, [65, 66, 700, 2], 0, 0),
    ("empty_seq", 3, 4, 2, 64, 16, [0, 33, 0], 0, 0),
    # one query head per kv head at every block size (the TMA-tensor kernel)
    ("mha_bs8_d128", 4, 6, 6, 128, 8, [9, 700, 1, 255], 0, 0),
    ("mha_bs32_d64", 4, 4, 4, 64, 32, [33, 31, 1100, 64], 0, 0),
    ("mha_bs16_parts", 3, 5, 5, 128, 16, [2000, 100, 513], 0, 64),
    ("mha_window", 3, 4, 4, 128, 16, [1000, 20, 777], 100, 0),
    ("mha_empty", 3, 2, 2, 64, 8, [0, 5, 0], 0, 0),
    # grouped heads, head_dim 128 (the tensor-core kernel for 16-bit K/V)
    ("tc_g2_bs32", 4, 4, 2, 128, 32, [129, 31, 1000, 257], 0, 0),
    ("tc_g4_parts", 3, 8, 2, 128, 16, [700, 129, 2049], 0, 64),
    ("tc_g8_bs8_window", 3, 16, 2, 128, 8, [5000, 77, 1300], 1000, 0),
    ("tc_empty", 3, 8, 1, 128, 8, [0, 300, 0], 0, 0),
    # many one-tile items of one or two blocks (16-token partitions at block 8),
    # empty and one-token sequences among them; up to 63 partitions per row
    ("tc_many_items", 24, 32, 8, 128, 8,
     [0, 1, 7, 8, 9, 16, 17, 100, 255, 256, 257, 0, 511, 512, 513, 3, 64, 1000, 129, 0, 33, 48, 2, 700], 0, 16),
    # long partitions: 64 / 128 / 256 blocks per item
    ("tc_g4_p1024", 3, 8, 2, 128, 16, [3000, 1100, 77], 0, 1024),
    ("tc_g8_bs32_p4096", 2, 16, 2, 128, 32, [5000, 2100], 0, 4096),
    ("mha_p2048", 2, 4, 4, 128, 8, [3000, 2100], 0, 2048),
]


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("case", EDGE_CASES, ids=[c[0] for c in EDGE_CASES])
def test_decode_edge_cases(case, dt):
    name, n, h, hkv, d, bs, lens, window, part = case
    sh = shape(name, n, h, hkv, d, bs, DT[dt], window=window, seed=17 + n + d + bs)
    inp = make_inputs(sh, lens)
    got, err = run_decode(inp, partition_size=part)
    assert err == 0
    compare(got, oracle_decode(inp), DT[dt])


@pytest.mark.parametrize("out_dt", ["f16", "bf16"])
def test_decode_low_precision_output(out_dt):
    sh = shape("lowout", 4, 8, 2, 128, 16, torch.bfloat16, seed=3)
    inp = make_inputs(sh, [300, 17, 600, 1])
    got, err = run_decode(inp, out_dtype=DT[out_dt])
    assert err == 0 and got.dtype == DT[out_dt]
    compare(got, oracle_decode(inp), torch.bfloat16)


def test_tiny_config():
    """4 sequences, 4 MHA heads, d 64, block 16, fp32, L ~ U[1,100], 64-block pool."""
    inp = wl.tiny()
    got, err = run_decode(inp)
    assert err == 0
    compare(got, oracle_decode(inp), torch.float32)


@pytest.mark.parametrize("hkv,d", [(4, 64), (2, 64), (2, 128)])
def test_invalid_table_entries_are_skipped_and_flagged(hkv, d):
    sh = shape("bad", 3, 4, hkv, d, 16, torch.float16, seed=8)
    inp = make_inputs(sh, [70, 40, 33])
    bt = inp.block_tables.clone()
    bt[0, 1] = inp.num_blocks + 5        # out of the pool
    bt[2, 0] = -7
    got, err = run_decode(inp, block_tables=bt)
    assert err & 1
    ref = oracle_decode(inp, block_tables=bt, invalid_policy=1)
    compare(got, ref, torch.float16)


def test_context_beyond_table_row_is_clamped_and_flagged():
    sh = shape("len", 2, 4, 4, 64, 16, torch.float32, seed=9)
    inp = make_inputs(sh, [40, 20])
    M = inp.block_tables.shape[1]
    cl = torch.tensor([M * 16 + 100, 20], dtype=torch.int32)
    got, err = run_decode(inp, context_lens=cl)
    assert err & 16
    # seq 0 is clamped to M*16 tokens; its table holds -1 beyond its 3 blocks
    ref = oracle_decode(inp, context_lens=torch.tensor([M * 16, 20], dtype=torch.int32), invalid_policy=1)
    compare(got, ref, torch.float32)


@pytest.mark.parametrize("hkv", [8, 2])
def test_table_entries_outside_the_window_are_never_read(hkv):
    """A sliding window touches only its own table entries: poison the rest."""
    sh = shape("win", 2, 8, hkv, 128, 16, torch.bfloat16, window=256, seed=10)
    inp = make_inputs(sh, [1000, 900])
    bt = inp.block_tables.clone()
    for s, L in enumerate([1000, 900]):
        first = (L - 256) // 16
        bt[s, :first] = 0x7FFFFFFF
    got, err = run_decode(inp, block_tables=bt)
    assert err == 0
    compare(got, oracle_decode(inp, block_tables=bt), torch.bfloat16)


def _sample_pairs(N, H, count, seed):
    idx = wl.permutation(seed, 1, N * H)[:count]
    return torch.stack([idx // H, idx % H], dim=1).to(torch.int32)


@pytest.mark.parametrize("name", ["opt13b", "gqa", "tiny_scaled"])
def test_full_size_config_sampled(name):
    """Full-size workloads in the launch configuration the benchmark times
    (inputs generated on the GPU); every output is finite and a sample of rows
    matches the oracle."""
    if name == "opt13b":
        inp = wl.decode_inputs(wl.SHAPES["opt13b"], device="cuda")
    elif name == "gqa":
        inp = wl.decode_inputs(wl.SHAPES["gqa"], device="cuda", room_for_append=False, fill=0.95,
                               with_append=False)
    else:
        inp = wl.decode_inputs(wl.SHAPES["tiny_scaled"], device="cuda")
    got, err = run_decode(inp)
    assert err == 0
    s = inp.shape
    pairs = _sample_pairs(s.num_seqs, s.num_heads, 96, seed=77)
    ref = oracle_decode(inp, pairs=pairs)
    sel = got[pairs[:, 0].long(), pairs[:, 1].long()]
    compare(sel, ref, s.dtype)


def test_full_gqa_batch_is_repeatable():
    """The tensor-core grouped-head kernel on the full GQA batch (items claimed
    from a counter), decoded twelve times: each item is computed by one CTA and
    partitions merge in a fixed order, so every run's output is bit-identical."""
    inp = wl.decode_inputs(wl.SHAPES["gqa"], device="cuda", room_for_append=False, fill=0.95, with_append=False)
    first, err = run_decode(inp)
    assert err == 0
    for _ in range(11):
        got, err = run_decode(inp)
        assert err == 0
        assert torch.equal(got, first)


@pytest.mark.parametrize("hkv", [8, 32])
def test_decode_replayed_from_a_cuda_graph(hkv):
    """pa_decode captured in a CUDA graph and replayed twenty times (no
    allocation or host synchronisation on the launch path; the item counter a
    launch claims from is returned to zero by its last CTA, so every replay
    starts from zero): every replay gives the eager result bit for bit (the
    grouped-head tensor-core kernel, hkv = 8, and the MHA kernel, hkv = 32),
    and the eager result matches the oracle."""
    from paged_kv_cache_251_gb300 import pa
    lens = [(37 * i * i + 300 * i) % 2100 + 1 for i in range(64)]  # 64 sequences: more items than CTAs
    sh = shape("graph", 64, 32, hkv, 128, 16, torch.bfloat16, seed=23)
    inp = make_inputs(sh, lens)
    dev = to_cuda(inp)
    out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pa.workspace_for(dev["q"], 16, dev["block_tables"].shape[1])

    def call():
        pa.pa_decode(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                     num_kv_heads=hkv, workspace=ws, err_word=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # eager, on the stream the capture will use
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(20):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert int(err.item()) == 0
    compare(eager.cpu(), oracle_decode(inp), torch.bfloat16)


def test_concurrent_launches_on_two_streams():
    """Two decode workloads (the tensor-core and the MHA kernel, each claiming
    items from a counter) launched ten times each on two streams without a
    synchronisation in between: launches in flight take different counter
    pairs, so both keep their single-stream results bit for bit."""
    from paged_kv_cache_251_gb300 import pa
    lens = [(37 * i * i + 300 * i) % 2100 + 1 for i in range(64)]
    cases = []
    for hkv, seed in ((8, 29), (32, 31)):
        inp = make_inputs(shape("streams", 64, 32, hkv, 128, 16, torch.bfloat16, seed=seed), lens)
        dev = to_cuda(inp)
        out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = pa.workspace_for(dev["q"], 16, dev["block_tables"].shape[1])
        cases.append((inp, dev, out, err, ws, hkv, torch.cuda.Stream()))

    def call(c):
        inp, dev, out, err, ws, hkv, st = c
        pa.pa_decode(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                     num_kv_heads=hkv, workspace=ws, err_word=err, stream=st)

    alone = []
    for c in cases:
        call(c)
        torch.cuda.synchronize()
        alone.append(c[2].clone())
    for c in cases:
        c[6].wait_stream(torch.cuda.current_stream())
    for _ in range(10):
        for c in cases:
            call(c)
    torch.cuda.synchronize()
    for c, ref in zip(cases, alone):
        assert int(c[3].item()) == 0
        assert torch.equal(c[2], ref)
    compare(cases[0][2].cpu(), oracle_decode(cases[0][0]), torch.bfloat16)


def test_graph_replays_overlap_more_than_4096_eager_launches():
    """A decode captured in a CUDA graph keeps its item counter for every
    replay, and eager launches take theirs round-robin from 4096 others, so
    the two never share one.  The graph (the MHA kernel) is replayed 100
    times on one stream while 4200 eager decodes (the tensor-core kernel; more
    launches than round-robin counters) run on another: every replay's output
    equals the eager result of the same inputs bit for bit, and both match
    the oracle."""
    from paged_kv_cache_251_gb300 import pa
    lens = [(37 * i * i + 300 * i) % 2100 + 1 for i in range(64)]   # more items than CTAs: counters in use
    cases = []
    for hkv, seed in ((32, 41), (8, 43)):
        inp = make_inputs(shape("overlap", 64, 32, hkv, 128, 16, torch.bfloat16, seed=seed), lens)
        dev = to_cuda(inp)
        out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = pa.workspace_for(dev["q"], 16, dev["block_tables"].shape[1])
        cases.append((inp, dev, out, err, ws, hkv))

    def call(c):
        inp, dev, out, err, ws, hkv = c
        pa.pa_decode(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                     num_kv_heads=hkv, workspace=ws, err_word=err)

    call(cases[0])
    torch.cuda.synchronize()
    ref_a = cases[0][2].clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(cases[0])
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    worst = torch.zeros((), dtype=torch.float32, device="cuda")
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    for i in range(4200):
        with torch.cuda.stream(sb):
            call(cases[1])
        if i % 42 == 0:
            with torch.cuda.stream(sa):
                cases[0][2].fill_(float("nan"))
                graph.replay()
                torch.maximum(worst, (cases[0][2] - ref_a).abs().amax().nan_to_num(float("inf")), out=worst)
    torch.cuda.synchronize()
    assert float(worst.item()) == 0.0
    assert int(cases[0][3].item()) == 0 and int(cases[1][3].item()) == 0
    compare(ref_a.cpu(), oracle_decode(cases[0][0]), torch.bfloat16)
    compare(cases[1][2].cpu(), oracle_decode(cases[1][0]), torch.bfloat16)


def test_full_opt13b_batch_is_repeatable():
    """The MHA kernel on the full OPT-13B-shaped batch (items claimed from a
    counter), decoded twelve times: block j of every item is summed by
    consumer warp j % 4 whatever the CTA ran before, and the warps merge in a
    fixed order, so every run's output is bit-identical."""
    inp = wl.decode_inputs(wl.SHAPES["opt13b"], device="cuda")
    first, err = run_decode(inp)
    assert err == 0
    for _ in range(11):
        got, err = run_decode(inp)
        assert err == 0
        assert torch.equal(got, first)


def test_decode_from_several_host_threads():
    """The library is called from four host threads at once, each on its own
    stream with its own workload (MHA and tensor-core decodes, an append, an
    8-bit decode): ctypes releases the GIL, so the calls really overlap on the
    host (per-thread tensor-map caches, the shared device facts and counter
    pool).  Every thread's results equal the single-threaded ones bit for bit."""
    import threading
    from paged_kv_cache_251_gb300 import pa
    lens = [(53 * i * i + 211 * i) % 1900 + 1 for i in range(32)]
    jobs = []
    for hkv, seed in ((8, 71), (32, 73), (4, 79)):
        inp = make_inputs(shape("threads", 32, 32, hkv, 128, 16, torch.bfloat16, seed=seed), lens)
        dev = to_cuda(inp)
        out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
        ws = pa.workspace_for(dev["q"], 16, dev["block_tables"].shape[1])
        jobs.append(("decode", inp, dev, out, ws, hkv))
    qinp = make_inputs(shape("threads_q", 32, 32, 8, 128, 16, torch.bfloat16, seed=83), lens)
    kq, vq = [t.cuda() for t in wl.quant_pools(qinp, "e4m3")]
    qdev = to_cuda(qinp)
    qout = torch.empty(qdev["q"].shape, dtype=torch.float32, device="cuda")
    qws = pa.workspace_for(qdev["q"], 16, qdev["block_tables"].shape[1])

    def run(job, stream, reps):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(reps):
            if job[0] == "decode":
                _, inp, dev, out, ws, hkv = job
                pa.pa_decode(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                             num_kv_heads=hkv, workspace=ws, err_word=err, stream=stream)
            else:
                pa.pa_decode_quant(qout, qdev["q"], kq, vq, qdev["block_tables"], qdev["context_lens"],
                                   num_kv_heads=8, workspace=qws, err_word=err, stream=stream)
        stream.synchronize()
        return int(err.item())

    all_jobs = jobs + [("quant",)]
    streams = [torch.cuda.Stream() for _ in all_jobs]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    alone = []
    for job, st in zip(all_jobs, streams):
        assert run(job, st, 1) == 0
        alone.append((job[3] if job[0] == "decode" else qout).clone())
    errs = [None] * len(all_jobs)

    def worker(i):
        errs[i] = run(all_jobs[i], streams[i], 25)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(all_jobs))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert errs == [0] * len(all_jobs)
    for job, ref in zip(all_jobs, alone):
        got = job[3] if job[0] == "decode" else qout
        assert torch.equal(got, ref)
    compare(jobs[0][3].cpu(), oracle_decode(jobs[0][1]), torch.bfloat16)
