"""GPU parity of the 8-bit KV cache (INT8 / E4M3 codes with one fp32 scale per
cached row, held in self-contained pages) against the oracle, through the C ABI:
  - quantise-on-append: whole page pools compared byte for byte;
  - decode over 8-bit pages: the attention tolerances of the 16-bit path,
    against the oracle reading every element as code * scale;
  - block copy and swap of page pools: bit-exact.
Decode inputs are random codes and scales from the seeded generator (no
quantiser on either side); the append-then-decode test runs the two steps in
sequence on each side."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare, shape

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
FMTS = ["int8", "e4m3"]


def _u8(t):
    return t.view(torch.uint8)


def _filled_pages(nb, hkv, bs, d, fmt, seed):
    """Page pools pre-filled with random codes and scales (so untouched rows are checked)."""
    shp = (nb, hkv, bs, d)
    return (wl.page_pool(wl.code_pool(seed, 1, shp, fmt), wl.scale_pool(seed, 3, shp[:3], fmt)),
            wl.page_pool(wl.code_pool(seed, 2, shp, fmt), wl.scale_pool(seed, 4, shp[:3], fmt)))


def _gpu_append(k, v, slots, pools, err=None):
    from paged_kv_cache_251_gb300 import pa
    dev = [t.cuda() for t in pools]
    pa.pa_append_kv_quant(k.cuda(), v.cuda(), slots.cuda(), *dev, err_word=err)
    torch.cuda.synchronize()
    return [t.cpu() for t in dev]


def _assert_pools_equal(got, want):
    for g, w, name in zip(got, want, ("K", "V")):
        assert torch.equal(_u8(g), _u8(w)), f"{name} pages differ"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("in_dt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("bs,d,hkv", [(16, 128, 8), (8, 64, 4), (32, 128, 40), (32, 64, 2)])
def test_append_quant_bit_exact(fmt, in_dt, bs, d, hkv):
    nb, T = 24, 37
    pools = _filled_pages(nb, hkv, bs, d, fmt, seed=bs + d + hkv)
    k = wl.normal_tensor(5, 1, (T, hkv, d), dtype=DT[in_dt])
    v = wl.normal_tensor(5, 2, (T, hkv, d), dtype=DT[in_dt]) * 3
    slots = wl.permutation(6, 1, nb * bs)[:T].clone()
    slots[3] = -1
    slots[10] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu_append(k, v, slots, pools, err)
    want = [t.clone() for t in pools]
    oracle.append_kv_quant(*want, k, v, slots)
    assert err.item() == 0
    _assert_pools_equal(got, want)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("in_dt", ["f16", "bf16"])
def test_append_quant_special_rows(fmt, in_dt):
    """Zero rows, constant rows, rows of tiny (subnormal) values, rows with
    exact ties, a single large element, negative zeros."""
    hkv, d, bs, nb = 1, 64, 16, 4
    rows = torch.zeros(8, hkv, d, dtype=torch.float32)
    rows[1] = 0.75                                         # constant
    rows[2] = torch.linspace(-1, 1, d) * 2.0 ** -20        # fp16 subnormals / bf16 tiny
    rows[3] = torch.arange(d, dtype=torch.float32) - 32    # integers (ties for INT8 after scaling)
    rows[4, 0, 7] = 1000.0                                 # one element dominates
    rows[4, 0, 8] = 0.001
    rows[5] = -0.0                                         # negative zeros
    rows[6] = torch.linspace(-3, 3, d)
    rows[7] = (torch.arange(d, dtype=torch.float32) % 7 - 3) * 0.5
    k = rows.to(DT[in_dt])
    v = (-rows).to(DT[in_dt])
    pools = _filled_pages(nb, hkv, bs, d, fmt, seed=77)
    slots = torch.tensor([0, 5, 16, 17, 33, 48, 63, 2], dtype=torch.int64)
    got = _gpu_append(k, v, slots, pools)
    want = [t.clone() for t in pools]
    oracle.append_kv_quant(*want, k, v, slots)
    _assert_pools_equal(got, want)


@pytest.mark.parametrize("fmt", FMTS)
def test_append_quant_out_of_range_slot_flagged_and_skipped(fmt):
    hkv, d, bs, nb = 2, 128, 16, 4
    pools = _filled_pages(nb, hkv, bs, d, fmt, seed=9)
    k = wl.normal_tensor(7, 1, (2, hkv, d), dtype=torch.float16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu_append(k, k, torch.tensor([nb * bs, 1 << 40]), pools, err)
    assert err.item() & 2
    _assert_pools_equal(got, pools)


def _quant_case(name, n, h, hkv, d, bs, lens, window, qdt, fmt, seed):
    sh = shape(name, n, h, hkv, d, bs, qdt, window=window, seed=seed)
    inp = wl.decode_inputs(sh, lens=torch.as_tensor(lens, dtype=torch.int32), room_for_append=False,
                           with_append=False)
    return inp, wl.quant_pools(inp, fmt)


def _gpu_decode_quant(inp, pools, out_dtype=torch.float32, window=None, partition_size=0, block_tables=None,
                      context_lens=None):
    from paged_kv_cache_251_gb300 import pa
    s = inp.shape
    q = inp.q.cuda()
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = (inp.block_tables if block_tables is None else block_tables).cuda().contiguous()
    cl = (inp.context_lens if context_lens is None else context_lens).cuda().contiguous()
    kp, vp = [t.cuda() for t in pools]
    pa.pa_decode_quant(out, q, kp, vp, bt, cl, num_kv_heads=s.num_kv_heads,
                       scale=1.0 / math.sqrt(s.head_dim), window=s.window if window is None else window,
                       partition_size=partition_size, err_word=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


def _oracle_decode_quant(inp, pools, block_tables=None, context_lens=None, invalid_policy=0, pairs=None):
    s = inp.shape
    kp, vp = pools
    return oracle.paged_attention(inp.q, kp, vp, inp.block_tables if block_tables is None else block_tables,
                                  inp.context_lens if context_lens is None else context_lens,
                                  num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim),
                                  window=s.window, invalid_policy=invalid_policy, pairs=pairs, threads=8)


# (name, N, H, H_kv, d, bs, lens, window, partition) — several tiles and a ragged tail each
QCASES = [
    ("mha_bs16", 6, 4, 4, 128, 16, [1, 15, 16, 17, 512, 513], 0, 0),
    ("mha_bs8_d64", 5, 4, 4, 64, 8, [7, 8, 9, 300, 1], 0, 0),
    ("mha_bs32_parts", 3, 5, 5, 128, 32, [2000, 33, 700], 0, 64),
    ("mha_window", 3, 4, 4, 128, 16, [1000, 20, 777], 100, 0),
    ("g2_bs32", 4, 4, 2, 128, 32, [129, 31, 1000, 257], 0, 0),
    ("g4_parts", 3, 8, 2, 128, 16, [700, 129, 2049], 0, 64),
    ("g8_bs8_window", 3, 16, 2, 128, 8, [3000, 77, 1300], 700, 0),
    ("g4_d64", 4, 8, 2, 64, 16, [65, 66, 700, 2], 0, 0),
    ("empty", 3, 8, 2, 128, 16, [0, 300, 0], 0, 0),
    # every (group, block size) corner of the TMA-fed kernel (head_dim 128, G <= 4)
    ("g1_bs8", 4, 6, 6, 128, 8, [9, 700, 1, 255], 0, 0),
    ("g2_bs16_window", 3, 8, 4, 128, 16, [1000, 5, 333], 200, 0),
    ("g2_bs8_parts", 3, 4, 2, 128, 8, [1500, 8, 9], 0, 64),
    ("g4_bs8", 3, 8, 2, 128, 8, [129, 1, 1000], 0, 0),
    ("g4_bs32_window", 3, 16, 4, 128, 32, [33, 2049, 64], 100, 0),
    ("g1_bs32_empty", 3, 2, 2, 128, 32, [0, 65, 0], 0, 0),
    # kv heads in fours, block size 16 / 32 (E4M3 with 16-bit queries: the
    # tensor-core kernel): partitions of 4 blocks (2 tiles) and of 3 blocks (a
    # last tile with one block), windows, empty sequences
    ("tc_g4_bs16_parts", 3, 16, 4, 128, 16, [700, 129, 2049], 0, 64),
    ("tc_g4_bs16_odd_parts", 3, 16, 4, 128, 16, [1000, 1, 47], 0, 48),
    ("tc_g4_window", 2, 16, 4, 128, 16, [3000, 77], 700, 0),
    ("tc_g2_bs32", 4, 8, 4, 128, 32, [129, 31, 1000, 257], 0, 0),
    ("tc_g1_bs32_parts", 3, 8, 8, 128, 32, [2000, 33, 700], 0, 64),
    ("tc_g4_hkv8_empty", 3, 32, 8, 128, 16, [0, 300, 0], 0, 0),
    # long partitions: 64 and 128 blocks per item (32 / 64 tiles of the tensor-core kernel)
    ("tc_g4_bs16_p1024", 3, 16, 4, 128, 16, [3000, 1100, 77], 0, 1024),
    ("tc_g4_bs32_p4096", 2, 16, 4, 128, 32, [5000, 2100], 0, 4096),
    ("g4_bs16_p2048", 3, 8, 2, 128, 16, [3000, 1100, 77], 0, 2048),
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("qdt", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("case", QCASES, ids=[c[0] for c in QCASES])
def test_decode_quant_edge_cases(case, qdt, fmt):
    name, n, h, hkv, d, bs, lens, window, part = case
    inp, pools = _quant_case(name, n, h, hkv, d, bs, lens, window, DT[qdt], fmt, seed=31 + n + d + bs)
    got, err = _gpu_decode_quant(inp, pools, partition_size=part)
    assert err == 0
    compare(got, _oracle_decode_quant(inp, pools), torch.float16)


def test_decode_quant_repeated_launches_reuse_item_counters():
    """The grouped-head E4M3 kernel claims items from a per-launch counter
    that each launch returns to zero; launches take counters round-robin from
    a pool of 4096.  5000 launches reuse every counter, and the last one's
    output still matches the oracle (a counter left non-zero would make a
    launch skip items)."""
    from paged_kv_cache_251_gb300 import pa
    inp, pools = _quant_case("reuse", 5, 16, 4, 128, 16, [700, 1, 2049, 33, 300], 0, torch.bfloat16, "e4m3",
                             seed=13)
    s = inp.shape
    q = inp.q.cuda()
    kp, vp = [t.cuda() for t in pools]
    bt, cl = inp.block_tables.cuda(), inp.context_lens.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    # 32-token partitions: about twice as many items as the GPU has CTAs of
    # this kernel, so the launches claim from a counter
    ws = torch.empty(pa.pa_decode_workspace_size(s.num_seqs, s.num_heads, s.head_dim, s.block_size,
                                                  bt.shape[1], 0, 32) // 4 + 4, dtype=torch.float32,
                     device="cuda")
    for i in range(5000):
        if i == 4999:
            out.fill_(float("nan"))
        pa.pa_decode_quant(out, q, kp, vp, bt, cl, num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim),
                           partition_size=32, workspace=ws, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    compare(out.cpu(), _oracle_decode_quant(inp, pools), torch.float16)


@pytest.mark.parametrize("out_dt", ["f16", "bf16"])
def test_decode_quant_low_precision_output(out_dt):
    inp, pools = _quant_case("lowout", 4, 8, 8, 128, 16, [300, 17, 600, 1], 0, torch.bfloat16, "e4m3", seed=3)
    got, err = _gpu_decode_quant(inp, pools, out_dtype=DT[out_dt])
    assert err == 0 and got.dtype == DT[out_dt]
    compare(got, _oracle_decode_quant(inp, pools), torch.bfloat16)


@pytest.mark.parametrize("hkv", [2, 4])
@pytest.mark.parametrize("fmt", FMTS)
def test_decode_quant_zero_scale_rows(fmt, hkv):
    """Rows stored with scale 0 (all-zero rows) read as zeros."""
    inp, pools = _quant_case("zeros", 2, 2 * hkv, hkv, 128, 16, [40, 70], 0, torch.float16, fmt, seed=4)
    kc, ks = oracle.unpack_pages(pools[0])
    vc, vs = oracle.unpack_pages(pools[1])
    ks[inp.block_tables[0, 0].item(), :, :5] = 0.0
    vs[inp.block_tables[1, 2].item(), 1, :] = 0.0
    pools = (wl.page_pool(kc, ks), wl.page_pool(vc, vs))
    got, err = _gpu_decode_quant(inp, pools)
    assert err == 0
    compare(got, _oracle_decode_quant(inp, pools), torch.float16)


@pytest.mark.parametrize("hkv", [2, 4])
@pytest.mark.parametrize("fmt", FMTS)
def test_decode_quant_invalid_table_entries_skipped_and_flagged(fmt, hkv):
    inp, pools = _quant_case("bad", 3, 2 * hkv, hkv, 128, 16, [70, 40, 33], 0, torch.float16, fmt, seed=8)
    bt = inp.block_tables.clone()
    bt[0, 1] = inp.num_blocks + 5
    bt[2, 0] = -7
    got, err = _gpu_decode_quant(inp, pools, block_tables=bt)
    assert err & 1
    compare(got, _oracle_decode_quant(inp, pools, block_tables=bt, invalid_policy=1), torch.float16)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("hkv", [8, 2])
def test_decode_quant_append_then_decode(fmt, hkv):
    """Quantise a whole fp16 pool token by token with pa_append_kv_quant (the
    pages must equal the oracle's bit for bit), then decode both."""
    from paged_kv_cache_251_gb300 import pa
    sh = shape("e2e", 3, 8, hkv, 128, 16, torch.float16, seed=12)
    inp = wl.decode_inputs(sh, lens=torch.tensor([300, 1, 517], dtype=torch.int32), room_for_append=False,
                           with_append=False)
    nb, bs = inp.num_blocks, 16
    code_dt = wl.CODE_DTYPES[fmt]
    shp = pa.quant_pool_shape(nb, hkv, bs, 128)
    zeros = [torch.zeros(shp, dtype=torch.uint8).view(code_dt), torch.zeros(shp, dtype=torch.uint8).view(code_dt)]
    # every slot of the pool as one appended token: rows [slot][H_kv][d]
    rows_k = inp.k_cache.permute(0, 2, 1, 3).reshape(nb * bs, hkv, 128).contiguous()
    rows_v = inp.v_cache.permute(0, 2, 1, 3).reshape(nb * bs, hkv, 128).contiguous()
    slots = torch.arange(nb * bs, dtype=torch.int64)
    got_pools = _gpu_append(rows_k, rows_v, slots, zeros)
    want_pools = [t.clone() for t in zeros]
    oracle.append_kv_quant(*want_pools, rows_k, rows_v, slots)
    _assert_pools_equal(got_pools, want_pools)
    got, err = _gpu_decode_quant(inp, got_pools)
    assert err == 0
    compare(got, _oracle_decode_quant(inp, want_pools), torch.float16)
    # the quantised cache stays close to the 16-bit one (context, not a parity bound)
    exact = oracle.paged_attention(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens,
                                   num_kv_heads=hkv, scale=1 / math.sqrt(128), threads=8)
    assert float(np.abs(got.double().numpy() - exact).max()) < (0.05 if fmt == "int8" else 0.25)


@pytest.mark.parametrize("fmt", FMTS)
def test_copy_blocks_quant_bit_exact(fmt):
    from paged_kv_cache_251_gb300 import pa
    nb, hkv, bs, d = 64, 8, 16, 128
    pools = _filled_pages(nb, hkv, bs, d, fmt, seed=21)
    perm = wl.permutation(9, 1, nb)
    pairs = torch.stack([perm[:20], perm[20:40]], dim=1).contiguous()
    pairs[5, 1] = nb + 3                                   # outside the pool: skipped, flagged
    dev = [t.cuda() for t in pools]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks_quant(pairs.cuda(), *dev, err_word=err)
    want = [t.clone() for t in pools]
    oracle.copy_blocks(want[0], want[1], pairs)
    torch.cuda.synchronize()
    assert err.item() & 4
    _assert_pools_equal([t.cpu() for t in dev], want)


@pytest.mark.parametrize("fmt", FMTS)
def test_swap_quant_to_pinned_host_and_back(fmt):
    from paged_kv_cache_251_gb300 import pa
    nb, hb, hkv, bs, d = 40, 24, 8, 16, 128
    pools = _filled_pages(nb, hkv, bs, d, fmt, seed=22)
    dev = [t.cuda() for t in pools]
    code_dt = wl.CODE_DTYPES[fmt]
    hshape = pa.quant_pool_shape(hb, hkv, bs, d)
    host = [torch.zeros(hshape, dtype=torch.uint8).view(code_dt).pin_memory() for _ in range(2)]
    want_host = [torch.zeros_like(t) for t in host]
    perm = wl.permutation(12, 1, nb)
    out_pairs = torch.stack([perm[:20], wl.permutation(13, 1, hb)[:20]], 1).contiguous()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_swap_blocks_quant(out_pairs.cuda(), *dev, *host, err_word=err)
    oracle.swap_blocks(pools[0], pools[1], want_host[0], want_host[1], out_pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    _assert_pools_equal(host, want_host)
    in_pairs = torch.stack([out_pairs[:, 1], perm[20:40]], 1).contiguous()
    pa.pa_swap_blocks_quant(in_pairs.cuda(), *host, *dev, err_word=err)
    want = [t.clone() for t in pools]
    oracle.swap_blocks(want_host[0], want_host[1], want[0], want[1], in_pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    _assert_pools_equal([t.cpu() for t in dev], want)


def _sample_pairs(N, H, count, seed):
    idx = wl.permutation(seed, 1, N * H)[:count]
    return torch.stack([idx // H, idx % H], dim=1).to(torch.int32)


@pytest.mark.parametrize("name,fmt", [("opt13b", "int8"), ("opt13b", "e4m3"), ("gqa", "e4m3"), ("gqa", "int8")])
def test_full_size_quant_sampled(name, fmt):
    """The full-size workloads with 8-bit pools (codes and scales generated on
    the GPU), in the launch configuration the benchmark times: every output
    finite, a sample of rows against the oracle."""
    from paged_kv_cache_251_gb300 import pa
    if name == "opt13b":
        inp = wl.decode_inputs(wl.SHAPES["opt13b"], device="cuda", with_append=False)
    else:
        inp = wl.decode_inputs(wl.SHAPES["gqa"], device="cuda", room_for_append=False, fill=0.95,
                               with_append=False)
    s = inp.shape
    inp.k_cache = inp.v_cache = None                      # the 16-bit pools are not needed
    torch.cuda.empty_cache()
    pools = wl.quant_pools(inp, fmt, device="cuda")
    q = inp.q
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    bt, cl = inp.block_tables.cuda(), inp.context_lens.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_quant(out, q, *pools, bt, cl, num_kv_heads=s.num_kv_heads, scale=1 / math.sqrt(s.head_dim),
                       err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0 and bool(torch.isfinite(out).all())
    pairs = _sample_pairs(s.num_seqs, s.num_heads, 48, seed=s.seed)
    cpu_pools = [t.cpu() for t in pools]
    ref = oracle.paged_attention(q.cpu(), cpu_pools[0], cpu_pools[1], inp.block_tables, inp.context_lens,
                                 num_kv_heads=s.num_kv_heads, scale=1 / math.sqrt(s.head_dim), pairs=pairs,
                                 threads=16)
    got = out.cpu()[pairs[:, 0].long(), pairs[:, 1].long()]
    compare(got, ref, torch.float16)


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_quant_full_gqa_batch_is_repeatable(fmt):
    """The full GQA batch (256 sequences of lognormal length, items claimed
    from a counter) decoded twelve times: every run's output is bit-identical
    (each item is computed by one CTA and partitions merge in a fixed order, so
    nothing but a race can change a bit), and a sample of rows matches the
    oracle.  A race in the tensor-core kernel's epilogue once corrupted one kv
    head's rows in about one run in five; twelve runs miss that with
    probability under 7 %."""
    from paged_kv_cache_251_gb300 import pa
    inp = wl.decode_inputs(wl.SHAPES["gqa"], device="cuda", room_for_append=False, fill=0.95, with_append=False)
    s = inp.shape
    q, bt, cl = inp.q, inp.block_tables.cuda(), inp.context_lens.cuda()
    inp.k_cache = inp.v_cache = None
    torch.cuda.empty_cache()
    kp, vp = wl.quant_pools(inp, fmt, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    runs = []
    for _ in range(12):
        out.fill_(float("nan"))
        pa.pa_decode_quant(out, q, kp, vp, bt, cl, num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim),
                           err_word=err)
        runs.append(out.clone())
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for r in runs[1:]:
        assert torch.equal(r, runs[0])
    pairs = torch.stack([torch.arange(0, s.num_seqs, 4), torch.arange(0, s.num_seqs, 4) % s.num_heads],
                        1).to(torch.int32)
    ref = oracle.paged_attention(q.cpu(), kp.cpu(), vp.cpu(), inp.block_tables, inp.context_lens,
                                 num_kv_heads=s.num_kv_heads, scale=1.0 / math.sqrt(s.head_dim), pairs=pairs,
                                 threads=8)
    got = runs[0].cpu()[pairs[:, 0].long(), pairs[:, 1].long()]
    compare(got, ref, torch.float16)


def _grown_quant_state(fmt, seed):
    """An 8-bit cache where each sequence gets one new token: its last, partly
    filled block is copied to a fresh one (copy-on-write), the token is
    quantised into the copy, and the decode reads the grown contexts.  Kv heads
    in fours with 16-bit queries, so E4M3 takes the tensor-core kernel."""
    N, H, hkv, bs, d = 4, 16, 4, 16, 128
    lens = [700, 1301, 43, 2100]                  # no context ends on a block boundary
    held = [(L + bs - 1) // bs for L in lens]
    nb = sum(held) + N + 4
    M = max(held) + 1
    perm = wl.permutation(seed, 1, nb).to(torch.int32)
    tables = torch.full((N, M), -1, dtype=torch.int32)
    at = 0
    for s in range(N):
        tables[s, :held[s]] = perm[at:at + held[s]]
        at += held[s]
    last = torch.tensor(held) - 1
    pairs = torch.stack([tables[torch.arange(N), last].to(torch.int64), perm[at:at + N].to(torch.int64)], 1)
    tables[torch.arange(N), last] = perm[at:at + N]
    slots = torch.tensor([int(tables[s, lens[s] // bs]) * bs + lens[s] % bs for s in range(N)], dtype=torch.int64)
    pools = _filled_pages(nb, hkv, bs, d, fmt, seed)
    kn = wl.normal_tensor(seed, 5, (N, hkv, d), dtype=torch.bfloat16)
    vn = wl.normal_tensor(seed, 6, (N, hkv, d), dtype=torch.bfloat16)
    q = wl.normal_tensor(seed, 7, (N, H, d), dtype=torch.bfloat16)
    return q, pools, kn, vn, pairs, slots, tables, torch.tensor(lens, dtype=torch.int32) + 1, hkv


@pytest.mark.parametrize("fmt", FMTS)
def test_quant_cache_step_captured_in_one_graph(fmt):
    """Block copy, quantise-on-append and decode of an 8-bit cache captured in
    one CUDA graph (every library kernel a programmatic dependent launch, the
    decode claiming items and merging partitions): each replay gives the eager
    step's pages and output bit for bit, and the eager step matches the oracle."""
    from paged_kv_cache_251_gb300 import pa
    q, pools, kn, vn, pairs, slots, tables, lens1, hkv = _grown_quant_state(fmt, seed=53)
    dev = {n: t.cuda() for n, t in dict(q=q, kn=kn, vn=vn, pairs=pairs, slots=slots, bt=tables, cl=lens1).items()}
    kp, vp = [t.cuda() for t in pools]
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pa.workspace_for(dev["q"], 16, tables.shape[1], 0, 0)

    def step():
        pa.pa_copy_blocks_quant(dev["pairs"], kp, vp, err_word=err)
        pa.pa_append_kv_quant(dev["kn"], dev["vn"], dev["slots"], kp, vp, err_word=err)
        pa.pa_decode_quant(out, dev["q"], kp, vp, dev["bt"], dev["cl"], num_kv_heads=hkv,
                           scale=1.0 / math.sqrt(128), workspace=ws, err_word=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    eager = (out.clone(), kp.clone(), vp.clone())

    want = [t.clone() for t in pools]
    oracle.copy_blocks(want[0], want[1], pairs)
    oracle.append_kv_quant(want[0], want[1], kn, vn, slots)
    _assert_pools_equal([eager[1].cpu(), eager[2].cpu()], want)
    ref = oracle.paged_attention(q, want[0], want[1], tables, lens1, num_kv_heads=hkv, scale=1.0 / math.sqrt(128),
                                 threads=8)
    compare(eager[0].cpu(), ref, torch.bfloat16)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(10):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager[0])
        assert torch.equal(_u8(kp), _u8(eager[1])) and torch.equal(_u8(vp), _u8(eager[2]))
    assert int(err.item()) == 0


def test_quant_concurrent_launches_on_two_streams():
    """INT8 and E4M3 decodes of GQA-shaped batches (the CUDA-core and the
    tensor-core 8-bit kernels, each claiming items from a counter) launched ten
    times each on two streams with no synchronisation in between: each keeps its
    single-stream result bit for bit."""
    from paged_kv_cache_251_gb300 import pa
    lens = [(37 * i * i + 300 * i) % 2100 + 1 for i in range(128)]
    cases = []
    for fmt, seed in (("int8", 61), ("e4m3", 67)):
        inp, pools = _quant_case("streams_" + fmt, 128, 32, 8, 128, 16, lens, 0, torch.bfloat16, fmt, seed=seed)
        q = inp.q.cuda()
        kp, vp = [t.cuda() for t in pools]
        bt, cl = inp.block_tables.cuda(), inp.context_lens.cuda()
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws = pa.workspace_for(q, 16, bt.shape[1])
        cases.append((inp, pools, q, kp, vp, bt, cl, out, err, ws, torch.cuda.Stream()))

    def call(c):
        inp, pools, q, kp, vp, bt, cl, out, err, ws, st = c
        pa.pa_decode_quant(out, q, kp, vp, bt, cl, num_kv_heads=8, scale=1.0 / math.sqrt(128), workspace=ws,
                           err_word=err, stream=st)

    alone = []
    for c in cases:
        call(c)
        torch.cuda.synchronize()
        alone.append(c[7].clone())
    for c in cases:
        c[10].wait_stream(torch.cuda.current_stream())
    for _ in range(10):
        for c in cases:
            call(c)
    torch.cuda.synchronize()
    for c, ref in zip(cases, alone):
        assert int(c[8].item()) == 0
        assert torch.equal(c[7], ref)
    inp, pools = cases[1][0], cases[1][1]
    pairs = torch.tensor([[s, h] for s in range(0, 128, 17) for h in (0, 13, 31)], dtype=torch.int32)
    ref = _oracle_decode_quant(inp, pools, pairs=pairs)
    got = cases[1][7].cpu()[pairs[:, 0].long(), pairs[:, 1].long()]
    compare(got, ref, torch.bfloat16)
