"""GPU parity of pa_decode_shared_prefix: the same attention as pa_decode,
with each group's shared prompt blocks read once.  Groups are built by the
block manager (a prompt, then forks that each append their own tokens), so
members' tables agree on the prompt's whole blocks."""
import math

import pytest
import torch

import oracle
from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare, make_groups

pytestmark = pytest.mark.gpu


CASES = [
    # prompts, samples, H, H_kv, bs, prompt lens, extra tokens per sample, partition
    (3, 8, 8, 8, 16, [700, 33, 1000], None, 0),
    (4, 4, 8, 4, 8, [130, 64, 9, 1500], None, 0),
    (2, 2, 8, 2, 32, [2000, 40], None, 128),
    (2, 8, 4, 4, 16, [0, 16], None, 0),            # an empty prompt and a one-block prompt
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_shared_prefix_matches_oracle_and_pa_decode(case, dtype):
    from paged_kv_cache_251_gb300 import pa
    prompts, samples, H, hkv, bs, plens, extra, part = case
    N = prompts * samples
    extra = extra or wl.randint(7, 1, N, 1, 300).tolist()
    tables, lens, k, v = make_groups(prompts, samples, plens, extra, bs, hkv, 128, dtype, seed=prompts * 31 + bs)
    q = wl.normal_tensor(9, 3, (N, H, 128), dtype=dtype)
    shared = torch.tensor([pl // bs * bs for pl in plens], dtype=torch.int32)
    out = torch.full((N, H, 128), float("nan"), device="cuda")
    ref_out = torch.empty_like(out)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = [t.cuda() for t in (q, k, v, tables, lens)]
    pa.pa_decode_shared_prefix(out, *dev, shared.cuda(), samples, num_kv_heads=hkv, partition_size=part,
                               err_word=err)
    pa.pa_decode(ref_out, *dev, num_kv_heads=hkv, partition_size=part)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.paged_attention(q, k, v, tables, lens, num_kv_heads=hkv, scale=1 / math.sqrt(128), threads=8)
    compare(out.cpu(), ref, dtype)
    compare(out.cpu(), ref_out.cpu().double().numpy(), dtype)


def test_shared_length_beyond_a_member_is_clamped_and_flagged():
    from paged_kv_cache_251_gb300 import pa
    bs, hkv, H = 16, 4, 8
    # group 0: a 320-token prompt (20 whole blocks); member 0 adds nothing, member 1 adds 50 tokens
    tables, lens, k, v = make_groups(2, 2, [320, 100], [0, 50, 3, 1], bs, hkv, 128, torch.bfloat16, seed=3)
    q = wl.normal_tensor(9, 3, (4, H, 128), dtype=torch.bfloat16)
    # claim more sharing than member 0's context (used: its 320 tokens, where the
    # tables still agree), and a length that is not whole blocks (used: 32)
    shared = torch.tensor([4000, 37], dtype=torch.int32)
    out = torch.empty((4, H, 128), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_shared_prefix(out, q.cuda(), k.cuda(), v.cuda(), tables.cuda(), lens.cuda(), shared.cuda(), 2,
                               num_kv_heads=hkv, err_word=err)
    torch.cuda.synchronize()
    assert err.item() & 16
    ref = oracle.paged_attention(q, k, v, tables, lens, num_kv_heads=hkv, scale=1 / math.sqrt(128))
    compare(out.cpu(), ref, torch.bfloat16)


def test_prefix_workload_full_size():
    """32 prompts x 2000 tokens x 8 samples after the copy-on-write step: the
    shared decode matches the oracle on sampled rows."""
    from paged_kv_cache_251_gb300 import pa, scenarios
    st = scenarios.prefix_state(16, device="cuda")
    s = st.shape
    pa.pa_copy_blocks(st.pairs.cuda(), st.k_cache, st.v_cache)
    pa.pa_append_kv(st.k_new, st.v_new, st.slots.cuda(), st.k_cache, st.v_cache)
    shared = torch.full((st.prompts,), st.prompt_len // 16 * 16, dtype=torch.int32, device="cuda")
    out = torch.empty((s.num_seqs, s.num_heads, s.head_dim), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_shared_prefix(out, st.q, st.k_cache, st.v_cache, st.block_tables.cuda(), st.context_lens.cuda(),
                               shared, st.samples, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    idx = wl.permutation(5, 1, s.num_seqs * s.num_heads)[:128]
    pairs = torch.stack([idx // s.num_heads, idx % s.num_heads], 1).to(torch.int32)
    ref = oracle.paged_attention(st.q.cpu(), st.k_cache.cpu(), st.v_cache.cpu(), st.block_tables,
                                 st.context_lens, num_kv_heads=s.num_kv_heads, scale=1 / math.sqrt(s.head_dim),
                                 pairs=pairs, threads=16)
    compare(out.cpu()[pairs[:, 0].long(), pairs[:, 1].long()], ref, s.dtype)


@pytest.mark.parametrize("H,hkv", [(8, 8), (8, 4)])
def test_shared_prefix_replayed_from_a_cuda_graph(H, hkv):
    """The shared-prefix call (its four kernels: prep, prefix pass, suffix pass,
    combine) captured in a CUDA graph and replayed: every replay gives the eager
    call's output bit for bit, which matches the oracle."""
    from paged_kv_cache_251_gb300 import pa
    prompts, samples, bs = 3, 4, 16
    N = prompts * samples
    plens = [1500, 40, 700]
    extra = wl.randint(17, 1, N, 1, 300).tolist()
    tables, lens, k, v = make_groups(prompts, samples, plens, extra, bs, hkv, 128, torch.bfloat16, seed=41 + hkv)
    q = wl.normal_tensor(19, 3, (N, H, 128), dtype=torch.bfloat16)
    shared = torch.tensor([pl // bs * bs for pl in plens], dtype=torch.int32)
    dev = [t.cuda() for t in (q, k, v, tables, lens)]
    sh = shared.cuda()
    out = torch.empty((N, H, 128), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = pa.pa_decode_shared_prefix_workspace_size(N, H, 128, bs, tables.shape[1], 0, samples, torch.bfloat16)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")

    def call():
        pa.pa_decode_shared_prefix(out, *dev, sh, samples, num_kv_heads=hkv, workspace=ws, err_word=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert err.item() == 0
    eager = out.clone()
    ref = oracle.paged_attention(q, k, v, tables, lens, num_kv_heads=hkv, scale=1 / math.sqrt(128), threads=8)
    compare(eager.cpu(), ref, torch.bfloat16)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(8):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert err.item() == 0
