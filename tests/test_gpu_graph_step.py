"""A whole cache step captured in one CUDA graph: copy-on-write block copy,
append of the next token, and decode over the grown contexts (partitioned, so
the partition merge runs too).  Every library kernel is a programmatic
dependent launch (it may be scheduled while the kernel before it runs, and
waits for it before touching memory), and the capture keeps those
dependences as graph edges.  Each replay must give the eager step's pools and
outputs bit for bit, and the eager step must match the oracle (bit-exact
pools, attention within the tolerances)."""
import math

import pytest
import torch

import oracle
from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare

pytestmark = pytest.mark.gpu


def _state(dtype, hkv, G, seed):
    N, bs, d = 4, 16, 128
    lens = [700, 1301, 43, 2100]                  # no context ends on a block boundary
    held = [(L + bs - 1) // bs for L in lens]
    nb = sum(held) + N + 4                        # + one copy destination per sequence
    M = max(held) + 1
    perm = wl.permutation(seed, 1, nb).to(torch.int32)
    tables = torch.full((N, M), -1, dtype=torch.int32)
    at = 0
    for s in range(N):
        tables[s, :held[s]] = perm[at:at + held[s]]
        at += held[s]
    # copy-on-write of every sequence's last (partly filled) block onto a fresh one
    dst = perm[at:at + N]
    pairs = torch.stack([tables[torch.arange(N), torch.tensor(held) - 1].to(torch.int64), dst.to(torch.int64)], 1)
    after = tables.clone()
    after[torch.arange(N), torch.tensor(held) - 1] = dst
    # token L of each sequence goes into its copied block
    slots = torch.tensor([int(after[s, lens[s] // bs]) * bs + lens[s] % bs for s in range(N)], dtype=torch.int64)
    k = wl.normal_tensor(seed, 2, (nb, hkv, bs, d), dtype=dtype)
    v = wl.normal_tensor(seed, 3, (nb, hkv, bs, d), dtype=dtype)
    kn = wl.normal_tensor(seed, 4, (N, hkv, d), dtype=dtype)
    vn = wl.normal_tensor(seed, 5, (N, hkv, d), dtype=dtype)
    q = wl.normal_tensor(seed, 6, (N, hkv * G, d), dtype=dtype)
    lens1 = torch.tensor(lens, dtype=torch.int32) + 1
    return k, v, kn, vn, q, pairs, slots, after, lens1


@pytest.mark.parametrize("dtype,hkv,G", [(torch.bfloat16, 2, 4), (torch.float16, 8, 1)])
def test_cache_step_captured_in_one_graph(dtype, hkv, G):
    from paged_kv_cache_251_gb300 import pa
    k, v, kn, vn, q, pairs, slots, after, lens1 = _state(dtype, hkv, G, seed=71 + hkv)
    dev = {n: t.cuda() for n, t in dict(k=k, v=v, kn=kn, vn=vn, q=q, pairs=pairs, slots=slots, bt=after,
                                         cl=lens1).items()}
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = pa.workspace_for(dev["q"], 16, after.shape[1], 0, 512)

    def step():
        pa.pa_copy_blocks(dev["pairs"], dev["k"], dev["v"], err_word=err)
        pa.pa_append_kv(dev["kn"], dev["vn"], dev["slots"], dev["k"], dev["v"], err_word=err)
        pa.pa_decode(out, dev["q"], dev["k"], dev["v"], dev["bt"], dev["cl"], num_kv_heads=hkv,
                     partition_size=512, workspace=ws, err_word=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                    # eager, on the stream the capture will use
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = (out.clone(), dev["k"].clone(), dev["v"].clone())
    assert int(err.item()) == 0

    # the oracle's step
    kr, vr = k.clone(), v.clone()
    oracle.copy_blocks(kr, vr, pairs)
    oracle.append_kv(kr, vr, kn, vn, slots)
    assert torch.equal(eager[1].cpu().view(torch.int16), kr.view(torch.int16))
    assert torch.equal(eager[2].cpu().view(torch.int16), vr.view(torch.int16))
    ref = oracle.paged_attention(q, kr, vr, after, lens1, num_kv_heads=hkv, scale=1 / math.sqrt(128), threads=8)
    compare(eager[0].cpu(), ref, dtype)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(10):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager[0])
        assert torch.equal(dev["k"], eager[1]) and torch.equal(dev["v"], eager[2])
    assert int(err.item()) == 0
