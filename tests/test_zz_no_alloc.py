"""pa_decode_noalloc: decode attention for callers that cannot allocate device
memory (for example a plugin whose host framework owns every allocation, or a
runtime with a fixed memory budget).  Its partials live in a scratch array
built into the library instead of a caller workspace.

Checked through the C ABI against pa_decode with a caller workspace and
against the fp64 oracle, within the parity tolerance, on two calls in a row
(different shapes, so the second call runs over the first call's leftovers
in the shared scratch); a warmed-up call leaves the device's free memory and
torch's allocated bytes unchanged.  This file is collected last so a failure
here leaves every other test already run.
"""
import pytest
import torch

from paritylib import compare, make_inputs, oracle_decode, shape, to_cuda

pytestmark = pytest.mark.gpu


def _both(inp, partition_size):
    from paged_kv_cache_251_gb300 import pa
    dev = to_cuda(inp)
    s = inp.shape
    args = (dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"])
    ref = torch.empty(inp.q.shape, dtype=torch.float32, device="cuda")
    got = torch.full(inp.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(ref, *args, num_kv_heads=s.num_kv_heads, window=s.window, partition_size=partition_size,
                 err_word=err)
    pa.pa_decode_noalloc(got, *args, num_kv_heads=s.num_kv_heads, window=s.window,
                         partition_size=partition_size, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    need = pa.pa_decode_workspace_size(s.num_seqs, s.num_heads, s.head_dim, s.block_size,
                                       inp.block_tables.shape[1], s.window, partition_size)
    return got.cpu(), ref.cpu(), need


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    from paged_kv_cache_251_gb300 import pa
    first = make_inputs(shape("na1", 6, 8, 2, 128, 16, torch.bfloat16, seed=31), [1500, 40, 700, 2100, 1, 513])
    second = make_inputs(shape("na2", 3, 4, 4, 64, 8, torch.float16, window=300, seed=32), [900, 64, 2000])
    for inp, part in ((first, 128), (second, 64)):
        got, ref, need = _both(inp, part)
        assert 0 < need <= pa.pa_decode_noalloc_max_scratch()   # the partition path really runs
        compare(got, ref.double().numpy(), inp.shape.dtype)
        compare(got, oracle_decode(inp), inp.shape.dtype)


def test_noalloc_call_allocates_no_device_memory():
    from paged_kv_cache_251_gb300 import pa
    inp = make_inputs(shape("na3", 4, 8, 2, 128, 16, torch.bfloat16, seed=33), [1500, 40, 700, 2100])
    dev = to_cuda(inp)
    s = inp.shape
    out = torch.empty(inp.q.shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        pa.pa_decode_noalloc(out, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                             dev["context_lens"], num_kv_heads=s.num_kv_heads, partition_size=128, err_word=err)

    call()   # first call on the device: module load and the scratch address lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0
    assert err.item() == 0
    compare(out.cpu(), oracle_decode(inp), s.dtype)


def test_noalloc_rejects_a_shape_beyond_its_scratch():
    from paged_kv_cache_251_gb300 import pa
    limit = pa.pa_decode_noalloc_max_scratch()
    # 4096 seqs x 64 heads x d 128 with 64-token partitions over 512-block rows
    need = pa.pa_decode_workspace_size(4096, 64, 128, 16, 512, 0, 64)
    assert need > limit
    q = torch.zeros((4096, 64, 128), dtype=torch.float16, device="cuda")
    kc = torch.zeros((1, 64, 16, 128), dtype=torch.float16, device="cuda")
    bt = torch.zeros((4096, 512), dtype=torch.int32, device="cuda")
    cl = torch.ones(4096, dtype=torch.int32, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_decode_noalloc(out, q, kc, kc, bt, cl, partition_size=64)
    assert e.value.status == pa.PA_ERR_WORKSPACE_TOO_SMALL
    assert "scratch" in str(e.value)
