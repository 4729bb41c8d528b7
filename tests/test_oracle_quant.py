"""Pins of the oracle's 8-bit KV cache: the E4M3 and INT8 codes, the per-row
quantiser, attention over a quantised cache and quantise-on-append.

Independent references: torch's own float8_e4m3fn / int8 conversions (library
routines), error bounds that follow from the definition of rounding, values
chosen so the exact codes are known by hand, and torch's fp64
scaled_dot_product_attention over values torch itself decodes.
"""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_251_gb300 import workloads as wl

GOLDEN = Path(__file__).parent / "golden"


def _e4m3_values():
    """Every finite E4M3 magnitude, by torch's decode."""
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)  # 0x7f is NaN
    return codes.view(torch.float8_e4m3fn).to(torch.float64)


def test_e4m3_decode_matches_torch_for_every_code():
    for c in range(256):
        want = torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).item()
        got = oracle.code_to_double(c, "e4m3")
        if math.isnan(want):
            assert math.isnan(got), c
        else:
            assert got == want, (c, got, want)
    # the format's landmarks: largest finite, smallest normal, smallest subnormal
    assert oracle.code_to_double(0x7E, "e4m3") == 448.0
    assert oracle.code_to_double(0x08, "e4m3") == 2.0 ** -6
    assert oracle.code_to_double(0x01, "e4m3") == 2.0 ** -9


def test_int8_decode_is_twos_complement():
    for c in range(256):
        assert oracle.code_to_double(c, "int8") == (c if c < 128 else c - 256)


def test_e4m3_encode_matches_torch_below_overflow():
    mags = _e4m3_values().numpy()
    mids = (mags[1:] + mags[:-1]) / 2                       # exact ties
    g = wl.uniform01(7, 1, 4000).double().numpy()              # random values in [0, 1)
    rnd = np.concatenate([g * 464.0, g * 2.0 ** -6, g * 2.0 ** -9 * 3])
    vals = np.concatenate([mags, mids, rnd, mids + 1e-9, mids - 1e-9])
    vals = vals[vals <= 464.0]
    vals = np.concatenate([vals, -vals, [-0.0]]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def test_e4m3_encode_saturates_and_rounds_ties_to_even():
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(470.0) == 0x7E                # past the last tie: saturated, not NaN
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00           # half the smallest subnormal -> 0 (even)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02       # 1.5 subnormal steps -> 2 (even)
    assert oracle.e4m3_encode(1.0625) == 0x38               # halfway 1 and 1.125 -> 1.0 (even)
    assert oracle.e4m3_encode(1.1875) == 0x3A               # halfway 1.125 and 1.25 -> 1.25 (even)
    assert oracle.e4m3_encode(-0.0) == 0x80


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_int8_rows_meet_the_rounding_bound(dtype):
    x = wl.normal_tensor(21, 1, (64, 128), dtype=dtype)
    codes, s = oracle.quantize_rows(x, "int8")
    c = codes.to(torch.int64)
    assert int(c.min()) >= -127 and int(c.max()) <= 127
    xf = x.double()
    amax = xf.abs().amax(dim=1)
    assert torch.equal(s, (amax.float() / 127.0))           # the scale as defined, in fp32
    # the largest element maps to +-127, every element to within half a step
    top = xf.abs().argmax(dim=1)
    assert torch.equal(c[torch.arange(64), top].abs(), torch.full((64,), 127))
    # (the quotient x / scale is rounded to fp32 first: up to 127 * 2^-24 of a step)
    err = (xf - c.double() * s.double()[:, None]).abs()
    assert bool((err <= s.double()[:, None] * (0.5 + 127 * 2.0 ** -24)).all())


def test_int8_exact_codes_by_hand():
    # amax = 127 -> scale exactly 1, so x / scale = x and the codes are rint(x)
    row = torch.tensor([[127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -126.4, 0.0]], dtype=torch.float32)
    codes, s = oracle.quantize_rows(row, "int8")
    assert float(s[0]) == 1.0
    assert codes[0].tolist() == [127, 2, 4, -2, 0, 2, -126, 0]
    zero, sz = oracle.quantize_rows(torch.zeros(2, 16), "int8")
    assert float(sz.abs().max()) == 0.0 and int(zero.view(torch.uint8).max()) == 0
    # integer rows with max 127 reproduce themselves exactly
    ints = (torch.arange(-127, 128, dtype=torch.float32)[torch.randperm(255, generator=torch.Generator().manual_seed(1))])
    codes, s = oracle.quantize_rows(ints.reshape(5, 51), "int8")
    for r in range(5):
        if float(ints.reshape(5, 51)[r].abs().max()) == 127.0:
            assert torch.equal(codes[r].to(torch.float32), ints.reshape(5, 51)[r])


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_e4m3_rows_meet_the_rounding_bound(dtype):
    x = wl.normal_tensor(22, 1, (64, 128), dtype=dtype)
    codes, s = oracle.quantize_rows(x, "e4m3")
    xf = x.double()
    assert torch.equal(s, xf.abs().amax(dim=1).float() / 448.0)
    dec = codes.to(torch.float64)                            # torch decodes the oracle's bytes
    v = (x.float() / s[:, None]).double()                    # the quotient the codes round
    assert float(dec.abs().max()) <= 448.0
    # half the spacing of the binade of v (subnormal spacing below 2^-6)
    b = torch.floor(torch.log2(v.abs().clamp_min(2.0 ** -6)))
    half = torch.pow(2.0, b - 4)
    assert bool(((dec - v).abs() <= half * (1 + 1e-12)).all())
    # torch's own conversion of the same fp32 quotient gives the same codes
    want = (x.float() / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(codes.view(torch.uint8), want)


def _quant_identity_case(n_seqs, n_heads, n_kv, d, bs, qdtype, fmt, lens, seed):
    """Identity-table case with 8-bit pages; also returns the codes and scales."""
    M = max(1, max((int(L) + bs - 1) // bs for L in lens))
    nb = n_seqs * M
    k = wl.normal_tensor(seed, 11, (nb, n_kv, bs, d), dtype=torch.float16)
    v = wl.normal_tensor(seed, 12, (nb, n_kv, bs, d), dtype=torch.float16)
    q = wl.normal_tensor(seed, 13, (n_seqs, n_heads, d), dtype=qdtype)
    kc, ks = oracle.quantize_rows(k, fmt)
    vc, vs = oracle.quantize_rows(v, fmt)
    tables = torch.arange(nb, dtype=torch.int32).reshape(n_seqs, M)
    return (q, oracle.pack_pages(kc, ks), oracle.pack_pages(vc, vs), kc, vc, ks, vs, tables,
            torch.tensor(lens, dtype=torch.int32), M)


def _torch_dequant(codes, scales):
    return codes.to(torch.float64) * scales.to(torch.float64)[..., None]


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("case", [(3, 8, 2, 128, 16, [40, 1, 77], 0), (2, 4, 4, 64, 8, [30, 12], 10),
                                  (2, 8, 1, 128, 32, [65, 64], 0), (2, 4, 2, 64, 32, [70, 33], 0)])
def test_quantised_cache_attention_equals_library_sdpa(fmt, case):
    n, H, hkv, d, bs, lens, window = case
    q, kp, vp, kc, vc, ks, vs, t, cl, M = _quant_identity_case(n, H, hkv, d, bs, torch.bfloat16, fmt, lens, seed=5)
    got = oracle.paged_attention(q, kp, vp, t, cl, num_kv_heads=hkv, scale=1 / math.sqrt(d), window=window)
    # torch decodes the codes and applies the row scales; fp64 SDPA on the contiguous view
    kd, vd = _torch_dequant(kc, ks), _torch_dequant(vc, vs)
    N, G = n, H // hkv
    kk = kd.reshape(N, M, hkv, bs, d).permute(0, 2, 1, 3, 4).reshape(N, hkv, M * bs, d)
    vv = vd.reshape(N, M, hkv, bs, d).permute(0, 2, 1, 3, 4).reshape(N, hkv, M * bs, d)
    for s in range(N):
        L = int(cl[s])
        lo = max(0, L - window) if window > 0 else 0
        ref = F.scaled_dot_product_attention(q[s].double().unsqueeze(1), kk[s, :, lo:L].repeat_interleave(G, 0),
                                             vv[s, :, lo:L].repeat_interleave(G, 0),
                                             scale=1 / math.sqrt(d)).squeeze(1)
        np.testing.assert_allclose(got[s], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_page_layout_by_hand():
    """The page of (block 1, head 0) at block 16, head_dim 128: rows 0-15 the
    codes, row 16 the 16 scales then zeros; the oracle reads element (token
    3, dim 5) of that page as code * scale."""
    codes = torch.zeros((2, 1, 16, 128), dtype=torch.int8)
    scales = torch.zeros((2, 1, 16))
    codes[1, 0, 3, 5] = -7
    scales[1, 0, 3] = 0.25
    pages = oracle.pack_pages(codes, scales)
    assert tuple(pages.shape) == (2, 1, 17, 128)
    raw = pages.view(torch.uint8)[1, 0]
    assert int(raw[3, 5]) == 256 - 7
    assert torch.equal(raw[16, 12:16], torch.tensor([0, 0, 128, 62], dtype=torch.uint8))  # 0.25f, little-endian
    assert int(raw[16, 64:].sum()) == 0
    # one token (3) attended through table [1]: the output is V's row 3 = code * scale
    q = torch.ones((1, 1, 128), dtype=torch.float16)
    t = torch.tensor([[1]], dtype=torch.int32)
    cl = torch.tensor([4], dtype=torch.int32)
    vcodes = torch.zeros_like(codes)
    vcodes[1, 0, 3] = 9
    vsc = torch.zeros_like(scales)
    vsc[1, 0, 3] = 0.5
    kp = oracle.pack_pages(torch.zeros_like(codes), torch.zeros_like(scales))
    out = oracle.paged_attention(q, kp, oracle.pack_pages(vcodes, vsc), t, cl, num_kv_heads=1, scale=1.0)
    np.testing.assert_allclose(out[0, 0], np.full(128, 4.5 / 4), rtol=0, atol=0)   # mean over 4 tokens


def test_quantised_cache_k_and_v_scales_are_not_interchangeable():
    # a V-only rescale must change the output by exactly that factor; K's scale
    # moves the softmax instead
    q, kp, vp, kc, vc, ks, vs, t, cl, M = _quant_identity_case(1, 2, 1, 64, 16, torch.float16, "int8", [20], seed=6)
    base = oracle.paged_attention(q, kp, vp, t, cl, num_kv_heads=1, scale=0.125)
    twice_v = oracle.paged_attention(q, kp, oracle.pack_pages(vc, vs * 2), t, cl, num_kv_heads=1, scale=0.125)
    np.testing.assert_allclose(twice_v, 2 * base, rtol=1e-14, atol=0)
    k_zero = oracle.paged_attention(q, oracle.pack_pages(kc, ks * 0), vp, t, cl, num_kv_heads=1, scale=0.125)
    vd = _torch_dequant(vc, vs)                                       # [M, 1, 16, 64], blocks in order
    mean_v = vd.permute(1, 0, 2, 3).reshape(1, -1, 64)[0, :20].mean(dim=0).numpy()  # zero scores -> mean of V
    np.testing.assert_allclose(k_zero[0, 0], mean_v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(k_zero[0, 1], mean_v, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_quantised_cache_block_permutation_is_bit_identical(fmt):
    q, kp, vp, *_, t, cl, M = _quant_identity_case(2, 4, 2, 64, 16, torch.float16, fmt, [50, 33], seed=8)
    base = oracle.paged_attention(q, kp, vp, t, cl, num_kv_heads=2, scale=0.125)
    perm = wl.permutation(9, 1, kp.shape[0])
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    # physical block p moves to slot inv[p]; tables follow
    got = oracle.paged_attention(q, kp[perm], vp[perm], inv[t.long()].to(torch.int32), cl, num_kv_heads=2,
                                 scale=0.125)
    assert np.array_equal(base, got)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("in_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("bs,d", [(16, 64), (32, 64), (8, 128)])
def test_append_quant_stores_the_row_quantisation_at_the_slot(fmt, in_dtype, bs, d):
    nb, hkv, T = 12, 2, 9
    code_dtype = torch.int8 if fmt == "int8" else torch.float8_e4m3fn
    rows = bs + oracle.scale_rows(bs, d)
    kp = torch.full((nb, hkv, rows, d), 0x55, dtype=torch.uint8).view(code_dtype)
    vp = torch.full_like(kp.view(torch.uint8), 0x66).view(code_dtype)
    k0, v0 = kp.clone(), vp.clone()
    k = wl.normal_tensor(30, 1, (T, hkv, d), dtype=in_dtype)
    v = wl.normal_tensor(30, 2, (T, hkv, d), dtype=in_dtype)
    slots = wl.permutation(31, 1, nb * bs)[:T].clone()
    slots[4] = -1
    assert oracle.append_kv_quant(kp, vp, k, v, slots) == 0
    kq, kqs = oracle.quantize_rows(k, fmt)
    vq, vqs = oracle.quantize_rows(v, fmt)
    kc, ks = oracle.unpack_pages(kp)
    vc, vs = oracle.unpack_pages(vp)
    kc0, ks0 = oracle.unpack_pages(k0)
    touched = torch.zeros((nb, bs), dtype=torch.bool)
    for i in range(T):
        sl = int(slots[i])
        if sl < 0:
            continue
        pb, o = sl // bs, sl % bs
        touched[pb, o] = True
        assert torch.equal(kc[pb, :, o].view(torch.uint8), kq[i].view(torch.uint8))
        assert torch.equal(vc[pb, :, o].view(torch.uint8), vq[i].view(torch.uint8))
        assert torch.equal(ks[pb, :, o], kqs[i]) and torch.equal(vs[pb, :, o], vqs[i])
    # untouched rows and scales keep their bytes; the padding after the scales too
    untouched = ~touched
    assert torch.equal(kc.view(torch.uint8).permute(0, 2, 1, 3)[untouched],
                       kc0.view(torch.uint8).permute(0, 2, 1, 3)[untouched])
    assert torch.equal(ks.permute(0, 2, 1)[untouched].view(torch.int32),
                       ks0.permute(0, 2, 1)[untouched].view(torch.int32))
    pad = kp.view(torch.uint8)[:, :, bs:].reshape(nb, hkv, -1)[:, :, 4 * bs:]
    assert bool((pad == 0x55).all())
    # duplicates refused, out-of-range counted
    with pytest.raises(ValueError):
        oracle.append_kv_quant(kp, vp, k[:2], v[:2], torch.tensor([3, 3]))
    assert oracle.append_kv_quant(kp, vp, k[:1], v[:1], torch.tensor([nb * bs])) == 1


def test_append_quant_worked_example_slot():
    """Token 34 through the page's table [7, 1, 3] (block size 16): its codes
    and scale land in the page of physical block 3, row 2."""
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    bs = g["block_size"]
    kp = torch.zeros((8, 1, bs + 1, 64), dtype=torch.int8)
    vp = torch.zeros_like(kp)
    row = torch.full((1, 1, 64), 3.0, dtype=torch.float16)
    slot = g["physical"] * bs + g["offset"]
    oracle.append_kv_quant(kp, vp, row, row, torch.tensor([slot]))
    kc, ks = oracle.unpack_pages(kp)
    assert float(ks[3, 0, 2]) == float(torch.tensor(3.0) / 127.0) and bool((kc[3, 0, 2] == 127).all())
    assert int((kc != 0).sum()) == 64 and int((ks != 0).sum()) == 1


def test_quantised_page_copy_moves_codes_and_scales():
    nb, hkv, bs, d = 6, 2, 8, 64
    codes = (wl.bits64(40, 1, nb * hkv * bs * d) & 0xFF).to(torch.uint8).reshape(nb, hkv, bs, d).view(torch.int8)
    kp = oracle.pack_pages(codes, torch.rand(nb, hkv, bs))
    vp = oracle.pack_pages(codes.flip(0), torch.rand(nb, hkv, bs))
    k0, v0 = kp.clone(), vp.clone()
    oracle.copy_blocks(kp, vp, [[1, 4]])
    assert torch.equal(kp[4], k0[1]) and torch.equal(vp[4], v0[1])
    keep = [0, 1, 2, 3, 5]
    assert torch.equal(kp[keep], k0[keep]) and torch.equal(vp[keep], v0[keep])
