"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins catch every one of them (the mistakes live only in the copies, which
are compiled and loaded by this test on the CPU)."""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from oracle import build as obuild

from test_oracle_pins import _identity_case, _sdpa_reference

GOLDEN = Path(__file__).parent / "golden"
SRC = (Path(oracle.__file__).parent / "pa_oracle.c").read_text()

MUTANTS = {
    "offset_uses_division": ("*offset = (int32_t)(token % block_size);",
                             "*offset = (int32_t)(token / block_size);"),
    "scale_dropped": ("x[i] = a->scale * dot;", "x[i] = dot;"),
    "wrong_kv_head": ("const int kvh = h / group;", "const int kvh = h % a->num_kv_heads;"),
    "softmax_sign": ("const double w = exp(x[i] - m);", "const double w = exp(m - x[i]);"),
    "window_off_by_one": ("start = L - a->window;", "start = L - a->window + 1;"),
    "cache_axes_transposed": (
        "row[i] = (((int64_t)phys * a->num_kv_heads + kvh) * a->block_size + off) * d;",
        "row[i] = (((int64_t)phys * a->block_size + off) * a->num_kv_heads + kvh) * d;"),
    "no_normalisation": ("out_row[j] /= denom;", "out_row[j] /= 1.0;"),
    "q_row_of_wrong_head": ("const int64_t q_base = ((int64_t)s * a->num_heads + h) * d;",
                            "const int64_t q_base = ((int64_t)s * a->num_heads + kvh) * d;"),
}


def _pins_pass(lib) -> bool:
    g = json.loads((GOLDEN / "locate_worked_example.json").read_text())
    try:
        if oracle.locate(g["block_table"], g["block_size"], g["token"], lib=lib) != (g["physical"], g["offset"]):
            return False
    except IndexError:
        return False
    for (n, H, hkv, d, bs, lens, window) in [(2, 8, 2, 64, 16, [40, 21], 0),
                                              (2, 4, 4, 64, 8, [30, 12], 10)]:
        q, k, v, t, cl, M = _identity_case(n, H, hkv, d, bs, torch.float32, lens, seed=3)
        try:
            got = oracle.paged_attention(q, k, v, t, cl, num_kv_heads=hkv, scale=1 / math.sqrt(d),
                                         window=window, lib=lib)
        except ValueError:
            return False
        ref = _sdpa_reference(q, k, v, cl, M, bs, hkv, window=window, scale=1 / math.sqrt(d))
        if not np.allclose(got, ref, rtol=1e-12, atol=1e-13):
            return False
    return True


def test_unmodified_oracle_passes_the_pins():
    assert _pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found"
    lib = oracle.load(obuild.build_from_text(SRC.replace(old, new), name))
    assert not _pins_pass(lib)


# ---------------------------------------------------------------------------
# 8-bit cache: mistakes in the quantiser, the code tables and the dequantised read

QUANT_MUTANTS = {
    "int8_scale_over_128": ("const float q = fmt == ORC_I8 ? 127.0f : 448.0f;",
                            "const float q = fmt == ORC_I8 ? 128.0f : 448.0f;"),
    "int8_truncates": ("float r = rintf(v);", "float r = truncf(v);"),
    "e4m3_bias_off_by_one": ("v = ldexp((double)(8 + mant), expo - 10);",
                             "v = ldexp((double)(8 + mant), expo - 9);"),
    "e4m3_ties_away_from_zero": ("const double r = nearbyint(a / quantum);",
                                 "const double r = floor(a / quantum + 0.5);"),
    "e4m3_no_subnormal_floor": ("    if (b < -6)\n        b = -6;\n    const double quantum",
                                "    const double quantum"),
    "scale_read_one_row_late": ("memcpy(&sc, pg + (int64_t)bs * d + 4 * r, 4);",
                                "memcpy(&sc, pg + (int64_t)bs * d + 4 * (r + 1), 4);"),
    "page_stride_without_scale_rows": (
        "const int64_t page_bytes = (int64_t)(bs + orc_scale_rows(bs, d)) * d;",
        "const int64_t page_bytes = (int64_t)bs * d;"),
    "append_k_codes_from_v": (
        "orc_quantize_row(k, in_dtype, src_row, head_dim, fmt, kp + off * head_dim, &ks);",
        "orc_quantize_row(v, in_dtype, src_row, head_dim, fmt, kp + off * head_dim, &ks);"),
}


def _quant_pins_pass(lib) -> bool:
    from test_oracle_quant import _quant_identity_case, _torch_dequant
    import torch.nn.functional as F
    from paged_kv_cache_251_gb300 import workloads as wl
    # code tables and the encoder against torch's float8_e4m3fn
    for c in range(256):
        want = torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).item()
        got = oracle.code_to_double(c, "e4m3", lib=lib)
        if not (math.isnan(want) and math.isnan(got)) and got != want:
            return False
    g = wl.uniform01(7, 1, 2000).double().numpy()
    vals = np.concatenate([g * 464.0, g * 2.0 ** -6, -g * 3.0]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ties = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10], dtype=np.float32)
    if any(oracle.e4m3_encode(float(v), lib=lib) != w for v, w in zip(vals, want)):
        return False
    if [oracle.e4m3_encode(float(v), lib=lib) for v in ties] != [0x38, 0x3A, 0x00, 0x02]:
        return False
    # int8 rows: scale, the largest element at +-127, the rounding bound
    x = wl.normal_tensor(21, 1, (16, 128), dtype=torch.float16)
    codes, s = oracle.quantize_rows(x, "int8", lib=lib)
    c, xf = codes.to(torch.int64), x.double()
    if not torch.equal(s, xf.abs().amax(dim=1).float() / 127.0):
        return False
    if not torch.equal(c[torch.arange(16), xf.abs().argmax(dim=1)].abs(), torch.full((16,), 127)):
        return False
    if not bool(((xf - c.double() * s.double()[:, None]).abs() <= s.double()[:, None] * (0.5 + 1e-5)).all()):
        return False
    # attention over a quantised cache against torch SDPA on torch-decoded values
    for fmt in ("int8", "e4m3"):
        q, kp, vp, kc, vc, ks, vs, t, cl, M = _quant_identity_case(2, 4, 2, 64, 16, torch.float16, fmt, [40, 21],
                                                                   seed=5)
        got = oracle.paged_attention(q, kp, vp, t, cl, num_kv_heads=2, scale=0.125, lib=lib)
        kd = _torch_dequant(kc, ks).reshape(2, M, 2, 16, 64).permute(0, 2, 1, 3, 4).reshape(2, 2, M * 16, 64)
        vd = _torch_dequant(vc, vs).reshape(2, M, 2, 16, 64).permute(0, 2, 1, 3, 4).reshape(2, 2, M * 16, 64)
        for si in range(2):
            L = int(cl[si])
            ref = F.scaled_dot_product_attention(q[si].double().unsqueeze(1), kd[si, :, :L].repeat_interleave(2, 0),
                                                 vd[si, :, :L].repeat_interleave(2, 0), scale=0.125).squeeze(1)
            if not np.allclose(got[si], ref.numpy(), rtol=1e-12, atol=1e-13):
                return False
    # quantise-on-append stores each row's quantisation at its slot
    kp = torch.zeros((4, 2, 17, 64), dtype=torch.int8)
    vp = torch.zeros_like(kp)
    k = wl.normal_tensor(30, 1, (3, 2, 64), dtype=torch.float16)
    v = wl.normal_tensor(30, 2, (3, 2, 64), dtype=torch.float16)
    oracle.append_kv_quant(kp, vp, k, v, torch.tensor([5, 17, 40]), lib=lib)
    kc, ks = oracle.unpack_pages(kp)
    vc, vs = oracle.unpack_pages(vp)
    kq, kqs = oracle.quantize_rows(k, "int8")
    vq, vqs = oracle.quantize_rows(v, "int8")
    for i, sl in enumerate([5, 17, 40]):
        p_, o_ = sl // 16, sl % 16
        if not (torch.equal(kc[p_, :, o_], kq[i]) and torch.equal(vc[p_, :, o_], vq[i])
                and torch.equal(ks[p_, :, o_], kqs[i]) and torch.equal(vs[p_, :, o_], vqs[i])):
            return False
    return True


def test_unmodified_oracle_passes_the_quant_pins():
    assert _quant_pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(QUANT_MUTANTS))
def test_planted_quantiser_mistake_is_caught(name):
    old, new = QUANT_MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found"
    lib = oracle.load(obuild.build_from_text(SRC.replace(old, new), name))
    assert not _quant_pins_pass(lib)
