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
