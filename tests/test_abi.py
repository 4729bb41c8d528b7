"""CPU checks of the C ABI: the library loads, exports every function that
include/*.h declares, and rejects bad arguments on the host before any CUDA
call (fake device addresses are never dereferenced on these paths)."""
import ctypes
import re
from pathlib import Path

import pytest

from paged_kv_cache_251_gb300 import build as pbuild

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    path = pbuild.build()
    return ctypes.CDLL(str(path))


def declared_functions():
    names = []
    for h in sorted((ROOT / "include").glob("*.h")):
        names += re.findall(r"^PA_API\s+[\w\s\*]+?\b(\w+)\s*\(", h.read_text(), flags=re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"pa_decode", "pa_append_kv", "pa_copy_blocks", "pa_decode_workspace_size",
            "pa_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def _decode_args(**over):
    a = dict(out=0x1000, q=0x2000, k=0x3000, v=0x4000, bt=0x5000, cl=0x6000, N=4, H=8, Hkv=2, d=128,
             bs=16, scale=0.088, window=0, dtype=1, out_dtype=0, M=8, nb=64, part=0, ws=0, wsb=0, err=0,
             stream=0)
    a.update(over)
    return a


def _call_decode(lib, **over):
    a = _decode_args(**over)
    P = ctypes.c_void_p
    f = lib.pa_decode
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, P, ctypes.c_size_t, P, P]
    return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["N"], a["H"], a["Hkv"], a["d"], a["bs"],
             a["scale"], a["window"], a["dtype"], a["out_dtype"], a["M"], a["nb"], a["part"], a["ws"],
             a["wsb"], a["err"], a["stream"])


def test_decode_host_validation(lib):
    INV, UNS, WS = 1, 2, 3
    assert _call_decode(lib, N=0) == 0                     # nothing to do, no launch
    assert _call_decode(lib, d=96) == UNS
    assert _call_decode(lib, bs=12) == UNS
    assert _call_decode(lib, H=12, Hkv=4) == UNS           # group of 3
    assert _call_decode(lib, H=9, Hkv=2) == INV            # not a multiple
    assert _call_decode(lib, q=0) == INV
    assert _call_decode(lib, k=0x3008) == INV              # misaligned cache
    assert _call_decode(lib, dtype=7) == INV
    assert _call_decode(lib, part=24) == INV               # not a multiple of the block size
    assert _call_decode(lib, part=16 * 257) == INV         # more than 256 blocks
    assert _call_decode(lib, M=100, ws=0, wsb=0) == WS     # 100 blocks span several partitions
    assert _call_decode(lib, window=-1) == INV
    assert _call_decode(lib, nb=0) == INV
    assert _call_decode(lib, scale=float("inf")) == INV


def test_workspace_size(lib):
    f = lib.pa_decode_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 7
    # one partition (<= 512 tokens at block 16): no workspace
    assert f(64, 40, 128, 16, 32, 0, 0) == 0
    # OPT-13B-shaped batch: table rows of 129 blocks -> 5 partitions of 32 blocks
    assert f(64, 40, 128, 16, 129, 0, 0) == 64 * 40 * 5 * (128 + 2) * 4
    # 4 x 131072 tokens, window 32768 (2049 blocks), 512-token partitions -> 65
    assert f(4, 32, 128, 16, 8192, 32768, 512) == 4 * 32 * 65 * 130 * 4
    assert f(4, 32, 96, 16, 8192, 0, 0) == 0                # unsupported -> 0


def test_cache_ops_host_validation(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    ap = lib.pa_append_kv
    ap.restype = I
    ap.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
    assert ap(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0, 8, 128, 16, 10, 1, None, None) == 0
    assert ap(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 4, 8, 100, 16, 10, 1, None, None) == 2
    assert ap(0x1000, 0x2004, 0x3000, 0x4000, 0x5000, 4, 8, 128, 16, 10, 1, None, None) == 1
    assert ap(0x1000, 0x2000, 0x3004, 0x4000, 0x5000, 4, 8, 128, 16, 10, 1, None, None) == 1
    cp = lib.pa_copy_blocks
    cp.restype = I
    cp.argtypes = [P, I, P, P, I, I, I, I, I, P, P]
    assert cp(0x1000, 0, 0x2000, 0x3000, 8, 128, 16, 10, 2, None, None) == 0
    assert cp(None, 3, 0x2000, 0x3000, 8, 128, 16, 10, 2, None, None) == 1
    assert cp(0x1000, 3, 0x2000, 0x3000, 8, 128, 24, 10, 2, None, None) == 2
    st = lib.pa_status_string
    st.restype = ctypes.c_char_p
    st.argtypes = [I]
    assert st(3) == b"PA_ERR_WORKSPACE_TOO_SMALL"


def _call_decode_quant(lib, **over):
    a = dict(out=0x1000, q=0x2000, k=0x3000, v=0x4000, bt=0x5000, cl=0x6000, N=4, H=8,
             Hkv=2, d=128, bs=16, scale=0.088, window=0, dtype=1, cdt=3, out_dtype=0, M=8, nb=64, part=0, ws=0,
             wsb=0, err=0, stream=0)
    a.update(over)
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.pa_decode_quant
    f.restype = I
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, ctypes.c_float, I, I, I, I, I, I, I, P, ctypes.c_size_t, P, P]
    return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["N"], a["H"], a["Hkv"],
             a["d"], a["bs"], a["scale"], a["window"], a["dtype"], a["cdt"], a["out_dtype"], a["M"], a["nb"],
             a["part"], a["ws"], a["wsb"], a["err"], a["stream"])


def test_decode_quant_host_validation(lib):
    INV, UNS, WS = 1, 2, 3
    assert _call_decode_quant(lib, N=0) == 0
    assert _call_decode_quant(lib, cdt=1) == INV           # a 16-bit dtype is not a code dtype
    assert _call_decode_quant(lib, cdt=5) == INV
    assert _call_decode_quant(lib, dtype=3) == INV         # q cannot be 8-bit
    assert _call_decode_quant(lib, k=0) == INV
    assert _call_decode_quant(lib, v=0x4008) == INV        # misaligned page pool
    assert _call_decode_quant(lib, d=96) == UNS
    assert _call_decode_quant(lib, H=12, Hkv=4) == UNS
    assert _call_decode_quant(lib, M=100) == WS


def test_quant_page_bytes(lib):
    f = lib.pa_quant_page_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int]
    # block_size code rows of head_dim bytes + ceil(4 * block_size / head_dim) scale rows
    assert f(128, 16) == 17 * 128
    assert f(128, 8) == 9 * 128
    assert f(128, 32) == 33 * 128
    assert f(64, 16) == 17 * 64
    assert f(64, 32) == 34 * 64
    assert f(96, 16) == 0 and f(128, 12) == 0


def test_append_quant_host_validation(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.pa_append_kv_quant
    f.restype = I
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, P]
    ok = dict(k=0x1000, v=0x2000, sl=0x3000, kc=0x4000, vc=0x5000, T=4, Hkv=2, d=128, bs=16, nb=8, dt=1, cdt=4)

    def call(**o):
        a = dict(ok, **o)
        return f(a["k"], a["v"], a["sl"], a["kc"], a["vc"], a["T"], a["Hkv"], a["d"], a["bs"], a["nb"], a["dt"],
                 a["cdt"], None, None)

    assert call(T=0) == 0
    assert call(cdt=2) == 1
    assert call(dt=4) == 1
    assert call(vc=0) == 1
    assert call(sl=0x3004) == 1
    assert call(d=32) == 2
    assert call(bs=4) == 2


def test_noalloc_reports_bad_arguments_before_the_scratch_limit(lib):
    """pa_decode_noalloc on a shape too large for its built-in scratch: a bad
    argument is reported as itself, and only a valid call comes back as
    PA_ERR_WORKSPACE_TOO_SMALL (nothing is launched on either path)."""
    INV, UNS, WS = 1, 2, 3
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.pa_decode_noalloc
    f.restype = I
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, ctypes.c_float, I, I, I, I, I, I, P, P]
    lim = lib.pa_decode_noalloc_max_scratch
    lim.restype = ctypes.c_size_t
    ws = lib.pa_decode_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [I] * 7
    # 4096 seqs x 64 heads x d 128, 64-token partitions over 512-block rows: far beyond the scratch
    big = dict(out=0x1000, q=0x2000, k=0x3000, v=0x4000, bt=0x5000, cl=0x6000, N=4096, H=64, Hkv=64, d=128,
               bs=16, scale=0.088, window=0, dtype=1, out_dtype=0, M=512, nb=64, part=64, err=None, stream=None)
    assert ws(4096, 64, 128, 16, 512, 0, 64) > lim()

    def call(**o):
        a = dict(big, **o)
        return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["cl"], a["N"], a["H"], a["Hkv"], a["d"], a["bs"],
                 a["scale"], a["window"], a["dtype"], a["out_dtype"], a["M"], a["nb"], a["part"], a["err"],
                 a["stream"])

    assert call() == WS
    assert call(q=0) == INV
    assert call(k=0x3008) == INV
    assert call(dtype=9) == INV
    assert call(H=48, Hkv=16) == UNS               # a group of 3
    assert call(nb=0) == INV
    assert call(scale=float("nan")) == INV


def test_contiguous_decode_host_validation(lib):
    INV, UNS, WS = 1, 2, 3
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.pa_decode_contiguous
    f.restype = I
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_float, I, I, I, I, P, ctypes.c_size_t, P, P]
    ok = dict(out=0x1000, q=0x2000, k=0x3000, v=0x4000, cl=0x6000, N=4, H=8, Hkv=2, d=128, L=256, scale=0.088,
              window=0, dtype=2, out_dtype=0, part=0, ws=None, wsb=0, err=None, stream=None)

    def call(**o):
        a = dict(ok, **o)
        return f(a["out"], a["q"], a["k"], a["v"], a["cl"], a["N"], a["H"], a["Hkv"], a["d"], a["L"], a["scale"],
                 a["window"], a["dtype"], a["out_dtype"], a["part"], a["ws"], a["wsb"], a["err"], a["stream"])

    assert call(N=0) == 0
    assert call(L=100) == INV                     # not a multiple of 16
    assert call(L=0) == INV
    assert call(cl=0) == INV
    assert call(k=0x3008) == INV
    assert call(H=12, Hkv=4) == UNS               # a group of 3
    assert call(dtype=0) == UNS                   # fp32 with grouped heads
    assert call(d=64) == UNS                      # head_dim 64 with grouped heads
    assert call(L=16 * 1000) == WS                # several partitions need a workspace
