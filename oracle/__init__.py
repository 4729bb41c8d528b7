"""CPU oracle for paged decode attention, KV append, block copy, copy-on-write
and the sliding-window ring.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It shares
no code with the CUDA library in ``paged_kv_cache_251_gb300`` and never
imports it.

The arithmetic lives in ``pa_oracle.c`` (fp64, one token at a time) and in
``cow.py`` (block-table bookkeeping as plain Python).  This module only moves
torch CPU tensors in and out of the C functions.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np
import torch

from . import build as _build
from .cow import CowModel, RingModel  # noqa: F401  (re-exported)

F32, F16, BF16, I8, E4M3 = 0, 1, 2, 3, 4
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
# 8-bit caches: the code pools are carried as int8 / float8_e4m3fn tensors
_CODE_FMT = {torch.int8: I8, torch.float8_e4m3fn: E4M3}
_FMT_DTYPE = {I8: torch.int8, E4M3: torch.float8_e4m3fn, "int8": torch.int8, "e4m3": torch.float8_e4m3fn}

_lib = None


def load(path: Path | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(str(_build.build())))
    return _lib


def _bind(lib):
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.orc_locate.argtypes = [P, I, I, I64, P, P]
    lib.orc_locate.restype = I
    lib.orc_paged_attention.argtypes = [P, P, P, P, P, P, I, I, I, I, I, D, I, I, I, I, I, P, I64, I, P]
    lib.orc_paged_attention.restype = I
    lib.orc_append_kv.argtypes = [P, P, P, P, P, I64, I, I, I, I, I]
    lib.orc_append_kv.restype = I64
    lib.orc_copy_blocks.argtypes = [P, P, P, I64, I, I, I, I, I]
    lib.orc_copy_blocks.restype = I64
    lib.orc_swap_blocks.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, I]
    lib.orc_swap_blocks.restype = I64
    lib.orc_element_to_double.argtypes = [P, I, I64]
    lib.orc_element_to_double.restype = D
    lib.orc_code_to_double.argtypes = [ctypes.c_uint8, I]
    lib.orc_code_to_double.restype = D
    lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_quantize_rows.argtypes = [P, I, I64, I, I, P, P]
    lib.orc_quantize_rows.restype = I
    lib.orc_paged_attention_cache.argtypes = [P, P, P, P, P, P, I, I, I, I, I, D, I, I, I, I, I, I,
                                              P, I64, I, P]
    lib.orc_paged_attention_cache.restype = I
    lib.orc_append_kv_quant.argtypes = [P, P, P, P, P, I64, I, I, I, I, I, I]
    lib.orc_append_kv_quant.restype = I64
    lib.orc_scale_rows.argtypes = [I, I]
    lib.orc_scale_rows.restype = I
    return lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu" or not t.is_contiguous():
        t = t.detach().to("cpu").contiguous()
    return t


def locate(block_table, block_size: int, token: int, lib=None) -> tuple[int, int]:
    """(physical block, offset) of a logical token through one block table."""
    lib = lib or load()
    tbl = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    phys, off = ctypes.c_int32(), ctypes.c_int32()
    rc = lib.orc_locate(tbl.ctypes.data, tbl.size, block_size, token,
                        ctypes.byref(phys), ctypes.byref(off))
    if rc != 0:
        raise IndexError(f"token {token} is beyond the block table")
    return phys.value, off.value


def to_double(t: torch.Tensor, lib=None) -> np.ndarray:
    """Exact fp64 values of a float32/float16/bfloat16 tensor, via the oracle's
    own element conversion."""
    lib = lib or load()
    t = _cpu(t)
    code = _DTYPE_CODE[t.dtype]
    flat = t.reshape(-1)
    out = np.empty(flat.numel(), dtype=np.float64)
    for i in range(flat.numel()):
        out[i] = lib.orc_element_to_double(ctypes.c_void_p(flat.data_ptr()), code, i)
    return out.reshape(tuple(t.shape))


def code_to_double(code: int, fmt, lib=None) -> float:
    """Value of one 8-bit code (fmt: "int8" / "e4m3" or I8 / E4M3)."""
    f = {"int8": I8, "e4m3": E4M3}.get(fmt, fmt)
    return (lib or load()).orc_code_to_double(int(code) & 0xFF, int(f))


def e4m3_encode(x: float, lib=None) -> int:
    """The oracle's fp32 -> E4M3 code (nearest, ties to even, saturating)."""
    return int((lib or load()).orc_e4m3_encode(float(x)))


def quantize_rows(x: torch.Tensor, fmt, lib=None):
    """Quantise the last axis of x (fp32/fp16/bf16) row by row.

    Returns (codes, scales): codes of x's shape as int8 ("int8") or
    float8_e4m3fn ("e4m3") holding the oracle's bytes, scales float32 of
    x.shape[:-1].  Dequantised row: codes * scales[..., None].
    """
    lib = lib or load()
    x = _cpu(x)
    code_dtype = _FMT_DTYPE[fmt]
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    codes = torch.zeros(x.shape, dtype=torch.uint8)
    scales = torch.zeros(x.shape[:-1], dtype=torch.float32)
    rc = lib.orc_quantize_rows(x.data_ptr(), _DTYPE_CODE[x.dtype], rows, d, _CODE_FMT[code_dtype],
                               codes.data_ptr(), scales.data_ptr())
    if rc != 0:
        raise ValueError(f"oracle quantize_rows failed with code {rc}")
    return codes.view(code_dtype), scales


def scale_rows(block_size: int, head_dim: int) -> int:
    """Rows of a page that hold its fp32 row scales: ceil(4 * block_size / head_dim)."""
    return (4 * block_size + head_dim - 1) // head_dim


def page_block_size(rows: int, head_dim: int) -> int:
    """block_size of a page with `rows` rows (codes + scale rows)."""
    for bs in (8, 16, 32):
        if bs + scale_rows(bs, head_dim) == rows:
            return bs
    raise ValueError(f"no block size gives a {rows}-row page at head_dim {head_dim}")


def pack_pages(codes: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """8-bit pages [nb, H_kv, bs + scale_rows, d] from codes [nb, H_kv, bs, d]
    (int8 / float8_e4m3fn) and scales float32 [nb, H_kv, bs]: the code rows,
    then the scales' bytes, then zeros."""
    nb, hkv, bs, d = codes.shape
    sr = scale_rows(bs, d)
    pages = torch.zeros((nb, hkv, bs + sr, d), dtype=torch.uint8)
    pages[:, :, :bs] = codes.view(torch.uint8)
    sb = scales.contiguous().view(torch.uint8).reshape(nb, hkv, 4 * bs)
    pages[:, :, bs:].reshape(nb, hkv, sr * d)[:, :, :4 * bs] = sb
    return pages.view(codes.dtype)


def unpack_pages(pages: torch.Tensor):
    """(codes [nb, H_kv, bs, d], scales float32 [nb, H_kv, bs]) of 8-bit pages."""
    nb, hkv, rows, d = pages.shape
    bs = page_block_size(rows, d)
    u8 = pages.view(torch.uint8)
    codes = u8[:, :, :bs].contiguous().view(pages.dtype)
    scales = u8[:, :, bs:].reshape(nb, hkv, -1)[:, :, :4 * bs].contiguous().view(torch.float32)
    return codes, scales


def dequantize(codes: torch.Tensor, scales: torch.Tensor, lib=None) -> np.ndarray:
    """fp64 values code * scale, codes decoded by the oracle's own tables."""
    lib = lib or load()
    codes, scales = _cpu(codes), _cpu(scales)
    fmt = _CODE_FMT[codes.dtype]
    table = np.array([lib.orc_code_to_double(c, fmt) for c in range(256)], dtype=np.float64)
    vals = table[codes.view(torch.uint8).numpy().astype(np.int64)]
    return vals * scales.numpy().astype(np.float64)[..., None]


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, *, num_kv_heads: int,
                    scale: float, window: int = 0, pairs=None, invalid_policy: int = 0,
                    threads: int = 1, lib=None, return_skipped: bool = False):
    """fp64 decode attention read through the block tables.

    q [N, H, d]; caches [num_blocks, H_kv, bs, d]; block_tables int32 [N, M];
    context_lens int32 [N].  ``pairs`` (int32 [P, 2] of (seq, head)) limits
    the work to those rows and returns [P, d]; otherwise [N, H, d].
    8-bit caches are int8 / float8_e4m3fn pages [num_blocks, H_kv, bs +
    scale_rows, d] (see pack_pages); every cached value is code * scale.
    """
    lib = lib or load()
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
    if k_cache.dtype in _CODE_FMT:
        if v_cache.dtype != k_cache.dtype:
            raise TypeError("both 8-bit pools must share one code dtype")
        return _paged_attention_cache(q, k_cache, v_cache, block_tables, context_lens, num_kv_heads, scale,
                                      window, pairs, invalid_policy, threads, lib, return_skipped)
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q, k_cache and v_cache must share one dtype")
    bt = _cpu(block_tables).to(torch.int32).contiguous()
    cl = _cpu(context_lens).to(torch.int32).contiguous()
    N, H, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d2 == d and hkv == num_kv_heads and tuple(v_cache.shape) == tuple(k_cache.shape)
    M = bt.shape[1]
    if pairs is not None:
        pr = torch.as_tensor(pairs, dtype=torch.int32).reshape(-1, 2).contiguous()
        out = np.zeros((pr.shape[0], d), dtype=np.float64)
        pptr, npairs = pr.data_ptr(), pr.shape[0]
    else:
        out = np.zeros((N, H, d), dtype=np.float64)
        pptr, npairs = None, 0
    skipped = ctypes.c_int64(0)
    rc = lib.orc_paged_attention(out.ctypes.data, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                 bt.data_ptr(), cl.data_ptr(), N, H, num_kv_heads, d, bs, float(scale),
                                 int(window), _DTYPE_CODE[q.dtype], M, nb, invalid_policy,
                                 pptr, npairs, threads, ctypes.byref(skipped))
    if rc != 0:
        raise ValueError(f"oracle paged_attention failed with code {rc}")
    return (out, skipped.value) if return_skipped else out


def _paged_attention_cache(q, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                           scale, window, pairs, invalid_policy, threads, lib, return_skipped):
    bt = _cpu(block_tables).to(torch.int32).contiguous()
    cl = _cpu(context_lens).to(torch.int32).contiguous()
    N, H, d = q.shape
    nb, hkv, rows, d2 = k_cache.shape
    bs = page_block_size(rows, d)
    assert d2 == d and hkv == num_kv_heads and tuple(v_cache.shape) == tuple(k_cache.shape)
    M = bt.shape[1]
    if pairs is not None:
        pr = torch.as_tensor(pairs, dtype=torch.int32).reshape(-1, 2).contiguous()
        out = np.zeros((pr.shape[0], d), dtype=np.float64)
        pptr, npairs = pr.data_ptr(), pr.shape[0]
    else:
        out = np.zeros((N, H, d), dtype=np.float64)
        pptr, npairs = None, 0
    skipped = ctypes.c_int64(0)
    rc = lib.orc_paged_attention_cache(out.ctypes.data, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       bt.data_ptr(), cl.data_ptr(),
                                       N, H, num_kv_heads, d, bs, float(scale), int(window),
                                       _DTYPE_CODE[q.dtype], _CODE_FMT[k_cache.dtype], M, nb, invalid_policy,
                                       pptr, npairs, threads, ctypes.byref(skipped))
    if rc != 0:
        raise ValueError(f"oracle paged_attention failed with code {rc}")
    return (out, skipped.value) if return_skipped else out


def append_kv_quant(k_pages: torch.Tensor, v_pages: torch.Tensor, k, v, slot_mapping, lib=None) -> int:
    """Quantise each token's K/V rows and store codes and scale in the slot's
    page, in place on CPU 8-bit pages (int8 / float8_e4m3fn [nb, H_kv, bs +
    scale_rows, d]).  Returns the out-of-range slots skipped."""
    lib = lib or load()
    for t in (k_pages, v_pages):
        assert t.device.type == "cpu" and t.is_contiguous()
    k, v = _cpu(k), _cpu(v)
    sm = _cpu(torch.as_tensor(slot_mapping)).to(torch.int64).contiguous()
    nb, hkv, rows, d = k_pages.shape
    bs = page_block_size(rows, d)
    rc = lib.orc_append_kv_quant(k_pages.data_ptr(), v_pages.data_ptr(), k.data_ptr(), v.data_ptr(),
                                 sm.data_ptr(), sm.numel(), hkv, d, bs, nb, _DTYPE_CODE[k.dtype],
                                 _CODE_FMT[k_pages.dtype])
    if rc < 0:
        raise ValueError(f"oracle append_kv_quant refused the input (code {rc})")
    return int(rc)


def _as_pool(t: torch.Tensor) -> torch.Tensor:
    # a scale pool [nb, H_kv, bs] is a pool of one-element rows
    return t.unsqueeze(-1) if t.dim() == 3 else t


def append_kv(k_cache: torch.Tensor, v_cache: torch.Tensor, k, v, slot_mapping, lib=None) -> int:
    """Byte-copy each token's K/V rows into its slot, in place on CPU tensors.
    Returns the number of out-of-range slots that were skipped."""
    lib = lib or load()
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous() and v_cache.is_contiguous()
    k, v = _cpu(k), _cpu(v)
    sm = _cpu(torch.as_tensor(slot_mapping)).to(torch.int64).contiguous()
    nb, hkv, bs, d = k_cache.shape
    rc = lib.orc_append_kv(k_cache.data_ptr(), v_cache.data_ptr(), k.data_ptr(), v.data_ptr(),
                           sm.data_ptr(), sm.numel(), hkv, d, bs, nb, k_cache.element_size())
    if rc < 0:
        raise ValueError(f"oracle append_kv refused the input (code {rc})")
    return int(rc)


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs, lib=None) -> int:
    """Copy whole blocks (all kv heads, K and V) for each (src, dst) pair, in
    place on CPU tensors.  Returns the number of out-of-range pairs skipped."""
    lib = lib or load()
    assert k_cache.device.type == "cpu" and k_cache.is_contiguous() and v_cache.is_contiguous()
    k_cache, v_cache = _as_pool(k_cache), _as_pool(v_cache)
    pr = _cpu(torch.as_tensor(src_dst_pairs)).to(torch.int64).reshape(-1, 2).contiguous()
    nb, hkv, bs, d = k_cache.shape
    rc = lib.orc_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), pr.data_ptr(), pr.shape[0],
                             hkv, d, bs, nb, k_cache.element_size())
    if rc < 0:
        raise ValueError(f"oracle copy_blocks refused the input (code {rc})")
    return int(rc)


def swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor, dst_v: torch.Tensor,
                src_dst_pairs, lib=None) -> int:
    """Copy block src of the source pool onto block dst of the destination
    pool (K and V), in place on CPU tensors.  Returns the out-of-range pairs."""
    lib = lib or load()
    assert dst_k.device.type == "cpu" and dst_k.is_contiguous() and dst_v.is_contiguous()
    src_k, src_v = _as_pool(_cpu(src_k)), _as_pool(_cpu(src_v))
    dst_k, dst_v = _as_pool(dst_k), _as_pool(dst_v)
    pr = _cpu(torch.as_tensor(src_dst_pairs)).to(torch.int64).reshape(-1, 2).contiguous()
    snb, hkv, bs, d = src_k.shape
    dnb = dst_k.shape[0]
    rc = lib.orc_swap_blocks(src_k.data_ptr(), src_v.data_ptr(), dst_k.data_ptr(), dst_v.data_ptr(), pr.data_ptr(),
                             pr.shape[0], snb, dnb, hkv, d, bs, src_k.element_size())
    if rc < 0:
        raise ValueError(f"oracle swap_blocks refused the input (code {rc})")
    return int(rc)
