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

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

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


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, *, num_kv_heads: int,
                    scale: float, window: int = 0, pairs=None, invalid_policy: int = 0,
                    threads: int = 1, lib=None, return_skipped: bool = False):
    """fp64 decode attention read through the block tables.

    q [N, H, d]; caches [num_blocks, H_kv, bs, d]; block_tables int32 [N, M];
    context_lens int32 [N].  ``pairs`` (int32 [P, 2] of (seq, head)) limits
    the work to those rows and returns [P, d]; otherwise [N, H, d].
    """
    lib = lib or load()
    q, k_cache, v_cache = _cpu(q), _cpu(k_cache), _cpu(v_cache)
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
    src_k, src_v = _cpu(src_k), _cpu(src_v)
    pr = _cpu(torch.as_tensor(src_dst_pairs)).to(torch.int64).reshape(-1, 2).contiguous()
    snb, hkv, bs, d = src_k.shape
    dnb = dst_k.shape[0]
    rc = lib.orc_swap_blocks(src_k.data_ptr(), src_v.data_ptr(), dst_k.data_ptr(), dst_v.data_ptr(), pr.data_ptr(),
                             pr.shape[0], snb, dnb, hkv, d, bs, src_k.element_size())
    if rc < 0:
        raise ValueError(f"oracle swap_blocks refused the input (code {rc})")
    return int(rc)
