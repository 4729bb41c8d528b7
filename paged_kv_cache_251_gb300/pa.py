"""Thin ctypes binding of libpa (include/pa.h): argument marshalling only.

Every function takes CUDA torch tensors, passes their device pointers and the
current torch stream to the C ABI, and raises ``PagedAttentionError`` on a
non-OK status.  There is no CPU path: the library must be built
(``paged_kv_cache_251_gb300.build``) and the tensors must live on a GPU.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path

import torch

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libpa.so"

PA_OK, PA_ERR_INVALID_ARGUMENT, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE_TOO_SMALL, PA_ERR_CUDA = range(5)
PA_F32, PA_F16, PA_BF16, PA_I8, PA_E4M3 = 0, 1, 2, 3, 4
DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT, DEVERR_BAD_PAIR, DEVERR_TIMEOUT, DEVERR_BAD_LEN, DEVERR_BAD_LAUNCH = 1, 2, 4, 8, 16, 32

DTYPE_CODE = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}
# 8-bit caches: code pools are int8 or float8_e4m3fn tensors, scales float32
CODE_DTYPE = {torch.int8: PA_I8, torch.float8_e4m3fn: PA_E4M3}


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{_lib.pa_status_string(status).decode()}: {detail}")
        self.status = status


def _load():
    if not LIB_PATH.exists():
        raise ImportError(f"libpa.so is not built ({LIB_PATH}); run paged_kv_cache_251_gb300.build.build()")
    lib = ctypes.CDLL(str(LIB_PATH))
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.pa_decode_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.pa_decode_workspace_size.restype = SZ
    lib.pa_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, I, I, I, I, P, SZ, P, P]
    lib.pa_decode.restype = I
    lib.pa_decode_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, I, I, I, I, P, P]
    lib.pa_decode_noalloc.restype = I
    lib.pa_decode_contiguous.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, I, I, P, SZ, P, P]
    lib.pa_decode_contiguous.restype = I
    lib.pa_decode_noalloc_max_scratch.argtypes = []
    lib.pa_decode_noalloc_max_scratch.restype = SZ
    lib.pa_append_kv.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.pa_append_kv.restype = I
    lib.pa_copy_blocks.argtypes = [P, I, P, P, I, I, I, I, I, P, P]
    lib.pa_copy_blocks.restype = I
    lib.pa_decode_shared_prefix.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, I, I, P, SZ, P, P]
    lib.pa_decode_shared_prefix.restype = I
    lib.pa_decode_shared_prefix_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.pa_decode_shared_prefix_workspace_size.restype = SZ
    lib.pa_swap_blocks.argtypes = [P, I, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.pa_swap_blocks.restype = I
    lib.pa_quant_page_bytes.argtypes = [I, I]
    lib.pa_quant_page_bytes.restype = SZ
    lib.pa_append_kv_quant.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, P]
    lib.pa_append_kv_quant.restype = I
    lib.pa_decode_quant.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, I, I, I, I, I, I, I, P, SZ, P, P]
    lib.pa_decode_quant.restype = I
    lib.pa_copy_blocks_quant.argtypes = [P, I, P, P, I, I, I, I, P, P]
    lib.pa_copy_blocks_quant.restype = I
    lib.pa_swap_blocks_quant.argtypes = [P, I, P, P, P, P, I, I, I, I, I, P, P]
    lib.pa_swap_blocks_quant.restype = I
    lib.pa_status_string.argtypes = [I]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_last_error_detail.argtypes = []
    lib.pa_last_error_detail.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    lib.pa_version.restype = I
    return lib


_lib = _load()


def _check(status: int) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, _lib.pa_last_error_detail().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("every tensor must be a contiguous CUDA tensor")


def pa_decode_workspace_size(num_seqs: int, num_heads: int, head_dim: int, block_size: int,
                             max_blocks_per_seq: int, window: int = 0, partition_size: int = 0) -> int:
    return int(_lib.pa_decode_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                             max_blocks_per_seq, window, partition_size))


def workspace_for(q: torch.Tensor, block_size: int, max_blocks_per_seq: int, window: int = 0,
                  partition_size: int = 0) -> torch.Tensor | None:
    """A workspace tensor sized by pa_decode_workspace_size (None if 0 bytes)."""
    N, H, d = q.shape
    n = pa_decode_workspace_size(N, H, d, block_size, max_blocks_per_seq, window, partition_size)
    if n == 0:
        return None
    return torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device=q.device)


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int | None = None,
              scale: float | None = None, window: int = 0, partition_size: int = 0,
              workspace: torch.Tensor | None = None, err_word: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """out[s, h] = softmax(scale * q[s, h] . K_s^T) V_s over sequence s's cached
    tokens, read through block_tables[s] (see include/pa.h)."""
    _cuda(out, q, k_cache, v_cache, block_tables, context_lens, workspace, err_word)
    N, H, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if num_kv_heads is None:
        num_kv_heads = hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    if workspace is None:
        workspace = workspace_for(q, bs, block_tables.shape[1], window, partition_size)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                          _ptr(context_lens), N, H, num_kv_heads, d, bs, float(scale), int(window),
                          DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype], block_tables.shape[1], nb,
                          int(partition_size), _ptr(workspace), ws_bytes, _ptr(err_word), _stream(stream)))
    return out


def pa_decode_shared_prefix_workspace_size(num_seqs: int, num_heads: int, head_dim: int, block_size: int,
                                           max_blocks_per_seq: int, partition_size: int, group_size: int,
                                           dtype: torch.dtype) -> int:
    return int(_lib.pa_decode_shared_prefix_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                                           max_blocks_per_seq, partition_size, group_size,
                                                           DTYPE_CODE[dtype]))


def pa_decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, context_lens: torch.Tensor, shared_lens: torch.Tensor,
                            group_size: int, num_kv_heads: int | None = None, scale: float | None = None,
                            partition_size: int = 0, workspace: torch.Tensor | None = None,
                            err_word: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_decode for consecutive groups of group_size sequences whose first
    shared_lens[g] tokens are the same blocks: each shared block is read once
    per group (see include/pa.h)."""
    _cuda(out, q, k_cache, v_cache, block_tables, context_lens, shared_lens, workspace, err_word)
    N, H, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if num_kv_heads is None:
        num_kv_heads = hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (block_tables, context_lens, shared_lens):
        if t.dtype != torch.int32:
            raise TypeError("block_tables, context_lens and shared_lens must be int32")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    if workspace is None:
        n = pa_decode_shared_prefix_workspace_size(N, H, d, bs, block_tables.shape[1], partition_size, group_size,
                                                   q.dtype)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    _check(_lib.pa_decode_shared_prefix(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                        _ptr(context_lens), _ptr(shared_lens), int(group_size), N, H, num_kv_heads,
                                        d, bs, float(scale), DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype],
                                        block_tables.shape[1], nb, int(partition_size), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _ptr(err_word),
                                        _stream(stream)))
    return out


def pa_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int | None = None,
                      scale: float | None = None, window: int = 0, partition_size: int = 0,
                      err_word: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_decode for callers that cannot allocate device memory: the partials'
    scratch is the library's built-in array (pa_decode_noalloc_max_scratch()
    bytes), shared by all calls on a device, so calls must not overlap on the
    GPU.  This wrapper allocates nothing either."""
    _cuda(out, q, k_cache, v_cache, block_tables, context_lens, err_word)
    N, H, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if num_kv_heads is None:
        num_kv_heads = hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    _check(_lib.pa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                  _ptr(context_lens), N, H, num_kv_heads, d, bs, float(scale), int(window),
                                  DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype], block_tables.shape[1], nb,
                                  int(partition_size), _ptr(err_word), _stream(stream)))
    return out


def pa_decode_contiguous(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         context_lens: torch.Tensor, num_kv_heads: int | None = None, scale: float | None = None,
                         window: int = 0, partition_size: int = 0, workspace: torch.Tensor | None = None,
                         err_word: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_decode over contiguous caches [N, H_kv, L, d] (no block table; see
    include/pa.h)."""
    _cuda(out, q, k_cache, v_cache, context_lens, workspace, err_word)
    N, H, d = q.shape
    n2, hkv, L, d2 = k_cache.shape
    if num_kv_heads is None:
        num_kv_heads = hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if context_lens.dtype != torch.int32:
        raise TypeError("context_lens must be int32")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("q, k_cache and v_cache must share one dtype")
    if workspace is None:
        n = pa_decode_workspace_size(N, H, d, 16, max(1, L // 16), window, partition_size)
        workspace = None if n == 0 else torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_contiguous(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(context_lens), N, H,
                                     num_kv_heads, d, L, float(scale), int(window), DTYPE_CODE[q.dtype],
                                     DTYPE_CODE[out.dtype], int(partition_size), _ptr(workspace), ws_bytes,
                                     _ptr(err_word), _stream(stream)))
    return out


def pa_decode_noalloc_max_scratch() -> int:
    return int(_lib.pa_decode_noalloc_max_scratch())


def pa_append_kv(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, err_word: torch.Tensor | None = None, stream=None) -> None:
    """Store token i's K/V rows at slot_mapping[i] (see include/pa.h)."""
    _cuda(k, v, slot_mapping, k_cache, v_cache, err_word)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise TypeError("k, v and the caches must share one dtype")
    nb, hkv, bs, d = k_cache.shape
    _check(_lib.pa_append_kv(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                             slot_mapping.numel(), hkv, d, bs, nb, DTYPE_CODE[k_cache.dtype],
                             _ptr(err_word), _stream(stream)))


def pa_copy_blocks(src_dst_pairs: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   err_word: torch.Tensor | None = None, stream=None) -> None:
    """Copy block src onto block dst (K and V, all kv heads) for every pair."""
    _cuda(src_dst_pairs, k_cache, v_cache, err_word)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    nb, hkv, bs, d = k_cache.shape
    _check(_lib.pa_copy_blocks(_ptr(src_dst_pairs), src_dst_pairs.numel() // 2, _ptr(k_cache),
                               _ptr(v_cache), hkv, d, bs, nb, DTYPE_CODE[k_cache.dtype],
                               _ptr(err_word), _stream(stream)))


def pa_swap_blocks(src_dst_pairs: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                   dst_v: torch.Tensor, err_word: torch.Tensor | None = None, stream=None) -> None:
    """Copy block src of (src_k, src_v) onto block dst of (dst_k, dst_v) for
    every pair.  Pools and pairs may be CUDA tensors or pinned host tensors
    (the GPU reads / writes host memory directly)."""
    for t in (src_dst_pairs, src_k, src_v, dst_k, dst_v):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("pools and pairs must be contiguous CUDA tensors or pinned host tensors")
    if err_word is not None:
        _cuda(err_word)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    if src_k.dtype != dst_k.dtype or src_v.dtype != src_k.dtype or dst_v.dtype != src_k.dtype:
        raise TypeError("both pools must share one dtype")
    snb, hkv, bs, d = src_k.shape
    dnb, hkv2, bs2, d2 = dst_k.shape
    if (hkv, bs, d) != (hkv2, bs2, d2) or src_v.shape != src_k.shape or dst_v.shape != dst_k.shape:
        raise ValueError("both pools must share the block layout")
    _check(_lib.pa_swap_blocks(_ptr(src_dst_pairs), src_dst_pairs.numel() // 2, _ptr(src_k), _ptr(src_v),
                               _ptr(dst_k), _ptr(dst_v), snb, dnb, hkv, d, bs, DTYPE_CODE[src_k.dtype],
                               _ptr(err_word), _stream(stream)))


def pa_quant_page_bytes(head_dim: int, block_size: int) -> int:
    """Bytes of one (block, kv head) page of an 8-bit pool: block_size code rows
    of head_dim bytes, then the rows holding their fp32 scales."""
    return int(_lib.pa_quant_page_bytes(head_dim, block_size))


def quant_pool_shape(num_blocks: int, num_kv_heads: int, block_size: int, head_dim: int) -> tuple:
    """Shape of an 8-bit pool tensor: [num_blocks, H_kv, page rows, head_dim]."""
    return (num_blocks, num_kv_heads, pa_quant_page_bytes(head_dim, block_size) // head_dim, head_dim)


def _pool_block_size(pool: torch.Tensor) -> int:
    if pool.dtype not in CODE_DTYPE or pool.dim() != 4:
        raise TypeError("8-bit pools are int8 / float8_e4m3fn tensors [num_blocks, H_kv, page rows, head_dim]")
    rows, d = pool.shape[2], pool.shape[3]
    for bs in (8, 16, 32):
        if pa_quant_page_bytes(d, bs) == rows * d:
            return bs
    raise ValueError(f"a {rows}-row page at head_dim {d} matches no block size")


def pa_append_kv_quant(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, err_word: torch.Tensor | None = None, stream=None) -> None:
    """Quantise token i's K/V rows (fp32/fp16/bf16) into the 8-bit pages at
    slot_mapping[i]: codes into the slot's row, the row scale into the page's
    scale rows (see include/pa.h)."""
    _cuda(k, v, slot_mapping, k_cache, v_cache, err_word)
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    bs = _pool_block_size(k_cache)
    if k.dtype != v.dtype or k_cache.dtype != v_cache.dtype or k_cache.shape != v_cache.shape:
        raise TypeError("k and v share one dtype, the page pools another and one shape")
    nb, hkv, _, d = k_cache.shape
    _check(_lib.pa_append_kv_quant(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                   slot_mapping.numel(), hkv, d, bs, nb, DTYPE_CODE[k.dtype],
                                   CODE_DTYPE[k_cache.dtype], _ptr(err_word), _stream(stream)))


def pa_decode_quant(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                    block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int | None = None,
                    scale: float | None = None, window: int = 0, partition_size: int = 0,
                    workspace: torch.Tensor | None = None, err_word: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """pa_decode over 8-bit pages: every cached element is code * scale of its
    row (see include/pa.h)."""
    _cuda(out, q, k_cache, v_cache, block_tables, context_lens, workspace, err_word)
    N, H, d = q.shape
    bs = _pool_block_size(k_cache)
    nb, hkv, _, d2 = k_cache.shape
    if num_kv_heads is None:
        num_kv_heads = hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if v_cache.dtype != k_cache.dtype or v_cache.shape != k_cache.shape:
        raise TypeError("k_cache and v_cache must share one code dtype and shape")
    if workspace is None:
        workspace = workspace_for(q, bs, block_tables.shape[1], window, partition_size)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.pa_decode_quant(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                _ptr(context_lens), N, H, num_kv_heads, d, bs, float(scale), int(window),
                                DTYPE_CODE[q.dtype], CODE_DTYPE[k_cache.dtype], DTYPE_CODE[out.dtype],
                                block_tables.shape[1], nb, int(partition_size), _ptr(workspace), ws_bytes,
                                _ptr(err_word), _stream(stream)))
    return out


def pa_copy_blocks_quant(src_dst_pairs: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                         err_word: torch.Tensor | None = None, stream=None) -> None:
    """pa_copy_blocks for 8-bit pools: whole pages (codes and scales)."""
    _cuda(src_dst_pairs, k_cache, v_cache, err_word)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    bs = _pool_block_size(k_cache)
    nb, hkv, _, d = k_cache.shape
    _check(_lib.pa_copy_blocks_quant(_ptr(src_dst_pairs), src_dst_pairs.numel() // 2, _ptr(k_cache),
                                     _ptr(v_cache), hkv, d, bs, nb, _ptr(err_word), _stream(stream)))


def pa_swap_blocks_quant(src_dst_pairs: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                         dst_v: torch.Tensor, err_word: torch.Tensor | None = None, stream=None) -> None:
    """pa_swap_blocks for 8-bit pools: whole pages (CUDA or pinned host tensors)."""
    for t in (src_dst_pairs, src_k, src_v, dst_k, dst_v):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("pools and pairs must be contiguous CUDA tensors or pinned host tensors")
    if err_word is not None:
        _cuda(err_word)
    if src_dst_pairs.dtype != torch.int64:
        raise TypeError("src_dst_pairs must be int64")
    bs = _pool_block_size(src_k)
    snb, hkv, rows, d = src_k.shape
    dnb, hkv2, rows2, d2 = dst_k.shape
    if (hkv, rows, d) != (hkv2, rows2, d2) or src_k.dtype != dst_k.dtype:
        raise ValueError("both pools must share the page layout and code dtype")
    _check(_lib.pa_swap_blocks_quant(_ptr(src_dst_pairs), src_dst_pairs.numel() // 2, _ptr(src_k), _ptr(src_v),
                                     _ptr(dst_k), _ptr(dst_v), snb, dnb, hkv, d, bs, _ptr(err_word),
                                     _stream(stream)))


def version() -> tuple[int, int, int]:
    v = _lib.pa_version()
    return (v >> 16) & 0xFF, (v >> 8) & 0xFF, v & 0xFF
