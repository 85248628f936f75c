"""Thin Python binding of libkvq (ctypes).

Argument marshalling only: torch tensors supply device pointers, sizes and
strides, and ``torch.cuda.current_stream()`` supplies the stream; every step
of the computation runs in the CUDA kernels behind ``include/kvq.h``.  If
``libkvq.so`` is missing or cannot be loaded the calls raise -- there is no
fallback path.

The operations keep the argument order of the pages' ops where there is
one:

* ``kvq_store_nvfp4(key, value, key_cache, value_cache, slot_mapping,
  k_scale, v_scale)`` -- vLLM ``reshape_and_cache_nvfp4_dispatch``
  (nvfp4_kv_cache_kernels.cu, commit 7ce4c8e): ``key_cache`` /
  ``value_cache`` are ``kv_cache[:, 0]`` / ``kv_cache[:, 1]`` in the logical
  order [num_blocks, block_size, num_heads, head_size/2 + head_size/16],
  their strides telling HND from NHD.
* ``kvq_gather_indexer_k(kv_cache, k_fp8, k_scale, block_table,
  cu_seq_lens)`` -- vLLM ``cp_gather_indexer_k_quant_cache`` (PR #25931,
  PR #26456).
* ``kvq_load_nvfp4(key_cache, value_cache, block_table, cu_seq_lens,
  k_scale, v_scale, key_out, value_out)`` -- the read side of the store.
* ``kvq_store_indexer_k(k, kv_cache, slot_mapping)`` -- the write side of
  the indexer cache the gather reads.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_NULL = -1
KVQ_ERR_SHAPE = -2
KVQ_ERR_ALIGN = -3
KVQ_ERR_DTYPE = -4
KVQ_ERR_LAYOUT = -5
KVQ_ERR_CUDA = -6
KVQ_ERR_ARG = -7
KVQ_ERR_SCRATCH = -8
KVQ_NOALLOC_SCRATCH_BYTES = 32 << 20

KVQ_LAYOUT_HND = 0
KVQ_LAYOUT_NHD = 1
KVQ_DTYPE_BF16 = 0
KVQ_DTYPE_FP16 = 1
KVQ_F_SWIZZLE_K_SCALE = 1
KVQ_F_PDL = 2
KVQ_F_PDL_EARLY_META = 4
KVQ_F_PDL_EARLY_READ = 1 << 4
KVQ_DEVERR_SLOT = 1
KVQ_DEVERR_BLOCK = 2
KVQ_DEVERR_SEQ = 4
KVQ_DEVERR_TIMEOUT = 8

_lock = threading.Lock()
_lib = None


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {kvq_status_string(status)} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libkvq.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m paged_quantized_kv_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        c = ctypes
        P = c.c_void_p
        L.kvq_store_nvfp4.argtypes = [
            P, c.c_int64, P, c.c_int64, c.c_int32, c.c_int32, c.c_int32,
            c.c_int32, P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, P,
            P, P, c.c_uint32, P, P]
        L.kvq_store_nvfp4.restype = c.c_int
        L.kvq_gather_indexer_k.argtypes = [
            P, c.c_int64, c.c_int64, c.c_int32, c.c_int32, P, c.c_int64,
            c.c_int32, P, c.c_int32, c.c_int64, P, P, c.c_uint32, P, P]
        L.kvq_gather_indexer_k.restype = c.c_int
        L.kvq_load_nvfp4.argtypes = [
            P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, c.c_int32,
            c.c_int32, P, c.c_int64, c.c_int32, P, c.c_int32, c.c_int64, P,
            P, c.c_int32, P, P, c.c_int64, c.c_uint32, P, P]
        L.kvq_load_nvfp4.restype = c.c_int
        L.kvq_store_indexer_k.argtypes = [
            P, c.c_int64, c.c_int32, c.c_int32, c.c_int32, P, c.c_int64,
            c.c_int32, c.c_int64, P, c.c_uint32, P, P]
        L.kvq_store_indexer_k.restype = c.c_int
        L.kvq_paged_attention_nvfp4.argtypes = [
            P, c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
            c.c_int32, P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, P,
            c.c_int64, c.c_int32, P, c.c_int32, P, P, c.c_float, c.c_int32,
            P, P, P, P, c.c_int64, c.c_uint32, P, P]
        L.kvq_paged_attention_nvfp4.restype = c.c_int
        L.kvq_paged_attention_nvfp4_noalloc.argtypes = [
            P, c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
            c.c_int32, P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, P,
            c.c_int64, c.c_int32, P, c.c_int32, P, P, c.c_float, c.c_int32,
            P, c.c_int64, c.c_uint32, P, P]
        L.kvq_paged_attention_nvfp4_noalloc.restype = c.c_int
        L.kvq_status_string.argtypes = [c.c_int]
        L.kvq_status_string.restype = c.c_char_p
        L.kvq_version.argtypes = []
        L.kvq_version.restype = c.c_int32
        _lib = L
        return L


def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(int(status)).decode()


def kvq_version() -> int:
    return int(lib().kvq_version())


def _stream_of(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check(fn: str, status: int) -> None:
    if status != KVQ_OK:
        raise KvqError(fn, status)


def kvq_store_nvfp4(key: torch.Tensor, value: torch.Tensor,
                    key_cache: torch.Tensor, value_cache: torch.Tensor,
                    slot_mapping: torch.Tensor, k_scale: torch.Tensor,
                    v_scale: torch.Tensor, flags: int = 0,
                    dev_error: torch.Tensor | None = None,
                    stream: int | None = None) -> None:
    """NVFP4 paged store (see ``include/kvq.h``).

    key, value: bf16 or fp16 [T, H, D], last two dims contiguous.  key_cache,
    value_cache: uint8 [num_blocks, block_size, H, D/2 + D/16] views whose
    stride(0) is the page stride and whose stride(2) > stride(1) marks HND.
    slot_mapping: int64 [T].  k_scale, v_scale: fp32 device scalars."""
    dtypes = {torch.bfloat16: KVQ_DTYPE_BF16, torch.float16: KVQ_DTYPE_FP16}
    if key.dtype not in dtypes or value.dtype != key.dtype:
        raise KvqError("kvq_store_nvfp4", KVQ_ERR_DTYPE)
    T, H, D = key.shape
    if (key.stride(2) != 1 or key.stride(1) != D or value.stride(2) != 1
            or value.stride(1) != D or tuple(value.shape) != (T, H, D)):
        raise KvqError("kvq_store_nvfp4", KVQ_ERR_SHAPE)
    if key_cache.dim() != 4 or key_cache.dtype != torch.uint8:
        raise KvqError("kvq_store_nvfp4", KVQ_ERR_SHAPE)
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() < T:
        raise KvqError("kvq_store_nvfp4", KVQ_ERR_SHAPE)
    layout = (KVQ_LAYOUT_HND if key_cache.stride(2) > key_cache.stride(1)
              else KVQ_LAYOUT_NHD)
    st = lib().kvq_store_nvfp4(
        key.data_ptr(), key.stride(0), value.data_ptr(), value.stride(0),
        dtypes[key.dtype], T, H, D, key_cache.data_ptr(),
        value_cache.data_ptr(), key_cache.stride(0), key_cache.size(1),
        key_cache.size(0), layout, slot_mapping.data_ptr(),
        k_scale.data_ptr(), v_scale.data_ptr(), int(flags),
        _ptr(dev_error), _stream_of(key) if stream is None else stream)
    _check("kvq_store_nvfp4", st)


def kvq_gather_indexer_k(kv_cache: torch.Tensor, k_fp8: torch.Tensor,
                         k_scale: torch.Tensor, block_table: torch.Tensor,
                         cu_seq_lens: torch.Tensor, block_size: int | None = None,
                         flags: int = 0,
                         dev_error: torch.Tensor | None = None,
                         stream: int | None = None) -> None:
    """Indexer-K gather (see ``include/kvq.h``).

    kv_cache: uint8 [num_blocks, block_size, head_dim + 4] (or
    [num_blocks, bytes] with ``block_size`` given); each block holds
    [block_size*head_dim K bytes | block_size*4 scale bytes].
    k_fp8: [total, head_dim] 1-byte elements; k_scale: [total, 4] uint8 (or
    [total] float32).  block_table int32 [num_seqs, max_blocks];
    cu_seq_lens int32 [num_seqs + 1]; total = k_fp8.size(0)."""
    if kv_cache.element_size() != 1 or k_fp8.element_size() != 1:
        raise KvqError("kvq_gather_indexer_k", KVQ_ERR_DTYPE)
    if block_table.dtype != torch.int32 or cu_seq_lens.dtype != torch.int32:
        raise KvqError("kvq_gather_indexer_k", KVQ_ERR_DTYPE)
    total, head_dim = k_fp8.shape
    if block_size is None:
        if kv_cache.dim() != 3:
            raise KvqError("kvq_gather_indexer_k", KVQ_ERR_SHAPE)
        block_size = kv_cache.size(1)
    if (k_fp8.stride(0) != head_dim or k_fp8.stride(1) != 1
            or k_scale.numel() * k_scale.element_size() < 4 * total
            or not k_scale.is_contiguous() or block_table.stride(1) != 1):
        raise KvqError("kvq_gather_indexer_k", KVQ_ERR_SHAPE)
    st = lib().kvq_gather_indexer_k(
        kv_cache.data_ptr(), kv_cache.stride(0), kv_cache.size(0),
        int(block_size), int(head_dim), block_table.data_ptr(),
        block_table.stride(0), block_table.size(1), cu_seq_lens.data_ptr(),
        cu_seq_lens.numel() - 1, int(total), k_fp8.data_ptr(),
        k_scale.data_ptr(), int(flags), _ptr(dev_error),
        _stream_of(kv_cache) if stream is None else stream)
    _check("kvq_gather_indexer_k", st)


def kvq_load_nvfp4(key_cache: torch.Tensor, value_cache: torch.Tensor,
                   block_table: torch.Tensor, cu_seq_lens: torch.Tensor,
                   k_scale: torch.Tensor, v_scale: torch.Tensor,
                   key_out: torch.Tensor, value_out: torch.Tensor,
                   flags: int = 0, dev_error: torch.Tensor | None = None,
                   stream: int | None = None) -> None:
    """NVFP4 paged load (see ``include/kvq.h``): the tokens the block table
    names, dequantised into key_out / value_out (bf16 [total, H, D], last two
    dims contiguous; total = key_out.size(0)).  key_cache / value_cache are
    the store's 4-D page views."""
    if key_out.dtype != torch.bfloat16 or value_out.dtype != torch.bfloat16:
        raise KvqError("kvq_load_nvfp4", KVQ_ERR_DTYPE)
    T, H, D = key_out.shape
    if (key_out.stride(2) != 1 or key_out.stride(1) != D
            or tuple(value_out.shape) != (T, H, D)
            or value_out.stride(0) != key_out.stride(0)
            or value_out.stride(2) != 1 or value_out.stride(1) != D):
        raise KvqError("kvq_load_nvfp4", KVQ_ERR_SHAPE)
    if key_cache.dim() != 4 or key_cache.dtype != torch.uint8:
        raise KvqError("kvq_load_nvfp4", KVQ_ERR_SHAPE)
    if block_table.dtype != torch.int32 or cu_seq_lens.dtype != torch.int32:
        raise KvqError("kvq_load_nvfp4", KVQ_ERR_DTYPE)
    layout = (KVQ_LAYOUT_HND if key_cache.stride(2) > key_cache.stride(1)
              else KVQ_LAYOUT_NHD)
    st = lib().kvq_load_nvfp4(
        key_cache.data_ptr(), value_cache.data_ptr(), key_cache.stride(0),
        key_cache.size(1), key_cache.size(0), layout, H, D,
        block_table.data_ptr(), block_table.stride(0), block_table.size(1),
        cu_seq_lens.data_ptr(), cu_seq_lens.numel() - 1, T,
        k_scale.data_ptr(), v_scale.data_ptr(), KVQ_DTYPE_BF16,
        key_out.data_ptr(), value_out.data_ptr(), key_out.stride(0),
        int(flags), _ptr(dev_error),
        _stream_of(key_out) if stream is None else stream)
    _check("kvq_load_nvfp4", st)


def kvq_store_indexer_k(k: torch.Tensor, kv_cache: torch.Tensor,
                        slot_mapping: torch.Tensor,
                        block_size: int | None = None, flags: int = 0,
                        dev_error: torch.Tensor | None = None,
                        stream: int | None = None) -> None:
    """Indexer-K store (see ``include/kvq.h``): k bf16/fp16 [T, head_dim]
    (last dim contiguous) into kv_cache uint8 [num_blocks, block_size,
    head_dim + 4] (or [num_blocks, bytes] with ``block_size`` given)."""
    dtypes = {torch.bfloat16: KVQ_DTYPE_BF16, torch.float16: KVQ_DTYPE_FP16}
    if k.dtype not in dtypes or kv_cache.element_size() != 1:
        raise KvqError("kvq_store_indexer_k", KVQ_ERR_DTYPE)
    T, D = k.shape
    if block_size is None:
        if kv_cache.dim() != 3:
            raise KvqError("kvq_store_indexer_k", KVQ_ERR_SHAPE)
        block_size = kv_cache.size(1)
    if (k.stride(1) != 1 or slot_mapping.dtype != torch.int64
            or slot_mapping.numel() < T):
        raise KvqError("kvq_store_indexer_k", KVQ_ERR_SHAPE)
    st = lib().kvq_store_indexer_k(
        k.data_ptr(), k.stride(0), dtypes[k.dtype], T, D,
        kv_cache.data_ptr(), kv_cache.stride(0), int(block_size),
        kv_cache.size(0), slot_mapping.data_ptr(), int(flags),
        _ptr(dev_error), _stream_of(k) if stream is None else stream)
    _check("kvq_store_indexer_k", st)


def attention_scratch(num_seqs: int, num_q_heads: int, max_context_len: int,
                      partition_size: int = 512, head_size: int = 128,
                      device="cuda"):
    """(exp_sums, max_logits, tmp_out) fp32 scratch for
    kvq_paged_attention_nvfp4, or (None, None, None) when every context fits
    one partition."""
    parts = -(-int(max_context_len) // int(partition_size))
    if parts <= 1:
        return None, None, None
    shape = (num_seqs, num_q_heads, parts)
    return (torch.empty(shape, dtype=torch.float32, device=device),
            torch.empty(shape, dtype=torch.float32, device=device),
            torch.empty(shape + (head_size,), dtype=torch.float32,
                        device=device))


def kvq_paged_attention_nvfp4(query: torch.Tensor, key_cache: torch.Tensor,
                              value_cache: torch.Tensor,
                              block_table: torch.Tensor,
                              context_lens: torch.Tensor,
                              k_scale: torch.Tensor, v_scale: torch.Tensor,
                              scale: float, out: torch.Tensor,
                              max_context_len: int,
                              partition_size: int = 512,
                              exp_sums: torch.Tensor | None = None,
                              max_logits: torch.Tensor | None = None,
                              tmp_out: torch.Tensor | None = None,
                              flags: int = 0,
                              dev_error: torch.Tensor | None = None,
                              stream: int | None = None) -> None:
    """Paged decode attention over the NVFP4 cache (see ``include/kvq.h``).

    query / out: bf16 or fp16 [num_seqs, Hq, 128] (last two dims
    contiguous); key_cache / value_cache: the store's 4-D page views;
    block_table int32 [num_seqs, max_blocks]; context_lens int32
    [num_seqs].  The fp32 scratch (``attention_scratch``) is allocated here
    when it is needed and not given."""
    dtypes = {torch.bfloat16: KVQ_DTYPE_BF16, torch.float16: KVQ_DTYPE_FP16}
    if query.dtype not in dtypes or out.dtype != query.dtype:
        raise KvqError("kvq_paged_attention_nvfp4", KVQ_ERR_DTYPE)
    n, Hq, D = query.shape
    if (query.stride(2) != 1 or query.stride(1) != D or out.stride(2) != 1
            or out.stride(1) != D or tuple(out.shape) != (n, Hq, D)):
        raise KvqError("kvq_paged_attention_nvfp4", KVQ_ERR_SHAPE)
    if key_cache.dim() != 4 or key_cache.dtype != torch.uint8:
        raise KvqError("kvq_paged_attention_nvfp4", KVQ_ERR_SHAPE)
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise KvqError("kvq_paged_attention_nvfp4", KVQ_ERR_DTYPE)
    layout = (KVQ_LAYOUT_HND if key_cache.stride(2) > key_cache.stride(1)
              else KVQ_LAYOUT_NHD)
    if exp_sums is None and max_logits is None and tmp_out is None:
        exp_sums, max_logits, tmp_out = attention_scratch(
            n, Hq, max_context_len, partition_size, D, query.device)
    st = lib().kvq_paged_attention_nvfp4(
        query.data_ptr(), query.stride(0), dtypes[query.dtype], n, Hq,
        key_cache.size(2), D, key_cache.data_ptr(), value_cache.data_ptr(),
        key_cache.stride(0), key_cache.size(1), key_cache.size(0), layout,
        block_table.data_ptr(), block_table.stride(0), block_table.size(1),
        context_lens.data_ptr(), int(max_context_len), k_scale.data_ptr(),
        v_scale.data_ptr(), float(scale), int(partition_size),
        _ptr(exp_sums), _ptr(max_logits), _ptr(tmp_out), out.data_ptr(),
        out.stride(0), int(flags), _ptr(dev_error),
        _stream_of(query) if stream is None else stream)
    _check("kvq_paged_attention_nvfp4", st)


def kvq_paged_attention_nvfp4_noalloc(query: torch.Tensor,
                                      key_cache: torch.Tensor,
                                      value_cache: torch.Tensor,
                                      block_table: torch.Tensor,
                                      context_lens: torch.Tensor,
                                      k_scale: torch.Tensor,
                                      v_scale: torch.Tensor, scale: float,
                                      out: torch.Tensor, max_context_len: int,
                                      partition_size: int = 512,
                                      flags: int = 0,
                                      dev_error: torch.Tensor | None = None,
                                      stream: int | None = None) -> None:
    """kvq_paged_attention_nvfp4 for callers that cannot allocate device
    memory (see ``include/kvq.h``): the same arguments without the scratch
    tensors; the library's built-in scratch array is used instead, and
    nothing is allocated here either."""
    dtypes = {torch.bfloat16: KVQ_DTYPE_BF16, torch.float16: KVQ_DTYPE_FP16}
    if query.dtype not in dtypes or out.dtype != query.dtype:
        raise KvqError("kvq_paged_attention_nvfp4_noalloc", KVQ_ERR_DTYPE)
    n, Hq, D = query.shape
    if (query.stride(2) != 1 or query.stride(1) != D or out.stride(2) != 1
            or out.stride(1) != D or tuple(out.shape) != (n, Hq, D)):
        raise KvqError("kvq_paged_attention_nvfp4_noalloc", KVQ_ERR_SHAPE)
    if key_cache.dim() != 4 or key_cache.dtype != torch.uint8:
        raise KvqError("kvq_paged_attention_nvfp4_noalloc", KVQ_ERR_SHAPE)
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise KvqError("kvq_paged_attention_nvfp4_noalloc", KVQ_ERR_DTYPE)
    layout = (KVQ_LAYOUT_HND if key_cache.stride(2) > key_cache.stride(1)
              else KVQ_LAYOUT_NHD)
    st = lib().kvq_paged_attention_nvfp4_noalloc(
        query.data_ptr(), query.stride(0), dtypes[query.dtype], n, Hq,
        key_cache.size(2), D, key_cache.data_ptr(), value_cache.data_ptr(),
        key_cache.stride(0), key_cache.size(1), key_cache.size(0), layout,
        block_table.data_ptr(), block_table.stride(0), block_table.size(1),
        context_lens.data_ptr(), int(max_context_len), k_scale.data_ptr(),
        v_scale.data_ptr(), float(scale), int(partition_size),
        out.data_ptr(), out.stride(0), int(flags), _ptr(dev_error),
        _stream_of(query) if stream is None else stream)
    _check("kvq_paged_attention_nvfp4_noalloc", st)


def alloc_nvfp4_cache(num_blocks: int, block_size: int, num_heads: int,
                      head_size: int, layout: int = KVQ_LAYOUT_HND,
                      device="cuda", fill: int | None = None):
    """Allocate an NVFP4 paged cache and return (kv_cache, key_cache,
    value_cache): kv_cache is the raw [num_blocks, 2, ...] uint8 tensor and
    key_cache / value_cache its two sides in the logical
    [num_blocks, block_size, num_heads, D/2 + D/16] order."""
    full = head_size // 2 + head_size // 16
    if layout == KVQ_LAYOUT_HND:
        kv = torch.empty(num_blocks, 2, num_heads, block_size, full,
                         dtype=torch.uint8, device=device)
        k, v = kv[:, 0].permute(0, 2, 1, 3), kv[:, 1].permute(0, 2, 1, 3)
    else:
        kv = torch.empty(num_blocks, 2, block_size, num_heads, full,
                         dtype=torch.uint8, device=device)
        k, v = kv[:, 0], kv[:, 1]
    if fill is not None:
        kv.fill_(fill)
    return kv, k, v
