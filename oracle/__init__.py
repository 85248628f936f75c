"""CPU oracle for the paged quantized KV-cache path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The library in
``paged_quantized_kv_gb300/`` shares no code with it and never calls it.

The arithmetic lives in ``kvq_oracle.c`` (plain C, fp32 IEEE operations, no
FMA contraction, table-search encoders); this module only compiles it with
gcc and marshals numpy arrays through ctypes.  The C file cites the page
passage each function restates:

* vLLM ``csrc/libtorch_stable/nvfp4_kv_cache_kernels.cu`` (commit 7ce4c8e):
  ``swizzle_scale_offset``, ``reshape_and_cache_nvfp4_kernel``,
  ``reshape_and_cache_nvfp4_dispatch``.
* vLLM PR #25931 "Add gather_indexer_k_quant_cache kernel" and PR #26456
  "[Deepseek-V3.2][Kernel] Integrate cuda indexer k cache gather".
* The NVFP4 paged load (the read side of the store) follows the same page
  layout and swizzle; its dequantisation rule is the plain inverse of the
  store's (the pages state none).
* The indexer-K store (the write side of the gathered cache) uses a
  per-token absmax rule (the pages state none): scale = amax / 448,
  q = e4m3_rn_satfinite(k / scale).
* Paged decode attention over the NVFP4 cache (vLLM PR #12348 "[ROCm]
  Faster Custom Paged Attention kernels" shows the op's signature only):
  plain softmax attention in double over the exactly dequantised cache.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(format tables against closed forms and torch's float8 cast, hand-worked
groups under ``tests/golden/``, the swizzle against the page's permute
statement, the dequantisation error bound, an independent numpy re-assembly
of the page layout, brute-force gather tracing), and
``tests/test_oracle_mutants.py`` shows those pins fail on planted mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "libkvq_oracle.so")

LAYOUT_HND = 0
LAYOUT_NHD = 1
DTYPE_BF16 = 0
DTYPE_F16 = 1
F_SWIZZLE_K_SCALE = 1

OK = 0
ERR_ARG = -1
ERR_NONFINITE = -2
ERR_BOUNDS = -3

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-Wall", "-Wextra"]


def compile_oracle(src: str, out: str) -> str:
    """gcc ``src`` into the shared object ``out`` (atomic replace)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``kvq_oracle.c`` into ``libkvq_oracle.so`` if stale."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE)):
        return _LIB
    return compile_oracle(SOURCE, _LIB)


def _ptr(a: np.ndarray, offset_bytes: int = 0) -> int:
    return a.ctypes.data + offset_bytes


class Oracle:
    """ctypes view of one compiled oracle shared object."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        c = ctypes
        P = c.c_void_p
        lib.kvqo_e4m3_decode.argtypes = [c.c_uint8]
        lib.kvqo_e4m3_decode.restype = c.c_double
        lib.kvqo_e2m1_decode.argtypes = [c.c_uint8]
        lib.kvqo_e2m1_decode.restype = c.c_double
        lib.kvqo_e4m3_encode.argtypes = [c.c_float]
        lib.kvqo_e4m3_encode.restype = c.c_uint8
        lib.kvqo_e2m1_encode.argtypes = [c.c_float]
        lib.kvqo_e2m1_encode.restype = c.c_uint8
        lib.kvqo_swizzle.argtypes = [c.c_int, c.c_int, c.c_int]
        lib.kvqo_swizzle.restype = c.c_int
        lib.kvqo_quantize_group.argtypes = [P, c.c_float, P, P]
        lib.kvqo_quantize_group.restype = c.c_int
        lib.kvqo_quantize_group_t.argtypes = [P, c.c_int, c.c_float, P, P]
        lib.kvqo_quantize_group_t.restype = c.c_int
        lib.kvqo_f16_decode.argtypes = [c.c_uint16]
        lib.kvqo_f16_decode.restype = c.c_double
        lib.kvqo_store_nvfp4.argtypes = [
            P, c.c_int64, P, c.c_int64, c.c_int32, c.c_int32, c.c_int32,
            c.c_int32, P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, P,
            c.c_float, c.c_float, c.c_uint32]
        lib.kvqo_store_nvfp4.restype = c.c_int
        lib.kvqo_gather_indexer_k.argtypes = [
            P, c.c_int64, c.c_int64, c.c_int32, c.c_int32, P, c.c_int64,
            c.c_int32, P, c.c_int32, c.c_int64, P, P]
        lib.kvqo_gather_indexer_k.restype = c.c_int
        lib.kvqo_float_to_bf16.argtypes = [c.c_float]
        lib.kvqo_float_to_bf16.restype = c.c_uint16
        lib.kvqo_load_nvfp4.argtypes = [
            P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, c.c_int32,
            c.c_int32, P, c.c_int64, c.c_int32, P, c.c_int32, c.c_int64,
            c.c_float, c.c_float, c.c_uint32, P, P, c.c_int64]
        lib.kvqo_load_nvfp4.restype = c.c_int
        lib.kvqo_store_indexer_k.argtypes = [
            P, c.c_int64, c.c_int32, c.c_int32, c.c_int32, P, c.c_int64,
            c.c_int32, c.c_int64, P]
        lib.kvqo_store_indexer_k.restype = c.c_int
        lib.kvqo_paged_attention_nvfp4.argtypes = [
            P, c.c_int64, c.c_int32, c.c_int32, c.c_int32, c.c_int32,
            c.c_int32, P, P, c.c_int64, c.c_int32, c.c_int64, c.c_int32, P,
            c.c_int64, c.c_int32, P, c.c_float, c.c_float, c.c_float,
            c.c_uint32, P, P]
        lib.kvqo_paged_attention_nvfp4.restype = c.c_int
        self.lib = lib
        self.path = lib_path

    # --- format tables ------------------------------------------------------
    def e4m3_decode(self, code: int) -> float:
        """Value of an e4m3 (fn) code; NaN for 0x7F / 0xFF."""
        return self.lib.kvqo_e4m3_decode(int(code) & 0xFF)

    def e2m1_decode(self, nibble: int) -> float:
        """Value of an e2m1 code (sign in bit 3)."""
        return self.lib.kvqo_e2m1_decode(int(nibble) & 0xF)

    def e4m3_encode(self, v: float) -> int:
        """fp32 -> e4m3, round to nearest even, saturate at 448."""
        return self.lib.kvqo_e4m3_encode(float(np.float32(v)))

    def e2m1_encode(self, v: float) -> int:
        """fp32 -> e2m1, round to nearest even, saturate at 6."""
        return self.lib.kvqo_e2m1_encode(float(np.float32(v)))

    def swizzle(self, t: int, s: int, S: int) -> int:
        """Swizzled offset of (token-in-page t, scale s) in a [B, S] tile."""
        return self.lib.kvqo_swizzle(int(t), int(s), int(S))

    def f16_decode(self, bits: int) -> float:
        """Value of an IEEE binary16 bit pattern."""
        return self.lib.kvqo_f16_decode(int(bits) & 0xFFFF)

    def quantize_group(self, x_bits: np.ndarray, g: float,
                       dtype: int = DTYPE_BF16):
        """Quantise 16 bf16 (or fp16) values, given as uint16 bit patterns,
        with global scale g.

        Returns (data: uint8[8], sf: int).  Raises on non-finite input."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        assert x.shape == (16,)
        data = np.zeros(8, dtype=np.uint8)
        sf = np.zeros(1, dtype=np.uint8)
        rc = self.lib.kvqo_quantize_group_t(_ptr(x), int(dtype),
                                            float(np.float32(g)),
                                            _ptr(data), _ptr(sf))
        if rc != OK:
            raise ValueError(f"kvqo_quantize_group failed: {rc}")
        return data, int(sf[0])

    def float_to_bf16(self, v: float) -> int:
        """fp32 -> bf16 bits, round to nearest even."""
        return int(self.lib.kvqo_float_to_bf16(float(np.float32(v))))

    # --- the operations -----------------------------------------------------
    def store_nvfp4(self, key_bits: np.ndarray, key_stride0: int,
                    value_bits: np.ndarray, value_stride0: int,
                    num_tokens: int, num_heads: int, head_size: int,
                    kv_cache: np.ndarray, key_offset: int, value_offset: int,
                    page_stride: int, block_size: int, num_blocks: int,
                    layout: int, slot_mapping: np.ndarray,
                    k_scale: float, v_scale: float, flags: int = 0,
                    key_base: int = 0, value_base: int = 0,
                    dtype: int = DTYPE_BF16) -> None:
        """NVFP4 paged store into ``kv_cache`` (uint8, modified in place).

        ``key_bits``/``value_bits`` are uint16 bf16 (or fp16, ``dtype``) bit
        patterns; key token
        t, head h, element d is ``key_bits[key_base + t*stride0 + h*D + d]``
        (value likewise).  ``key_offset``/``value_offset`` are the byte
        offsets of the K side and the V side of page 0 inside ``kv_cache``."""
        assert kv_cache.dtype == np.uint8 and kv_cache.flags.c_contiguous
        assert key_bits.dtype == np.uint16 and value_bits.dtype == np.uint16
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert slots.size >= num_tokens
        rc = self.lib.kvqo_store_nvfp4(
            _ptr(key_bits, 2 * key_base), int(key_stride0),
            _ptr(value_bits, 2 * value_base), int(value_stride0),
            int(dtype), int(num_tokens), int(num_heads), int(head_size), _ptr(kv_cache, key_offset),
            _ptr(kv_cache, value_offset), int(page_stride), int(block_size),
            int(num_blocks), int(layout), _ptr(slots),
            float(np.float32(k_scale)), float(np.float32(v_scale)),
            int(flags))
        if rc != OK:
            raise ValueError(f"kvqo_store_nvfp4 failed: {rc}")

    def gather_indexer_k(self, cache: np.ndarray, block_stride: int,
                         num_blocks: int, block_size: int, head_dim: int,
                         block_table: np.ndarray, cu_seq_lens: np.ndarray,
                         total_tokens: int, k_fp8: np.ndarray,
                         k_scale: np.ndarray) -> None:
        """Indexer-K gather into ``k_fp8`` [total, head_dim] and ``k_scale``
        [total*4] (uint8 arrays, modified in place)."""
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
        assert bt.ndim == 2
        assert k_fp8.dtype == np.uint8 and k_fp8.flags.c_contiguous
        assert k_scale.dtype == np.uint8 and k_scale.flags.c_contiguous
        assert k_fp8.size >= total_tokens * head_dim
        assert k_scale.size >= total_tokens * 4
        rc = self.lib.kvqo_gather_indexer_k(
            _ptr(cache), int(block_stride), int(num_blocks), int(block_size),
            int(head_dim), _ptr(bt), int(bt.shape[1]), int(bt.shape[1]),
            _ptr(cu), int(cu.size - 1), int(total_tokens), _ptr(k_fp8),
            _ptr(k_scale))
        if rc != OK:
            raise ValueError(f"kvqo_gather_indexer_k failed: {rc}")

    def store_indexer_k(self, k_bits: np.ndarray, k_stride0: int,
                        num_tokens: int, head_dim: int, cache: np.ndarray,
                        block_stride: int, block_size: int, num_blocks: int,
                        slot_mapping: np.ndarray, dtype: int = DTYPE_BF16,
                        k_base: int = 0) -> None:
        """Indexer-K store into ``cache`` (uint8, modified in place): token
        t (bits at ``k_base + t*k_stride0``) -> block slot / B, row slot % B
        of [B*D fp8 K | B*4 fp32 scale] blocks."""
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert cache.dtype == np.uint8 and cache.flags.c_contiguous
        rc = self.lib.kvqo_store_indexer_k(
            _ptr(k_bits, 2 * k_base), int(k_stride0), int(dtype),
            int(num_tokens), int(head_dim), _ptr(cache), int(block_stride),
            int(block_size), int(num_blocks), _ptr(slots))
        if rc != OK:
            raise ValueError(f"kvqo_store_indexer_k failed: {rc}")

    def load_nvfp4(self, kv_cache: np.ndarray, key_offset: int,
                   value_offset: int, page_stride: int, block_size: int,
                   num_blocks: int, layout: int, num_heads: int,
                   head_size: int, block_table: np.ndarray,
                   cu_seq_lens: np.ndarray, total_tokens: int,
                   k_scale: float, v_scale: float, flags: int = 0):
        """NVFP4 paged load: returns (key, value) bf16 bit arrays
        [total_tokens, H, D] (uint16), rows of sequences in cu_seq_lens order;
        rows no sequence covers stay 0."""
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cu = np.ascontiguousarray(cu_seq_lens, dtype=np.int32)
        H, D = num_heads, head_size
        k = np.zeros((max(total_tokens, 1), H, D), dtype=np.uint16)
        v = np.zeros((max(total_tokens, 1), H, D), dtype=np.uint16)
        rc = self.lib.kvqo_load_nvfp4(
            _ptr(kv_cache, key_offset), _ptr(kv_cache, value_offset),
            int(page_stride), int(block_size), int(num_blocks), int(layout),
            int(H), int(D), _ptr(bt), int(bt.shape[1]), int(bt.shape[1]),
            _ptr(cu), int(cu.size - 1), int(total_tokens),
            float(np.float32(k_scale)), float(np.float32(v_scale)), int(flags),
            _ptr(k), _ptr(v), H * D)
        if rc != OK:
            raise ValueError(f"kvqo_load_nvfp4 failed: {rc}")
        return k[:total_tokens], v[:total_tokens]

    def paged_attention_nvfp4(self, query_bits: np.ndarray, kv_cache: np.ndarray,
                              key_offset: int, value_offset: int,
                              page_stride: int, block_size: int,
                              num_blocks: int, layout: int, num_kv_heads: int,
                              block_table: np.ndarray,
                              context_lens: np.ndarray, k_scale: float,
                              v_scale: float, scale: float, flags: int = 0,
                              dtype: int = DTYPE_BF16):
        """Paged decode attention over the NVFP4 cache.

        ``query_bits``: uint16 bf16 (or fp16) bits [num_seqs, Hq, D].
        Returns (out, mag), float64 [num_seqs, Hq, D]: the exact attention
        output and sum_t p_t |V^[t, d]|."""
        q = np.ascontiguousarray(query_bits, dtype=np.uint16)
        assert q.ndim == 3
        n, Hq, D = q.shape
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        assert bt.ndim == 2 and bt.shape[0] >= n
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        assert lens.size >= n
        out = np.zeros((max(n, 1), Hq, D), dtype=np.float64)
        mag = np.zeros((max(n, 1), Hq, D), dtype=np.float64)
        rc = self.lib.kvqo_paged_attention_nvfp4(
            _ptr(q), Hq * D, int(dtype), int(n), int(Hq), int(num_kv_heads),
            int(D), _ptr(kv_cache, key_offset), _ptr(kv_cache, value_offset),
            int(page_stride), int(block_size), int(num_blocks), int(layout),
            _ptr(bt), int(bt.shape[1]), int(bt.shape[1]), _ptr(lens),
            float(np.float32(k_scale)), float(np.float32(v_scale)),
            float(np.float32(scale)), int(flags), _ptr(out), _ptr(mag))
        if rc != OK:
            raise ValueError(f"kvqo_paged_attention_nvfp4 failed: {rc}")
        return out[:n], mag[:n]


_default = None
_lock = threading.Lock()


def get() -> Oracle:
    """The oracle built from ``kvq_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default

