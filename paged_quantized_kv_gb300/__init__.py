"""GB300-native paged quantized KV-cache kernels.

Two memory-bound CUDA kernels for sm_103a behind a C-ABI library
(``libkvq.so``, declared in ``include/kvq.h``):

* ``kvq_store_nvfp4`` -- bf16 K/V -> NVFP4 (e2m1 data + e4m3 group scales),
  scattered by ``slot_mapping`` into pages laid out as
  [K_data | K_scale | V_data | V_scale].
* ``kvq_gather_indexer_k`` -- fp8 indexer-K rows and their fp32 scales
  gathered from a paged cache into contiguous outputs through
  ``block_table`` and ``cu_seq_lens``.

``paged_quantized_kv_gb300.kvq`` is the thin Python binding (ctypes; torch
tensors only supply device pointers and the current stream).  Importing the
package itself loads nothing; the library is opened on first use and the
binding raises if it is missing -- there is no fallback.
"""

__all__ = ["kvq", "workloads"]
