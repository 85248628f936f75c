// kvq_internal.h -- launch parameters and device helpers shared by the
// libkvq translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

// ---------------------------------------------------------------------------
// NVFP4 store
// ---------------------------------------------------------------------------
struct StoreParams {
  const uint16_t* src[2];  // key, value (bf16 or fp16 bit patterns)
  int64_t src_stride[2];   // row stride in elements
  uint8_t* side[2];        // page 0 of the K side / V side
  const int64_t* slots;
  const float* scale[2];   // device k_scale / v_scale
  int32_t* dev_error;      // nullable
  int64_t page_stride;     // bytes
  int64_t num_slots;       // num_blocks * block_size
  int64_t data_per_side;   // H * B * D/2: offset of the scale region
  int64_t dhs, dts;        // data head / token strides (bytes)
  int64_t shs, sts;        // scale head / token strides (bytes)
  int32_t num_tokens;
  int32_t H, D, S, B;
  int32_t b_shift;         // log2(B) when B is a power of two, else -1
  int32_t gpt;             // 16-element groups per token, both sides
  int32_t tpp;             // tokens per pass (gpt <= 256: 256 / gpt)
  int32_t slices_log2;     // passes per token = 1 << slices_log2
  int32_t num_passes;
  uint32_t swizzle_sides;  // bit s set: side s's scales are swizzled
  bool pdl;                // launch with programmatic dependent launch
  bool early_read;         // load the first groups before waiting (PDL)
  bool f16;                // inputs are IEEE fp16 (else bf16)
};

cudaError_t launch_store_nvfp4(const StoreParams& p, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Indexer-K gather
// ---------------------------------------------------------------------------
struct GatherParams {
  const uint8_t* cache;
  int64_t block_stride;
  int64_t num_blocks;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* cu;
  uint8_t* k_fp8;
  uint8_t* k_scale;
  int32_t* dev_error;
  int64_t total;
  int32_t B, D;
  int32_t max_blocks;
  int32_t num_seqs;
  bool pdl;                // launch with programmatic dependent launch
  bool early_meta;         // read metadata before waiting on the predecessor
  bool early_read;         // ... and the cache rows too (wait before writes)
};

cudaError_t launch_gather_indexer_k(const GatherParams& p,
                                    cudaStream_t stream);

// ---------------------------------------------------------------------------
// NVFP4 paged load (dequantise pages back to bf16 rows)
// ---------------------------------------------------------------------------
struct LoadParams {
  const uint8_t* side[2];  // page 0 of the K side / V side
  uint16_t* out[2];        // bf16 key / value rows
  const float* scale[2];   // device k_scale / v_scale
  const int32_t* block_table;
  const int32_t* cu;
  int32_t* dev_error;      // nullable
  int64_t bt_stride;
  int64_t page_stride;
  int64_t num_blocks;
  int64_t data_per_side;
  int64_t dhs, dts, shs, sts;
  int64_t out_stride0;     // elements
  int64_t total;
  int32_t H, D, S, B;
  int32_t b_shift;
  int32_t upt;             // thread roles per row (two groups each): H * S
  int32_t tpp, slices_log2, num_passes;
  int32_t num_seqs, max_blocks;
  uint32_t swizzle_sides;
  bool pdl, early_meta;
};

cudaError_t launch_load_nvfp4(const LoadParams& p, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Indexer-K store (bf16/fp16 K -> e4m3 row + fp32 scale per token)
// ---------------------------------------------------------------------------
struct IndexerStoreParams {
  const uint16_t* k;       // [num_tokens, D] bit patterns, row stride below
  int64_t k_stride0;       // elements
  uint8_t* cache;          // block 0: [B*D e4m3 | B*4 scale bytes]
  int64_t block_stride;
  const int64_t* slots;
  int32_t* dev_error;      // nullable
  int64_t num_slots;       // num_blocks * B
  int64_t num_tokens;
  int32_t D, B, b_shift;
  bool f16, pdl;
  bool vec32;              // rows start 32-byte aligned (256-bit loads)
  bool early_read;         // load the first rows before waiting (PDL)
};

cudaError_t launch_store_indexer_k(const IndexerStoreParams& p,
                                   cudaStream_t stream);

// ---------------------------------------------------------------------------
// Paged decode attention over the NVFP4 cache
// ---------------------------------------------------------------------------
struct AttnParams {
  const uint16_t* q;       // [num_seqs, Hq, D] bf16/fp16 bits
  int64_t q_stride0;       // elements
  const uint8_t* side[2];  // page 0 of the K side / V side
  int64_t page_stride;
  int64_t num_blocks;
  int64_t scale_off;       // H * B * D/2: offset of a side's scale region
  int64_t dhs, dts, shs, sts;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* lens;     // context_lens [num_seqs]
  const float* k_scale;    // device scalars
  const float* v_scale;
  float scale;             // softmax scale
  float* exp_sums;         // [num_seqs, Hq, max_parts]  (max_parts > 1)
  float* max_logits;       // [num_seqs, Hq, max_parts]
  float* tmp_out;          // [num_seqs, Hq, max_parts, D]
  uint16_t* out;           // [num_seqs, Hq, D], rows out_stride0 apart
  int64_t out_stride0;
  int32_t* dev_error;      // nullable
  int32_t num_seqs, Hq, Hkv, G, B, b_shift;
  int32_t part;            // partition size (multiple of 128, <= 512)
  int32_t max_parts;       // partitions of the longest allowed context
  int32_t len_cap;         // min(max_context_len, max_blocks * B)
  bool swizzle_k;          // K scales stored swizzled too
  bool f16;                // query / out are fp16 (else bf16)
  bool pdl;
  bool early_meta;         // lengths, block ids, query read before the wait
};

cudaError_t launch_paged_attention_mma(const AttnParams& p,
                                       cudaStream_t stream);
// The argument checks of kvq_paged_attention_nvfp4 other than those of its
// scratch pointers (KVQ_OK when they pass); kvq_paged_attention_nvfp4_noalloc
// runs them before it checks its scratch capacity.
kvq_status attention_check(
    const void* query, int64_t query_stride0, int32_t dtype, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    const uint8_t* key_cache, const uint8_t* value_cache, int64_t page_stride,
    int32_t block_size, int64_t num_blocks, int32_t layout,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const float* k_scale, const float* v_scale,
    float scale, int32_t partition_size, const void* out, int64_t out_stride0,
    uint32_t flags);

// The partition merge of the attention (PDL launch).
cudaError_t launch_attention_merge(const AttnParams& p, cudaStream_t stream);

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Launch `kernel<<<grid, block, smem, stream>>>(params)`, with programmatic
// dependent launch when `pdl` is set.
template <typename Params>
cudaError_t launch_kernel(void (*kernel)(Params), dim3 grid,
                          unsigned block, size_t smem, cudaStream_t stream,
                          bool pdl, const Params& params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, params);
}

// First thing every kernel does: wait until the grid it depends on (when
// launched with programmatic dependent launch) has completed and its writes
// are visible -- a no-op otherwise -- then let a dependent grid start its
// own launch.
__device__ __forceinline__ void pdl_prologue() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace kvq
