// kvq_api.cu -- the extern "C" boundary of libkvq: host-side argument
// validation (no device memory is touched), stride/pointer derivation as in
// vLLM reshape_and_cache_nvfp4_dispatch (nvfp4_kv_cache_kernels.cu, commit
// 7ce4c8e), and the launch on the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "kvq.h"
#include "kvq_internal.h"

namespace kvq {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  int& n = cached[dev & 63];
  if (n == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        v < 1)
      v = 1;
    n = v;
  }
  return n;
}

namespace {

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

int ilog2_exact(int64_t v) {  // log2(v) if v is a power of two, else -1
  if (v <= 0 || (v & (v - 1)) != 0) return -1;
  int s = 0;
  while ((int64_t{1} << s) < v) ++s;
  return s;
}

}  // namespace

// Every check kvq_paged_attention_nvfp4 makes except those of its three
// scratch pointers, in the same order; KVQ_OK when they all pass.
kvq_status attention_check(
    const void* query, int64_t query_stride0, int32_t dtype, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    const uint8_t* key_cache, const uint8_t* value_cache, int64_t page_stride,
    int32_t block_size, int64_t num_blocks, int32_t layout,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const float* k_scale, const float* v_scale,
    float scale, int32_t partition_size, const void* out, int64_t out_stride0,
    uint32_t flags) {
  if (dtype != KVQ_DTYPE_BF16 && dtype != KVQ_DTYPE_FP16) return KVQ_ERR_DTYPE;
  if (layout != KVQ_LAYOUT_HND && layout != KVQ_LAYOUT_NHD)
    return KVQ_ERR_LAYOUT;
  if ((flags & ~static_cast<uint32_t>(KVQ_F_SWIZZLE_K_SCALE | KVQ_F_PDL |
                                     KVQ_F_PDL_EARLY_META)) != 0u)
    return KVQ_ERR_ARG;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_size <= 0 || block_size <= 0 || num_blocks < 0 ||
      max_blocks_per_seq < 0 || block_table_stride < max_blocks_per_seq ||
      max_context_len < 0)
    return KVQ_ERR_SHAPE;
  if (head_size != 128 || block_size % 4 != 0) return KVQ_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0 || num_q_heads / num_kv_heads > 16)
    return KVQ_ERR_SHAPE;
  if (partition_size <= 0 || partition_size % 128 != 0 ||
      partition_size > 512)
    return KVQ_ERR_SHAPE;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return KVQ_ERR_ARG;
  const int64_t H = num_kv_heads, D = head_size, B = block_size;
  const int64_t S = D / 16;
  if (page_stride < H * B * (D / 2 + S)) return KVQ_ERR_SHAPE;
  if (query_stride0 < num_q_heads * D || out_stride0 < num_q_heads * D)
    return KVQ_ERR_SHAPE;
  const int64_t max_parts =
      (static_cast<int64_t>(max_context_len) + partition_size - 1) /
      partition_size;
  if (num_seqs > 65535 || num_kv_heads > 65535 || max_parts > (1 << 20) ||
      static_cast<int64_t>(num_seqs) * num_kv_heads * max_parts >= INT32_MAX)
    return KVQ_ERR_SHAPE;
  if (num_seqs == 0) return KVQ_OK;
  if (query == nullptr || key_cache == nullptr || value_cache == nullptr ||
      block_table == nullptr || context_lens == nullptr ||
      k_scale == nullptr || v_scale == nullptr || out == nullptr)
    return KVQ_ERR_NULL;
  if (!aligned(query, 16) || query_stride0 % 8 != 0 || !aligned(out, 16) ||
      out_stride0 % 8 != 0 || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || page_stride % 16 != 0 ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return KVQ_ERR_ALIGN;
  return KVQ_OK;
}

}  // namespace kvq

extern "C" {

kvq_status kvq_store_nvfp4(const void* key, int64_t key_stride0,
                           const void* value, int64_t value_stride0,
                           int32_t dtype, int32_t num_tokens,
                           int32_t num_heads, int32_t head_size,
                           uint8_t* key_cache, uint8_t* value_cache,
                           int64_t page_stride, int32_t block_size,
                           int64_t num_blocks, int32_t layout,
                           const int64_t* slot_mapping, const float* k_scale,
                           const float* v_scale, uint32_t flags,
                           int32_t* dev_error, void* stream) {
  using namespace kvq;
  if (dtype != KVQ_DTYPE_BF16 && dtype != KVQ_DTYPE_FP16) return KVQ_ERR_DTYPE;
  if (layout != KVQ_LAYOUT_HND && layout != KVQ_LAYOUT_NHD)
    return KVQ_ERR_LAYOUT;
  if ((flags & ~static_cast<uint32_t>(KVQ_F_SWIZZLE_K_SCALE | KVQ_F_PDL |
                                      KVQ_F_PDL_EARLY_READ)) !=
      0u)
    return KVQ_ERR_ARG;
  if (num_tokens < 0 || num_heads <= 0 || head_size <= 0 || block_size <= 0 ||
      num_blocks < 0)
    return KVQ_ERR_SHAPE;
  // S = head_size/16 must split into 4 swizzle column groups; the swizzle
  // works on 4-token bands of the page.
  if (head_size % 64 != 0 || block_size % 4 != 0) return KVQ_ERR_SHAPE;
  const int64_t H = num_heads, D = head_size, B = block_size;
  const int64_t S = D / 16;
  const int64_t side_bytes = H * B * (D / 2 + S);
  if (page_stride < side_bytes) return KVQ_ERR_SHAPE;
  if (key_stride0 < 0 || value_stride0 < 0) return KVQ_ERR_SHAPE;
  const int64_t gpt = 2 * H * D / 16;  // 16-element groups per token
  if (gpt > (int64_t{1} << 20)) return KVQ_ERR_SHAPE;
  if (num_tokens == 0) return KVQ_OK;

  if (key == nullptr || value == nullptr || key_cache == nullptr ||
      value_cache == nullptr || slot_mapping == nullptr ||
      k_scale == nullptr || v_scale == nullptr)
    return KVQ_ERR_NULL;
  if (!aligned(key, 16) || !aligned(value, 16) || key_stride0 % 8 != 0 ||
      value_stride0 % 8 != 0 || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || page_stride % 16 != 0 ||
      !aligned(slot_mapping, 8) || !aligned(k_scale, 4) ||
      !aligned(v_scale, 4))
    return KVQ_ERR_ALIGN;

  StoreParams p{};
  p.src[0] = static_cast<const uint16_t*>(key);
  p.src[1] = static_cast<const uint16_t*>(value);
  p.src_stride[0] = key_stride0;
  p.src_stride[1] = value_stride0;
  p.side[0] = key_cache;
  p.side[1] = value_cache;
  p.slots = slot_mapping;
  p.scale[0] = k_scale;
  p.scale[1] = v_scale;
  p.dev_error = dev_error;
  p.page_stride = page_stride;
  p.num_slots = num_blocks * B;
  p.data_per_side = H * B * (D / 2);
  if (layout == KVQ_LAYOUT_HND) {
    p.dhs = B * (D / 2);
    p.dts = D / 2;
    p.shs = B * S;
    p.sts = S;
  } else {
    p.dhs = D / 2;
    p.dts = H * (D / 2);
    p.shs = S;
    p.sts = H * S;
  }
  p.num_tokens = num_tokens;
  p.H = num_heads;
  p.D = head_size;
  p.S = static_cast<int32_t>(S);
  p.B = block_size;
  p.b_shift = ilog2_exact(B);
  p.gpt = static_cast<int32_t>(gpt);
  if (gpt <= 256) {
    p.tpp = static_cast<int32_t>(256 / gpt);
    p.slices_log2 = 0;
  } else {
    p.tpp = 1;
    int sl = 0;
    while ((int64_t{256} << sl) < gpt) ++sl;
    p.slices_log2 = sl;
  }
  const int64_t passes =
      ((num_tokens + p.tpp - 1) / p.tpp) << p.slices_log2;
  if (passes >= (int64_t{1} << 31)) return KVQ_ERR_SHAPE;
  p.num_passes = static_cast<int32_t>(passes);
  p.swizzle_sides = 2u | ((flags & KVQ_F_SWIZZLE_K_SCALE) ? 1u : 0u);
  p.early_read = (flags & KVQ_F_PDL_EARLY_READ) != 0u;
  p.pdl = p.early_read || (flags & KVQ_F_PDL) != 0u;
  p.f16 = dtype == KVQ_DTYPE_FP16;

  const cudaError_t err =
      launch_store_nvfp4(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_gather_indexer_k(const uint8_t* kv_cache, int64_t block_stride,
                                int64_t num_blocks, int32_t block_size,
                                int32_t head_dim, const int32_t* block_table,
                                int64_t block_table_stride,
                                int32_t max_blocks_per_seq,
                                const int32_t* cu_seq_lens, int32_t num_seqs,
                                int64_t total_tokens, uint8_t* k_fp8,
                                uint8_t* k_scale, uint32_t flags,
                                int32_t* dev_error, void* stream) {
  using namespace kvq;
  if ((flags & ~static_cast<uint32_t>(KVQ_F_PDL | KVQ_F_PDL_EARLY_META |
                                      KVQ_F_PDL_EARLY_READ)) !=
      0u)
    return KVQ_ERR_ARG;
  if (block_size <= 0 || head_dim <= 0 || num_seqs < 0 || total_tokens < 0 ||
      num_blocks < 0 || max_blocks_per_seq < 0 ||
      block_table_stride < max_blocks_per_seq)
    return KVQ_ERR_SHAPE;
  if (head_dim % 16 != 0) return KVQ_ERR_SHAPE;
  if (block_stride < static_cast<int64_t>(block_size) * (head_dim + 4))
    return KVQ_ERR_SHAPE;
  if (total_tokens >= (int64_t{1} << 31)) return KVQ_ERR_SHAPE;
  if (total_tokens == 0) return KVQ_OK;
  if (num_seqs == 0) return KVQ_ERR_ARG;  // rows but no sequence
  if (kv_cache == nullptr || block_table == nullptr ||
      cu_seq_lens == nullptr || k_fp8 == nullptr || k_scale == nullptr)
    return KVQ_ERR_NULL;
  if (!aligned(kv_cache, 16) || block_stride % 16 != 0 ||
      !aligned(k_fp8, 16) || !aligned(k_scale, 4) ||
      !aligned(block_table, 4) || !aligned(cu_seq_lens, 4))
    return KVQ_ERR_ALIGN;

  GatherParams p{};
  p.cache = kv_cache;
  p.block_stride = block_stride;
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.bt_stride = block_table_stride;
  p.cu = cu_seq_lens;
  p.k_fp8 = k_fp8;
  p.k_scale = k_scale;
  p.dev_error = dev_error;
  p.total = total_tokens;
  p.B = block_size;
  p.D = head_dim;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.early_read = (flags & KVQ_F_PDL_EARLY_READ) != 0u;
  p.early_meta = p.early_read || (flags & KVQ_F_PDL_EARLY_META) != 0u;
  p.pdl = p.early_meta || (flags & KVQ_F_PDL) != 0u;
  const cudaError_t err =
      launch_gather_indexer_k(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_load_nvfp4(const uint8_t* key_cache, const uint8_t* value_cache,
                          int64_t page_stride, int32_t block_size,
                          int64_t num_blocks, int32_t layout,
                          int32_t num_heads, int32_t head_size,
                          const int32_t* block_table,
                          int64_t block_table_stride,
                          int32_t max_blocks_per_seq,
                          const int32_t* cu_seq_lens, int32_t num_seqs,
                          int64_t total_tokens, const float* k_scale,
                          const float* v_scale, int32_t out_dtype,
                          void* key_out, void* value_out, int64_t out_stride0,
                          uint32_t flags, int32_t* dev_error, void* stream) {
  using namespace kvq;
  if (out_dtype != KVQ_DTYPE_BF16) return KVQ_ERR_DTYPE;
  if (layout != KVQ_LAYOUT_HND && layout != KVQ_LAYOUT_NHD)
    return KVQ_ERR_LAYOUT;
  if ((flags & ~static_cast<uint32_t>(KVQ_F_SWIZZLE_K_SCALE | KVQ_F_PDL |
                                      KVQ_F_PDL_EARLY_META)) != 0u)
    return KVQ_ERR_ARG;
  if (num_heads <= 0 || head_size <= 0 || block_size <= 0 ||
      num_blocks < 0 || num_seqs < 0 || total_tokens < 0 ||
      max_blocks_per_seq < 0 || block_table_stride < max_blocks_per_seq)
    return KVQ_ERR_SHAPE;
  if (head_size % 64 != 0 || block_size % 4 != 0) return KVQ_ERR_SHAPE;
  const int64_t H = num_heads, D = head_size, B = block_size;
  const int64_t S = D / 16;
  if (page_stride < H * B * (D / 2 + S)) return KVQ_ERR_SHAPE;
  if (out_stride0 < H * D) return KVQ_ERR_SHAPE;
  const int64_t gpt = 2 * H * S;
  if (gpt > (int64_t{1} << 20) || total_tokens >= (int64_t{1} << 31))
    return KVQ_ERR_SHAPE;
  if (total_tokens == 0) return KVQ_OK;
  if (num_seqs == 0) return KVQ_ERR_ARG;
  if (key_cache == nullptr || value_cache == nullptr ||
      block_table == nullptr || cu_seq_lens == nullptr ||
      k_scale == nullptr || v_scale == nullptr || key_out == nullptr ||
      value_out == nullptr)
    return KVQ_ERR_NULL;
  if (!aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      page_stride % 16 != 0 || !aligned(key_out, 16) ||
      !aligned(value_out, 16) || out_stride0 % 8 != 0 ||
      !aligned(block_table, 4) || !aligned(cu_seq_lens, 4) ||
      !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return KVQ_ERR_ALIGN;

  LoadParams p{};
  p.side[0] = key_cache;
  p.side[1] = value_cache;
  p.out[0] = static_cast<uint16_t*>(key_out);
  p.out[1] = static_cast<uint16_t*>(value_out);
  p.scale[0] = k_scale;
  p.scale[1] = v_scale;
  p.block_table = block_table;
  p.cu = cu_seq_lens;
  p.dev_error = dev_error;
  p.bt_stride = block_table_stride;
  p.page_stride = page_stride;
  p.num_blocks = num_blocks;
  p.data_per_side = H * B * (D / 2);
  if (layout == KVQ_LAYOUT_HND) {
    p.dhs = B * (D / 2);
    p.dts = D / 2;
    p.shs = B * S;
    p.sts = S;
  } else {
    p.dhs = D / 2;
    p.dts = H * (D / 2);
    p.shs = S;
    p.sts = H * S;
  }
  p.out_stride0 = out_stride0;
  p.total = total_tokens;
  p.H = num_heads;
  p.D = head_size;
  p.S = static_cast<int32_t>(S);
  p.B = block_size;
  p.b_shift = ilog2_exact(B);
  const int64_t upt = gpt / 2;  // two groups per thread role
  p.upt = static_cast<int32_t>(upt);
  if (upt <= 256) {
    p.tpp = static_cast<int32_t>(256 / upt);
    p.slices_log2 = 0;
  } else {
    p.tpp = 1;
    int sl = 0;
    while ((int64_t{256} << sl) < upt) ++sl;
    p.slices_log2 = sl;
  }
  const int64_t passes =
      ((total_tokens + p.tpp - 1) / p.tpp) << p.slices_log2;
  if (passes >= (int64_t{1} << 31)) return KVQ_ERR_SHAPE;
  p.num_passes = static_cast<int32_t>(passes);
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.swizzle_sides = 2u | ((flags & KVQ_F_SWIZZLE_K_SCALE) ? 1u : 0u);
  p.early_meta = (flags & KVQ_F_PDL_EARLY_META) != 0u;
  p.pdl = p.early_meta || (flags & KVQ_F_PDL) != 0u;
  const cudaError_t err =
      launch_load_nvfp4(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_store_indexer_k(const void* k, int64_t k_stride0,
                               int32_t dtype, int32_t num_tokens,
                               int32_t head_dim, uint8_t* kv_cache,
                               int64_t block_stride, int32_t block_size,
                               int64_t num_blocks,
                               const int64_t* slot_mapping, uint32_t flags,
                               int32_t* dev_error, void* stream) {
  using namespace kvq;
  if (dtype != KVQ_DTYPE_BF16 && dtype != KVQ_DTYPE_FP16) return KVQ_ERR_DTYPE;
  if ((flags & ~static_cast<uint32_t>(KVQ_F_PDL | KVQ_F_PDL_EARLY_READ)) !=
      0u)
    return KVQ_ERR_ARG;
  if (num_tokens < 0 || block_size <= 0 || num_blocks < 0 || k_stride0 < 0)
    return KVQ_ERR_SHAPE;
  if (head_dim != 16 && head_dim != 32 && head_dim != 64 && head_dim != 128 &&
      head_dim != 256)
    return KVQ_ERR_SHAPE;
  if (block_stride < static_cast<int64_t>(block_size) * (head_dim + 4))
    return KVQ_ERR_SHAPE;
  if (num_tokens == 0) return KVQ_OK;
  if (k == nullptr || kv_cache == nullptr || slot_mapping == nullptr)
    return KVQ_ERR_NULL;
  if (!aligned(k, 16) || k_stride0 % 8 != 0 || !aligned(kv_cache, 16) ||
      block_stride % 16 != 0 || !aligned(slot_mapping, 8))
    return KVQ_ERR_ALIGN;
  IndexerStoreParams p{};
  p.k = static_cast<const uint16_t*>(k);
  p.k_stride0 = k_stride0;
  p.cache = kv_cache;
  p.block_stride = block_stride;
  p.slots = slot_mapping;
  p.dev_error = dev_error;
  p.num_slots = num_blocks * block_size;
  p.num_tokens = num_tokens;
  p.D = head_dim;
  p.B = block_size;
  p.b_shift = ilog2_exact(block_size);
  p.f16 = dtype == KVQ_DTYPE_FP16;
  p.early_read = (flags & KVQ_F_PDL_EARLY_READ) != 0u;
  p.pdl = p.early_read || (flags & KVQ_F_PDL) != 0u;
  p.vec32 = aligned(k, 32) && k_stride0 % 16 == 0;
  const cudaError_t err =
      launch_store_indexer_k(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_paged_attention_nvfp4(
    const void* query, int64_t query_stride0, int32_t dtype, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    const uint8_t* key_cache, const uint8_t* value_cache, int64_t page_stride,
    int32_t block_size, int64_t num_blocks, int32_t layout,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const float* k_scale, const float* v_scale,
    float scale, int32_t partition_size, float* exp_sums, float* max_logits,
    float* tmp_out, void* out, int64_t out_stride0, uint32_t flags,
    int32_t* dev_error, void* stream) {
  using namespace kvq;
  const kvq_status st = attention_check(
      query, query_stride0, dtype, num_seqs, num_q_heads, num_kv_heads,
      head_size, key_cache, value_cache, page_stride, block_size, num_blocks,
      layout, block_table, block_table_stride, max_blocks_per_seq,
      context_lens, max_context_len, k_scale, v_scale, scale, partition_size,
      out, out_stride0, flags);
  if (st != KVQ_OK || num_seqs == 0) return st;
  const int64_t H = num_kv_heads, D = head_size, B = block_size;
  const int64_t S = D / 16;
  const int64_t max_parts =
      (static_cast<int64_t>(max_context_len) + partition_size - 1) /
      partition_size;
  if (max_parts > 1 &&
      (exp_sums == nullptr || max_logits == nullptr || tmp_out == nullptr))
    return KVQ_ERR_NULL;
  if (max_parts > 1 && (!aligned(exp_sums, 4) || !aligned(max_logits, 4) ||
                        !aligned(tmp_out, 16)))
    return KVQ_ERR_ALIGN;

  AttnParams p{};
  p.q = static_cast<const uint16_t*>(query);
  p.q_stride0 = query_stride0;
  p.side[0] = key_cache;
  p.side[1] = value_cache;
  p.page_stride = page_stride;
  p.num_blocks = num_blocks;
  p.scale_off = H * B * (D / 2);
  if (layout == KVQ_LAYOUT_HND) {
    p.dhs = B * (D / 2);
    p.dts = D / 2;
    p.shs = B * S;
    p.sts = S;
  } else {
    p.dhs = D / 2;
    p.dts = H * (D / 2);
    p.shs = S;
    p.sts = H * S;
  }
  p.block_table = block_table;
  p.bt_stride = block_table_stride;
  p.lens = context_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.scale = scale;
  p.exp_sums = exp_sums;
  p.max_logits = max_logits;
  p.tmp_out = tmp_out;
  p.out = static_cast<uint16_t*>(out);
  p.out_stride0 = out_stride0;
  p.dev_error = dev_error;
  p.num_seqs = num_seqs;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = num_q_heads / num_kv_heads;
  p.B = block_size;
  p.b_shift = ilog2_exact(B);
  p.part = partition_size;
  p.max_parts = static_cast<int32_t>(max_parts > 0 ? max_parts : 1);
  const int64_t cap = std::min<int64_t>(
      max_context_len, static_cast<int64_t>(max_blocks_per_seq) * B);
  p.len_cap = static_cast<int32_t>(std::min<int64_t>(cap, INT32_MAX));
  p.swizzle_k = (flags & KVQ_F_SWIZZLE_K_SCALE) != 0u;
  p.f16 = dtype == KVQ_DTYPE_FP16;
  p.early_meta = (flags & KVQ_F_PDL_EARLY_META) != 0u;
  p.pdl = p.early_meta || (flags & KVQ_F_PDL) != 0u;
  const cudaError_t err =
      launch_paged_attention_mma(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_NULL: return "a required pointer is NULL";
    case KVQ_ERR_SHAPE: return "invalid size or divisibility";
    case KVQ_ERR_ALIGN: return "pointer or stride misaligned";
    case KVQ_ERR_DTYPE: return "unsupported element type";
    case KVQ_ERR_LAYOUT: return "unknown cache layout";
    case KVQ_ERR_CUDA: return "CUDA launch error";
    case KVQ_ERR_ARG: return "invalid flags or inconsistent arguments";
    case KVQ_ERR_SCRATCH: return "needs more than the built-in scratch array";
  }
  return "unknown status";
}

int32_t kvq_version(void) { return 100; }

}  // extern "C"
