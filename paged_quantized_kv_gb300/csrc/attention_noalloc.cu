// attention_noalloc.cu -- paged decode attention for callers that must not
// allocate device memory.
//
// kvq_paged_attention_nvfp4 needs fp32 scratch (per-partition maxima, sums
// and partial outputs) whenever a context spans more than one partition,
// and it takes that scratch from the caller.  Some callers cannot provide
// it: code that runs after an engine has reserved all device memory for
// itself, or inside a runtime whose rules forbid device allocation once it
// is serving.  This file gives them one entry point that uses a scratch
// array built into the library instead: a file-scope device array of a
// fixed size, which every GPU that loads the library holds until the
// process exits.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine; the work is done by kvq_paged_attention_nvfp4 itself,
// unchanged, pointed at sub-ranges of the array.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

// The scratch.  Host code sees only a stand-in for this name; the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_attn_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;  // taken only until a device's address is known
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the array on the current device; looked up once per
// device (the first call on a device does it, with that device current).
// Once known, the address is read without a lock.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      err = cudaGetSymbolAddress(&p, g_attn_scratch);
      if (err != cudaSuccess) return err;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_paged_attention_nvfp4_noalloc(
    const void* query, int64_t query_stride0, int32_t dtype, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    const uint8_t* key_cache, const uint8_t* value_cache, int64_t page_stride,
    int32_t block_size, int64_t num_blocks, int32_t layout,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const float* k_scale, const float* v_scale,
    float scale, int32_t partition_size, void* out, int64_t out_stride0,
    uint32_t flags, int32_t* dev_error, void* stream) {
  // the plain entry point's own checks first, so that a call it would
  // reject gets the same code here (whatever the scratch it would need)
  const kvq_status st = kvq::attention_check(
      query, query_stride0, dtype, num_seqs, num_q_heads, num_kv_heads,
      head_size, key_cache, value_cache, page_stride, block_size, num_blocks,
      layout, block_table, block_table_stride, max_blocks_per_seq,
      context_lens, max_context_len, k_scale, v_scale, scale, partition_size,
      out, out_stride0, flags);
  if (st != KVQ_OK || num_seqs == 0) return st;
  float* exp_sums = nullptr;
  float* max_logits = nullptr;
  float* tmp_out = nullptr;
  const int64_t parts =
      (static_cast<int64_t>(max_context_len) + partition_size - 1) /
      partition_size;
  if (parts > 1) {
    // tmp_out [rows, head_size] first (16-byte aligned), then the sums and
    // maxima [rows] each: (head_size + 2) floats per row
    const int64_t cap = static_cast<int64_t>(KVQ_NOALLOC_SCRATCH_BYTES) /
                        ((static_cast<int64_t>(head_size) + 2) * 4);
    const int64_t rows =
        static_cast<int64_t>(num_seqs) * num_q_heads * parts;
    if (rows > cap) return KVQ_ERR_SCRATCH;
    void* base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return KVQ_ERR_CUDA;
    tmp_out = static_cast<float*>(base);
    exp_sums = tmp_out + rows * head_size;
    max_logits = exp_sums + rows;
  }
  return kvq_paged_attention_nvfp4(
      query, query_stride0, dtype, num_seqs, num_q_heads, num_kv_heads,
      head_size, key_cache, value_cache, page_stride, block_size, num_blocks,
      layout, block_table, block_table_stride, max_blocks_per_seq,
      context_lens, max_context_len, k_scale, v_scale, scale, partition_size,
      exp_sums, max_logits, tmp_out, out, out_stride0, flags, dev_error,
      stream);
}
