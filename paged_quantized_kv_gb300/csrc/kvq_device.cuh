// kvq_device.cuh -- device helpers shared by the kernels that read paged
// metadata (cu_seq_lens, block_table): TMA bulk staging into shared memory
// with a bounded mbarrier wait, and the sequence search.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {
namespace dev {

constexpr size_t kMaxMetaSmem = 48 * 1024;  // no opt-in needed

// Time limit of a bounded mbarrier wait (ns of %globaltimer).
#ifndef KVQ_WAIT_LIMIT_NS
#define KVQ_WAIT_LIMIT_NS 1000000000ull
#endif
// Test builds only: expect this many bytes more than the bulk copies
// deliver, so that the bounded wait runs out (0 in the library).
#ifndef KVQ_TEST_EXTRA_TX
#define KVQ_TEST_EXTRA_TX 0
#endif

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One non-blocking test of phase `parity` of the mbarrier at `bar`.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of the mbarrier at `bar`, for at most
// KVQ_WAIT_LIMIT_NS of wall time (and at most 2^24 polls, in case the
// timer stood still); false on timeout.  The timer is read only once the
// first test has failed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t start = global_ns();
  for (uint32_t polls = 0; polls < (1u << 24); ++polls) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - start > KVQ_WAIT_LIMIT_NS) return false;
  }
  return false;
}

// Largest b in [0, n] with cu[b] <= r (cu[0] == 0 <= r); cu in shared
// memory (kShared) or global memory.
template <bool kShared>
__device__ __forceinline__ int find_seq(const int32_t* cu, int n, int64_t r) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int32_t v = kShared ? cu[mid] : __ldg(cu + mid);
    if (static_cast<int64_t>(v) <= r)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Where the kernel reads its metadata from.
enum MetaMode {
  kMetaGlobal = 0,     // cu_seq_lens and block_table from global memory
  kMetaSharedCu = 1,   // cu_seq_lens staged in shared memory
  kMetaSharedCuBt = 2  // cu_seq_lens and the (contiguous) block table
};

// Shared-memory image of an int32 range: it starts at base + (src % 16) so
// that every 16-byte-aligned source address maps to a 16-byte-aligned
// shared address; the range needs at most 16 + 4 * n bytes, rounded to 16.
__host__ __device__ constexpr size_t region_bytes(int64_t n) {
  return (16 + 4 * static_cast<size_t>(n) + 15) & ~size_t{15};
}

struct RangeSplit {
  int head;  // entries before the first 16-byte boundary
  int body;  // entries in whole 16-byte chunks
};

__device__ __forceinline__ RangeSplit split_range(const int32_t* src, int n) {
  const int mis = static_cast<int>(reinterpret_cast<uintptr_t>(src) & 15);
  int head = ((16 - mis) & 15) >> 2;
  if (head > n) head = n;
  const int body = ((n - head) >> 2) << 2;
  return {head, body};
}

// Stage cu_seq_lens (and the block table) into shared memory.  Thread 0
// arms the mbarrier and issues the bulk copies of the aligned bodies; warp
// 1 copies the unaligned heads and tails (the CTA needs at least 44
// threads).  Every thread of the CTA must call it.  Returns false if the
// bulk copy did not complete within the poll budget.
__device__ __forceinline__ bool stage_meta(uint8_t* smem, uint64_t* bar,
                                           const int32_t* cu, int ncu,
                                           const int32_t* bt, int nbt,
                                           int32_t** s_cu, int32_t** s_bt) {
  const int tid = threadIdx.x;
  int32_t* dcu = reinterpret_cast<int32_t*>(
      smem + (reinterpret_cast<uintptr_t>(cu) & 15));
  uint8_t* bt_base = smem + region_bytes(ncu);
  int32_t* dbt = reinterpret_cast<int32_t*>(
      bt_base + (reinterpret_cast<uintptr_t>(bt) & 15));
  *s_cu = dcu;
  *s_bt = dbt;
  const RangeSplit rc = split_range(cu, ncu);
  const RangeSplit rb =
      nbt > 0 ? split_range(bt, nbt) : RangeSplit{0, 0};
  const uint32_t bytes = 4u * static_cast<uint32_t>(rc.body + rb.body);
  const uint32_t expect = bytes > 0 ? bytes + KVQ_TEST_EXTRA_TX : 0;
  const uint32_t b = smem_addr(bar);

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0 && bytes > 0) {
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
        ::"r"(b), "r"(expect)
        : "memory");
    if (rc.body > 0)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1], %2, [%3];" ::"r"(smem_addr(dcu + rc.head)),
          "l"(cu + rc.head), "r"(4u * rc.body), "r"(b)
          : "memory");
    if (rb.body > 0)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1], %2, [%3];" ::"r"(smem_addr(dbt + rb.head)),
          "l"(bt + rb.head), "r"(4u * rb.body), "r"(b)
          : "memory");
  }
  // unaligned heads and tails: at most 3 + 3 entries per range
  if (tid >= 32 && tid < 32 + 12) {
    const int k = tid - 32;
    const int32_t* src = k < 6 ? cu : bt;
    int32_t* dst = k < 6 ? dcu : dbt;
    const int n = k < 6 ? ncu : nbt;
    const RangeSplit r = k < 6 ? rc : rb;
    const int j = k % 6;
    const int i = j < 3 ? j : r.head + r.body + (j - 3);
    if ((j < 3 && i < r.head) || (j >= 3 && i < n)) dst[i] = __ldg(src + i);
  }
  bool ok = true;
  if (bytes > 0) {
    ok = mbar_wait(b, 0);
    // on a timeout, give a copy that may still be in flight a second term
    // before the CTA (and its shared memory) goes away
    if (!ok) mbar_wait(b, 0);
  }
  __syncthreads();
  return ok;
}

}  // namespace dev
}  // namespace kvq
