// gather_indexer_k.cu -- paged fp8 indexer-K + fp32 scale gather, sm_103a.
//
// Operation: vLLM PR #25931 "Add gather_indexer_k_quant_cache kernel"
// (cp_gather_indexer_k_quant_cache(kv_cache, k_fp8, k_scale, block_table,
// cu_seq_lens)) and PR #26456 (k_scale handed on as raw bytes viewed as
// float32).  Output row i = cu_seq_lens[b] + p takes the K row and the scale
// of token p of sequence b from block block_table[b, p / B], offset p % B.
// The first published version of this op launched too few blocks for long
// sequences; here every output row belongs to exactly one warp unit, so the
// grid covers total_tokens by construction.
//
// GB300 design: a pure copy, HBM-bound (2 x (D + 4) bytes per row), whose
// time at tens of MB is dominated by the fixed launch cost and by the
// dependent-load chain before the first row load (cu_seq_lens ->
// block_table -> K rows), since the whole grid fits in one wave.
//   * Each CTA stages cu_seq_lens -- and, when it is contiguous and fits,
//     the used block table -- in shared memory: the 16-byte-aligned body of
//     each range with one TMA bulk copy (cp.async.bulk, completion counted
//     on an mbarrier, waited on with a bounded poll), the few unaligned
//     head/tail entries with plain loads.  Row resolution (binary search,
//     block lookup) then costs one memory round trip and few instructions.
//     Ranges beyond 48 KB fall back to global reads.
//   * With KVQ_F_PDL the kernel waits for its predecessor (griddepcontrol)
//     before touching memory; with KVQ_F_PDL_EARLY_META it stages and
//     resolves the metadata first and waits only before the cache reads and
//     any write, overlapping that round trip with the predecessor's tail;
//     with KVQ_F_PDL_EARLY_READ it also issues the cache reads first and
//     waits only before its first write.
//   * One warp owns 32 consecutive output rows: lane l resolves row r0 + l,
//     then the warp moves the 32 rows as 16-byte vectors -- all loads of the
//     unit issued before its stores, 32 x D bytes in flight per warp -- and
//     each lane copies its row's 4 scale bytes.  Destination rows are
//     contiguous, so every store is a full sector.  Row loads are
//     L2-evict-first and row stores streaming: nothing here is read twice.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

using namespace kvq::dev;

#ifndef KVQ_GATHER_THREADS
#define KVQ_GATHER_THREADS 256
#endif
constexpr int kThreads = KVQ_GATHER_THREADS;
constexpr int kWarps = kThreads / 32;

// Cache rows are read once: each 16-byte load carries an L2 evict-first
// policy (created next to the load), and the K rows are stored streaming
// (.cs).  Measured back to back with KVQ_F_PDL_EARLY_READ on the
// long-context gather: 7.1 us with default policies, 5.6 us with both (a
// variant that created the policy once per thread, and also hinted the
// 4-byte scale load and store, measured 7.2 us; hinting the scales on top
// of this form, 5.7 us).
__device__ __forceinline__ uint4 ld_nc_16(const void* p) {
  uint4 v;
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(pol));
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 "
      "{%0, %1, %2, %3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_16(void* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// When the kernel waits for its predecessor (programmatic dependent
// launch): before anything (0), after resolving its rows from the
// metadata (1, KVQ_F_PDL_EARLY_META), or after issuing its cache reads,
// just before its first write (2, KVQ_F_PDL_EARLY_READ; with a runtime row
// width it waits before the reads instead).
enum { kWaitFirst = 0, kWaitMeta = 1, kWaitWrites = 2 };

// CPR = 16-byte chunks per K row (head_dim / 16); 0 = runtime value.
template <int CPR, int kMode, int kEarly>
__global__ void __launch_bounds__(kThreads)
gather_indexer_k_kernel(const GatherParams p) {
  extern __shared__ __align__(16) uint8_t s_raw[];
  __shared__ __align__(8) uint64_t s_bar;

  if constexpr (kEarly == kWaitFirst) pdl_prologue();
  const int32_t* cu = p.cu;
  int32_t* s_cu = nullptr;
  int32_t* s_bt = nullptr;
  bool staged = true;
  if constexpr (kMode != kMetaGlobal) {
    staged = stage_meta(s_raw, &s_bar, p.cu, p.num_seqs + 1, p.block_table,
                        kMode == kMetaSharedCuBt ? p.num_seqs * p.max_blocks
                                                 : 0,
                        &s_cu, &s_bt);
    cu = s_cu;
  }
  const int lane = threadIdx.x & 31;
  const int64_t unit =
      static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t r0 = unit * 32;

  // ---- resolve this lane's row (metadata only) ---------------------------
  const int64_t r = r0 + lane;
  const uint8_t* src_row = nullptr;
  const uint8_t* src_scale = nullptr;
  int err = 0;
  if (!staged) {
    err = KVQ_DEVERR_TIMEOUT;
  } else if (r < p.total) {
    const int b = find_seq<kMode != kMetaGlobal>(cu, p.num_seqs, r);
    if (b >= p.num_seqs) {
      err = KVQ_DEVERR_SEQ;  // no sequence covers this row
    } else {
      const int64_t pos64 = r - cu[b];
      const int32_t pos = static_cast<int32_t>(pos64);
      const int32_t kb = pos / p.B;
      const int32_t off = pos - kb * p.B;
      if (pos64 < 0 || pos64 >= (int64_t{1} << 31) || kb >= p.max_blocks) {
        err = KVQ_DEVERR_SEQ;
      } else {
        const int64_t blk =
            kMode == kMetaSharedCuBt
                ? s_bt[b * p.max_blocks + kb]
                : __ldg(p.block_table + b * p.bt_stride + kb);
        if (blk < 0 || blk >= p.num_blocks) {
          err = KVQ_DEVERR_BLOCK;
        } else {
          const uint8_t* base = p.cache + blk * p.block_stride;
          src_row = base + static_cast<int64_t>(off) * p.D;
          src_scale = base + static_cast<int64_t>(p.B) * p.D + off * 4;
        }
      }
    }
  }
  const bool total_mismatch = unit == 0 && lane == 0 && staged &&
                              static_cast<int64_t>(cu[p.num_seqs]) != p.total;

  // ---- from here on: cache reads and writes ------------------------------
  constexpr bool kWaitBeforeReads =
      kEarly == kWaitMeta || (kEarly == kWaitWrites && CPR == 0);
  if constexpr (kWaitBeforeReads) pdl_prologue();
  auto flag_errors = [&]() {
    if (p.dev_error != nullptr) {
      if (err != 0) atomicOr(p.dev_error, err);
      if (total_mismatch) atomicOr(p.dev_error, KVQ_DEVERR_SEQ);
    }
  };
  constexpr bool kFlagAfterReads = kEarly == kWaitWrites && CPR > 0;
  if constexpr (!kFlagAfterReads) flag_errors();
  // whole warp leaves together (a warp past the last row has nothing to
  // flag: its rows do not exist)
  if (r0 >= p.total) return;
  if (!staged) {
    if constexpr (kFlagAfterReads) {
      pdl_prologue();  // the timeout flag is a write: after the wait
      flag_errors();
    }
    return;
  }

  // the scale load goes out first, alongside the row loads below
  uint32_t scale_bits = 0;
  if (src_scale != nullptr) scale_bits = ld_nc_u32(src_scale);

  // ---- copy the 32 K rows as 16-byte vectors ---------------------------
  const int cpr = CPR > 0 ? CPR : (p.D >> 4);
  const unsigned long long my_src =
      reinterpret_cast<unsigned long long>(src_row);
  if constexpr (CPR > 0) {
    // all CPR loads of this lane first, then the stores
    uint4 v[CPR];
    const uint8_t* s[CPR];
#pragma unroll
    for (int i = 0; i < CPR; ++i) {
      const int c = i * 32 + lane;
      const int row = c / CPR;
      s[i] = reinterpret_cast<const uint8_t*>(
          __shfl_sync(0xFFFFFFFFu, my_src, row));
      if (s[i] != nullptr) v[i] = ld_nc_16(s[i] + (c % CPR) * 16);
    }
    if constexpr (kEarly == kWaitWrites) {
      pdl_prologue();  // the reads are in flight; no write before the wait
      flag_errors();
    }
#pragma unroll
    for (int i = 0; i < CPR; ++i) {
      const int c = i * 32 + lane;
      const int row = c / CPR;
      if (s[i] != nullptr)
        st_16(p.k_fp8 + (r0 + row) * p.D + (c % CPR) * 16, v[i]);
    }
  } else {
    for (int c = lane; c < 32 * cpr; c += 32) {
      const int row = c / cpr;
      const uint8_t* s = reinterpret_cast<const uint8_t*>(
          __shfl_sync(0xFFFFFFFFu, my_src, row));
      if (s != nullptr) {
        const uint4 v = ld_nc_16(s + (c % cpr) * 16);
        st_16(p.k_fp8 + (r0 + row) * p.D + (c % cpr) * 16, v);
      }
    }
  }

  // ---- the row's 4 scale bytes -----------------------------------------
  if (src_scale != nullptr)
    *reinterpret_cast<uint32_t*>(p.k_scale + r * 4) = scale_bits;
}

// ---------------------------------------------------------------------------
// Bulk-copy form (build option KVQ_GATHER_BULK=1): one CTA of one warp per
// (sequence, block of its table).  The block's rows of that sequence -- at
// most B of them, contiguous in the cache and in k_fp8 -- move with two TMA
// bulk copies (cache -> shared memory, completion counted on an mbarrier
// waited on with the bounded poll; shared memory -> k_fp8), and their scale
// bytes (contiguous in the cache, starting at any 4-byte row of k_scale)
// with one bulk load and 4-byte stores; taken when the rows and scales of a
// block fit in 48 KB.  Measured on GB300 against the per-row form above
// (long-context gather, 34.6 MB): a cold single launch 3-8 % faster (ncu:
// 8.58 against 9.31 us, 9.38 against 9.63 in another capture), back to back
// with KVQ_F_PDL_EARLY_READ 15 % slower (6.41 against 5.57 us: its 8.4 KB
// per-warp CTAs find less room beside the finishing predecessor), equal
// without PDL -- so the per-row form is the default.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int64_t bulk_scale_bytes(int B) {
  return (static_cast<int64_t>(B) * 4 + 15) & ~int64_t{15};
}

template <int kEarly>
__global__ void __launch_bounds__(32)
gather_bulk_kernel(const GatherParams p) {
  extern __shared__ __align__(128) uint8_t s_buf[];  // rows, then scales
  __shared__ __align__(8) uint64_t s_bar;
  if constexpr (kEarly == kWaitFirst) pdl_prologue();
  const int lane = threadIdx.x;
  const int64_t unit = blockIdx.x;
  const int b = static_cast<int>(unit / p.max_blocks);
  const int kb = static_cast<int>(unit - static_cast<int64_t>(b) * p.max_blocks);
  const int64_t c0 = __ldg(p.cu + b);
  const int64_t len = static_cast<int64_t>(__ldg(p.cu + b + 1)) - c0;
  const int64_t pos0 = static_cast<int64_t>(kb) * p.B;
  const int64_t row0 = c0 + pos0;  // first output row of the unit
  int err = 0;
  int n = 0;
  const uint8_t* src = nullptr;
  if (c0 < 0) {
    err = len > 0 ? KVQ_DEVERR_SEQ : 0;
  } else if (len > pos0) {
    n = static_cast<int>(len - pos0 < p.B ? len - pos0 : p.B);
    if (row0 + n > p.total) {  // rows past total_tokens are not written
      err = KVQ_DEVERR_SEQ;
      n = row0 >= p.total ? 0 : static_cast<int>(p.total - row0);
    }
    const int32_t blk = __ldg(p.block_table + b * p.bt_stride + kb);
    if (blk < 0 || blk >= p.num_blocks) {
      err |= KVQ_DEVERR_BLOCK;
      n = 0;
    } else {
      src = p.cache + static_cast<int64_t>(blk) * p.block_stride;
    }
  }
  // positions past the block table's last column, and cu_seq_lens that
  // does not end at total_tokens, are flagged once
  if (kb == p.max_blocks - 1 && len > static_cast<int64_t>(p.max_blocks) * p.B)
    err |= KVQ_DEVERR_SEQ;
  if (unit == 0 && static_cast<int64_t>(__ldg(p.cu + p.num_seqs)) != p.total)
    err |= KVQ_DEVERR_SEQ;

  const uint32_t kbytes = static_cast<uint32_t>(n) * p.D;
  const uint32_t sbytes = static_cast<uint32_t>((n * 4 + 15) & ~15);
  const uint32_t bar = smem_addr(&s_bar);
  uint8_t* s_scales = s_buf + static_cast<int64_t>(p.B) * p.D;
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  auto issue_loads = [&]() {
    if (lane != 0 || n == 0) return;
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
        ::"r"(bar), "r"(kbytes + sbytes + KVQ_TEST_EXTRA_TX)
        : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(smem_addr(s_buf)),
        "l"(src), "r"(kbytes),
        "r"(bar)
        : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(smem_addr(s_scales)),
        "l"(src + static_cast<int64_t>(p.B) * p.D), "r"(sbytes), "r"(bar)
        : "memory");
  };
  if constexpr (kEarly == kWaitWrites) {
    issue_loads();  // reads while the predecessor finishes
    pdl_prologue();
  } else {
    if constexpr (kEarly == kWaitMeta) pdl_prologue();
    issue_loads();
  }
  if (lane == 0 && err != 0 && p.dev_error != nullptr)
    atomicOr(p.dev_error, err);
  if (n == 0) return;
  if (!mbar_wait(bar, 0)) {
    // give a copy that may still be in flight a second term before the
    // shared memory goes away; write nothing
    mbar_wait(bar, 0);
    if (lane == 0 && p.dev_error != nullptr)
      atomicOr(p.dev_error, KVQ_DEVERR_TIMEOUT);
    return;
  }
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile(
        "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
            p.k_fp8 + row0 * p.D),
        "r"(smem_addr(s_buf)), "r"(kbytes)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  for (int i = lane; i < n; i += 32)
    *reinterpret_cast<uint32_t*>(p.k_scale + (row0 + i) * 4) =
        *reinterpret_cast<const uint32_t*>(s_scales + 4 * i);
  // the bulk store must have read the shared memory before the CTA ends
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

template <int kEarly>
cudaError_t launch_bulk(const GatherParams& p, cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(p.num_seqs) * p.max_blocks;
  const size_t smem = static_cast<size_t>(p.B) * p.D + bulk_scale_bytes(p.B);
  return launch_kernel(gather_bulk_kernel<kEarly>,
                       dim3(static_cast<unsigned>(units)), 32, smem, stream,
                       p.pdl, p);
}

template <int CPR, int kEarly>
cudaError_t launch_mode(const GatherParams& p, unsigned grid,
                        cudaStream_t stream) {
  const int64_t ncu = static_cast<int64_t>(p.num_seqs) + 1;
  const int64_t nbt = static_cast<int64_t>(p.num_seqs) * p.max_blocks;
  const size_t both = region_bytes(ncu) + region_bytes(nbt);
  if (p.bt_stride == p.max_blocks && both <= kMaxMetaSmem)
    return launch_kernel(
        gather_indexer_k_kernel<CPR, kMetaSharedCuBt, kEarly>, grid,
        kThreads, both, stream, p.pdl, p);
  if (region_bytes(ncu) <= kMaxMetaSmem)
    return launch_kernel(
        gather_indexer_k_kernel<CPR, kMetaSharedCu, kEarly>, grid,
        kThreads, region_bytes(ncu), stream, p.pdl, p);
  return launch_kernel(gather_indexer_k_kernel<CPR, kMetaGlobal, kEarly>,
                       grid, kThreads, 0, stream, p.pdl, p);
}

template <int CPR>
cudaError_t launch_cpr(const GatherParams& p, unsigned grid,
                       cudaStream_t stream) {
  if (p.early_read) return launch_mode<CPR, kWaitWrites>(p, grid, stream);
  if (p.early_meta) return launch_mode<CPR, kWaitMeta>(p, grid, stream);
  return launch_mode<CPR, kWaitFirst>(p, grid, stream);
}

}  // namespace

#ifndef KVQ_GATHER_BULK
#define KVQ_GATHER_BULK 0
#endif

cudaError_t launch_gather_indexer_k(const GatherParams& p,
                                    cudaStream_t stream) {
  if (KVQ_GATHER_BULK && p.max_blocks > 0 &&
      static_cast<int64_t>(p.B) * p.D + bulk_scale_bytes(p.B) <=
          static_cast<int64_t>(kMaxMetaSmem) &&
      static_cast<int64_t>(p.num_seqs) * p.max_blocks < (int64_t{1} << 31)) {
    if (p.early_read) return launch_bulk<kWaitWrites>(p, stream);
    if (p.early_meta) return launch_bulk<kWaitMeta>(p, stream);
    return launch_bulk<kWaitFirst>(p, stream);
  }
  const int64_t units = (p.total + 31) / 32;
  const unsigned grid = static_cast<unsigned>((units + kWarps - 1) / kWarps);
  return p.D == 128 ? launch_cpr<8>(p, grid, stream)
                    : launch_cpr<0>(p, grid, stream);
}

}  // namespace kvq
