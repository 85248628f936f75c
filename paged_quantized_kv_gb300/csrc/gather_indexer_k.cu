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

cudaError_t launch_gather_indexer_k(const GatherParams& p,
                                    cudaStream_t stream) {
  const int64_t units = (p.total + 31) / 32;
  const unsigned grid = static_cast<unsigned>((units + kWarps - 1) / kWarps);
  return p.D == 128 ? launch_cpr<8>(p, grid, stream)
                    : launch_cpr<0>(p, grid, stream);
}

}  // namespace kvq
