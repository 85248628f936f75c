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
// time is dominated by the dependent-load chain before the first row load
// (cu_seq_lens -> block_table -> K rows), since the whole grid fits in one
// wave.  Each CTA first stages cu_seq_lens -- and, when it is contiguous
// and fits, the used block table -- in shared memory with one batch of
// coalesced loads (48 KB at most; otherwise the reads go to global memory),
// so the per-row binary search and the block lookup cost one memory round
// trip together instead of one per search level plus one.  One warp owns 32 consecutive output rows: lane l
// resolves row r0 + l (search, one block-table read, bounds checks), then the
// warp moves the 32 rows as 16-byte vectors -- every load of a unit issued
// before its stores, 32 x D bytes in flight per warp -- and each lane copies
// its row's 4 scale bytes.  Destination rows are contiguous, so every store
// is a full sector.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

#ifndef KVQ_GATHER_THREADS
#define KVQ_GATHER_THREADS 256
#endif
constexpr int kThreads = KVQ_GATHER_THREADS;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_nc_16(const void* p) {
  uint4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st_16(void* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
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

// int32 metadata entries staged in shared memory at most (48 KB, no opt-in).
constexpr int kMaxSharedInts = 12288;
constexpr int kStageBatch = 16;

// Where the kernel reads its metadata from.
enum MetaMode {
  kMetaGlobal = 0,       // cu_seq_lens and block_table from global memory
  kMetaSharedCu = 1,     // cu_seq_lens staged in shared memory
  kMetaSharedCuBt = 2    // cu_seq_lens and the (contiguous) block table
};

// Copy int32 ranges a[0, na) and b[0, nb) into dst[0, na + nb): every load
// of a batch is issued before its stores, so both ranges arrive in about
// one memory round trip.
__device__ __forceinline__ void stage_meta(int32_t* dst, const int32_t* a,
                                           int na, const int32_t* b,
                                           int nb) {
  const int total = na + nb;
  for (int base = threadIdx.x; base < total; base += kThreads * kStageBatch) {
    int32_t v[kStageBatch];
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const int i = base + k * kThreads;
      v[k] = 0;
      if (i < na)
        v[k] = __ldg(a + i);
      else if (i < total)
        v[k] = __ldg(b + (i - na));
    }
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const int i = base + k * kThreads;
      if (i < total) dst[i] = v[k];
    }
  }
}

// CPR = 16-byte chunks per K row (head_dim / 16); 0 = runtime value.
template <int CPR, int kMode>
__global__ void __launch_bounds__(kThreads)
gather_indexer_k_kernel(const GatherParams p) {
  extern __shared__ int32_t s_meta[];
  pdl_prologue();
  const int32_t* cu = p.cu;
  const int32_t* s_bt = nullptr;
  if constexpr (kMode != kMetaGlobal) {
    const int ncu = p.num_seqs + 1;
    const int nbt =
        kMode == kMetaSharedCuBt ? p.num_seqs * p.max_blocks : 0;
    stage_meta(s_meta, p.cu, ncu, p.block_table, nbt);
    __syncthreads();
    cu = s_meta;
    s_bt = s_meta + ncu;
  }
  const int lane = threadIdx.x & 31;
  const int64_t unit =
      static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t r0 = unit * 32;
  if (r0 >= p.total) return;  // whole warp leaves together

  if (unit == 0 && lane == 0 && p.dev_error != nullptr &&
      static_cast<int64_t>(cu[p.num_seqs]) != p.total)
    atomicOr(p.dev_error, KVQ_DEVERR_SEQ);

  // ---- resolve this lane's row ----------------------------------------
  const int64_t r = r0 + lane;
  const uint8_t* src_row = nullptr;
  const uint8_t* src_scale = nullptr;
  if (r < p.total) {
    const int b = find_seq<kMode != kMetaGlobal>(cu, p.num_seqs, r);
    int err = 0;
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
    if (err != 0 && p.dev_error != nullptr) atomicOr(p.dev_error, err);
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

template <int CPR>
cudaError_t launch_cpr(const GatherParams& p, unsigned grid,
                       cudaStream_t stream) {
  const int64_t ncu = static_cast<int64_t>(p.num_seqs) + 1;
  const int64_t nbt = static_cast<int64_t>(p.num_seqs) * p.max_blocks;
  if (p.bt_stride == p.max_blocks && ncu + nbt <= kMaxSharedInts) {
    const size_t smem = static_cast<size_t>(ncu + nbt) * sizeof(int32_t);
    return launch_kernel(gather_indexer_k_kernel<CPR, kMetaSharedCuBt>, grid,
                         kThreads, smem, stream, p.pdl, p);
  }
  if (ncu <= kMaxSharedInts) {
    const size_t smem = static_cast<size_t>(ncu) * sizeof(int32_t);
    return launch_kernel(gather_indexer_k_kernel<CPR, kMetaSharedCu>, grid,
                         kThreads, smem, stream, p.pdl, p);
  }
  return launch_kernel(gather_indexer_k_kernel<CPR, kMetaGlobal>, grid,
                       kThreads, 0, stream, p.pdl, p);
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
