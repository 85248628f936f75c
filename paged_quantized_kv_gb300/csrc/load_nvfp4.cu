// load_nvfp4.cu -- NVFP4 paged cache -> bf16 rows (the read side of the
// store), sm_103a.
//
// Operation: the pages written by reshape_and_cache_nvfp4 (vLLM
// csrc/libtorch_stable/nvfp4_kv_cache_kernels.cu, commit 7ce4c8e: page
// layout [K_data | K_scale | V_data | V_scale], HND/NHD strides, V scales
// swizzled inside each head's [block_size, S] tile) are read back for the
// tokens a block table names and dequantised.  The pages state no
// dequantisation rule; this takes the plain inverse of the store's:
// x' = bf16_rn(e2m1(q) * (float(sf) * k_scale)) -- the scale product and
// the element product are each one fp32 rounding, then round-to-nearest-even
// to bf16.  Output row cu_seq_lens[b] + p is token p of sequence b, read
// from page block_table[b, p / B], offset p % B.
//
// GB300 design: HBM-bound, 0.5625 B read and 2 B written per element.
//   * Persistent grid; every thread owns one fixed role -- two 16-element
//     groups of one side, 32 groups apart, so the per-row work (sequence
//     step, bounds checks, page addressing) is shared by 32 elements and
//     each warp store instruction writes 1 KB contiguous; output rows come in
//     chunks of kChunk row groups dealt round-robin to the CTAs, walked
//     kUnroll rows at a time (16 data bytes + 2 scale bytes each in flight
//     before any of them is used).
//   * cu_seq_lens and the block table are staged in shared memory once per
//     CTA (TMA bulk copies, shared with the indexer gather); a thread finds
//     its first row's sequence with one binary search and then only steps
//     it forward (its rows only increase), so row resolution costs a few
//     instructions per row.
//   * e2m1 -> f16x2 with cvt.rn.f16x2.e2m1x2 (exact), widened to fp32,
//     times the group's fp32 scale with mul.rn.f32x2, packed to bf16x2 with
//     cvt.rn.bf16x2.f32; each thread writes its group's 32 bytes with one
//     256-bit store when the rows are 32-byte aligned.
//   * KVQ_F_PDL / KVQ_F_PDL_EARLY_META as for the gather (the scales and the
//     cache are read only after the wait).
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

using namespace kvq::dev;

constexpr int kThreads = 256;
#ifndef KVQ_LOAD_UNROLL
#define KVQ_LOAD_UNROLL 4
#endif
#ifndef KVQ_LOAD_MIN_BLOCKS
#define KVQ_LOAD_MIN_BLOCKS 1
#endif
constexpr int kUnroll = KVQ_LOAD_UNROLL;
constexpr int kChunk = 16;  // row groups (tpp rows each) per chunk

__device__ __forceinline__ void ld_nc_8(const void* p, uint32_t& a,
                                        uint32_t& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(a), "=r"(b)
               : "l"(p));
}

__device__ __forceinline__ uint32_t ld_nc_u8(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// e4m3 code -> fp32 (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  float f;
  asm("{ .reg .f16 lo, hi;\n"
      "  mov.b32 {lo, hi}, %1;\n"
      "  cvt.f32.f16 %0, lo; }"
      : "=f"(f)
      : "r"(h2));
  return f;
}

// Four bytes of e2m1 pairs (element 2k in the low nibble of byte k) times c
// -> four bf16x2 words, element 2k in the low half of word k.
__device__ __forceinline__ void dequant4(uint32_t bytes, uint64_t cc,
                                         uint32_t (&out)[4]) {
  asm("{ .reg .b8 q0, q1, q2, q3;\n"
      "  .reg .b32 h0, h1, h2, h3;\n"
      "  .reg .f16 a0, b0, a1, b1, a2, b2, a3, b3;\n"
      "  .reg .f32 l0, u0, l1, u1, l2, u2, l3, u3;\n"
      "  .reg .b64 x0, x1, x2, x3;\n"
      "  mov.b32 {q0, q1, q2, q3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 h0, q0;  cvt.rn.f16x2.e2m1x2 h1, q1;\n"
      "  cvt.rn.f16x2.e2m1x2 h2, q2;  cvt.rn.f16x2.e2m1x2 h3, q3;\n"
      "  mov.b32 {a0, b0}, h0;  mov.b32 {a1, b1}, h1;\n"
      "  mov.b32 {a2, b2}, h2;  mov.b32 {a3, b3}, h3;\n"
      "  cvt.f32.f16 l0, a0;  cvt.f32.f16 u0, b0;\n"
      "  cvt.f32.f16 l1, a1;  cvt.f32.f16 u1, b1;\n"
      "  cvt.f32.f16 l2, a2;  cvt.f32.f16 u2, b2;\n"
      "  cvt.f32.f16 l3, a3;  cvt.f32.f16 u3, b3;\n"
      "  mov.b64 x0, {l0, u0};  mov.b64 x1, {l1, u1};\n"
      "  mov.b64 x2, {l2, u2};  mov.b64 x3, {l3, u3};\n"
      "  mul.rn.f32x2 x0, x0, %5;  mul.rn.f32x2 x1, x1, %5;\n"
      "  mul.rn.f32x2 x2, x2, %5;  mul.rn.f32x2 x3, x3, %5;\n"
      "  mov.b64 {l0, u0}, x0;  mov.b64 {l1, u1}, x1;\n"
      "  mov.b64 {l2, u2}, x2;  mov.b64 {l3, u3}, x3;\n"
      "  cvt.rn.bf16x2.f32 %0, u0, l0;  cvt.rn.bf16x2.f32 %1, u1, l1;\n"
      "  cvt.rn.bf16x2.f32 %2, u2, l2;  cvt.rn.bf16x2.f32 %3, u3, l3; }"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(bytes), "l"(cc));
}

template <bool kVec32>
__device__ __forceinline__ void store_group(uint16_t* p,
                                            const uint32_t (&w)[8]) {
  if constexpr (kVec32) {
    asm volatile(
        "st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
        "r"(w[6]), "r"(w[7])
        : "memory");
  } else {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p + 8),
                 "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  }
}

template <int kMode, bool kEarlyMeta, bool kVec32>
__global__ void __launch_bounds__(kThreads, KVQ_LOAD_MIN_BLOCKS)
load_nvfp4_kernel(const LoadParams p) {
  extern __shared__ __align__(16) uint8_t s_raw[];
  __shared__ __align__(8) uint64_t s_bar;

  if constexpr (!kEarlyMeta) pdl_prologue();
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
  if constexpr (kEarlyMeta) pdl_prologue();
  if (!staged) {
    if (threadIdx.x == 0 && p.dev_error != nullptr)
      atomicOr(p.dev_error, KVQ_DEVERR_TIMEOUT);
    return;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.dev_error != nullptr &&
      static_cast<int64_t>(cu[p.num_seqs]) != p.total)
    atomicOr(p.dev_error, KVQ_DEVERR_SEQ);

  // ---- this thread's fixed role inside a row ------------------------------
  // A thread owns two 16-element groups of one side, gA and gB = gA + P
  // (P = 32 when the side has a multiple of 64 groups, else half the side),
  // so each of a warp's two 256-bit store instructions writes one contiguous
  // run of 32 groups' output (1 KB).
  const int tid = threadIdx.x;
  const int slices = 1 << p.slices_log2;
  int unit_in_tok, tok_sub;
  if (slices == 1) {
    tok_sub = tid / p.upt;
    unit_in_tok = tid - tok_sub * p.upt;
  } else {
    tok_sub = 0;
    unit_in_tok = (static_cast<int>(blockIdx.x) & (slices - 1)) * kThreads + tid;
  }
  if (tok_sub >= p.tpp || unit_in_tok >= p.upt) return;  // idle role
  const int ups = p.upt >> 1;  // units per side
  const int side = unit_in_tok >= ups ? 1 : 0;
  const int i = unit_in_tok - side * ups;
  const int gps = 2 * ups;  // groups per side
  const int P = (gps % 64 == 0) ? 32 : ups;
  const int gA = (i / P) * 2 * P + (i % P);
  const int gB = gA + P;
  const int headA = gA / p.S, jA = gA - headA * p.S;
  const int headB = gB / p.S, jB = gB - headB * p.S;
  const int q = p.S >> 2;
  const bool swz = (p.swizzle_sides >> side) & 1u;

  const uint8_t* const side_base = p.side[side];
  const uint8_t* const data_roleA = side_base + headA * p.dhs + jA * 8;
  const uint8_t* const data_roleB = side_base + headB * p.dhs + jB * 8;
  const uint8_t* const scale_side = side_base + p.data_per_side;
  const uint8_t* const scale_roleA =
      scale_side + headA * p.shs +
      (swz ? (jA / q) * p.sts + (jA % q) * 4 : static_cast<int64_t>(jA));
  const uint8_t* const scale_roleB =
      scale_side + headB * p.shs +
      (swz ? (jB / q) * p.sts + (jB % q) * 4 : static_cast<int64_t>(jB));
  uint16_t* const out_roleA = p.out[side] + headA * p.D + jA * 16;
  uint16_t* const out_roleB = p.out[side] + headB * p.D + jB * 16;
  const float kscale = __ldg(p.scale[side]);

  // ---- rows: small contiguous chunks dealt round-robin to CTAs -----------
  // Within a chunk a thread's rows advance by tpp; across chunks they jump
  // forward by the grid's span.  The thread finds its first row's sequence
  // with one binary search and afterwards only steps the sequence forward,
  // while the round-robin deal keeps every SM's share spread over the
  // whole output (balanced across SMs and memory partitions).
  const int64_t T = p.total;
  const int64_t tgroups = (T + p.tpp - 1) / p.tpp;
  const int64_t nchunks = (tgroups + kChunk - 1) / kChunk;
  const int64_t cstride = gridDim.x >> p.slices_log2;
  const int64_t c_first = blockIdx.x >> p.slices_log2;
  const int n = p.num_seqs;
  int b = c_first < nchunks
              ? find_seq<kMode != kMetaGlobal>(
                    cu, n, c_first * kChunk * p.tpp + tok_sub)
              : n;
  int64_t seq_lo = b < n ? cu[b] : 0;
  int64_t seq_hi = b < n ? cu[b + 1] : 0;
  const int64_t tstep = p.tpp;

  for (int64_t c = c_first; c < nchunks; c += cstride) {
   int64_t row_hi = (c + 1) * kChunk * p.tpp;
   if (row_hi > T) row_hi = T;
   for (int64_t t0 = c * kChunk * p.tpp + tok_sub; t0 < row_hi;
        t0 += kUnroll * tstep) {
    uint4 d[kUnroll];
    uint32_t sf0[kUnroll], sf1[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t row = t0 + u * tstep;
      ok[u] = false;
      d[u] = make_uint4(0u, 0u, 0u, 0u);
      sf0[u] = sf1[u] = 0u;
      if (row >= row_hi) continue;
      while (b < n && row >= seq_hi) {  // next non-empty sequence
        ++b;
        seq_lo = seq_hi;
        if (b < n) seq_hi = cu[b + 1];
      }
      int err = 0;
      if (b >= n) {
        err = KVQ_DEVERR_SEQ;  // no sequence covers this row
      } else {
        const int64_t pos = row - seq_lo;
        int64_t kb, off;
        if (p.b_shift >= 0) {
          kb = pos >> p.b_shift;
          off = pos & (p.B - 1);
        } else {
          kb = pos / p.B;
          off = pos - kb * p.B;
        }
        if (pos < 0 || kb >= p.max_blocks) {
          err = KVQ_DEVERR_SEQ;
        } else {
          const int64_t blk =
              kMode == kMetaSharedCuBt
                  ? s_bt[b * p.max_blocks + kb]
                  : __ldg(p.block_table + b * p.bt_stride + kb);
          if (blk < 0 || blk >= p.num_blocks) {
            err = KVQ_DEVERR_BLOCK;
          } else {
            const int64_t page = blk * p.page_stride;
            const int64_t doff = page + off * p.dts;
            ld_nc_8(data_roleA + doff, d[u].x, d[u].y);
            ld_nc_8(data_roleB + doff, d[u].z, d[u].w);
            const int64_t soff =
                page + (swz ? (off & ~int64_t{3}) * p.sts + (off & 3)
                            : off * p.sts);
            sf0[u] = ld_nc_u8(scale_roleA + soff);
            sf1[u] = ld_nc_u8(scale_roleB + soff);
            ok[u] = true;
          }
        }
      }
      if (err != 0 && p.dev_error != nullptr && i == 0)
        atomicOr(p.dev_error, err);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (!ok[u]) continue;
      const int64_t orow = (t0 + u * tstep) * p.out_stride0;
      const float c0 = __fmul_rn(e4m3_value(sf0[u]), kscale);
      const float c1 = __fmul_rn(e4m3_value(sf1[u]), kscale);
      const uint64_t cc0 =
          (static_cast<uint64_t>(__float_as_uint(c0)) << 32) |
          __float_as_uint(c0);
      const uint64_t cc1 =
          (static_cast<uint64_t>(__float_as_uint(c1)) << 32) |
          __float_as_uint(c1);
      uint32_t w[8];
      uint32_t a[4], b2[4];
      dequant4(d[u].x, cc0, a);
      dequant4(d[u].y, cc0, b2);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[k] = a[k];
        w[4 + k] = b2[k];
      }
      store_group<kVec32>(out_roleA + orow, w);
      dequant4(d[u].z, cc1, a);
      dequant4(d[u].w, cc1, b2);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[k] = a[k];
        w[4 + k] = b2[k];
      }
      store_group<kVec32>(out_roleB + orow, w);
    }
   }
  }
}

template <int kMode, bool kEarlyMeta, bool kVec32>
cudaError_t launch_variant(const LoadParams& p, size_t smem,
                           cudaStream_t stream) {
  static int ctas_per_sm[64] = {0};  // register-limited, per device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int& occ_regs = ctas_per_sm[dev & 63];
  if (occ_regs == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ_regs, load_nvfp4_kernel<kMode, kEarlyMeta, kVec32>, kThreads,
        0);
    if (err != cudaSuccess) return err;
    if (occ_regs < 1) occ_regs = 1;
  }
  // shared-memory limit for this launch's metadata (228 KB per SM, 1 KB
  // reserved per CTA)
  int occ = occ_regs;
  const int by_smem = static_cast<int>((228 * 1024) / (smem + 1024 + 64));
  if (by_smem < occ) occ = by_smem < 1 ? 1 : by_smem;
  const int slices = 1 << p.slices_log2;
  int64_t grid = static_cast<int64_t>(sm_count()) * occ;
  if (grid > p.num_passes) grid = p.num_passes;
  grid = (grid / slices) * slices;
  if (grid < slices) grid = slices;
  return launch_kernel(load_nvfp4_kernel<kMode, kEarlyMeta, kVec32>,
                       static_cast<unsigned>(grid), kThreads, smem, stream,
                       p.pdl, p);
}

template <bool kEarlyMeta, bool kVec32>
cudaError_t launch_mode(const LoadParams& p, cudaStream_t stream) {
  const int64_t ncu = static_cast<int64_t>(p.num_seqs) + 1;
  const int64_t nbt = static_cast<int64_t>(p.num_seqs) * p.max_blocks;
  const size_t both = region_bytes(ncu) + region_bytes(nbt);
  if (p.bt_stride == p.max_blocks && both <= kMaxMetaSmem)
    return launch_variant<kMetaSharedCuBt, kEarlyMeta, kVec32>(p, both,
                                                               stream);
  if (region_bytes(ncu) <= kMaxMetaSmem)
    return launch_variant<kMetaSharedCu, kEarlyMeta, kVec32>(
        p, region_bytes(ncu), stream);
  return launch_variant<kMetaGlobal, kEarlyMeta, kVec32>(p, 0, stream);
}

}  // namespace

cudaError_t launch_load_nvfp4(const LoadParams& p, cudaStream_t stream) {
  // 256-bit stores need every group start 32-byte aligned
  const bool vec32 = (reinterpret_cast<uintptr_t>(p.out[0]) % 32 == 0) &&
                     (reinterpret_cast<uintptr_t>(p.out[1]) % 32 == 0) &&
                     (p.out_stride0 % 16 == 0);
  if (p.early_meta)
    return vec32 ? launch_mode<true, true>(p, stream)
                 : launch_mode<true, false>(p, stream);
  return vec32 ? launch_mode<false, true>(p, stream)
               : launch_mode<false, false>(p, stream);
}

}  // namespace kvq
