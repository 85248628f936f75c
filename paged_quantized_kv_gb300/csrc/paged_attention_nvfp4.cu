// paged_attention_nvfp4.cu -- paged decode attention over the NVFP4 KV
// cache, sm_103a, on the 5th-generation tensor cores.
//
// Operation: the paged_attention op of vLLM PR #12348 "[ROCm] Faster Custom
// Paged Attention kernels" (out, exp_sums, max_logits, tmp_out, query,
// key_cache, value_cache, num_kv_heads, scale, block_tables, context_lens,
// block_size, max_context_len, k_scale, v_scale, partition_size), read over
// the NVFP4 pages of vLLM nvfp4_kv_cache_kernels.cu (commit 7ce4c8e).  For
// sequence b (one query token) and query head h, KV head h / G:
//   out[b, h] = sum_t softmax_t(scale * q . K^[t]) V^[t],
//   K^ = e2m1(code) * float(sf) * k_scale  (V^ with v_scale),
// over the first context_lens[b] tokens.  A context longer than one
// partition is split: each (sequence, KV head, partition) CTA writes the
// partition's max logit, exp-sum and normalised output to the caller's
// scratch, and a second small kernel merges the partitions.
//
// This file holds the two tcgen05 kernels (KVQ_F_ATTN_TCGEN05 and
// KVQ_F_ATTN_PIPELINED) and the partition merge; the default kernel, on
// warp-level MMAs, is in paged_attention_mma.cu.
//
// GB300 design -- one CTA of 4 warps per (partition of <= 512 tokens, KV
// head, sequence), 3 CTAs per SM (56 KB of shared memory, 128 TMEM columns
// each):
//   * Every thread owns one token of a 128-token tile and reads its 64 data
//     bytes and 8 scale bytes straight from HBM into registers, two tiles
//     ahead of their use (measured: two tiles in flight at 3 CTAs/SM beat
//     one tile at 4 CTAs/SM by 16 %, and three tiles at 2 CTAs/SM).  K
//     tiles, then V tiles, stream through one shared-memory operand buffer.
//   * e2m1 -> fp16 with cvt.rn.f16x2.e2m1x2, times the group's e4m3 scale
//     (cvt.rn.f16x2.e4m3x2) with one packed multiply: e2m1 * sf has at most
//     6 significant bits and lies in [2^-10, 2688], so the fp16 operand is
//     exact.  k_scale and v_scale are applied to the fp32 results.
//   * tcgen05.mma kind::f16 with fp32 accumulators in tensor memory, issued
//     by one thread and tracked by tcgen05.commit on an mbarrier:
//       S^T[128 tokens x 16] = K'[128 x 128] . Q'^T   (K-major operands;
//                              the group's G <= 16 query heads on N)
//       O^T[128 dims x 16]  += V'^T . P^T            (MN-major operands:
//                              V' is read in the layout it was written in)
//     Operands use the no-swizzle canonical layout (8 rows x 16 bytes core
//     matrices); every thread's 16-byte stores into it are conflict-free.
//   * The whole partition's logits stay in tensor memory (16 columns per
//     tile), so the softmax max is exact before any P.V product and the
//     output accumulator is never rescaled.  P is rounded to fp16 and the
//     denominator sums the rounded values (the weights sum to one).
//   * Every mbarrier wait is bounded (KVQ_DEVERR_TIMEOUT); on a timeout the
//     CTA waits once more, frees its tensor memory and writes nothing.
// KVQ_F_ATTN_PIPELINED selects the persistent, warp-specialised kernel
// further down instead (same contract).  Measured on GB300, the per-CTA one
// is the faster of the two: per 128-token tile a single thread's 8
// tcgen05.mma issues cost ~750 cycles and each mbarrier test ~300, which
// several independent CTAs per SM hide better than one pipelined CTA does.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

using namespace kvq::dev;

constexpr int kThreads = 128;
constexpr int kTile = 128;                          // tokens per MMA tile
constexpr int kD = 128;                             // head_size
constexpr int kMaxTiles = 4;                        // partition <= 512
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kOCol = 64;                      // O^T at columns 64..79
constexpr int kKVBytes = kTile * kD * 2;            // K' or V' tile, fp16
constexpr int kPGroup = kMaxTiles * kTile * 8 * 2;  // P^T, one 8-head group
constexpr int kPBytes = 2 * kPGroup;
constexpr int kQBytes = 16 * kD * 2;                // Q' [16 x 128] fp16
constexpr int kRedFloats = 2 * 4 * 16;
constexpr int kSmemBytes = kKVBytes + kPBytes + kQBytes + kRedFloats * 4 + 16;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// tcgen05 / shared-memory helpers
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor, no-swizzle canonical layout: `lbo` is the
// byte distance between core matrices adjacent along K, `sbo` along M / N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo,
                                              uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) |
         (uint64_t{1} << 46);  // descriptor version; base offset 0, no swizzle
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, M = 128, N = 16.
__host__ __device__ constexpr uint32_t instr_desc(bool a_mn, bool b_mn) {
  return (1u << 4) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u) |
         ((16u >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a,
                                        uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64"
      " [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Columns [col, col + N) of this warp's 32 TMEM lanes, one lane per thread.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t addr, float (&v)[N]) {
  uint32_t r[N];
  if constexpr (N == 4) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(addr));
  } else if constexpr (N == 8) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(addr));
  } else {
    static_assert(N == 16, "4, 8 or 16 columns");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
          "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(addr));
  }
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a,
                                             uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b,
                                         uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two e4m3 codes (low byte first) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair) {
  uint32_t h;
  const uint16_t in = static_cast<uint16_t>(pair & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
  return h;
}

// Four bytes of e2m1 pairs (element 2k in the low nibble of byte k) times
// the f16x2 scale `sf2` -> four f16x2 words, element 2k in the low half.
// Exact: the products have at most 6 significant bits.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t sf2,
                                             uint32_t (&o)[4]) {
  asm("{ .reg .b8 q0, q1, q2, q3;\n"
      "  .reg .b32 h0, h1, h2, h3;\n"
      "  mov.b32 {q0, q1, q2, q3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 h0, q0;  cvt.rn.f16x2.e2m1x2 h1, q1;\n"
      "  cvt.rn.f16x2.e2m1x2 h2, q2;  cvt.rn.f16x2.e2m1x2 h3, q3;\n"
      "  mul.rn.f16x2 %0, h0, %5;  mul.rn.f16x2 %1, h1, %5;\n"
      "  mul.rn.f16x2 %2, h2, %5;  mul.rn.f16x2 %3, h3, %5; }"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w), "r"(sf2));
}

// Two fp32 -> f16x2, round to nearest even; `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  return h;
}

__device__ __forceinline__ void unpack_f16x2(uint32_t h, float& lo,
                                             float& hi) {
  asm("{ .reg .f16 a, b;\n"
      "  mov.b32 {a, b}, %2;\n"
      "  cvt.f32.f16 %0, a;\n"
      "  cvt.f32.f16 %1, b; }"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
}

// bf16x2 -> f16x2 (round to nearest; exact for bf16 values inside the fp16
// normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16),
                    __uint_as_float(w & 0xFFFF0000u));
}

template <bool kF16>
__device__ __forceinline__ uint16_t float_to_out(float f) {
  uint16_t h;
  if constexpr (kF16)
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(f));
  else
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// ---------------------------------------------------------------------------
// One token's raw NVFP4 bytes of one side
// ---------------------------------------------------------------------------
struct Raw {
  uint4 d[4];     // 64 data bytes: group j in bytes 8j .. 8j+7
  uint32_t s[8];  // linear: s[0..1] = the 8 scale bytes; swizzled: the
                  // token's 4-row band, scale j = byte (off % 4) of s[j]
  uint32_t r;     // off % 4
  int ok;         // token inside the context with a valid block id
};

__device__ __forceinline__ void load_raw(const AttnParams& p, int b, int kh,
                                         int t, int t_end, bool is_v,
                                         Raw& raw) {
  raw.ok = 0;
  if (t >= t_end) return;
  const int idx = p.b_shift >= 0 ? (t >> p.b_shift) : t / p.B;
  const int32_t blk = __ldg(p.block_table + b * p.bt_stride + idx);
  if (blk < 0 || blk >= p.num_blocks) {
    if (p.dev_error != nullptr) atomicOr(p.dev_error, KVQ_DEVERR_BLOCK);
    return;
  }
  const int off = t - idx * p.B;
  const uint8_t* page =
      p.side[is_v ? 1 : 0] + static_cast<int64_t>(blk) * p.page_stride;
  const uint8_t* dp = page + kh * p.dhs + off * p.dts;
#pragma unroll
  for (int c = 0; c < 4; ++c) raw.d[c] = ld_nc_v4(dp + 16 * c);
  const uint8_t* sp = page + p.scale_off + kh * p.shs;
  if (!is_v && !p.swizzle_k) {
    const uint2 w = ld_nc_v2(sp + off * p.sts);
    raw.s[0] = w.x;
    raw.s[1] = w.y;
  } else {
    const uint8_t* band = sp + (off & ~3) * p.sts;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const uint2 w = ld_nc_v2(band + a * p.sts);
      raw.s[2 * a] = w.x;
      raw.s[2 * a + 1] = w.y;
    }
  }
  raw.r = static_cast<uint32_t>(off & 3);
  raw.ok = 1;
}

// Convert one token row into the operand buffer: K' (K-major A operand,
// row = token) or V' (MN-major A operand of O^T, K = token).  Chunk c holds
// dims 8c .. 8c+7.
__device__ __forceinline__ void convert_raw(const Raw& raw, bool linear,
                                            uint32_t base, uint32_t cstride) {
  if (!raw.ok) {
#pragma unroll
    for (int c = 0; c < 16; ++c) st_shared_v4(base + c * cstride, 0, 0, 0, 0);
    return;
  }
  const uint32_t sel = raw.r | ((raw.r + 4u) << 4);
#pragma unroll
  for (int m = 0; m < 4; ++m) {  // groups 2m and 2m+1
    uint32_t pair;
    if (linear)
      pair = (m & 1) ? (raw.s[m >> 1] >> 16) : raw.s[m >> 1];
    else
      pair = prmt(raw.s[2 * m], raw.s[2 * m + 1], sel);
    const uint32_t sf = e4m3x2_to_f16x2(pair);
    const uint32_t sf_even = prmt(sf, sf, 0x1010u);
    const uint32_t sf_odd = prmt(sf, sf, 0x3232u);
    uint32_t o[4];
    dequant_word(raw.d[m].x, sf_even, o);
    st_shared_v4(base + (4 * m + 0) * cstride, o[0], o[1], o[2], o[3]);
    dequant_word(raw.d[m].y, sf_even, o);
    st_shared_v4(base + (4 * m + 1) * cstride, o[0], o[1], o[2], o[3]);
    dequant_word(raw.d[m].z, sf_odd, o);
    st_shared_v4(base + (4 * m + 2) * cstride, o[0], o[1], o[2], o[3]);
    dequant_word(raw.d[m].w, sf_odd, o);
    st_shared_v4(base + (4 * m + 3) * cstride, o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------------------
// Main kernel: one (partition, KV head, sequence) per CTA
// ---------------------------------------------------------------------------
template <int NG, bool kF16>
__global__ void __launch_bounds__(kThreads, 3)
paged_attention_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* kv_s = smem;
  uint8_t* p_s = smem + kKVBytes;
  uint8_t* q_s = p_s + kPBytes;
  float* red = reinterpret_cast<float*>(q_s + kQBytes);  // [2][4 warps][16]
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + kRedFloats);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int part = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
  pdl_prologue();

  int L = __ldg(p.lens + b);
  if (L < 0 || L > p.len_cap) {
    if (p.dev_error != nullptr && part == 0 && kh == 0 && tid == 0)
      atomicOr(p.dev_error, KVQ_DEVERR_SEQ);
    L = L < 0 ? 0 : p.len_cap;
  }
  const int p0 = part * p.part;
  if (p0 >= L) {
    if (part == 0) {  // empty context: the output is zero
      for (int i = tid; i < p.G * kD; i += kThreads)
        p.out[b * p.out_stride0 + (kh * p.G) * kD + i] = 0;
    }
    return;
  }
  const int ntok = min(p.part, L - p0);
  const int ntiles = (ntok + kTile - 1) / kTile;
  const int nparts = (L + p.part - 1) / p.part;
  const int t_end = p0 + ntok;

  // the first two tiles' loads go out before the set-up work; every later
  // tile's loads are issued two tiles ahead of its use
  Raw cur, nxt, nx2;
  load_raw(p, b, kh, p0 + tid, t_end, false, cur);
  if (2 * ntiles > 1) {
    const bool nv = ntiles == 1;  // tile 1 is V tile 0 of a 1-tile unit
    load_raw(p, b, kh, p0 + (nv ? 0 : 1) * kTile + tid, t_end, nv, nxt);
  }

  if (warp == 0) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
        ::"r"(smem_addr(slot)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  const uint32_t bar_a = smem_addr(bar);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_a));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // Q' [16 x 128] fp16, K-major: row n = query head kh*G + n (zero n >= G)
  const uint32_t q_a = smem_addr(q_s), p_a = smem_addr(p_s),
                 kv_a = smem_addr(kv_s);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = tid + kThreads * i;
    const int n = c >> 4, kc = c & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < p.G) {
      v = *reinterpret_cast<const uint4*>(
          p.q + b * p.q_stride0 + (kh * p.G + n) * kD + kc * 8);
      if constexpr (!kF16) {
        v.x = bf16x2_to_f16x2(v.x);
        v.y = bf16x2_to_f16x2(v.y);
        v.z = bf16x2_to_f16x2(v.z);
        v.w = bf16x2_to_f16x2(v.w);
      }
    }
    st_shared_v4(q_a + (n >> 3) * 2048 + kc * 128 + (n & 7) * 16, v.x, v.y,
                 v.z, v.w);
  }
  if constexpr (NG == 8) {  // heads 8..15 of P^T stay zero
#pragma unroll
    for (int i = 0; i < 4; ++i)
      st_shared_v4(p_a + kPGroup + (tid * 4 + i) * 16, 0, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  float m[NG], l[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) { m[g] = 0.f; l[g] = 0.f; }
  const float k_scale = __ldg(p.k_scale);
  const int nu = 2 * ntiles;
  bool bad = false;
  uint32_t kvalid = 0;  // bit i: this thread's token of K tile i is usable
  for (int u = 0; u < nu; ++u) {
    const bool is_v = u >= ntiles;
    const int tile = is_v ? u - ntiles : u;
    if (u + 2 < nu) {
      const bool nv = u + 2 >= ntiles;
      const int nt = nv ? u + 2 - ntiles : u + 2;
      load_raw(p, b, kh, p0 + nt * kTile + tid, t_end, nv, nx2);
    }
    if (u > 0 && !mbar_wait(bar_a, (u - 1) & 1)) bad = true;
    if (__syncthreads_or(bad)) break;

    if (u == ntiles) {
      // ---- softmax over the partition's logits -------------------------
      tc_fence_after();
      float x[kMaxTiles][NG];
#pragma unroll
      for (int i = 0; i < kMaxTiles; ++i)
        if (i < ntiles) tmem_ld<NG>(tmem + lane_base + 16 * i, x[i]);
      tmem_wait_ld();
      const float c2 = p.scale * k_scale * kLog2e;
#pragma unroll
      for (int i = 0; i < kMaxTiles; ++i) {
        const bool valid = i < ntiles && ((kvalid >> i) & 1u);
#pragma unroll
        for (int g = 0; g < NG; ++g)
          x[i][g] = valid ? x[i][g] * c2 : -INFINITY;
      }
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        float v = x[0][g];
#pragma unroll
        for (int i = 1; i < kMaxTiles; ++i) v = fmaxf(v, x[i][g]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
          v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
        m[g] = v;
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < NG; ++g) red[warp * 16 + g] = m[g];
      }
      __syncthreads();
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        float v = fmaxf(fmaxf(red[g], red[16 + g]),
                        fmaxf(red[32 + g], red[48 + g]));
        m[g] = v == -INFINITY ? 0.f : v;
      }
#pragma unroll
      for (int i = 0; i < kMaxTiles; ++i) {
        if (i >= ntiles) break;
        uint32_t h[NG / 2];
#pragma unroll
        for (int g = 0; g < NG; g += 2) {
          h[g / 2] = pack_f16x2(ex2(x[i][g] - m[g]),
                                ex2(x[i][g + 1] - m[g + 1]));
          float lo, hi;
          unpack_f16x2(h[g / 2], lo, hi);
          l[g] += lo;
          l[g + 1] += hi;
        }
        const uint32_t row = p_a + (i * 16 + (tid >> 3)) * 128 + (tid & 7) * 16;
        st_shared_v4(row, h[0], h[1], h[2], h[3]);
        if constexpr (NG == 16)
          st_shared_v4(row + kPGroup, h[4], h[5], h[6], h[7]);
      }
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        float v = l[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
          v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        l[g] = v;
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < NG; ++g) red[64 + warp * 16 + g] = l[g];
      }
      __syncthreads();
#pragma unroll
      for (int g = 0; g < NG; ++g)
        l[g] = (red[64 + g] + red[80 + g]) + (red[96 + g] + red[112 + g]);
    }

    // ---- this tile's operand: K' (row = token) or V' (K = token) --------
    const uint32_t tbase =
        is_v ? kv_a + (tid >> 3) * 128 + (tid & 7) * 16
             : kv_a + (tid >> 3) * 2048 + (tid & 7) * 16;
    convert_raw(cur, !is_v && !p.swizzle_k, tbase, is_v ? 2048u : 128u);
    if (!is_v) kvalid |= static_cast<uint32_t>(cur.ok) << tile;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      if (!is_v) {
        constexpr uint32_t id = instr_desc(false, false);
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)
          mma_f16(tmem + 16 * tile, smem_desc(kv_a + s * 256, 128, 2048),
                  smem_desc(q_a + s * 256, 128, 2048), id, s > 0);
      } else {
        constexpr uint32_t id = instr_desc(true, true);
#pragma unroll
        for (int s = 0; s < kTile / 16; ++s)
          mma_f16(tmem + kOCol, smem_desc(kv_a + s * 256, 128, 2048),
                  smem_desc(p_a + (16 * tile + 2 * s) * 128, 128, kPGroup),
                  id, (tile > 0 || s > 0) ? 1u : 0u);
      }
      mma_commit(bar_a);
    }
    cur = nxt;
    nxt = nx2;
  }

  // ---- output ----------------------------------------------------------
  if (!bad && !mbar_wait(bar_a, (nu - 1) & 1)) bad = true;
  if (__syncthreads_or(bad)) {
    if (p.dev_error != nullptr && tid == 0)
      atomicOr(p.dev_error, KVQ_DEVERR_TIMEOUT);
    mbar_wait(bar_a, (nu - 1) & 1);  // give in-flight MMAs one more chance
  } else {
    tc_fence_after();
    float o[NG];
    tmem_ld<NG>(tmem + lane_base + kOCol, o);
    tmem_wait_ld();
    const int d = tid;
    if (nparts == 1) {
      const float v_scale = __ldg(p.v_scale);
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (g < p.G) {
          const float y = l[g] > 0.f ? o[g] * (1.0f / l[g]) * v_scale : 0.f;
          p.out[b * p.out_stride0 + (kh * p.G + g) * kD + d] =
              float_to_out<kF16>(y);
        }
      }
    } else {
      const int64_t row0 =
          (static_cast<int64_t>(b) * p.Hq + kh * p.G) * p.max_parts + part;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        if (g < p.G) {
          const int64_t r = row0 + static_cast<int64_t>(g) * p.max_parts;
          p.tmp_out[r * kD + d] = l[g] > 0.f ? o[g] * (1.0f / l[g]) : 0.f;
          if (tid == g) {
            p.max_logits[r] = m[g];
            p.exp_sums[r] = l[g];
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(tmem), "r"(kTmemCols));
}

// ---------------------------------------------------------------------------
// Pipelined kernel: one persistent CTA per SM, 8 converter warps and one MMA
// warp.
//
// Converters (256 threads, two per token of a 128-token tile: dims 0..63
// and 64..127) walk this CTA's work units tile by tile -- the unit's K
// tiles, then its V tiles -- and for each tile
//   * copy their own half row (32 code bytes, the 4 scale bytes or the 16
//     band bytes) global -> shared with cp.async, kDepth tiles ahead, into
//     a private slot (each thread reads back only what it copied, so the
//     slots need no barrier and their reads are conflict-free); the
//     block-table entry of a tile is fetched the same way kDepth tiles
//     before its data;
//   * dequantise the half row and write K' into tensor memory (tcgen05.st,
//     lane = token: the MMA reads its A operand there) or V' into one of two
//     shared-memory buffers (MN-major A operand of O^T = V'^T . P^T);
//   * arrive on the buffer's "ready" mbarrier.
// The MMA warp waits for "ready", issues the tile's MMAs from one thread and
// commits them to the buffer's "done" mbarrier, which the converters wait
// on before reusing the buffer, before the softmax (last K tile) and before
// the output (last V tile).  Softmax and output are split by head columns:
// warps 0..3 take the first half, warps 4..7 the second.
// Context lengths are staged in shared memory once; a unit's query rows are
// loaded while the previous unit runs.  Every wait is bounded; after a
// timeout the CTA stops waiting, still walks its units to the end (so every
// barrier is reached), writes no output and flags KVQ_DEVERR_TIMEOUT.
// ---------------------------------------------------------------------------
constexpr int kDepth = 6;            // tiles in flight per thread
constexpr int kConsumers = 256;
constexpr int kPipeThreads = kConsumers + 32;
constexpr int kMaxLensSmem = 4096;   // context lengths staged when they fit
constexpr uint32_t kPipeTmemCols = 256;  // S 0..63, O 64..79, K' 128..255
constexpr uint32_t kKCol = 128;
constexpr int kSlotBytes = 3 * kConsumers * 16;          // one tile, 12 KB
constexpr int kOffSlots = 0;
constexpr int kOffBt = kOffSlots + kDepth * kSlotBytes;  // [2*kDepth][256]
constexpr int kOffV = kOffBt + 2 * kDepth * kConsumers * 4;
constexpr int kOffP = kOffV + 2 * kKVBytes;
constexpr int kOffQ = kOffP + kPBytes;
constexpr int kOffLens = kOffQ + kQBytes;
constexpr int kOffRed = kOffLens + kMaxLensSmem * 4;     // [2][8 warps][8]
constexpr int kOffBar = kOffRed + 2 * 8 * 8 * 4;         // ready[2], done[2]
constexpr int kOffSlot = kOffBar + 4 * 8;
constexpr int kOffAbort = kOffSlot + 4;
constexpr int kPipeSmem = kOffAbort + 4;
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kOffV % 1024 == 0, "operand alignment");

struct Unit {
  int b, kh, part, L, p0, ntok, nt;
};

// Work unit u (partition fastest, then KV head, then sequence); false when
// the partition starts past the (clamped) context.
__device__ __forceinline__ bool unit_at(const AttnParams& p,
                                        const int32_t* lens, int u, Unit& w) {
  w.part = u % p.max_parts;
  const int r = u / p.max_parts;
  w.kh = r % p.Hkv;
  w.b = r / p.Hkv;
  int L = lens[w.b];
  L = L < 0 ? 0 : (L > p.len_cap ? p.len_cap : L);
  w.L = L;
  w.p0 = w.part * p.part;
  if (w.p0 >= L) return false;
  w.ntok = min(p.part, L - w.p0);
  w.nt = (w.ntok + kTile - 1) / kTile;
  return true;
}

// Position in this CTA's walk: tile k (K tiles, then V tiles) of unit u.
struct Cursor {
  int u, k;
  Unit w;
};

__device__ __forceinline__ void cursor_seek(const AttnParams& p,
                                            const int32_t* lens, int U,
                                            Cursor& c) {
  while (c.u < U && !unit_at(p, lens, c.u, c.w)) c.u += gridDim.x;
}

__device__ __forceinline__ void cursor_next(const AttnParams& p,
                                            const int32_t* lens, int U,
                                            Cursor& c) {
  if (c.u >= U) return;
  if (++c.k < 2 * c.w.nt) return;
  c.k = 0;
  c.u += gridDim.x;
  cursor_seek(p, lens, U, c);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// A operand in tensor memory: kind::f16, fp32 accumulate.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem,
                                           uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

// 32 columns of this warp's 32 TMEM lanes, one lane per thread.
__device__ __forceinline__ void tmem_st32(uint32_t addr,
                                          const uint32_t (&w)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(addr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
      "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]),
      "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]),
      "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
      "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]),
      "r"(w[30]), "r"(w[31])
      : "memory");
}

// Half a token row (4 groups = 64 dims) -> 32 f16x2 words, dims 2c, 2c+1 in
// word c.  d0, d1: the 32 code bytes; sw: the scale words (linear: one word
// whose bytes are the 4 groups' scales; swizzled: 4 band words, scale =
// byte r of each).
__device__ __forceinline__ void dequant_half(uint4 d0, uint4 d1,
                                             const uint32_t (&sw)[4],
                                             bool linear, uint32_t r,
                                             uint32_t (&w)[32]) {
  const uint32_t sel = r | ((r + 4u) << 4);
#pragma unroll
  for (int m = 0; m < 2; ++m) {  // groups 2m, 2m+1 of this half
    const uint32_t pair =
        linear ? (m ? sw[0] >> 16 : sw[0]) : prmt(sw[2 * m], sw[2 * m + 1], sel);
    const uint32_t sf = e4m3x2_to_f16x2(pair);
    const uint32_t sf_even = prmt(sf, sf, 0x1010u);
    const uint32_t sf_odd = prmt(sf, sf, 0x3232u);
    const uint4 d = m ? d1 : d0;
    uint32_t o[4];
    dequant_word(d.x, sf_even, o);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[16 * m + i] = o[i];
    dequant_word(d.y, sf_even, o);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[16 * m + 4 + i] = o[i];
    dequant_word(d.z, sf_odd, o);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[16 * m + 8 + i] = o[i];
    dequant_word(d.w, sf_odd, o);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[16 * m + 12 + i] = o[i];
  }
}

// Token of this thread in the cursor's tile, or -1 past the partition.
__device__ __forceinline__ int cursor_token(const Cursor& c, int U, int r) {
  if (c.u >= U) return -1;
  const int tile = c.k >= c.w.nt ? c.k - c.w.nt : c.k;
  const int t = c.w.p0 + tile * kTile + r;
  return t < c.w.p0 + c.w.ntok ? t : -1;
}

template <int NG, bool kF16>
__global__ void __launch_bounds__(kPipeThreads, 1)
paged_attention_pipe_kernel(const AttnParams p) {
  constexpr int NH = NG / 2;  // head columns per half
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t s_a = smem_addr(smem);
  const uint32_t v_a = s_a + kOffV, p_a = s_a + kOffP, q_a = s_a + kOffQ;
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  const uint32_t bar0 = s_a + kOffBar;
  auto ready = [&](uint32_t x) { return bar0 + 8u * x; };
  auto done = [&](uint32_t x) { return bar0 + 16u + 8u * x; };
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  volatile int* abort_flag = reinterpret_cast<int*>(smem + kOffAbort);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int U = p.num_seqs * p.Hkv * p.max_parts;
  pdl_prologue();

  const int32_t* lens = p.lens;
  if (p.num_seqs <= kMaxLensSmem) {
    int32_t* s_lens = reinterpret_cast<int32_t*>(smem + kOffLens);
    for (int i = tid; i < p.num_seqs; i += kPipeThreads)
      s_lens[i] = __ldg(p.lens + i);
    lens = s_lens;
  }
  if (warp == 0) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
        ::"r"(smem_addr(slot)), "r"(kPipeTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(ready(x)));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(done(x)));
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (NG == 8) {  // heads 8..15 of P^T stay zero
    if (tid < kConsumers)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        st_shared_v4(p_a + kPGroup + (tid * 2 + i) * 16, 0, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  // bounded wait; after any timeout in the CTA every wait fails at once
  auto wait_ok = [&](uint32_t bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    if (p.dev_error != nullptr) atomicOr(p.dev_error, KVQ_DEVERR_TIMEOUT);
    return false;
  };

  if (warp == kConsumers / 32) {
    // =========================== MMA warp ================================
    Cursor c{static_cast<int>(blockIdx.x), 0, {}};
    cursor_seek(p, lens, U, c);
    uint32_t g = 0;
    while (c.u < U) {
      const uint32_t x = g & 1u;
      int go = 1;
      if (lane == 0) go = wait_ok(ready(x), (g >> 1) & 1u);
      if (!__shfl_sync(0xFFFFFFFFu, go, 0)) break;
      tc_fence_after();
      if (lane == 0) {
        const bool is_v = c.k >= c.w.nt;
        const int tile = is_v ? c.k - c.w.nt : c.k;
        const uint32_t buf = v_a + x * kKVBytes;
        if (!is_v) {
          constexpr uint32_t id = instr_desc(false, false);
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks)
            mma_f16_ta(tmem + 16 * tile, tmem + kKCol + 64 * x + 8 * ks,
                       smem_desc(q_a + ks * 256, 128, 2048), id, ks > 0);
        } else {
          constexpr uint32_t id = instr_desc(true, true);
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            mma_f16(tmem + kOCol, smem_desc(buf + ks * 256, 128, 2048),
                    smem_desc(p_a + (16 * tile + 2 * ks) * 128, 128, kPGroup),
                    id, (tile > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(done(x));
      }
      __syncwarp();
      cursor_next(p, lens, U, c);
      ++g;
    }
    // the last commits complete before the CTA can free tensor memory
    if (lane == 0 && g > 0) {
      mbar_wait(done((g - 1) & 1u), ((g - 1) >> 1) & 1u);
      if (g > 1) mbar_wait(done(g & 1u), ((g - 2) >> 1) & 1u);
    }
  } else {
    // ========================== converter warps ==========================
    const int r = tid & (kTile - 1);  // token of the tile
    const int h = tid >> 7;           // dims 64h .. 64h+63
    const int wq = warp & 3;          // TMEM lane quarter
    const int half = warp >> 2;       // head columns [half*NH, half*NH+NH)
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float k_scale = __ldg(p.k_scale);
    const float v_scale = __ldg(p.v_scale);
    const float c2 = p.scale * k_scale * kLog2e;
    const int qn = tid >> 4, qkc = tid & 15;  // this thread's Q' chunk
    const uint32_t my_slot = s_a + kOffSlots + tid * 16;
    const uint32_t my_bt = s_a + kOffBt + tid * 4;

    // empty contexts: zero output; contexts past the cap: flagged
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
      Unit w;
      if (unit_at(p, lens, u, w) || w.part != 0) continue;
      if (w.L == 0)
        for (int i = tid; i < p.G * kD; i += kConsumers)
          p.out[w.b * p.out_stride0 + (w.kh * p.G) * kD + i] = 0;
    }
    if (tid == 0 && p.dev_error != nullptr) {
      for (int u = blockIdx.x; u < U; u += gridDim.x) {
        if (u % p.max_parts != 0 || (u / p.max_parts) % p.Hkv != 0) continue;
        const int raw = lens[u / p.max_parts / p.Hkv];
        if (raw < 0 || raw > p.len_cap) atomicOr(p.dev_error, KVQ_DEVERR_SEQ);
      }
    }

    // block-table entry of this thread's token of the cursor's tile
    auto issue_bt = [&](const Cursor& c, int slot_i) {
      const int t = cursor_token(c, U, r);
      if (t < 0) return;
      const int idx = p.b_shift >= 0 ? t >> p.b_shift : t / p.B;
      cp_async4(my_bt + slot_i * (kConsumers * 4),
                p.block_table + c.w.b * p.bt_stride + idx);
    };
    // this thread's half row of the cursor's tile; false if nothing copied
    auto issue_data = [&](const Cursor& c, int slot_i, int bt_i) -> bool {
      const int t = cursor_token(c, U, r);
      if (t < 0) return false;
      const int32_t blk = static_cast<int32_t>(
          ld_shared_u32(my_bt + bt_i * (kConsumers * 4)));
      if (blk < 0 || blk >= p.num_blocks) {
        if (p.dev_error != nullptr) atomicOr(p.dev_error, KVQ_DEVERR_BLOCK);
        return false;
      }
      const bool is_v = c.k >= c.w.nt;
      const int idx = p.b_shift >= 0 ? t >> p.b_shift : t / p.B;
      const int off = t - idx * p.B;
      const uint8_t* page =
          p.side[is_v ? 1 : 0] + static_cast<int64_t>(blk) * p.page_stride;
      const uint8_t* dp = page + c.w.kh * p.dhs + off * p.dts + h * 32;
      const uint32_t dst = my_slot + slot_i * kSlotBytes;
      cp_async16(dst, dp);
      cp_async16(dst + kConsumers * 16, dp + 16);
      const uint8_t* sp = page + p.scale_off + c.w.kh * p.shs;
      if (!is_v && !p.swizzle_k) {
        cp_async4(dst + 2 * kConsumers * 16, sp + off * p.sts + h * 4);
      } else {  // band rows 2h and 2h+1 of the token's 4-row band
        const uint8_t* band = sp + (off & ~3) * p.sts;
        cp_async8(dst + 2 * kConsumers * 16, band + (2 * h) * p.sts);
        cp_async8(dst + 2 * kConsumers * 16 + 8, band + (2 * h + 1) * p.sts);
      }
      return true;
    };

    Cursor cp{static_cast<int>(blockIdx.x), 0, {}};
    cursor_seek(p, lens, U, cp);
    Cursor cd = cp, cb = cp;
    // prologue: entries of tiles 0 .. 2D-1, then data of tiles 0 .. D-1
    for (int i = 0; i < 2 * kDepth; ++i) {
      issue_bt(cb, i);
      cursor_next(p, lens, U, cb);
    }
    cp_async_commit();
    cp_async_wait<0>();
    uint32_t okmask = 0;  // bit j: data slot j holds a copied half row
    for (int i = 0; i < kDepth; ++i) {
      okmask |= static_cast<uint32_t>(issue_data(cd, i, i)) << i;
      cursor_next(p, lens, U, cd);
      cp_async_commit();
    }
    uint4 qv = make_uint4(0, 0, 0, 0);
    auto load_q = [&](const Unit& w) {
      qv = make_uint4(0, 0, 0, 0);
      if (qn < p.G)
        qv = *reinterpret_cast<const uint4*>(
            p.q + w.b * p.q_stride0 + (w.kh * p.G + qn) * kD + qkc * 8);
    };
    if (cp.u < U) load_q(cp.w);

    uint32_t g = 0;          // tiles processed
    int ds = 0, bs = 0;      // data slot g % D, entry slot g % 2D
    uint32_t kvalid = 0;
    float m[NH], l[NH];
#pragma unroll
    for (int i = 0; i < NH; ++i) { m[i] = 0.f; l[i] = 0.f; }
    while (cp.u < U) {
      // ---- keep kDepth tiles in flight --------------------------------
      cp_async_wait<kDepth - 1>();  // tile g's data and tile g+D's entry
      {
        const int ds_new = ds;  // slot of tile g, reused by tile g + D
        const int bt_new = bs + kDepth >= 2 * kDepth ? bs - kDepth
                                                     : bs + kDepth;
        const uint4 d0 = ld_shared_v4(my_slot + ds * kSlotBytes);
        const uint4 d1 =
            ld_shared_v4(my_slot + ds * kSlotBytes + kConsumers * 16);
        const uint4 sc =
            ld_shared_v4(my_slot + ds * kSlotBytes + 2 * kConsumers * 16);
        const bool ok_g = (okmask >> ds) & 1u;
        // tile g's bytes are in registers: the slot takes tile g + D
        okmask &= ~(1u << ds_new);
        okmask |= static_cast<uint32_t>(issue_data(cd, ds_new, bt_new))
                  << ds_new;
        issue_bt(cb, bs);  // tile g + 2D into the entry slot of tile g
        cp_async_commit();
        cursor_next(p, lens, U, cd);
        cursor_next(p, lens, U, cb);

        const Unit& w = cp.w;
        const bool is_v = cp.k >= w.nt;
        const int tile = is_v ? cp.k - w.nt : cp.k;
        const uint32_t x = g & 1u;
        if (cp.k == 0) {
          // a new unit: its query rows (every MMA of the previous unit has
          // completed), and the next unit's rows start loading
          if constexpr (!kF16) {
            qv.x = bf16x2_to_f16x2(qv.x);
            qv.y = bf16x2_to_f16x2(qv.y);
            qv.z = bf16x2_to_f16x2(qv.z);
            qv.w = bf16x2_to_f16x2(qv.w);
          }
          st_shared_v4(q_a + (qn >> 3) * 2048 + qkc * 128 + (qn & 7) * 16,
                       qv.x, qv.y, qv.z, qv.w);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          Cursor nx = cp;
          nx.k = 0;
          nx.u += gridDim.x;
          cursor_seek(p, lens, U, nx);
          if (nx.u < U) load_q(nx.w);
          kvalid = 0;
        }
        if (is_v && tile == 0) {
          // ---- softmax, once the last K tile's MMAs have completed ------
          wait_ok(done((g - 1) & 1u), ((g - 1) >> 1) & 1u);
          tc_fence_after();
          float xv[kMaxTiles][NH];
#pragma unroll
          for (int i = 0; i < kMaxTiles; ++i)
            if (i < w.nt)
              tmem_ld<NH>(tmem + lane_base + 16 * i + half * NH, xv[i]);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kMaxTiles; ++i) {
            const bool valid = i < w.nt && ((kvalid >> i) & 1u);
#pragma unroll
            for (int gg = 0; gg < NH; ++gg)
              xv[i][gg] = valid ? xv[i][gg] * c2 : -INFINITY;
          }
#pragma unroll
          for (int gg = 0; gg < NH; ++gg) {
            float v = xv[0][gg];
#pragma unroll
            for (int i = 1; i < kMaxTiles; ++i) v = fmaxf(v, xv[i][gg]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
              v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
            if (lane == 0) red[warp * 8 + gg] = v;
          }
          consumers_sync();
#pragma unroll
          for (int gg = 0; gg < NH; ++gg) {
            const float* rr = red + half * 32 + gg;
            const float v = fmaxf(fmaxf(rr[0], rr[8]), fmaxf(rr[16], rr[24]));
            m[gg] = v == -INFINITY ? 0.f : v;
            l[gg] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < kMaxTiles; ++i) {
            if (i >= w.nt) break;
            uint32_t hh[NH / 2];
#pragma unroll
            for (int gg = 0; gg < NH; gg += 2) {
              hh[gg / 2] = pack_f16x2(ex2(xv[i][gg] - m[gg]),
                                      ex2(xv[i][gg + 1] - m[gg + 1]));
              float lo, hi;
              unpack_f16x2(hh[gg / 2], lo, hi);
              l[gg] += lo;
              l[gg + 1] += hi;
            }
            const int kt = i * kTile + r;  // token of the partition
            const uint32_t row = p_a + (kt >> 3) * 128 + (kt & 7) * 16;
            if constexpr (NH == 4) {
              asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(
                               row + half * 8),
                           "r"(hh[0]), "r"(hh[1])
                           : "memory");
            } else {
              st_shared_v4(row + half * kPGroup, hh[0], hh[1], hh[2], hh[3]);
            }
          }
#pragma unroll
          for (int gg = 0; gg < NH; ++gg) {
            float v = l[gg];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
              v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane == 0) red[64 + warp * 8 + gg] = v;
          }
          consumers_sync();
#pragma unroll
          for (int gg = 0; gg < NH; ++gg) {
            const float* rr = red + 64 + half * 32 + gg;
            l[gg] = (rr[0] + rr[8]) + (rr[16] + rr[24]);
          }
        }

        // ---- the operand buffer of tile g is free once tile g-2's MMAs
        // have completed ------------------------------------------------
        if (g >= 2) wait_ok(done(x), ((g >> 1) - 1) & 1u);
        uint32_t wv[32];
        if (ok_g) {
          const bool linear = !is_v && !p.swizzle_k;
          const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
          dequant_half(d0, d1, sw, linear,
                       static_cast<uint32_t>((w.p0 + r) & 3), wv);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) wv[i] = 0;
        }
        if (!is_v) {
          // K' -> tensor memory: lane = token, 32 columns per half row
          tmem_st32(tmem + lane_base + kKCol + 64 * x + 32 * h, wv);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          kvalid |= static_cast<uint32_t>(ok_g) << tile;
        } else {
          // V' -> shared memory, MN-major for O^T = V'^T . P^T
          const uint32_t tb =
              v_a + x * kKVBytes + (r >> 3) * 128 + (r & 7) * 16;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(tb + (8 * h + c) * 2048, wv[4 * c], wv[4 * c + 1],
                         wv[4 * c + 2], wv[4 * c + 3]);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ready(x));

        if (is_v && tile == w.nt - 1) {
          // ---- output of this unit -------------------------------------
          const bool ok = wait_ok(done(x), (g >> 1) & 1u);
          tc_fence_after();
          float o[NH];
          tmem_ld<NH>(tmem + lane_base + kOCol + half * NH, o);
          tmem_wait_ld();
          tc_fence_before();
          const int d = wq * 32 + lane;
          const int nparts = (w.L + p.part - 1) / p.part;
          if (ok && nparts == 1) {
#pragma unroll
            for (int gg = 0; gg < NH; ++gg) {
              const int hg = half * NH + gg;
              if (hg < p.G) {
                const float y =
                    l[gg] > 0.f ? o[gg] * (1.0f / l[gg]) * v_scale : 0.f;
                p.out[w.b * p.out_stride0 + (w.kh * p.G + hg) * kD + d] =
                    float_to_out<kF16>(y);
              }
            }
          } else if (ok) {
            const int64_t row0 =
                (static_cast<int64_t>(w.b) * p.Hq + w.kh * p.G) *
                    p.max_parts + w.part;
#pragma unroll
            for (int gg = 0; gg < NH; ++gg) {
              const int hg = half * NH + gg;
              if (hg < p.G) {
                const int64_t rr =
                    row0 + static_cast<int64_t>(hg) * p.max_parts;
                p.tmp_out[rr * kD + d] =
                    l[gg] > 0.f ? o[gg] * (1.0f / l[gg]) : 0.f;
                if (wq == 0 && lane == gg) {
                  p.max_logits[rr] = m[gg];
                  p.exp_sums[rr] = l[gg];
                }
              }
            }
          }
        }
        ds = ds + 1 == kDepth ? 0 : ds + 1;
        bs = bs + 1 == 2 * kDepth ? 0 : bs + 1;
        cursor_next(p, lens, U, cp);
        ++g;
      }
    }
    cp_async_wait<0>();  // no copy may land after the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(tmem), "r"(kPipeTmemCols));
}

// ---------------------------------------------------------------------------
// Merge of the partitions of contexts longer than one partition
// ---------------------------------------------------------------------------
// 16 rows (sequence, query head) per CTA of 256 threads, a half-warp per
// row and 8 head dims per lane, so that one wave of CTAs covers a whole
// decode batch.  The context length is read before the wait for the
// attention kernel, which writes none of it; every thread waits before it
// may leave.  Per dim, the sums run over the partitions in order.
constexpr int kMergeThreads = 256;
constexpr int kMergeRows = kMergeThreads / 16;
// Rows of at most this many partitions issue all their loads at once.
constexpr int kMergeFew = 4;

template <bool kF16>
__global__ void __launch_bounds__(kMergeThreads)
attention_merge_kernel(const AttnParams p) {
  const int sub = threadIdx.x & 15;  // dims 8 sub .. 8 sub + 7
  const int64_t row =
      static_cast<int64_t>(blockIdx.x) * kMergeRows + (threadIdx.x >> 4);
  const bool live = row < static_cast<int64_t>(p.num_seqs) * p.Hq;
  const int b = live ? static_cast<int>(row / p.Hq) : 0;
  const int h = live ? static_cast<int>(row - static_cast<int64_t>(b) * p.Hq)
                     : 0;
  int L = live ? __ldg(p.lens + b) : 0;
  pdl_prologue();
  L = L < 0 ? 0 : (L > p.len_cap ? p.len_cap : L);
  const int nparts = (L + p.part - 1) / p.part;
  if (!live || nparts <= 1) return;
  const int64_t row0 = row * p.max_parts;
  float M = -INFINITY;
  float den = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  auto add = [&](float w, const float4& x, const float4& y) {
    den += w;
    acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
    acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
  };
  if (nparts <= kMergeFew) {
    // every load of the row in one round trip, then the same sums in order
    float ml[kMergeFew], es[kMergeFew];
    float4 xs[kMergeFew], ys[kMergeFew];
#pragma unroll
    for (int i = 0; i < kMergeFew; ++i) {
      if (i < nparts) {
        ml[i] = p.max_logits[row0 + i];
        es[i] = p.exp_sums[row0 + i];
        const float4* src = reinterpret_cast<const float4*>(
            p.tmp_out + (row0 + i) * kD + 8 * sub);
        xs[i] = src[0];
        ys[i] = src[1];
      }
    }
#pragma unroll
    for (int i = 0; i < kMergeFew; ++i)
      if (i < nparts) M = fmaxf(M, ml[i]);
#pragma unroll
    for (int i = 0; i < kMergeFew; ++i)
      if (i < nparts) add(es[i] * ex2(ml[i] - M), xs[i], ys[i]);
  } else {
#pragma unroll 4
    for (int i = 0; i < nparts; ++i) M = fmaxf(M, p.max_logits[row0 + i]);
#pragma unroll 2
    for (int i = 0; i < nparts; ++i) {
      const float4* src = reinterpret_cast<const float4*>(
          p.tmp_out + (row0 + i) * kD + 8 * sub);
      add(p.exp_sums[row0 + i] * ex2(p.max_logits[row0 + i] - M), src[0],
          src[1]);
    }
  }
  const float f = den > 0.f ? 1.0f / den : 0.f;
  const float vs = __ldg(p.v_scale);
  uint32_t packed[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float y0 = den > 0.f ? acc[2 * k] * f * vs : 0.f;
    const float y1 = den > 0.f ? acc[2 * k + 1] * f * vs : 0.f;
    packed[k] = static_cast<uint32_t>(float_to_out<kF16>(y0)) |
                (static_cast<uint32_t>(float_to_out<kF16>(y1)) << 16);
  }
  *reinterpret_cast<uint4*>(p.out + b * p.out_stride0 + h * kD + 8 * sub) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

template <int NG, bool kF16>
cudaError_t launch_pipe(const AttnParams& p, cudaStream_t stream) {
  auto kernel = paged_attention_pipe_kernel<NG, kF16>;
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (!configured[dev & 63]) {
    err = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPipeSmem);
    if (err != cudaSuccess) return err;
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel,
                                                        kPipeThreads, kPipeSmem);
    if (err != cudaSuccess) return err;
    if (occ < 1 || occ * kPipeTmemCols > 512)
      return cudaErrorInvalidConfiguration;
    configured[dev & 63] = true;
  }
  const int64_t units =
      static_cast<int64_t>(p.num_seqs) * p.Hkv * p.max_parts;
  const unsigned grid =
      static_cast<unsigned>(std::min<int64_t>(units, sm_count()));
  err = launch_kernel(kernel, dim3(grid), kPipeThreads, kPipeSmem, stream,
                      p.pdl, p);
  if (err != cudaSuccess || p.max_parts <= 1) return err;
  return launch_attention_merge(p, stream);
}

template <int NG, bool kF16>
cudaError_t launch_ng(const AttnParams& p, cudaStream_t stream) {
  if (p.kernel == kAttnPipelined) return launch_pipe<NG, kF16>(p, stream);
  auto kernel = paged_attention_kernel<NG, kF16>;
  static bool configured[64] = {false};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (!configured[dev & 63]) {
    err = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    // tensor memory: at most 512 columns may be held per SM at once
    int occ = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel,
                                                        kThreads, kSmemBytes);
    if (err != cudaSuccess) return err;
    if (occ * kTmemCols > 512) return cudaErrorInvalidConfiguration;
    configured[dev & 63] = true;
  }
  const dim3 grid(p.max_parts, p.Hkv, p.num_seqs);
  err = launch_kernel(kernel, grid, kThreads, kSmemBytes, stream, p.pdl, p);
  if (err != cudaSuccess || p.max_parts <= 1) return err;
  return launch_attention_merge(p, stream);
}

}  // namespace

cudaError_t launch_attention_merge(const AttnParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.num_seqs) * p.Hq;
  const dim3 grid(static_cast<unsigned>((rows + kMergeRows - 1) / kMergeRows));
  return p.f16 ? launch_kernel(attention_merge_kernel<true>, grid,
                               kMergeThreads, 0, stream, true, p)
               : launch_kernel(attention_merge_kernel<false>, grid,
                               kMergeThreads, 0, stream, true, p);
}

cudaError_t launch_paged_attention_nvfp4(const AttnParams& p,
                                         cudaStream_t stream) {
  if (p.kernel == kAttnWarpMma) return launch_paged_attention_mma(p, stream);
  if (p.G <= 8)
    return p.f16 ? launch_ng<8, true>(p, stream)
                 : launch_ng<8, false>(p, stream);
  return p.f16 ? launch_ng<16, true>(p, stream)
               : launch_ng<16, false>(p, stream);
}

}  // namespace kvq
