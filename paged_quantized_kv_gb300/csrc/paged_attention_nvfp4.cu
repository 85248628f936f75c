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
// GB300 design -- one CTA of 4 warps per (partition of <= 512 tokens, KV
// head, sequence), 4 CTAs per SM (52 KB of shared memory, 128 TMEM columns
// each):
//   * Every thread owns one token of a 128-token tile and reads its 64 data
//     bytes and 8 scale bytes straight from HBM into registers; the next
//     tile's loads are in flight while the current tile is converted.  K
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
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

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
  if constexpr (N == 8) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(addr));
  } else {
    static_assert(N == 16, "8 or 16 columns");
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
__global__ void __launch_bounds__(kThreads, 4)
paged_attention_kernel(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
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

  // first tile's loads go out before the set-up work
  Raw cur, nxt;
  load_raw(p, b, kh, p0 + tid, t_end, false, cur);

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
  for (int u = 0; u < nu; ++u) {
    const bool is_v = u >= ntiles;
    const int tile = is_v ? u - ntiles : u;
    if (u + 1 < nu) {
      const bool nv = u + 1 >= ntiles;
      const int nt = nv ? u + 1 - ntiles : u + 1;
      load_raw(p, b, kh, p0 + nt * kTile + tid, t_end, nv, nxt);
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
        const bool valid = i < ntiles && i * kTile + tid < ntok;
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
// Merge of the partitions of contexts longer than one partition
// ---------------------------------------------------------------------------
template <bool kF16>
__global__ void __launch_bounds__(kD)
attention_merge_kernel(const AttnParams p) {
  pdl_prologue();
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  int L = __ldg(p.lens + b);
  L = L < 0 ? 0 : (L > p.len_cap ? p.len_cap : L);
  const int nparts = (L + p.part - 1) / p.part;
  if (nparts <= 1) return;
  const int64_t row0 = (static_cast<int64_t>(b) * p.Hq + h) * p.max_parts;
  float M = -INFINITY;
  for (int i = 0; i < nparts; ++i) M = fmaxf(M, p.max_logits[row0 + i]);
  float den = 0.f, acc = 0.f;
  for (int i = 0; i < nparts; ++i) {
    const float w = p.exp_sums[row0 + i] * ex2(p.max_logits[row0 + i] - M);
    den += w;
    acc += w * p.tmp_out[(row0 + i) * kD + d];
  }
  const float y = den > 0.f ? acc * (1.0f / den) * __ldg(p.v_scale) : 0.f;
  p.out[b * p.out_stride0 + h * kD + d] = float_to_out<kF16>(y);
}

template <int NG, bool kF16>
cudaError_t launch_ng(const AttnParams& p, cudaStream_t stream) {
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
  return launch_kernel(attention_merge_kernel<kF16>, dim3(p.Hq, p.num_seqs),
                       kD, 0, stream, true, p);
}

}  // namespace

cudaError_t launch_paged_attention_nvfp4(const AttnParams& p,
                                         cudaStream_t stream) {
  if (p.G <= 8)
    return p.f16 ? launch_ng<8, true>(p, stream)
                 : launch_ng<8, false>(p, stream);
  return p.f16 ? launch_ng<16, true>(p, stream)
               : launch_ng<16, false>(p, stream);
}

}  // namespace kvq
