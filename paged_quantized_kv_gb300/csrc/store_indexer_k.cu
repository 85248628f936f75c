// store_indexer_k.cu -- bf16/fp16 indexer K -> fp8 e4m3 + per-token fp32
// scale in a paged indexer cache, sm_103a.  The write side of the cache
// that cp_gather_indexer_k_quant_cache reads (vLLM PR #25931 "Add
// gather_indexer_k_quant_cache kernel": "quantized k/k_scale" in blocks of
// [block_size * head_dim fp8 K | block_size * 4 scale bytes]).
//
// The pages give no quantisation rule; per-token absmax scaling is taken:
// scale = amax / 448 (IEEE fp32 division), q_i = e4m3_rn_satfinite(k_i /
// scale) (IEEE division), q = 0 when amax = 0.  Token t with slot s >= 0
// goes to block s / B, row s % B; s < 0 is skipped.
//
// GB300 design: HBM-bound, ~2 bytes read and ~1.03 written per element; the
// per-element division of the rule is replaced by products whose result is
// proven equal (below), which keeps the instruction stream short.  A token is
// L = head_dim / 16 lanes (8 for head_dim 128; 4 tokens per warp), each
// holding 16 elements from one 256-bit load; amax is a packed max.bf16x2 /
// max.f16x2 tree plus an xor-shuffle reduction over the L lanes; the
// codes come from cvt.rn.satfinite.e4m3x2.f32.  Each lane writes its 16
// code bytes (the token's row is one contiguous run) and the first lane the
// scale.  The grid is persistent, trimmed so its last iteration is as full
// as the others; each lane keeps kUnroll tokens' loads in flight.
//
// Division-free quotients, checked exhaustively.  With y = RN(1/scale)
// (one IEEE reciprocal per token), q0 = RN(k y), r = RN(k - q0 scale) and
// q1 = RN(q0 + r y) (two fused multiply-adds: P. Markstein's quotient
// correction, IBM J. Res. Dev. 34(1), 1990), and the sign bit of k put back
// on the code (q1 of k = -0 is +0), e4m3(q1) equals e4m3(RN32(k / scale))
// for every pair of finite bf16 or fp16 inputs with |k| <= amax and
// scale >= 2^-90 -- about 2 x 10^9 pairs per type, enumerated by
// tests/quotient_exhaustive.c.  Tokens with a smaller scale (1/scale may
// overflow, residuals may underflow) take IEEE divisions.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
#ifndef KVQ_ISTORE_UNROLL
#define KVQ_ISTORE_UNROLL 2
#endif
constexpr int kUnroll = KVQ_ISTORE_UNROLL;

// 16 elements (32 bytes) of a row: one 256-bit load when 32-byte aligned.
__device__ __forceinline__ void load16(const uint16_t* p, uint32_t (&w)[8],
                                       bool vec32) {
  if (vec32) {
    asm volatile(
        "ld.global.nc.L1::no_allocate.v8.u32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]),
          "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "l"(p));
  } else {
    asm volatile(
        "ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
        : "l"(p));
    asm volatile(
        "ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "l"(p + 8));
  }
}

__device__ __forceinline__ int64_t ld_nc_s64(const int64_t* p) {
  int64_t v;
  asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

template <bool kF16>
__device__ __forceinline__ uint32_t half2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (kF16)
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Packed pair -> two fp32 values (exact for both element types).
template <bool kF16>
__device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi) {
  if constexpr (kF16) {
    asm("{ .reg .f16 a, b;\n"
        "  mov.b32 {a, b}, %2;\n"
        "  cvt.f32.f16 %0, a;\n"
        "  cvt.f32.f16 %1, b; }"
        : "=f"(lo), "=f"(hi)
        : "r"(w));
  } else {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
  }
}

// Two fp32 -> e4m3 codes, rn, satfinite; `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi),
      "f"(lo));
  return pair;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) |
         (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}

// Four elements (two packed pairs) -> their four e4m3 codes, element 0 in
// the low byte: q0 = k y, r = k + q0 (-scale), q1 = q0 + r y as packed IEEE
// products and fused multiply-adds (two elements per f32x2 instruction),
// then cvt.rn.satfinite.e4m3x2.f32.  y2 = {y, y}, ns2 = {-scale, -scale}.
__device__ __forceinline__ uint32_t codes4(uint64_t x01, uint64_t x23,
                                           uint64_t y2, uint64_t ns2) {
  uint32_t out;
  asm("{ .reg .b64 p, q, r, t;\n"
      "  .reg .f32 p0, p1, q0, q1;\n"
      "  .reg .b16 c0, c1;\n"
      "  mul.rn.f32x2 p, %1, %3;\n"
      "  mul.rn.f32x2 q, %2, %3;\n"
      "  fma.rn.f32x2 r, p, %4, %1;\n"
      "  fma.rn.f32x2 t, q, %4, %2;\n"
      "  fma.rn.f32x2 p, r, %3, p;\n"
      "  fma.rn.f32x2 q, t, %3, q;\n"
      "  mov.b64 {p0, p1}, p;\n"
      "  mov.b64 {q0, q1}, q;\n"
      "  cvt.rn.satfinite.e4m3x2.f32 c0, p1, p0;\n"
      "  cvt.rn.satfinite.e4m3x2.f32 c1, q1, q0;\n"
      "  mov.b32 %0, {c0, c1}; }"
      : "=r"(out)
      : "l"(x01), "l"(x23), "l"(y2), "l"(ns2));
  return out;
}

// The sign bits of four packed 16-bit elements (two words, element 0 in the
// low half of wa) as the top bits of four bytes.
__device__ __forceinline__ uint32_t signs4(uint32_t wa, uint32_t wb) {
  return __byte_perm(wa, wb, 0x7531) & 0x80808080u;
}

// The rule written out for one lane's 16 elements: an IEEE division per
// element.  Out of line: it runs only for tokens whose scale is below
// 2^-90.
template <bool kF16>
__device__ __noinline__ uint4 codes16_exact(uint4 w0, uint4 w1,
                                            float scale) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a, b, d, e;
    widen2<kF16>(w[2 * k], a, b);
    widen2<kF16>(w[2 * k + 1], d, e);
    c[k] = e4m3x2(__fdiv_rn(a, scale), __fdiv_rn(b, scale)) |
           (e4m3x2(__fdiv_rn(d, scale), __fdiv_rn(e, scale)) << 16);
  }
  return make_uint4(c[0], c[1], c[2], c[3]);
}

// kEarlyRead (KVQ_F_PDL_EARLY_READ): the first iteration's slot and row
// loads go out before the wait on the predecessor kernel; every write
// (cache bytes, dev_error) comes after it.  A thread with no token writes
// nothing and needs no wait.  Measured back to back on the long-context
// shape: 10.2 us with the wait first, 9.0 us with the reads first.
template <bool kF16, int L, bool kEarlyRead>
__global__ void __launch_bounds__(kThreads)
store_indexer_k_kernel(const IndexerStoreParams p) {
  if constexpr (!kEarlyRead) pdl_prologue();
  bool waited = !kEarlyRead;
  constexpr int kTokPerWarp = 32 / L;
  const int lane = threadIdx.x & 31;
  const int sub = lane / L;      // token slot inside the warp
  const int part = lane % L;     // 16-element chunk of the row
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) +
                       (threadIdx.x >> 5);
  const int64_t tstep = warps * kTokPerWarp;
  const uint32_t seg_mask =
      L == 32 ? 0xFFFFFFFFu : (((1u << L) - 1u) << (sub * L));

  for (int64_t t0 = warp * kTokPerWarp + sub; t0 - sub < p.num_tokens;
       t0 += kUnroll * tstep) {
    uint32_t raw[kUnroll][8];
    int64_t slot[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t t = t0 + u * tstep;
#pragma unroll
      for (int k = 0; k < 8; ++k) raw[u][k] = 0u;
      slot[u] = -1;
      if (t < p.num_tokens) {
        slot[u] = ld_nc_s64(p.slots + t);
        load16(p.k + t * p.k_stride0 + part * 16, raw[u], p.vec32);
      }
    }
    if (!waited) {  // reads of the first tokens are in flight
      pdl_prologue();
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      // amax over the token's L lanes (every lane of the segment takes part)
      uint32_t m = raw[u][0] & 0x7FFF7FFFu;
#pragma unroll
      for (int k = 1; k < 8; ++k)
        m = half2_max<kF16>(m, raw[u][k] & 0x7FFF7FFFu);
      float lo, hi;
      widen2<kF16>(m, lo, hi);
      float amax = fmaxf(lo, hi);
#pragma unroll
      for (int o = L / 2; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(seg_mask, amax, o));
      if (slot[u] < 0) continue;
      if (slot[u] >= p.num_slots) {
        if (p.dev_error != nullptr && part == 0)
          atomicOr(p.dev_error, KVQ_DEVERR_SLOT);
        continue;
      }
      const float scale = __fdiv_rn(amax, 448.0f);
      uint32_t codes[4] = {0u, 0u, 0u, 0u};
      if (amax != 0.0f) {
        if (scale >= 0x1p-90f) {
          const float y = __frcp_rn(scale);
          const uint64_t y2 = pack2(y, y);
          const uint64_t ns2 = pack2(-scale, -scale);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float a, b, d, e;
            widen2<kF16>(raw[u][2 * k], a, b);
            widen2<kF16>(raw[u][2 * k + 1], d, e);
            codes[k] = codes4(pack2(a, b), pack2(d, e), y2, ns2) |
                       signs4(raw[u][2 * k], raw[u][2 * k + 1]);
          }
        } else {
          const uint4 c = codes16_exact<kF16>(
              make_uint4(raw[u][0], raw[u][1], raw[u][2], raw[u][3]),
              make_uint4(raw[u][4], raw[u][5], raw[u][6], raw[u][7]), scale);
          codes[0] = c.x;
          codes[1] = c.y;
          codes[2] = c.z;
          codes[3] = c.w;
        }
      }
      int64_t blk, off;
      if (p.b_shift >= 0) {
        blk = slot[u] >> p.b_shift;
        off = slot[u] & (p.B - 1);
      } else {
        blk = slot[u] / p.B;
        off = slot[u] - blk * p.B;
      }
      uint8_t* const base = p.cache + blk * p.block_stride;
      asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(
                       base + off * L * 16 + part * 16),
                   "r"(codes[0]), "r"(codes[1]), "r"(codes[2]),
                   "r"(codes[3])
                   : "memory");
      if (part == 0)
        *reinterpret_cast<float*>(base + static_cast<int64_t>(p.B) * L * 16 +
                                  off * 4) = scale;
    }
  }
}

template <bool kF16, int L, bool kEarlyRead>
cudaError_t launch(const IndexerStoreParams& p, cudaStream_t stream) {
  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int& occ = ctas_per_sm[dev & 63];
  if (occ == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ, store_indexer_k_kernel<kF16, L, kEarlyRead>, kThreads, 0);
    if (err != cudaSuccess) return err;
    if (occ < 1) occ = 1;
  }
  // tokens per CTA per loop iteration; the grid is trimmed so the last
  // iteration is as full as the others
  const int64_t per_cta = (kThreads / 32) * (32 / L) * kUnroll;
  const int64_t resident = static_cast<int64_t>(sm_count()) * occ;
  const int64_t iters =
      (p.num_tokens + resident * per_cta - 1) / (resident * per_cta);
  int64_t grid = (p.num_tokens + iters * per_cta - 1) / (iters * per_cta);
  if (grid < 1) grid = 1;
  return launch_kernel(store_indexer_k_kernel<kF16, L, kEarlyRead>,
                       static_cast<unsigned>(grid), kThreads, 0, stream,
                       p.pdl, p);
}

template <bool kF16, bool kEarlyRead>
cudaError_t launch_dim(const IndexerStoreParams& p, cudaStream_t stream) {
  switch (p.D) {  // L = head_dim / 16 lanes per token
    case 16: return launch<kF16, 1, kEarlyRead>(p, stream);
    case 32: return launch<kF16, 2, kEarlyRead>(p, stream);
    case 64: return launch<kF16, 4, kEarlyRead>(p, stream);
    case 128: return launch<kF16, 8, kEarlyRead>(p, stream);
    default: return launch<kF16, 16, kEarlyRead>(p, stream);  // 256
  }
}

}  // namespace

cudaError_t launch_store_indexer_k(const IndexerStoreParams& p,
                                   cudaStream_t stream) {
  if (p.early_read)
    return p.f16 ? launch_dim<true, true>(p, stream)
                 : launch_dim<false, true>(p, stream);
  return p.f16 ? launch_dim<true, false>(p, stream)
               : launch_dim<false, false>(p, stream);
}

}  // namespace kvq
