// store_nvfp4.cu -- bf16 K/V -> NVFP4 paged-cache store for sm_103a.
//
// Operation: vLLM csrc/libtorch_stable/nvfp4_kv_cache_kernels.cu (commit
// 7ce4c8e), reshape_and_cache_nvfp4_kernel / _dispatch: per token, per side
// (K, V), per head, per 16-element group: amax, e4m3 scale
// sf = rn_satfinite((amax / 6) * g), e2m1 codes of x * (g / sf), two codes a
// byte (even element low nibble), 8 data bytes + 1 scale byte into the page
// chosen by slot_mapping; V scales go to the swizzled position of the head's
// [block_size, S] tile.
//
// GB300 design (this file's own, not the page's one-CTA-per-token loop):
//   * HBM-bound at ~2.6 B per element, so the budget is instructions per
//     byte: the grid is persistent (SMs x resident CTAs) and every thread
//     owns one fixed 16-element group "role" (side, head, group) of a token,
//     computes all role addresses once and walks tokens with a grid stride,
//     issuing kUnroll independent loads (one 256-bit load per group when the
//     rows are 32-byte aligned) before using any of them.
//   * Inputs are bf16 or IEEE fp16 (a template parameter); both widen to
//     fp32 exactly.  amax: sign bits cleared, a tree of max.bf16x2 /
//     max.f16x2, one final max.
//   * amax / 6 in three instructions that equal the IEEE quotient for every
//     finite bf16 amax: q0 = amax * RN(1/6), the exact residual
//     r = fma(-q0, 6, amax), q = fma(r, RN(1/6), q0) -- the quotient
//     correction step of P. Markstein, "Computation of elementary functions
//     on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990;
//     checked exhaustively over every finite non-negative bf16 and fp16
//     value by tests/test_div6.py.
//   * g = 1/k_scale and g / float(sf) are IEEE divisions; the second one is
//     read from a 2 x 256 shared-memory table filled once per CTA with
//     __fdiv_rn (exactly the per-group quotient, since sf has 256 codes).
//   * x * r as packed mul.rn.f32x2 (two IEEE products per instruction), codes
//     from cvt.rn.satfinite.e2m1x2.f32 / cvt.rn.satfinite.e4m3x2.f32; the
//     sf == 0 case is a select.
//   * Each thread stores its group's 8 data bytes (a warp writes whole
//     sectors of head rows) and its scale byte.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

#ifndef KVQ_STORE_UNROLL
#define KVQ_STORE_UNROLL 4
#endif
#ifndef KVQ_STORE_MIN_BLOCKS
#define KVQ_STORE_MIN_BLOCKS 1
#endif
constexpr int kThreads = 256;
constexpr int kUnroll = KVQ_STORE_UNROLL;
constexpr uint32_t kInv6Bits = 0x3E2AAAABu;  // RN(1/6) in fp32

// 16 bf16 of one group into w[0..7] (element 2k in the low half of w[k]).
template <bool kVec32>
__device__ __forceinline__ void load_group(const uint16_t* p,
                                           uint32_t (&w)[8]) {
  if constexpr (kVec32) {
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

// Packed max of two pairs of non-negative half-precision values (bf16 or
// IEEE fp16 bit patterns).
template <bool kF16>
__device__ __forceinline__ uint32_t half2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  if constexpr (kF16)
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  else
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Low half of a packed pair -> fp32 (exact for both types).
template <bool kF16>
__device__ __forceinline__ float half_lo_to_float(uint32_t w) {
  if constexpr (kF16) {
    float f;
    asm("{ .reg .f16 lo, hi;\n"
        "  mov.b32 {lo, hi}, %1;\n"
        "  cvt.f32.f16 %0, lo; }"
        : "=f"(f)
        : "r"(w));
    return f;
  } else {
    return __uint_as_float(w << 16);
  }
}

// e4m3 code -> fp32 (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
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

// fp32 -> e4m3, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t float_to_e4m3(float v) {
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f),
      "f"(v));
  return pair & 0xFFu;  // the second operand lands in the low byte
}

// Four packed pairs (bf16, or fp16 with kF16) times r (IEEE fp32 products,
// two per mul.f32x2) -> four bytes of e2m1 codes, element 2k in the low
// nibble of byte k.  Both element types widen to fp32 exactly.
template <bool kF16>
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1,
                                           uint32_t w2, uint32_t w3,
                                           uint64_t rr) {
  uint32_t out;
  if constexpr (kF16) {
    asm("{ .reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n"
        "  .reg .f16 a0, b0_, a1, b1_, a2, b2_, a3, b3_;\n"
        "  .reg .b64 x0, x1, x2, x3;\n"
        "  .reg .b8 b0, b1, b2, b3;\n"
        "  mov.b32 {a0, b0_}, %1;  mov.b32 {a1, b1_}, %2;\n"
        "  mov.b32 {a2, b2_}, %3;  mov.b32 {a3, b3_}, %4;\n"
        "  cvt.f32.f16 l0, a0;  cvt.f32.f16 h0, b0_;\n"
        "  cvt.f32.f16 l1, a1;  cvt.f32.f16 h1, b1_;\n"
        "  cvt.f32.f16 l2, a2;  cvt.f32.f16 h2, b2_;\n"
        "  cvt.f32.f16 l3, a3;  cvt.f32.f16 h3, b3_;\n"
        "  mov.b64 x0, {l0, h0};  mov.b64 x1, {l1, h1};\n"
        "  mov.b64 x2, {l2, h2};  mov.b64 x3, {l3, h3};\n"
        "  mul.rn.f32x2 x0, x0, %5;  mul.rn.f32x2 x1, x1, %5;\n"
        "  mul.rn.f32x2 x2, x2, %5;  mul.rn.f32x2 x3, x3, %5;\n"
        "  mov.b64 {l0, h0}, x0;  mov.b64 {l1, h1}, x1;\n"
        "  mov.b64 {l2, h2}, x2;  mov.b64 {l3, h3}, x3;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b0, h0, l0;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b1, h1, l1;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b2, h2, l2;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b3, h3, l3;\n"
        "  mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(out)
        : "r"(w0), "r"(w1), "r"(w2), "r"(w3), "l"(rr));
  } else {
    asm("{ .reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n"
        "  .reg .b64 x0, x1, x2, x3;\n"
        "  .reg .b8 b0, b1, b2, b3;\n"
        "  shl.b32 l0, %1, 16;  and.b32 h0, %1, 0xFFFF0000;\n"
        "  shl.b32 l1, %2, 16;  and.b32 h1, %2, 0xFFFF0000;\n"
        "  shl.b32 l2, %3, 16;  and.b32 h2, %3, 0xFFFF0000;\n"
        "  shl.b32 l3, %4, 16;  and.b32 h3, %4, 0xFFFF0000;\n"
        "  mov.b64 x0, {l0, h0};  mov.b64 x1, {l1, h1};\n"
        "  mov.b64 x2, {l2, h2};  mov.b64 x3, {l3, h3};\n"
        "  mul.rn.f32x2 x0, x0, %5;  mul.rn.f32x2 x1, x1, %5;\n"
        "  mul.rn.f32x2 x2, x2, %5;  mul.rn.f32x2 x3, x3, %5;\n"
        "  mov.b64 {l0, h0}, x0;  mov.b64 {l1, h1}, x1;\n"
        "  mov.b64 {l2, h2}, x2;  mov.b64 {l3, h3}, x3;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b0, h0, l0;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b1, h1, l1;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b2, h2, l2;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 b3, h3, l3;\n"
        "  mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(out)
        : "r"(w0), "r"(w1), "r"(w2), "r"(w3), "l"(rr));
  }
  return out;
}

__device__ __forceinline__ void st_v2(uint8_t* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b)
               : "memory");
}

// kEarlyRead (KVQ_F_PDL_EARLY_READ): the scale table and the first
// iteration's slot and row loads happen before the wait on the predecessor
// kernel; every write (cache bytes, dev_error) after it.  An idle role
// writes nothing and needs no wait.  Measured back to back on the
// long-context store: 105.5 us with the wait first, 102.8 us with the reads
// first (the step with the early-read gather: 110.0 -> 108.0 us).
template <bool kVec32, bool kF16, bool kEarlyRead>
__global__ void __launch_bounds__(kThreads, KVQ_STORE_MIN_BLOCKS)
store_nvfp4_kernel(const StoreParams p) {
  __shared__ float s_ratio[2][256];  // g_side / float(e4m3 code)

  if constexpr (!kEarlyRead) pdl_prologue();
  bool waited = !kEarlyRead;
  const int tid = threadIdx.x;
  {
    const float g0 = __fdiv_rn(1.0f, __ldg(p.scale[0]));
    const float g1 = __fdiv_rn(1.0f, __ldg(p.scale[1]));
    for (int i = tid; i < 512; i += kThreads) {
      const float v = e4m3_to_float(static_cast<uint32_t>(i & 255));
      const float g = (i < 256) ? g0 : g1;
      s_ratio[i >> 8][i & 255] =
          (v == 0.0f || v != v) ? 0.0f : __fdiv_rn(g, v);
    }
  }
  __syncthreads();

  // ---- this thread's fixed role inside a token ---------------------------
  const int slices = 1 << p.slices_log2;
  int grp_in_tok, tok_sub;
  if (slices == 1) {
    tok_sub = tid / p.gpt;
    grp_in_tok = tid - tok_sub * p.gpt;
  } else {
    tok_sub = 0;
    grp_in_tok = (static_cast<int>(blockIdx.x) & (slices - 1)) * kThreads + tid;
  }
  if (tok_sub >= p.tpp || grp_in_tok >= p.gpt) return;  // idle role
  const int gps = p.gpt >> 1;  // groups per side
  const int side = grp_in_tok >= gps ? 1 : 0;
  const int e = grp_in_tok - side * gps;
  const int head = e / p.S;  // S = groups per head
  const int j = e - head * p.S;
  const int q = p.S >> 2;
  const bool swz = (p.swizzle_sides >> side) & 1u;

  const uint16_t* const src_role = p.src[side] + head * p.D + j * 16;
  const int64_t src_stride = p.src_stride[side];
  uint8_t* const data_role = p.side[side] + head * p.dhs + j * 8;
  uint8_t* const scale_role =
      p.side[side] + p.data_per_side + head * p.shs +
      (swz ? (j / q) * p.sts + (j % q) * 4 : static_cast<int64_t>(j));
  const float* const ratio = s_ratio[side];
  const float g = __fdiv_rn(1.0f, __ldg(p.scale[side]));
  const float inv6 = __uint_as_float(kInv6Bits);

  const int64_t T = p.num_tokens;
  const int64_t tstep =
      static_cast<int64_t>(gridDim.x >> p.slices_log2) * p.tpp;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x >> p.slices_log2) *
                        p.tpp + tok_sub;
       t0 < T; t0 += kUnroll * tstep) {
    uint32_t w[kUnroll][8];
    int64_t slot[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t t = t0 + u * tstep;
      slot[u] = -1;
      if (t < T) {
        slot[u] = ld_nc_s64(p.slots + t);
        load_group<kVec32>(src_role + t * src_stride, w[u]);
      }
    }
    if (!waited) {  // reads of the first tokens are in flight
      pdl_prologue();
      waited = true;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (slot[u] < 0) continue;  // skipped token, or past the end
      if (slot[u] >= p.num_slots) {
        if (p.dev_error != nullptr) atomicOr(p.dev_error, KVQ_DEVERR_SLOT);
        continue;
      }
      // amax of the 16 magnitudes
      const uint32_t m = half2_max<kF16>(
          half2_max<kF16>(half2_max<kF16>(w[u][0] & 0x7FFF7FFFu,
                                          w[u][1] & 0x7FFF7FFFu),
                          half2_max<kF16>(w[u][2] & 0x7FFF7FFFu,
                                          w[u][3] & 0x7FFF7FFFu)),
          half2_max<kF16>(half2_max<kF16>(w[u][4] & 0x7FFF7FFFu,
                                          w[u][5] & 0x7FFF7FFFu),
                          half2_max<kF16>(w[u][6] & 0x7FFF7FFFu,
                                          w[u][7] & 0x7FFF7FFFu)));
      const float amax = half_lo_to_float<kF16>(half2_max<kF16>(m, m >> 16));
      // IEEE amax / 6 (see the header comment), then * g
      const float q0 = __fmul_rn(amax, inv6);
      const float res = __fmaf_rn(-q0, 6.0f, amax);
      const float d6 = __fmaf_rn(res, inv6, q0);
      const uint32_t sf = float_to_e4m3(__fmul_rn(d6, g));
      const float r = ratio[sf];
      const uint64_t rr = (static_cast<uint64_t>(__float_as_uint(r)) << 32) |
                          __float_as_uint(r);
      uint32_t lo = quant4<kF16>(w[u][0], w[u][1], w[u][2], w[u][3], rr);
      uint32_t hi = quant4<kF16>(w[u][4], w[u][5], w[u][6], w[u][7], rr);
      lo = sf != 0u ? lo : 0u;
      hi = sf != 0u ? hi : 0u;

      int64_t blk, off;
      if (p.b_shift >= 0) {
        blk = slot[u] >> p.b_shift;
        off = slot[u] & (p.B - 1);
      } else {
        blk = slot[u] / p.B;
        off = slot[u] - blk * p.B;
      }
      const int64_t page = blk * p.page_stride;
      st_v2(data_role + page + off * p.dts, lo, hi);
      const int64_t soff =
          swz ? (off & ~int64_t{3}) * p.sts + (off & 3) : off * p.sts;
      scale_role[page + soff] = static_cast<uint8_t>(sf);
    }
  }
}

template <bool kVec32, bool kF16, bool kEarlyRead>
cudaError_t launch(const StoreParams& p, cudaStream_t stream) {
  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int& occ = ctas_per_sm[dev & 63];
  if (occ == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ, store_nvfp4_kernel<kVec32, kF16, kEarlyRead>, kThreads, 0);
    if (err != cudaSuccess) return err;
    if (occ < 1) occ = 1;
  }
  const int slices = 1 << p.slices_log2;
  int64_t grid = static_cast<int64_t>(sm_count()) * occ;
  if (grid > p.num_passes) grid = p.num_passes;
  grid = (grid / slices) * slices;  // every CTA keeps one slice of a token
  if (grid < slices) grid = slices;
  return launch_kernel(store_nvfp4_kernel<kVec32, kF16, kEarlyRead>,
                       static_cast<unsigned>(grid), kThreads, 0, stream,
                       p.pdl, p);
}

}  // namespace

cudaError_t launch_store_nvfp4(const StoreParams& p, cudaStream_t stream) {
  // 256-bit loads need every group start 32-byte aligned
  const bool vec32 =
      (reinterpret_cast<uintptr_t>(p.src[0]) % 32 == 0) &&
      (reinterpret_cast<uintptr_t>(p.src[1]) % 32 == 0) &&
      (p.src_stride[0] % 16 == 0) && (p.src_stride[1] % 16 == 0);
  if (p.early_read) {
    if (p.f16)
      return vec32 ? launch<true, true, true>(p, stream)
                   : launch<false, true, true>(p, stream);
    return vec32 ? launch<true, false, true>(p, stream)
                 : launch<false, false, true>(p, stream);
  }
  if (p.f16)
    return vec32 ? launch<true, true, false>(p, stream)
                 : launch<false, true, false>(p, stream);
  return vec32 ? launch<true, false, false>(p, stream)
               : launch<false, false, false>(p, stream);
}

}  // namespace kvq
