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
//   * HBM-bound: ~2 B read per element, 0.5625 B written.  The grid is
//     persistent (a multiple of the SM count x resident CTAs); every thread
//     owns one fixed 16-byte chunk "role" (side, head, group half) of a token
//     and walks tokens with a grid stride, issuing UNROLL independent 16-byte
//     streaming loads before using any of them, so each SM keeps tens of KB
//     of reads in flight.
//   * A 16-element group is two adjacent lanes (8 bf16 = one 16-byte load
//     each); amax is a packed unsigned max on the sign-cleared bf16 bits
//     (non-negative bf16 order == integer order) plus one xor-1 shuffle.
//   * g = 1/k_scale and g / float(sf) are IEEE divisions; the second one is
//     taken from a 2 x 256-entry shared-memory table filled once per CTA with
//     __fdiv_rn (exactly the per-group IEEE quotient, since sf has only 256
//     codes), so the hot loop holds one division (amax / 6).
//   * e4m3 and e2m1 codes come from the sm_100-family cvt instructions
//     (cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32), round-to-nearest-even.
//   * Each lane stores its 4 packed bytes (a warp writes whole 32-byte
//     sectors of a head row); the even lane of a pair stores the scale byte.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile(
      "ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ int64_t ld_nc_s64(const int64_t* p) {
  int64_t v;
  asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
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
  return pair & 0xFFu;  // second operand lands in the low byte
}

// Eight fp32 -> eight e2m1 codes, element 2k in the low nibble of byte k.
__device__ __forceinline__ uint32_t pack_e2m1x8(const float (&y)[8]) {
  uint32_t out;
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "  cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "  mov.b32 %0, {b0, b1, b2, b3}; }"
      : "=r"(out)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]),
        "f"(y[6]), "f"(y[7]));
  return out;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kThreads)
store_nvfp4_kernel(const StoreParams p) {
  __shared__ float s_ratio[2][256];  // g_side / float(e4m3 code)

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
  int chunk, tok_sub;
  if (slices == 1) {
    tok_sub = tid / p.cpt;
    chunk = tid - tok_sub * p.cpt;
  } else {
    tok_sub = 0;
    chunk = (static_cast<int>(blockIdx.x) & (slices - 1)) * kThreads + tid;
  }
  const bool role_ok = (tok_sub < p.tpp) && (chunk < p.cpt);
  const int cps = p.cpt >> 1;          // chunks per side
  const int side = chunk >= cps ? 1 : 0;
  const int e = chunk - side * cps;
  const int cph = p.D >> 3;            // chunks per head
  const int head = e / cph;
  const int ch = e - head * cph;
  const int grp = ch >> 1;
  const int half = ch & 1;
  const int q = p.S >> 2;
  const bool swz = (p.swizzle_sides >> side) & 1u;

  const uint16_t* src_base = p.src[side] + head * p.D + ch * 8;
  const int64_t src_stride = p.src_stride[side];
  uint8_t* const data_base = p.side[side] + head * p.dhs + grp * 8 + half * 4;
  uint8_t* const scale_base =
      p.side[side] + p.data_per_side + head * p.shs +
      (swz ? (grp / q) * p.sts + (grp % q) * 4 : static_cast<int64_t>(grp));
  const float* ratio = s_ratio[side];
  const float g = __fdiv_rn(1.0f, __ldg(p.scale[side]));

  const int grid = gridDim.x;
  for (int p0 = blockIdx.x; p0 < p.num_passes; p0 += kUnroll * grid) {
    uint4 raw[kUnroll];
    int64_t slot[kUnroll];
    bool act[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int pass = p0 + u * grid;
      const int t = (pass >> p.slices_log2) * p.tpp + tok_sub;
      act[u] = role_ok && pass < p.num_passes && t < p.num_tokens;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      slot[u] = -1;
      if (act[u]) {
        slot[u] = ld_nc_s64(p.slots + t);
        raw[u] = ld_stream_16(src_base + static_cast<int64_t>(t) * src_stride);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      // group amax over the lane pair (all lanes take part in the shuffle)
      const uint32_t m01 = __vmaxu2(raw[u].x & 0x7FFF7FFFu,
                                    raw[u].y & 0x7FFF7FFFu);
      const uint32_t m23 = __vmaxu2(raw[u].z & 0x7FFF7FFFu,
                                    raw[u].w & 0x7FFF7FFFu);
      const uint32_t m = __vmaxu2(m01, m23);
      uint32_t a = max(m & 0xFFFFu, m >> 16);
      a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));

      if (!act[u] || slot[u] < 0) continue;
      if (slot[u] >= p.num_slots) {
        if (p.dev_error != nullptr && half == 0)
          atomicOr(p.dev_error, KVQ_DEVERR_SLOT);
        continue;
      }
      const float amax = __uint_as_float(a << 16);
      const float sfv = __fmul_rn(__fdiv_rn(amax, 6.0f), g);
      const uint32_t sf = float_to_e4m3(sfv);

      uint32_t packed = 0u;
      if (sf != 0u) {
        const float r = ratio[sf];
        float y[8];
        y[0] = __fmul_rn(bf16_lo(raw[u].x), r);
        y[1] = __fmul_rn(bf16_hi(raw[u].x), r);
        y[2] = __fmul_rn(bf16_lo(raw[u].y), r);
        y[3] = __fmul_rn(bf16_hi(raw[u].y), r);
        y[4] = __fmul_rn(bf16_lo(raw[u].z), r);
        y[5] = __fmul_rn(bf16_hi(raw[u].z), r);
        y[6] = __fmul_rn(bf16_lo(raw[u].w), r);
        y[7] = __fmul_rn(bf16_hi(raw[u].w), r);
        packed = pack_e2m1x8(y);
      }
      int64_t blk, off;
      if (p.b_shift >= 0) {
        blk = slot[u] >> p.b_shift;
        off = slot[u] & (p.B - 1);
      } else {
        blk = slot[u] / p.B;
        off = slot[u] - blk * p.B;
      }
      const int64_t page = blk * p.page_stride;
      *reinterpret_cast<uint32_t*>(data_base + page + off * p.dts) = packed;
      if (half == 0) {
        const int64_t soff = swz ? (off & ~int64_t{3}) * p.sts + (off & 3)
                                 : off * p.sts;
        scale_base[page + soff] = static_cast<uint8_t>(sf);
      }
    }
  }
}

}  // namespace

cudaError_t launch_store_nvfp4(const StoreParams& p, cudaStream_t stream) {
  static int ctas_per_sm[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int& occ = ctas_per_sm[dev & 63];
  if (occ == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &occ, store_nvfp4_kernel, kThreads, 0);
    if (err != cudaSuccess) return err;
    if (occ < 1) occ = 1;
  }
  const int slices = 1 << p.slices_log2;
  int64_t grid = static_cast<int64_t>(sm_count()) * occ;
  if (grid > p.num_passes) grid = p.num_passes;
  grid = (grid / slices) * slices;  // every CTA keeps one slice of a token
  if (grid < slices) grid = slices;
  store_nvfp4_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
