/*
 * kvq_oracle.c -- plain, slow CPU oracle for the paged quantized KV-cache
 * write/read path.  TEST INFRASTRUCTURE ONLY: the library under
 * paged_quantized_kv_gb300/ never links, loads or calls this file; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg do.
 *
 * It restates, step by step and without blocking, fusion or reordering, the
 * operations described on these pages:
 *   [nvfp4-cu]  vLLM csrc/libtorch_stable/nvfp4_kv_cache_kernels.cu
 *               (commit 7ce4c8e): "swizzle_scale_offset" comment block,
 *               "reshape_and_cache_nvfp4_kernel" and
 *               "reshape_and_cache_nvfp4_dispatch".
 *   [pr25931]   vLLM PR #25931 "Add gather_indexer_k_quant_cache kernel".
 *   [pr26456]   vLLM PR #26456 "[Deepseek-V3.2][Kernel] Integrate cuda
 *               indexer k cache gather" (k_scale viewed as float32).
 *   [rocm-cpa]  vLLM PR #12348 "[ROCm] Faster Custom Paged Attention
 *               kernels": the paged_attention op signature (decode
 *               attention over a paged, quantised KV cache).
 *
 * The per-group quantiser (cvt_warp_fp16_to_fp4) is named but not shown on
 * the pages; its rule is taken as: amax over the 16 values,
 * sf = e4m3_rn_satfinite((amax / 6) * g) with g = 1 / k_scale, every element
 * e2m1_rn_satfinite(x * (g / float(sf))) or 0 when sf == 0, two elements per
 * byte with the even element in the low nibble.  Every division is an IEEE
 * fp32 division, every product one fp32 rounding, no fused multiply-add
 * (build with -ffp-contract=off, no -ffast-math).
 *
 * Format tables are built from the bit-level definitions of the two formats
 * (OCP 8-bit e4m3 "fn" variant: bias 7, no infinities, 0x7F/0xFF NaN, max
 * 448; e2m1: bias 1, no inf/NaN, max 6) and every encoding is a search over
 * the table with round-to-nearest, ties to the even code, saturating to the
 * largest finite magnitude.
 *
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVQO_OK 0
#define KVQO_ERR_ARG (-1)
#define KVQO_ERR_NONFINITE (-2)
#define KVQO_ERR_BOUNDS (-3)

#define KVQO_LAYOUT_HND 0
#define KVQO_LAYOUT_NHD 1
#define KVQO_DTYPE_BF16 0
#define KVQO_DTYPE_F16 1
#define KVQO_F_SWIZZLE_K_SCALE 1u

/* ------------------------------------------------------------------------ */
/* Format tables                                                            */
/* ------------------------------------------------------------------------ */

/* Non-negative finite e4m3 codes 0x00..0x7E and e2m1 codes 0..7. */
static double e4m3_val[127];
static double e2m1_val[8];
static int tables_ready = 0;

static void build_tables(void) {
  if (tables_ready) return;
  for (int c = 0; c < 127; ++c) {
    int e = (c >> 3) & 0xF, m = c & 7;
    /* subnormal: m/8 * 2^(1-7); normal: (1 + m/8) * 2^(e-7) */
    e4m3_val[c] = (e == 0) ? ldexp((double)m / 8.0, 1 - 7)
                           : ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  for (int c = 0; c < 8; ++c) {
    int e = (c >> 1) & 3, m = c & 1;
    /* subnormal: m/2 * 2^(1-1); normal: (1 + m/2) * 2^(e-1) */
    e2m1_val[c] = (e == 0) ? ldexp((double)m / 2.0, 1 - 1)
                           : ldexp(1.0 + (double)m / 2.0, e - 1);
  }
  tables_ready = 1;
}

/* Round |v| to the nearest table entry, ties to the even code, saturating
 * at the top entry.  vals[] is strictly increasing, vals[0] == 0. */
static int encode_magnitude(double a, const double* vals, int n) {
  if (a >= vals[n - 1]) return n - 1;
  int c = 0;
  while (!(vals[c] <= a && a < vals[c + 1])) ++c;
  double mid = 0.5 * (vals[c] + vals[c + 1]); /* exact in double */
  if (a < mid) return c;
  if (a > mid) return c + 1;
  return (c % 2 == 0) ? c : c + 1;
}

double kvqo_e4m3_decode(uint8_t code) {
  build_tables();
  int mag = code & 0x7F;
  if (mag == 0x7F) return NAN;
  double v = e4m3_val[mag];
  return (code & 0x80) ? -v : v;
}

double kvqo_e2m1_decode(uint8_t nibble) {
  build_tables();
  double v = e2m1_val[nibble & 7];
  return (nibble & 8) ? -v : v;
}

/* e4m3 round-to-nearest-even, satfinite; the sign of v (including -0) is
 * kept.  Saturation covers infinities (+-inf -> +-448); NaN returns 0x7F. */
uint8_t kvqo_e4m3_encode(float v) {
  build_tables();
  if (isnan(v)) return 0x7F;
  int mag = encode_magnitude(fabs((double)v), e4m3_val, 127);
  return (uint8_t)((signbit(v) ? 0x80 : 0x00) | mag);
}

/* e2m1 round-to-nearest-even, satfinite; the sign of v (including -0) is
 * kept in bit 3.  Saturation covers infinities (+-inf -> +-6); e2m1 has no
 * NaN, so NaN input returns 0xF. */
uint8_t kvqo_e2m1_encode(float v) {
  build_tables();
  if (isnan(v)) return 0xF;
  int mag = encode_magnitude(fabs((double)v), e2m1_val, 8);
  return (uint8_t)((signbit(v) ? 0x8 : 0x0) | mag);
}

/* bf16 bits -> fp32 (exact). */
static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* IEEE binary16 bits -> fp32 (exact): 1 sign, 5 exponent (bias 15),
 * 10 mantissa; subnormals m * 2^-24; exponent 31 is inf / NaN. */
static float f16_to_float(uint16_t h) {
  int sign = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = (m == 0) ? INFINITY : NAN;
  else
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  return (float)(sign ? -v : v);
}

double kvqo_f16_decode(uint16_t h) { return (double)f16_to_float(h); }

static float element_to_float(uint16_t x, int dtype) {
  return dtype == KVQO_DTYPE_F16 ? f16_to_float(x) : bf16_to_float(x);
}

/* ------------------------------------------------------------------------ */
/* Scale-tile swizzle ([nvfp4-cu] "swizzle_scale_offset" comment):          */
/* the [T, S] tile viewed as [T/4, 4, 4, S/4], permuted (0, 2, 3, 1) and    */
/* read back as [T, S].  Returns row * S + col of the swizzled position.    */
/* ------------------------------------------------------------------------ */
int kvqo_swizzle(int t, int s, int S) {
  int q = S / 4;
  int row = (t / 4) * 4 + s / q;
  int col = (s % q) * 4 + t % 4;
  return row * S + col;
}

/* ------------------------------------------------------------------------ */
/* One 16-element group ([nvfp4-cu] kernel: load group, quantise, pack).     */
/* x: 16 bf16 (or fp16, dtype) bit patterns.  g: global scale (1/k_scale).  */
/* data8: 8 output bytes.  *sf: e4m3 scale code.                             */
/* ------------------------------------------------------------------------ */
int kvqo_quantize_group_t(const uint16_t* x, int dtype, float g,
                          uint8_t* data8, uint8_t* sf_out) {
  float xs[16];
  for (int i = 0; i < 16; ++i) {
    xs[i] = element_to_float(x[i], dtype);
    if (!isfinite(xs[i])) return KVQO_ERR_NONFINITE;
  }
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = fabsf(xs[i]);
    if (a > amax) amax = a;
  }
  float sfv = (amax / 6.0f) * g; /* two IEEE fp32 roundings */
  uint8_t sf = kvqo_e4m3_encode(sfv);
  uint8_t q[16];
  if (sf == 0) {
    for (int i = 0; i < 16; ++i) q[i] = 0;
  } else {
    float r = g / (float)kvqo_e4m3_decode(sf); /* IEEE fp32 division */
    for (int i = 0; i < 16; ++i) q[i] = kvqo_e2m1_encode(xs[i] * r);
  }
  for (int k = 0; k < 8; ++k)
    data8[k] = (uint8_t)(q[2 * k] | (q[2 * k + 1] << 4));
  *sf_out = sf;
  return KVQO_OK;
}

int kvqo_quantize_group(const uint16_t* x, float g, uint8_t* data8,
                        uint8_t* sf_out) {
  return kvqo_quantize_group_t(x, KVQO_DTYPE_BF16, g, data8, sf_out);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 paged store ([nvfp4-cu] kernel and dispatch).                      */
/*                                                                          */
/* key/value: bf16 (dtype 0) or fp16 (dtype 1) bits [num_tokens, H, D],    */
/*   row stride key_stride0 /                                               */
/*   value_stride0 elements, heads and elements contiguous.                 */
/* key_cache/value_cache: base of the K side and of the V side of page 0    */
/*   (kv_cache[:, 0] and kv_cache[:, 1]); pages are page_stride bytes apart. */
/*   Inside one side: data region [H, B, D/2] (HND) or [B, H, D/2] (NHD),    */
/*   then the scale region at +H*B*D/2, [H, B, S] or [B, H, S].              */
/* slot_mapping: int64 per token; slot < 0 skips the token.                 */
/* k_scale/v_scale: the per-tensor scales; g = 1/k_scale, 1/v_scale.         */
/* flags & KVQO_F_SWIZZLE_K_SCALE: K scales also swizzled (default linear). */
/* Bytes of the cache that no token owns are left as they were.             */
/* ------------------------------------------------------------------------ */
int kvqo_store_nvfp4(const uint16_t* key, int64_t key_stride0,
                     const uint16_t* value, int64_t value_stride0,
                     int32_t dtype, int32_t num_tokens, int32_t num_heads,
                     int32_t head_size,
                     uint8_t* key_cache, uint8_t* value_cache,
                     int64_t page_stride, int32_t block_size,
                     int64_t num_blocks, int32_t layout,
                     const int64_t* slot_mapping, float k_scale, float v_scale,
                     uint32_t flags) {
  if (num_tokens < 0 || num_heads <= 0 || head_size <= 0 || block_size <= 0)
    return KVQO_ERR_ARG;
  if (head_size % 64 != 0 || block_size % 4 != 0) return KVQO_ERR_ARG;
  if (layout != KVQO_LAYOUT_HND && layout != KVQO_LAYOUT_NHD)
    return KVQO_ERR_ARG;
  if (dtype != KVQO_DTYPE_BF16 && dtype != KVQO_DTYPE_F16) return KVQO_ERR_ARG;

  const int64_t H = num_heads, D = head_size, B = block_size;
  const int64_t data_dim = D / 2, S = D / 16;
  const int64_t groups_per_head = D / 16;

  /* Inner strides of one side ([nvfp4-cu] dispatch, layout detection). */
  int64_t dhs, dts, shs, sts;
  if (layout == KVQO_LAYOUT_HND) {
    dhs = B * data_dim; dts = data_dim;
    shs = B * S;        sts = S;
  } else {
    dhs = data_dim;     dts = H * data_dim;
    shs = S;            sts = H * S;
  }
  const int64_t data_per_side = H * B * data_dim;

  /* S2: global scale per side. */
  const float g_side[2] = {1.0f / k_scale, 1.0f / v_scale};

  for (int64_t t = 0; t < num_tokens; ++t) {
    /* S1: slot decode, skip rule. */
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / B;
    const int64_t off = slot % B;
    if (blk >= num_blocks) return KVQO_ERR_BOUNDS;

    for (int side = 0; side < 2; ++side) {
      const uint16_t* src = (side == 0) ? key + t * key_stride0
                                        : value + t * value_stride0;
      uint8_t* side_base = (side == 0) ? key_cache : value_cache;
      uint8_t* data_page = side_base + blk * page_stride;
      uint8_t* scale_page = data_page + data_per_side;
      const float g = g_side[side];
      const int swizzle = (side == 1) || (flags & KVQO_F_SWIZZLE_K_SCALE);

      for (int64_t h = 0; h < H; ++h) {
        for (int64_t j = 0; j < groups_per_head; ++j) {
          /* S3..S5 */
          uint8_t packed[8], sf;
          int rc = kvqo_quantize_group_t(src + h * D + 16 * j, dtype, g,
                                         packed, &sf);
          if (rc != KVQO_OK) return rc;
          /* S6: 8 data bytes of group j. */
          uint8_t* dst = data_page + h * dhs + off * dts + 8 * j;
          for (int k = 0; k < 8; ++k) dst[k] = packed[k];
          /* S7: scale byte, linear or swizzled inside the head's tile. */
          uint8_t* sdst;
          if (!swizzle) {
            sdst = scale_page + h * shs + off * sts + j;
          } else {
            int pos = kvqo_swizzle((int)off, (int)j, (int)S);
            int64_t row = pos / S, col = pos % S;
            sdst = scale_page + h * shs + row * sts + col;
          }
          *sdst = sf;
        }
      }
    }
  }
  return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* Indexer-K gather ([pr25931] cp_gather_indexer_k_quant_cache; [pr26456]   */
/* scale bytes viewed as float32 by the consumer).                          */
/*                                                                          */
/* cache: blocks block_stride bytes apart; block = [B*D fp8 K | B*4 scale]. */
/* block_table: int32 [num_seqs, bt_stride]; cu_seq_lens: int32 [num_seqs+1]*/
/* Sequence b's token p (0 <= p < len_b) is output row cu[b] + p:           */
/*   k_fp8[row, 0:D]      = K bytes of (block_table[b, p/B], p%B)            */
/*   k_scale[4*row, +4]   = the 4 scale bytes of that token (raw copy).      */
/* Rows at or beyond total_tokens are not written.                          */
/* ------------------------------------------------------------------------ */
int kvqo_gather_indexer_k(const uint8_t* cache, int64_t block_stride,
                          int64_t num_blocks, int32_t block_size,
                          int32_t head_dim, const int32_t* block_table,
                          int64_t bt_stride, int32_t max_blocks_per_seq,
                          const int32_t* cu_seq_lens, int32_t num_seqs,
                          int64_t total_tokens, uint8_t* k_fp8,
                          uint8_t* k_scale) {
  if (num_seqs < 0 || block_size <= 0 || head_dim <= 0 || total_tokens < 0)
    return KVQO_ERR_ARG;
  const int64_t B = block_size, D = head_dim;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int64_t start = cu_seq_lens[b];
    const int64_t len = (int64_t)cu_seq_lens[b + 1] - start;
    for (int64_t p = 0; p < len; ++p) {
      const int64_t row = start + p;
      if (row < 0 || row >= total_tokens) return KVQO_ERR_BOUNDS;
      if (p / B >= max_blocks_per_seq) return KVQO_ERR_BOUNDS;
      const int64_t blk = block_table[b * bt_stride + p / B];
      const int64_t off = p % B;
      if (blk < 0 || blk >= num_blocks) return KVQO_ERR_BOUNDS;
      const uint8_t* block = cache + blk * block_stride;
      for (int64_t d = 0; d < D; ++d) k_fp8[row * D + d] = block[off * D + d];
      for (int k = 0; k < 4; ++k)
        k_scale[row * 4 + k] = block[B * D + off * 4 + k];
    }
  }
  return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* NVFP4 paged load -- the read side of the store ([nvfp4-cu] page layout   */
/* and swizzle; the pages give no dequantisation rule, so this is the plain */
/* inverse of the store's: x' = e2m1(q) * (float(sf) * k_scale), the scale  */
/* product and the element product each one fp32 rounding, then rounded to  */
/* bf16, nearest-even).                                                     */
/*                                                                          */
/* Sequence b's token p (0 <= p < cu[b+1]-cu[b]) is output row cu[b] + p,   */
/* read from page block_table[b*bt_stride + p/B], offset p%B.  key_out /     */
/* value_out: bf16 bits [total, H, D] with row stride out_stride0 elements. */
/* ------------------------------------------------------------------------ */

/* fp32 -> bf16 bits, round to nearest even (NaN -> quiet NaN). */
static uint16_t float_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

uint16_t kvqo_float_to_bf16(float f) { return float_to_bf16(f); }

int kvqo_load_nvfp4(const uint8_t* key_cache, const uint8_t* value_cache,
                    int64_t page_stride, int32_t block_size,
                    int64_t num_blocks, int32_t layout, int32_t num_heads,
                    int32_t head_size, const int32_t* block_table,
                    int64_t bt_stride, int32_t max_blocks_per_seq,
                    const int32_t* cu_seq_lens, int32_t num_seqs,
                    int64_t total_tokens, float k_scale, float v_scale,
                    uint32_t flags, uint16_t* key_out, uint16_t* value_out,
                    int64_t out_stride0) {
  if (num_heads <= 0 || head_size <= 0 || block_size <= 0 || num_seqs < 0)
    return KVQO_ERR_ARG;
  if (head_size % 64 != 0 || block_size % 4 != 0) return KVQO_ERR_ARG;
  if (layout != KVQO_LAYOUT_HND && layout != KVQO_LAYOUT_NHD)
    return KVQO_ERR_ARG;
  const int64_t H = num_heads, D = head_size, B = block_size;
  const int64_t data_dim = D / 2, S = D / 16;
  int64_t dhs, dts, shs, sts;
  if (layout == KVQO_LAYOUT_HND) {
    dhs = B * data_dim; dts = data_dim;
    shs = B * S;        sts = S;
  } else {
    dhs = data_dim;     dts = H * data_dim;
    shs = S;            sts = H * S;
  }
  const int64_t data_per_side = H * B * data_dim;
  const float side_scale[2] = {k_scale, v_scale};

  for (int32_t b = 0; b < num_seqs; ++b) {
    const int64_t start = cu_seq_lens[b];
    const int64_t len = (int64_t)cu_seq_lens[b + 1] - start;
    for (int64_t p = 0; p < len; ++p) {
      const int64_t row = start + p;
      if (row < 0 || row >= total_tokens) return KVQO_ERR_BOUNDS;
      if (p / B >= max_blocks_per_seq) return KVQO_ERR_BOUNDS;
      const int64_t blk = block_table[b * bt_stride + p / B];
      const int64_t off = p % B;
      if (blk < 0 || blk >= num_blocks) return KVQO_ERR_BOUNDS;
      for (int side = 0; side < 2; ++side) {
        const uint8_t* page =
            (side == 0 ? key_cache : value_cache) + blk * page_stride;
        const uint8_t* scale_page = page + data_per_side;
        uint16_t* out = (side == 0 ? key_out : value_out) + row * out_stride0;
        const int swizzle = (side == 1) || (flags & KVQO_F_SWIZZLE_K_SCALE);
        for (int64_t h = 0; h < H; ++h) {
          for (int64_t j = 0; j < S; ++j) {
            const uint8_t* sptr;
            if (!swizzle) {
              sptr = scale_page + h * shs + off * sts + j;
            } else {
              int pos = kvqo_swizzle((int)off, (int)j, (int)S);
              sptr = scale_page + h * shs + (pos / S) * sts + pos % S;
            }
            const float c = (float)kvqo_e4m3_decode(*sptr) * side_scale[side];
            const uint8_t* dptr = page + h * dhs + off * dts + 8 * j;
            for (int k = 0; k < 16; ++k) {
              const uint8_t byte = dptr[k / 2];
              const uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
              const float v = (float)kvqo_e2m1_decode(nib) * c;
              out[h * D + 16 * j + k] = float_to_bf16(v);
            }
          }
        }
      }
    }
  }
  return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* Indexer-K store -- the write side of the cache the gather reads          */
/* ([pr25931]: "quantized k/k_scale" in a paged indexer cache of blocks     */
/* [B*D fp8 K | B*4 fp32 scale]).  The pages give no quantisation rule; the */
/* reading taken is per-token absmax scaling: scale = amax / 448 (fp32      */
/* IEEE division), q_i = e4m3_rn_satfinite(k_i / scale) (IEEE division),   */
/* or q_i = 0 when amax = 0.  Token t with slot s >= 0 goes to block s / B, */
/* row s % B; slot < 0 is skipped.                                          */
/* ------------------------------------------------------------------------ */
int kvqo_store_indexer_k(const uint16_t* k, int64_t k_stride0, int32_t dtype,
                         int32_t num_tokens, int32_t head_dim, uint8_t* cache,
                         int64_t block_stride, int32_t block_size,
                         int64_t num_blocks, const int64_t* slot_mapping) {
  if (num_tokens < 0 || head_dim <= 0 || block_size <= 0) return KVQO_ERR_ARG;
  if (dtype != KVQO_DTYPE_BF16 && dtype != KVQO_DTYPE_F16) return KVQO_ERR_ARG;
  const int64_t B = block_size, D = head_dim;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t blk = slot / B, off = slot % B;
    if (blk >= num_blocks) return KVQO_ERR_BOUNDS;
    const uint16_t* row = k + t * k_stride0;
    float amax = 0.0f;
    for (int64_t d = 0; d < D; ++d) {
      const float x = element_to_float(row[d], dtype);
      if (!isfinite(x)) return KVQO_ERR_NONFINITE;
      if (fabsf(x) > amax) amax = fabsf(x);
    }
    const float scale = amax / 448.0f; /* IEEE fp32 division */
    uint8_t* dst = cache + blk * block_stride + off * D;
    for (int64_t d = 0; d < D; ++d) {
      const float x = element_to_float(row[d], dtype);
      dst[d] = (amax == 0.0f) ? 0 : kvqo_e4m3_encode(x / scale);
    }
    memcpy(cache + blk * block_stride + B * D + off * 4, &scale, 4);
  }
  return KVQO_OK;
}

/* ------------------------------------------------------------------------ */
/* Paged decode attention over the NVFP4 cache ([rocm-cpa]: vLLM PR #12348  */
/* "[ROCm] Faster Custom Paged Attention kernels", the paged_attention op   */
/* signature: out, query, key_cache, value_cache, num_kv_heads, scale,      */
/* block_tables, context_lens, block_size, k_scale, v_scale).  The page     */
/* shows the signature only; the computation taken is plain softmax         */
/* attention of each sequence's one query token over its first              */
/* context_lens[b] cached tokens, on the cache dequantised exactly:         */
/*   K^[t, d] = e2m1(q) * float(sf) * k_scale  (V^ with v_scale),           */
/* sf read where the store put it (K linear unless KVQO_F_SWIZZLE_K_SCALE,  */
/* V swizzled).  Query head h reads KV head h / (Hq / Hkv).  Everything in  */
/* double:                                                                  */
/*   s_t = scale * sum_d q[h, d] * K^[t, d];   m = max_t s_t                */
/*   p_t = exp(s_t - m) / sum_u exp(s_u - m);  out[h, d] = sum_t p_t V^[t,d] */
/* context_lens[b] == 0 gives out = 0.  mag[h, d] = sum_t p_t |V^[t, d]|    */
/* is returned beside out (the scale of the rounding error of any          */
/* finite-precision evaluation).  query: bf16 / fp16 bits [num_seqs, Hq, D] */
/* with row stride q_stride0 elements; out, mag: double [num_seqs, Hq, D].  */
/* ------------------------------------------------------------------------ */

/* One token's dequantised row (head h, page blk, offset off) of one side. */
static void nvfp4_row_exact(const uint8_t* side_base, int64_t page_stride,
                            int64_t blk, int64_t off, int64_t h, int64_t H,
                            int64_t B, int64_t D, int32_t layout,
                            int swizzle, double side_scale, double* row) {
  const int64_t data_dim = D / 2, S = D / 16;
  int64_t dhs, dts, shs, sts;
  if (layout == KVQO_LAYOUT_HND) {
    dhs = B * data_dim; dts = data_dim;
    shs = B * S;        sts = S;
  } else {
    dhs = data_dim;     dts = H * data_dim;
    shs = S;            sts = H * S;
  }
  const uint8_t* page = side_base + blk * page_stride;
  const uint8_t* scale_page = page + H * B * data_dim;
  for (int64_t j = 0; j < S; ++j) {
    const uint8_t* sptr;
    if (!swizzle) {
      sptr = scale_page + h * shs + off * sts + j;
    } else {
      int pos = kvqo_swizzle((int)off, (int)j, (int)S);
      sptr = scale_page + h * shs + (pos / S) * sts + pos % S;
    }
    const double sf = kvqo_e4m3_decode(*sptr);
    const uint8_t* dptr = page + h * dhs + off * dts + 8 * j;
    for (int k = 0; k < 16; ++k) {
      const uint8_t byte = dptr[k / 2];
      const uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
      row[16 * j + k] = kvqo_e2m1_decode(nib) * sf * side_scale;
    }
  }
}

int kvqo_paged_attention_nvfp4(
    const uint16_t* query, int64_t q_stride0, int32_t q_dtype,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_size, const uint8_t* key_cache, const uint8_t* value_cache,
    int64_t page_stride, int32_t block_size, int64_t num_blocks,
    int32_t layout, const int32_t* block_table, int64_t bt_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens, float k_scale,
    float v_scale, float scale, uint32_t flags, double* out, double* mag) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_size <= 0 || block_size <= 0)
    return KVQO_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0) return KVQO_ERR_ARG;
  if (head_size % 64 != 0 || block_size % 4 != 0) return KVQO_ERR_ARG;
  if (layout != KVQO_LAYOUT_HND && layout != KVQO_LAYOUT_NHD)
    return KVQO_ERR_ARG;
  if (q_dtype != KVQO_DTYPE_BF16 && q_dtype != KVQO_DTYPE_F16)
    return KVQO_ERR_ARG;
  const int64_t Hq = num_q_heads, Hkv = num_kv_heads, D = head_size;
  const int64_t B = block_size, G = Hq / Hkv;
  const int k_swizzle = (flags & KVQO_F_SWIZZLE_K_SCALE) != 0;
  double* krow = malloc(sizeof(double) * D);
  double* vrow = malloc(sizeof(double) * D);
  if (!krow || !vrow) { free(krow); free(vrow); return KVQO_ERR_ARG; }
  int rc = KVQO_OK;

  for (int32_t b = 0; b < num_seqs && rc == KVQO_OK; ++b) {
    const int64_t L = context_lens[b];
    if (L < 0 || (L + B - 1) / B > max_blocks_per_seq) {
      rc = KVQO_ERR_BOUNDS;
      break;
    }
    double* s = malloc(sizeof(double) * (L > 0 ? L : 1));
    if (!s) { rc = KVQO_ERR_ARG; break; }
    for (int64_t h = 0; h < Hq && rc == KVQO_OK; ++h) {
      const int64_t kh = h / G;
      const uint16_t* q = query + b * q_stride0 + h * D;
      double* o = out + (b * Hq + h) * D;
      double* mg = mag + (b * Hq + h) * D;
      for (int64_t d = 0; d < D; ++d) { o[d] = 0.0; mg[d] = 0.0; }
      if (L == 0) continue;
      /* logits */
      for (int64_t t = 0; t < L; ++t) {
        const int64_t blk = block_table[b * bt_stride + t / B];
        if (blk < 0 || blk >= num_blocks) { rc = KVQO_ERR_BOUNDS; break; }
        nvfp4_row_exact(key_cache, page_stride, blk, t % B, kh, Hkv, B, D,
                        layout, k_swizzle, (double)k_scale, krow);
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
          dot += (double)element_to_float(q[d], q_dtype) * krow[d];
        s[t] = (double)scale * dot;
      }
      if (rc != KVQO_OK) break;
      /* softmax */
      double m = s[0];
      for (int64_t t = 1; t < L; ++t) if (s[t] > m) m = s[t];
      double l = 0.0;
      for (int64_t t = 0; t < L; ++t) l += exp(s[t] - m);
      /* weighted sum of values */
      for (int64_t t = 0; t < L; ++t) {
        const int64_t blk = block_table[b * bt_stride + t / B];
        nvfp4_row_exact(value_cache, page_stride, blk, t % B, kh, Hkv, B, D,
                        layout, 1, (double)v_scale, vrow);
        const double p = exp(s[t] - m) / l;
        for (int64_t d = 0; d < D; ++d) {
          o[d] += p * vrow[d];
          mg[d] += p * fabs(vrow[d]);
        }
      }
    }
    free(s);
  }
  free(krow);
  free(vrow);
  return rc;
}
