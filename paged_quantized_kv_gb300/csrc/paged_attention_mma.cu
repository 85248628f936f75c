// paged_attention_mma.cu -- paged decode attention over the NVFP4 KV cache,
// sm_103a, on warp-level tensor-core MMAs (mma.sync m16n8k16, fp16
// operands, fp32 accumulators) with register fragments.
//
// Operation: the paged_attention op of vLLM PR #12348 "[ROCm] Faster Custom
// Paged Attention kernels" (out, exp_sums, max_logits, tmp_out, query,
// key_cache, value_cache, num_kv_heads, scale, block_tables, context_lens,
// block_size, max_context_len, k_scale, v_scale, partition_size), read over
// the NVFP4 pages of vLLM nvfp4_kv_cache_kernels.cu (commit 7ce4c8e): for
// sequence b and query head h (KV head h / G) over the first
// context_lens[b] tokens, out = softmax(scale * q . K^) V^ with
// K^ = e2m1(code) * float(sf) * k_scale (V^ with v_scale).  A context
// longer than one CTA's stretch is split: each stretch writes its max
// logit, exp-sum and normalised output to the caller's scratch, and a
// second small kernel (the partition merge, at the end of this file)
// combines them.
//
// Why warp-level MMAs here: a decode step multiplies each 128-token tile by
// at most 16 query heads, so every MMA is tiny (N = 8 or 16).  Measured on
// GB300, one thread issues tcgen05.mma at 43-89 cycles per instruction at
// that shape (the tensor core finishes each in ~25), and the handshakes
// around tensor memory (commit, mbarrier wake-up ~300 cycles) sit on every
// tile's critical path; mma.sync.m16n8k16 runs at 2 cycles per instruction
// per SM with its operands already in registers and needs no handshake.
// Two tcgen05 designs of this operation (one CTA per partition with the
// logits held in tensor memory; a persistent warp-specialised one) measured
// 0.25 and 0.11 of the HBM roofline against this kernel's 0.66 (0.78 now)
// on the Llama-70B-shaped step, and 0.20 / 0.10 against 0.39 (0.45 now)
// with 16 query heads per KV head, so they were retired.
//
// Design, per CTA of 4 warps = one (stretch of context, KV head, sequence):
// on contiguous pages (a power-of-two block_size >= 16: HND, whose 16-token
// halves are contiguous, or NHD, whose token rows are copied row by row; K
// scales linear or swizzled) a context of L tokens is split into
// n = ceil(L / KVQ_ATTN_MMA_PART)
// stretches (KVQ_ATTN_MMA_PART = 1792; boundaries at multiples of 32
// tokens) in the proportions 4 : ... : 4 : 1, elsewhere into the caller's
// partitions (<= 512 tokens); the CTAs are launched stretch-major (every
// context's first stretch, then the second ones, ...), so that the CTAs
// that start last, when the SMs begin to fall idle, are the short last
// stretches; a stretch's tokens are split evenly over the warps, which walk
// them in steps of 32 tokens:
//   * Loads: cp.async into the warp's own shared-memory slots, kDepth steps
//     ahead; the warp waits with cp.async.wait_group only.  Block ids of the
//     warp's range are loaded once (one or two per lane) and shuffled.  On
//     contiguous pages one block id serves 16 tokens and the pages' bytes
//     keep their order (16-byte copies, a step's scales in one or two
//     copies per lane; a bad block id zero-filled); elsewhere every thread
//     copies exactly the bytes its own MMA fragments need, zero-filled for
//     tokens past the context or with a bad block id.  The query fragments
//     are staged in shared memory once per CTA.
//   * Logits S^T[16 tokens x 8 heads] = K' Q'^T per n-block of 8 query
//     heads: A = K' (rows = tokens), B = Q'^T (k = head dims).  The head
//     dims are permuted (the same way for K and Q): in k-step s, lane
//     (g, t) holds dims 32t + 4s .. 32t + 4s + 3, so one lane's bytes of a
//     token are the contiguous 16 bytes 16t .. 16t + 15 (groups 2t, 2t+1).
//   * e2m1 -> fp16 with cvt.rn.f16x2.e2m1x2 times the group scale
//     (cvt.rn.f16x2.e4m3x2, one packed multiply): e2m1 * sf has at most 6
//     significant bits and lies in [2^-10, 2688], so the operand is exact.
//   * Online softmax over the warp's steps (exp2 of the scaled logits minus
//     a running reference, rounded to fp16; the denominator sums the
//     rounded weights, by an MMA of an all-ones A with the weights; the
//     reference moves, and the accumulators are rescaled, only when a
//     step's maximum exceeds it by more than 8, so weights stay below
//     2^8 and most steps skip the rescale).  The fp16
//     weights P^T (tokens x heads, in the logits' accumulator layout) are
//     transposed into the B fragment of the second product with
//     movmatrix.
//   * O^T += V'^T P^T per 8-token block, with the contraction index running
//     over (token, e) pairs so that a V byte (dims 2p, 2p+1 of a token) is
//     one A register as it stands: the same A meets a B holding each
//     token's weight at e = 0 (this product sums the even dims) and one
//     holding it at e = 1 (the odd dims).  Lane (g, t) reads the 8
//     contiguous bytes 8g .. 8g+7 (group g) of tokens 2t and 2t+1 of each
//     block; the rows of m-block mb are bytes 2mb and 2mb+1 of the group.
//   * A step none of whose tokens is left out (all in the warp's range,
//     every block id valid -- every step but a partial last one) runs a
//     form with no per-token test at all.
//   * The 4 warps' (max, sum, O) merge in shared memory (each warp writes
//     its own into its copy slots, one barrier, every output thread
//     combines the four for its head); a stretch of a longer context is
//     written to the caller's scratch (rows max_parts apart, as for the
//     caller's partitions: a stretch covers at least one partition, so
//     fewer rows are used) and merged by the partition-merge kernel.
//   * Start-up: the query loads go out with the block-id loads and are
//     staged once the first step's copies are issued; with
//     KVQ_F_PDL_EARLY_META the context length, block ids, query and scales
//     are read before the PDL wait.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "kvq_internal.h"
#include "kvq.h"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kD = 128;          // head_size
constexpr int kStep = 32;        // tokens per warp step
#ifndef KVQ_ATTN_MMA_DEPTH
#define KVQ_ATTN_MMA_DEPTH 2
#endif
constexpr int kDepth = KVQ_ATTN_MMA_DEPTH;  // steps in flight per warp
// Contiguous pages: a context of up to this many tokens is one stretch;
// longer ones are split (see kLastShare).
#ifndef KVQ_ATTN_MMA_PART
#define KVQ_ATTN_MMA_PART 1792
#endif
// Contiguous pages: the last of a context's n > 1 stretches gets 1 /
// kLastShare of the share of each of the others.
#ifndef KVQ_ATTN_MMA_LAST_SHARE
#define KVQ_ATTN_MMA_LAST_SHARE 4
#endif
constexpr int kLastShare = KVQ_ATTN_MMA_LAST_SHARE;
// the longest stretch (the first of two, 2 kLastShare S / (kLastShare + 1)
// tokens) leaves each warp at most 1024 tokens: 64 blocks of 16
static_assert(2 * kLastShare * KVQ_ATTN_MMA_PART / (kLastShare + 1) <=
                  4 * 64 * 16,
              "stretch too long for a warp's block ids");
// The stretch length on contiguous pages with block_size 8.
constexpr int kPartB8 = 1280;
static_assert(2 * kLastShare * kPartB8 / (kLastShare + 1) <= 4 * 64 * 8,
              "stretch too long for a warp's block ids");
// One step's slots of one warp.  On contiguous pages the step's 32
// tokens arrive in the pages' own order (whichever lane copies a chunk,
// its bytes keep their place), as 16-byte copies:
//   K data  4 x 512 B: tokens 16h + 8r + 0..7 (j = 2h + r), 64 B each;
//           lane (g, t) reads bytes 16t .. 16t+15 of token g
//   V data  4 x 512 B: tokens 16h + 8q + 0..7, 16-byte chunk k of the
//           piece at chunk k ^ (bit 3 of k, moved to bit 2), so that the
//           reads of token 2t (+1), bytes 8g .. 8g+7, meet no bank conflict
//   scales  512 B: per half h, 128 B of K scale rows (8 B per token) then
//           the 128 B of the half's V scales as the page holds them
//           (4-token bands of 32 B)
// Elsewhere every lane copies its own fragments into private,
// lane-contiguous slots:
//   K data  4 x 16 B (tokens g + 8j, bytes 16t .. 16t+15)
//   V data  8 x  8 B (tokens 16h + {2t, 2t+1, 2t+8, 2t+9}, bytes 8g .. 8g+7)
//   K scale 4 x  8 B (the 8-byte scale row holding groups 2t, 2t+1)
//   V scale 4 x  4 B (the word holding group g of a token pair)
// followed, after every warp's slots, by the query fragments of the CTA:
// [n-block][i][lane] x 16 B = lane (g, t)'s dims 32t + 8i .. + 7 of query
// head 8n + g as fp16, and 16 bytes for v_scale (read at the start, used
// at the end).
// The warps' partial outputs at the end, in each warp's own slots: one row
// of head dims per head, rows kMergeRow floats apart and dim d at column
// merge_col(d) (bits 1-2 of d XOR bits 5-6), so that both the
// fragment-layout float2 stores (lane (g, t) writes dims 16g + 4mb + e and
// 16g + 4mb + 2 + e of head 2t + c) and the readers (a quarter-warp reads
// 128 contiguous bytes of a row) meet no bank conflict.
constexpr int kMergeRow = kD + 4;
__host__ __device__ constexpr int merge_col(int d) {
  return d ^ (((d >> 5) & 3) << 1);
}
constexpr int kKdOff = 0;
constexpr int kVdOff = kKdOff + 4 * 16 * 32;
constexpr int kKsOff = kVdOff + 8 * 8 * 32;
__host__ __device__ constexpr int vchunk(int k) {
  return k ^ (((k >> 3) & 1) << 2);
}
template <bool kContig>
struct Slots {
  static constexpr int kVsOff = kKsOff + 4 * 8 * 32;  // not contiguous
  static constexpr int kStage = kContig ? kKsOff + 512 : kVsOff + 4 * 4 * 32;
  static constexpr int kWarp = kDepth * kStage;
  static constexpr int kQOff = kWarps * kWarp;
  __host__ __device__ static constexpr int kVsc(int NB) {
    return kQOff + NB * 4 * 32 * 16;
  }
  template <int NB>
  static constexpr int smem() { return kVsc(NB) + 16; }
  // a warp's partial result (16 rows of kMergeRow floats, then 16 maxima
  // and 16 sums) reuses its own copy slots
  static_assert(kWarp >= (16 * kMergeRow + 32) * 4, "");
};
constexpr float kLog2e = 1.4426950408889634f;


// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async of `bytes` (4, 8 or 16) from src to dst; src_bytes = 0 fills the
// destination with zeros and reads nothing.
template <int kBytes>
__device__ __forceinline__ void cp_async(uint32_t dst, const void* src,
                                         bool valid) {
  const uint32_t n = valid ? kBytes : 0u;
  if constexpr (kBytes == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"(src), "r"(n)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst),
                 "l"(src), "n"(kBytes), "r"(n)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b,
                                         uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four bytes of e2m1 pairs (element 2k in the low nibble of byte k) times
// half kHalf of the f16x2 scale pair `sfp` (both lanes of the multiply take
// that half) -> four f16x2 words, element 2k in the low half.  Exact: the
// products have at most 6 significant bits.
template <int kHalf>
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t sfp,
                                             uint32_t (&o)[4]) {
  if constexpr (kHalf == 0)
    asm("{ .reg .b8 q0, q1, q2, q3;\n"
        "  .reg .b32 h0, h1, h2, h3, sb;\n"
        "  .reg .b16 s0, s1;\n"
        "  mov.b32 {s0, s1}, %5;\n"
        "  mov.b32 sb, {s0, s0};\n"
        "  mov.b32 {q0, q1, q2, q3}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 h0, q0;  cvt.rn.f16x2.e2m1x2 h1, q1;\n"
        "  cvt.rn.f16x2.e2m1x2 h2, q2;  cvt.rn.f16x2.e2m1x2 h3, q3;\n"
        "  mul.rn.f16x2 %0, h0, sb;  mul.rn.f16x2 %1, h1, sb;\n"
        "  mul.rn.f16x2 %2, h2, sb;  mul.rn.f16x2 %3, h3, sb; }"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w), "r"(sfp));
  else
    asm("{ .reg .b8 q0, q1, q2, q3;\n"
        "  .reg .b32 h0, h1, h2, h3, sb;\n"
        "  .reg .b16 s0, s1;\n"
        "  mov.b32 {s0, s1}, %5;\n"
        "  mov.b32 sb, {s1, s1};\n"
        "  mov.b32 {q0, q1, q2, q3}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 h0, q0;  cvt.rn.f16x2.e2m1x2 h1, q1;\n"
        "  cvt.rn.f16x2.e2m1x2 h2, q2;  cvt.rn.f16x2.e2m1x2 h3, q3;\n"
        "  mul.rn.f16x2 %0, h0, sb;  mul.rn.f16x2 %1, h1, sb;\n"
        "  mul.rn.f16x2 %2, h2, sb;  mul.rn.f16x2 %3, h3, sb; }"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w), "r"(sfp));
}

__device__ __forceinline__ uint16_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// Two e4m3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint16_t pair) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(pair));
  return h;
}

// A pair of fp16 weights {P_lo, P_hi} -> the B registers of the even-dim
// product ({P_lo, 0}, {P_hi, 0}) and of the odd-dim one ({0, P_lo},
// {0, P_hi}): packed multiplies by {1, 0} / {0, 1} (exact; the weights are
// finite and non-negative).
__device__ __forceinline__ void split_weights(uint32_t w, uint32_t (&b)[4]) {
  asm("{ .reg .b16 l, h;\n"
      "  .reg .b32 ll, hh;\n"
      "  mov.b32 {l, h}, %4;\n"
      "  mov.b32 ll, {l, l};\n"
      "  mov.b32 hh, {h, h};\n"
      "  mul.rn.f16x2 %0, ll, %5;  mul.rn.f16x2 %1, hh, %5;\n"
      "  mul.rn.f16x2 %2, ll, %6;  mul.rn.f16x2 %3, hh, %6; }"
      : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
      : "r"(w), "r"(0x00003C00u), "r"(0x3C000000u));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> f16x2, round to nearest even; `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// bf16x2 -> f16x2 (round to nearest; exact for bf16 values inside the fp16
// normal range).
__device__ __forceinline__ uint32_t bf16x2_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  return pack_f16x2(lo, hi);
}

// The 8 x 8 b16 matrix whose row r / columns (2c, 2c+1) lane 4r + c holds,
// transposed (mma fragment layout in and out).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;"
               : "=r"(d)
               : "r"(x));
  return d;
}

// D += A . B, m16n8k16, fp16 A/B, fp32 D.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0,
                                         uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
// The kernel: one (partition, KV head, sequence) per CTA of 4 warps
// ---------------------------------------------------------------------------
// Logits of an empty (or fully invalid) range: ex2 of it minus any finite
// maximum is 0, and ex2(0) times a zero sum stays 0 when every range is
// empty.
constexpr float kNoLogit = -3.0e38f;
constexpr uint32_t kOnes2 = 0x3C003C00u;  // f16x2 {1, 1}
// A step's logits may exceed the running reference by up to this much (log2
// units) before the accumulators are rescaled: weights stay below 2^8, far
// inside fp16, and their rounding is still relative (2^-11).
constexpr float kLazy = 8.0f;

// kContig (kPages != 0): pages whose rows a warp copies as whole 8- or
// 16-token pieces in the pages' own order, one block id and lane-constant
// offsets per piece.
// kPages: 0 = other pages; 1, 2 = contiguous (HND, a power-of-two
// block_size >= 16); 3, 4 = token rows (NHD, the same block sizes: a
// head's 64-byte data rows and 8-byte scale rows H rows apart, copied row
// by row into the same shared-memory layout); 2 and 4 with block_size 16,
// where (warp ranges starting at multiples of 32 tokens) half h of a
// warp's step i is its block 2i + h, whole; 5 .. 8 = 1 .. 4 with the K
// scales swizzled like the V scales (the same bytes copied, read as
// bands); 9, 10 = 1, 3 with block_size 8 (linear K scales): 8-token piece
// j of step i is block 4i + j, and a stretch is kPartB8 tokens long, so
// that a warp's range spans at most 64 blocks.
template <int NG, bool kF16, int kPages>
__global__ void __launch_bounds__(kThreads, NG == 8 ? 4 : 3)
paged_attention_mma_kernel(const AttnParams p) {
  constexpr bool kB8 = kPages >= 9;
  constexpr bool kSwzK = kPages >= 5 && !kB8;
  constexpr int kForm = kB8 ? (kPages == 9 ? 1 : 3) : kSwzK ? kPages - 4
                                                            : kPages;
  constexpr bool kContig = kForm != 0, kB16 = kForm == 2 || kForm == 4;
  constexpr bool kRows = kForm >= 3;
  constexpr int NB = NG / 8;  // n-blocks of 8 query heads
  using SL = Slots<kContig>;
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  // stretch-major launch order: (stretch, sequence, KV head), KV head
  // fastest
  const int kh = static_cast<int>(blockIdx.x % p.Hkv);
  const int sb = static_cast<int>(blockIdx.x / p.Hkv);
  const int b = sb % p.num_seqs, part = sb / p.num_seqs;
  // PDL: wait for the kernel before here, or -- when the caller promised
  // that it writes none of the query, block table, context lengths and
  // scales (KVQ_F_PDL_EARLY_META) -- only before the first read of the
  // pages and the first write, so that the lengths, block ids and query
  // load while it finishes.  The next kernel may launch only after the
  // wait, as everywhere here: a kernel two launches back has then always
  // finished when another early read starts.
  const bool early = p.early_meta;
  if (!early) pdl_prologue();

  int L = __ldg(p.lens + b);
  const bool bad_len = L < 0 || L > p.len_cap;
  if (bad_len) L = L < 0 ? 0 : p.len_cap;
  // flags a clamped length (once per sequence); a write, so after the wait
  auto flag_len = [&]() {
    if (bad_len && p.dev_error != nullptr && part == 0 && kh == 0 &&
        tid == 0)
      atomicOr(p.dev_error, KVQ_DEVERR_SEQ);
  };
  // stretch length: fixed on contiguous pages (the host sets p.part to it)
  const int S = kB8 ? kPartB8 : kContig ? KVQ_ATTN_MMA_PART : p.part;
  const int nparts = (L + S - 1) / S;
  if (part >= nparts) {
    if (early) pdl_prologue();
    flag_len();
    if (part == 0) {  // empty context: the output is zero
      for (int i = tid; i < p.G * kD; i += kThreads)
        p.out[b * p.out_stride0 + (kh * p.G) * kD + i] = 0;
    }
    return;
  }
  // This CTA's stretch [p0, p1): on contiguous pages the context is split
  // over its nparts stretches in the proportions kLastShare : ... :
  // kLastShare : 1 (boundary i at kLastShare i L / (kLastShare (nparts-1) +
  // 1), rounded down to a multiple of 32 tokens; the last stretch of two
  // holds more than S / (kLastShare + 1) tokens), so that no CTA carries a
  // remainder of a few tokens with three of its warps idle and the last
  // stretches, launched last, are short; elsewhere the caller's partitions.
  int p0, p1;
  if constexpr (kContig) {
    const int64_t den = static_cast<int64_t>(kLastShare) * (nparts - 1) + 1;
    p0 = static_cast<int>(static_cast<int64_t>(kLastShare) * part * L / den) &
         ~31;
    p1 = part + 1 == nparts
             ? L
             : static_cast<int>(static_cast<int64_t>(kLastShare) *
                                (part + 1) * L / den) &
                   ~31;
  } else {
    p0 = part * S;
    p1 = min(L, p0 + S);
  }
  // the stretch's tokens split evenly over the warps, in whole steps
  const int ntok = p1 - p0;
  const int quarter =
      (ntok + kWarps * kStep - 1) / (kWarps * kStep) * kStep;
  const int w0 = p0 + warp * quarter;
  const int w1 = min(w0 + quarter, p1);
  const int nsteps = w1 > w0 ? (w1 - w0 + kStep - 1) / kStep : 0;

  // block ids of the warp's range, one or two per lane: blocks e0 + lane
  // and, on contiguous pages (ranges of up to 64 blocks), e0 + 32 + lane;
  // elsewhere a range spans at most 32 blocks
  const int e0 = p.b_shift >= 0 ? (w0 >> p.b_shift) : w0 / p.B;
  int32_t bt_lane = -1, bt_hi = -1;
  bool lane_in = false, hi_in = false;  // the block holds tokens of the range
  if (nsteps > 0) {
    const int e1 = p.b_shift >= 0 ? ((w1 - 1) >> p.b_shift) : (w1 - 1) / p.B;
    const int32_t* row = p.block_table + b * p.bt_stride;
    lane_in = e0 + lane <= e1;
    if (lane_in) bt_lane = __ldg(row + e0 + lane);
    if constexpr (kContig) {
      hi_in = e0 + 32 + lane <= e1;
      if (hi_in) bt_hi = __ldg(row + e0 + 32 + lane);
    }
  }

  // Logit scale in log2 units, made positive so that the maximum of the
  // unscaled logits gives the maximum of the scaled ones: a negative scale
  // negates the staged query (exact), a zero one zeroes it (every logit 0).
  float c2 = p.scale * __ldg(p.k_scale) * kLog2e;
  const uint32_t qflip = c2 < 0.f ? 0x80008000u : 0u;
  const bool qzero = c2 == 0.f;
  c2 = qzero ? 1.f : fabsf(c2);

  // query fragments, staged in shared memory once per CTA: entry (n, i,
  // lane) = lane (g, t)'s dims 32t + 8i .. + 7 of head 8n + g, as fp16.
  // Thread tid stages entries tid + 128n (i = its warp, lane = its lane);
  // they are loaded here and stored once the first copies are out, so that
  // their latency overlaps that of the block ids.  v_scale, needed only at
  // the end, is read now as well.
  const uint32_t qbase = smem_u32(smem) + SL::kQOff;
  uint4 qv[NB];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    qv[n] = make_uint4(0u, 0u, 0u, 0u);
    if (8 * n + g < p.G)
      qv[n] = __ldg(reinterpret_cast<const uint4*>(
          p.q + b * p.q_stride0 + (kh * p.G + 8 * n + g) * kD + 32 * t +
          8 * warp));
  }
  const float v_scale_in = tid == 0 ? __ldg(p.v_scale) : 0.f;
  if (early) pdl_prologue();
  flag_len();

  const uint32_t wbase = smem_u32(smem) + warp * SL::kWarp;
  const uint8_t* const kside = p.side[0];
  const uint8_t* const vside = p.side[1];

  // Where token `tok` of a side lives; every lane of the warp must call it
  // (the block id comes by shuffle).  ok: inside the range, valid block.
  auto locate = [&](int tok, const uint8_t* side, const uint8_t*& data,
                    const uint8_t*& sc, int& off) -> bool {
    const int idx = p.b_shift >= 0 ? (tok >> p.b_shift) : tok / p.B;
    const int32_t blk = __shfl_sync(0xFFFFFFFFu, bt_lane, (idx - e0) & 31);
    off = tok - idx * p.B;
    const bool ok = tok < w1 && blk >= 0 && blk < p.num_blocks;
    const uint8_t* page = side + static_cast<int64_t>(blk) * p.page_stride;
    data = page + kh * p.dhs + static_cast<int64_t>(off) * p.dts;
    sc = page + p.scale_off + kh * p.shs;
    if (!ok) {  // zero-filled copy: point it at memory that surely exists
      data = reinterpret_cast<const uint8_t*>(p.q);
      sc = data;
      off = 0;
    }
    return ok;
  };

  // bit e: the warp's block e0 + e has a valid id.  Every block of the
  // warp's range holds some of its tokens, so a bad id among them is
  // flagged here, once (its tokens are left out below).
  const uint32_t bmask =
      __ballot_sync(0xFFFFFFFFu, bt_lane >= 0 && bt_lane < p.num_blocks);
  const uint64_t bmask64 =
      bmask | static_cast<uint64_t>(__ballot_sync(
                  0xFFFFFFFFu, bt_hi >= 0 && bt_hi < p.num_blocks))
                  << 32;
  const uint64_t rmask64 =
      __ballot_sync(0xFFFFFFFFu, lane_in) |
      static_cast<uint64_t>(__ballot_sync(0xFFFFFFFFu, hi_in)) << 32;
  const bool bad_block = (rmask64 & ~bmask64) != 0u;
  if (lane == 0 && p.dev_error != nullptr && bad_block)
    atomicOr(p.dev_error, KVQ_DEVERR_BLOCK);

  // Whether token `tok` takes part (inside the range, valid block id);
  // every lane must call it.
  auto usable = [&](int tok) -> bool {
    const int idx = p.b_shift >= 0 ? (tok >> p.b_shift) : tok / p.B;
    return tok < w1 && ((bmask >> ((idx - e0) & 31)) & 1u) != 0u;
  };

  // contiguous pages: where this lane's copy lands in a V piece, and where
  // its fragments are read from (V data of token 2t + e of a piece; K
  // scale word of token g; V scale word of tokens 2t, 2t+1)
  const int v_dst = vchunk(lane) * 16;
  // contiguous pages: lane e's blocks e0 + e and e0 + 32 + e as the K-side
  // bases of this KV head (block 0 stands in for a bad id, whose half is
  // zero-filled from the query instead), V data at + vdelta, the K scale
  // rows at + sdelta
  const uint8_t* const kb_lane =
      kside + static_cast<int64_t>((bmask >> lane) & 1u ? bt_lane : 0) *
                  p.page_stride + kh * p.dhs;
  const uint8_t* const kb_hi =
      kside + static_cast<int64_t>((bmask64 >> (32 + lane)) & 1u ? bt_hi : 0) *
                  p.page_stride + kh * p.dhs;
  const int64_t vdelta = vside - kside;
  const int64_t sdelta = p.scale_off + kh * p.shs - kh * p.dhs;
  // contiguous pages: bytes between the data (scale) rows of consecutive
  // tokens of the head, and this lane's 16 bytes of the first 8 tokens'
  // data rows (token lane / 4, chunk lane % 4; 16 lane on HND pages)
  const int64_t dts = kRows ? p.dts : kD / 2;
  const int64_t sts = kRows ? p.sts : kD / 16;
  const int64_t lane_doff = (lane >> 2) * dts + (lane & 3) * 16;
  const int v_rd0 = vchunk(8 * t + (g >> 1)) * 16 + (g & 1) * 8;
  const int v_rd1 = vchunk(8 * t + 4 + (g >> 1)) * 16 + (g & 1) * 8;
  // contiguous pages: this lane's scale pairs (K: groups 2t, 2t+1 of token
  // g's row; V: tokens 2t, 2t+1 of group g in their 4-token band)
  const int ks_rd16 = g * 8 + 2 * t;
  const int ks_rd64 = (g >> 2) * 32 + 8 * t;  // K scales swizzled
  const int vs_rd16 = 128 + 32 * (t >> 1) + 4 * g + 2 * (t & 1);

  // Issue the copies of step i (tokens w0 + 32i ..) into its slots and
  // commit them as one group (an empty group past the last step).
  // kValid: every block id of the warp's range is valid (no test).
  auto issue = [&](int i, auto valid_tag) {
    constexpr bool kValid = decltype(valid_tag)::value;
    static_cast<void>(kValid);  // (only the contiguous forms test it)
    if (i >= nsteps) {
      // nothing to copy
    } else if constexpr (kB8) {
      // blocks of 8 tokens: piece 2h + u of step i (tokens 16h + 8u ..) is
      // the warp's block 4i + 2h + u, whole, copied as on block_size 16
      const uint32_t st = wbase + (i % kDepth) * SL::kStage;
      const uint8_t* qz = reinterpret_cast<const uint8_t*>(p.q);
      const uint8_t* sbp[4];
      bool okp[4];
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const int e = 4 * i + pc;  // < 64, warp-uniform
        const uint64_t kl =
            reinterpret_cast<uint64_t>(e < 32 ? kb_lane : kb_hi);
        const uint32_t lo =
            __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(kl), e & 31);
        const uint32_t hi =
            __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(kl >> 32), e & 31);
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(
            (static_cast<uint64_t>(hi) << 32) | lo);
        okp[pc] = kValid || ((bmask64 >> e) & 1u) != 0u;
        sbp[pc] = kb + sdelta;
        const uint32_t kd = st + kKdOff + pc * 512 + lane * 16;
        const uint32_t vd = st + kVdOff + pc * 512 + v_dst;
        const uint8_t* ka = kb + lane_doff;
        if (okp[pc]) {
          cp_async<16>(kd, ka, true);
          cp_async<16>(vd, ka + vdelta, true);
        } else {
          cp_async<16>(kd, qz, false);
          cp_async<16>(vd, qz, false);
        }
      }
      // the step's scales: lanes 16h .. 16h+15 take half h
      const int sh = lane >> 4, li = lane & 15;
      // the piece whose scales this lane copies
      const int pc = 2 * sh + (kRows ? li >> 3 : (li >> 2) & 1);
      const bool sok = pc == 0 ? okp[0] : pc == 1 ? okp[1]
                       : pc == 2 ? okp[2] : okp[3];
      const uint8_t* const sbs = pc == 0 ? sbp[0] : pc == 1 ? sbp[1]
                                 : pc == 2 ? sbp[2] : sbp[3];
      if constexpr (kRows) {
        // the K row of token li and V row li of the half: row li % 8 of
        // its block
        const uint8_t* so = sbs + (li & 7) * sts;
        const uint32_t sd = st + kKsOff + 256 * sh + 8 * li;
        cp_async<8>(sd, sok ? so : qz, sok);
        cp_async<8>(sd + 128, sok ? so + vdelta : qz, sok);
      } else {
        // lanes 0-3 / 4-7 the K scale rows of the half's two blocks, 8-11
        // / 12-15 their V scale bands, 16 contiguous bytes each
        const uint8_t* so = sbs + 16 * (li & 3) + ((li & 8) ? vdelta : 0);
        cp_async<16>(st + kKsOff + lane * 16, sok ? so : qz, sok);
      }
    } else if constexpr (kContig) {
      // whole 16-token halves: a block with a valid id is copied as it is
      // (tokens past the range are left out of the softmax and their V
      // scales zeroed when read), a bad one zero-filled from memory that
      // surely exists (the query)
      const uint32_t st = wbase + (i % kDepth) * SL::kStage;
      const uint8_t* qz = reinterpret_cast<const uint8_t*>(p.q);
      const uint8_t* sb[2];
      bool bok[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int T = w0 + kStep * i + 16 * h;
        // (contiguous pages have a power-of-two block size)
        const int idx = kB16 ? e0 + 2 * i + h : T >> p.b_shift;
        const int e = idx - e0;  // 0 .. 63, warp-uniform
        const uint64_t kl =
            reinterpret_cast<uint64_t>(e < 32 ? kb_lane : kb_hi);
        const uint32_t lo =
            __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(kl), e & 31);
        const uint32_t hi =
            __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(kl >> 32), e & 31);
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(
            (static_cast<uint64_t>(hi) << 32) | lo);
        // one block holds the whole half: the branch is warp-uniform
        bok[h] = kValid || ((bmask64 >> e) & 1u) != 0u;
        const int tok = kB16 ? 0 : T & (p.B - 1);  // the half's first row
        const uint32_t kd = st + kKdOff + 2 * h * 512 + lane * 16;
        const uint32_t vd = st + kVdOff + 2 * h * 512 + v_dst;
        // this lane's first K copy and the distance to its second (8
        // tokens on); two forms of the same addresses on HND pages (the
        // first measured faster with block_size 16, the second with 32)
        const uint8_t* ka;
        int64_t k8;
        if constexpr (kRows || kB16) {
          sb[h] = kb + sdelta + tok * sts;
          ka = kb + tok * dts + lane_doff;
          k8 = 8 * dts;
        } else {
          sb[h] = kb + sdelta + tok * (kD / 16);
          ka = kb + tok * (kD / 2) + 16 * lane;
          k8 = 512;
        }
        if (bok[h]) {
          const uint8_t* va = ka + vdelta;
          cp_async<16>(kd, ka, true);
          cp_async<16>(kd + 512, ka + k8, true);
          cp_async<16>(vd, va, true);
          cp_async<16>(vd + 512, va + k8, true);
        } else {
          cp_async<16>(kd, qz, false);
          cp_async<16>(kd + 512, qz, false);
          cp_async<16>(vd, qz, false);
          cp_async<16>(vd + 512, qz, false);
        }
      }
      // the step's scales: lanes 16h .. 16h+15 take half h
      const int sh = lane >> 4;
      const bool sok = sh ? bok[1] : bok[0];
      const uint8_t* const sbh = sh ? sb[1] : sb[0];
      if constexpr (kRows) {
        // scale row lane % 16 of the half: the K row of its token and V
        // row lane % 16 (4-token band lane % 16 / 4), 8 bytes each
        const uint8_t* so = sbh + (lane & 15) * sts;
        const uint32_t sd = st + kKsOff + 256 * sh + 8 * (lane & 15);
        cp_async<8>(sd, sok ? so : qz, sok);
        cp_async<8>(sd + 128, sok ? so + vdelta : qz, sok);
      } else {
        // the first 8 lanes the half's K scale rows, the other 8 its V
        // scale bands, 16 contiguous bytes each
        const uint8_t* so = sbh + 16 * (lane & 7) + ((lane & 8) ? vdelta : 0);
        cp_async<16>(st + kKsOff + lane * 16, sok ? so : qz, sok);
      }
    } else {
      const uint32_t st = wbase + (i % kDepth) * SL::kStage;
      const int T0 = w0 + kStep * i;
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // K: tokens T0 + g + 8j
        const uint8_t *data, *sc;
        int off;
        const bool ok = locate(T0 + g + 8 * j, kside, data, sc, off);
        cp_async<16>(st + kKdOff + j * 512 + lane * 16, data + 16 * t, ok);
        const uint8_t* srow =
            p.swizzle_k ? sc + static_cast<int64_t>((off & ~3) + t) * p.sts
                        : sc + static_cast<int64_t>(off) * p.sts;
        cp_async<8>(st + kKsOff + j * 256 + lane * 8, srow, ok);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // V: tokens T0 + 16h + 8q + 2t (+1)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint8_t *data, *sc;
          int off;
          const int tok = T0 + 16 * h + 8 * q + 2 * t;
          const bool ok0 = locate(tok, vside, data, sc, off);
          const bool ok1 = ok0 && tok + 1 < w1;
          const int piece = 4 * h + 2 * q;
          cp_async<8>(st + kVdOff + piece * 256 + lane * 8, data + 8 * g, ok0);
          cp_async<8>(st + kVdOff + (piece + 1) * 256 + lane * 8,
                      data + p.dts + 8 * g, ok1);
          cp_async<4>(st + SL::kVsOff + (2 * h + q) * 128 + lane * 4,
                      sc + static_cast<int64_t>((off & ~3) + (g >> 1)) * p.sts +
                          (g & 1) * 4,
                      ok0);
        }
      }
    }
    cp_async_commit();
  };

  // running softmax state of heads 8n + 2t + c, and O^T fragments:
  // o[mb][e][n] = rows dims 16g + 4mb + e (c0, c1) and 16g + 4mb + 2 + e
  // (c2, c3), columns heads 8n + 2t, 8n + 2t + 1
  // lacc[n][c]: running denominator of head 8n + 2t + c, already summed
  // over the warp's tokens by the tensor cores (c2, c3 repeat it and are
  // not read)
  // m_neg: -m_run, or 0 while m_run is -inf (no usable token yet)
  // m_thr: (m_run + kLazy) / c2, the unscaled logit above which a step
  // moves the reference
  float m_run[NB][2], m_neg[NB][2], m_thr[NB][2], lacc[NB][4];
  float o[4][2][NB][4];
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    m_run[n][0] = m_run[n][1] = -INFINITY;
    m_thr[n][0] = m_thr[n][1] = -INFINITY;
    m_neg[n][0] = m_neg[n][1] = 0.f;
    lacc[n][0] = lacc[n][1] = lacc[n][2] = lacc[n][3] = 0.f;
#pragma unroll
    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        o[mb][e][n][0] = o[mb][e][n][1] = o[mb][e][n][2] =
            o[mb][e][n][3] = 0.f;
  }
  // byte selectors (pages that are not contiguous): K scales of groups 2t,
  // 2t+1 (linear: bytes 2t, 2t+1 of the row; swizzled: bytes off%4 and
  // 4 + off%4 of the band row, off%4 = g%4 because steps start at multiples
  // of 32 and B % 4 == 0); V scales of a token pair: bytes 2t%4, 2t%4 + 1
  // of the word
  const uint32_t ksel =
      p.swizzle_k ? static_cast<uint32_t>((g & 3) | ((4 + (g & 3)) << 4))
                  : static_cast<uint32_t>((2 * t) | ((2 * t + 1) << 4));
  const uint32_t vsel =
      static_cast<uint32_t>(((2 * t) & 3) | ((((2 * t) & 3) + 1) << 4));

  // One step of 32 tokens.  kMasked: some token of the step is past the
  // warp's range or in a block with a bad id (its logit becomes -inf and,
  // past the range, its V scales are zeroed); otherwise no per-token test
  // is made at all.
  auto step = [&](int i, auto masked_tag) {
    constexpr bool kMasked = decltype(masked_tag)::value;
    // the unmasked steps run only when no block id of the range is bad
    issue(i + kDepth - 1, std::integral_constant<bool, !kMasked>{});
    cp_async_wait<kDepth - 1>();
    const uint32_t st = wbase + (i % kDepth) * SL::kStage;
    const int T0 = w0 + kStep * i;

    // ---- logits S^T[16 tokens x 8 heads] of the two 16-token halves -------
    // word by word: the query fragments of two k-steps (one 16-byte shared
    // load), the two tokens' e2m1 words dequantised, two MMAs -- few
    // registers live at a time
    float sacc[2][NB][4];
    uint32_t kvalid = 0xFu;  // bit j: K token T0 + g + 8j is usable
    if constexpr (kMasked && kB8) {
      // 8-token piece j of the step is the warp's block 4i + j
      const uint32_t vb = static_cast<uint32_t>(bmask64 >> (4 * i)) & 0xFu;
      const int rem = w1 - T0 - g;  // token T0 + g + 8j usable: 8j < rem
      kvalid = (vb & 1u & static_cast<uint32_t>(rem > 0)) |
               (((vb >> 1) & 1u & static_cast<uint32_t>(rem > 8)) << 1) |
               (((vb >> 2) & 1u & static_cast<uint32_t>(rem > 16)) << 2) |
               (((vb >> 3) & 1u & static_cast<uint32_t>(rem > 24)) << 3);
    } else if constexpr (kMasked && kContig) {
      // each 16-token half lies in one block
      const int i0 = kB16 ? e0 + 2 * i : T0 >> p.b_shift;
      const int i1 = kB16 ? i0 + 1 : (T0 + 16) >> p.b_shift;
      const uint32_t v0 = static_cast<uint32_t>(bmask64 >> (i0 - e0)) & 1u;
      const uint32_t v1 = static_cast<uint32_t>(bmask64 >> (i1 - e0)) & 1u;
      const int rem = w1 - T0 - g;  // token T0 + g + 8j usable: 8j < rem
      kvalid = (v0 & static_cast<uint32_t>(rem > 0)) |
               ((v0 & static_cast<uint32_t>(rem > 8)) << 1) |
               ((v1 & static_cast<uint32_t>(rem > 16)) << 2) |
               ((v1 & static_cast<uint32_t>(rem > 24)) << 3);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 kd[2];
      uint32_t sfw[2];  // [row]: groups 2t | 2t+1 scales as f16x2
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = 2 * h + r;
        kd[r] = lds128(st + kKdOff + j * 512 + lane * 16);
        uint16_t pair;
        if constexpr (kContig && kSwzK) {
          // band (2r + g / 4), row t: scales 2t, 2t+1 of token 8r + g at
          // bytes g % 4 and 4 + g % 4
          const uint2 ks = lds64(st + kKsOff + 256 * h + 64 * r + ks_rd64);
          pair = static_cast<uint16_t>(prmt(ks.x, ks.y, ksel));
        } else if constexpr (kContig) {
          pair = lds16(st + kKsOff + 256 * h + 64 * r + ks_rd16);
        } else {
          const uint2 ks = lds64(st + kKsOff + j * 256 + lane * 8);
          pair = static_cast<uint16_t>(prmt(ks.x, ks.y, ksel));
        }
        if constexpr (kMasked && !kContig) {
          if (r == 0 && h == 0) kvalid = 0u;
          kvalid |= static_cast<uint32_t>(usable(T0 + g + 8 * j)) << j;
        }
        sfw[r] = e4m3x2_f16x2(pair);
      }
      // two accumulators (even / odd k-steps) halve the dependent chain
      float e2[NB][4];
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int r = 0; r < 4; ++r) sacc[h][n][r] = e2[n][r] = 0.f;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {  // word wd: k-steps 2wd, 2wd+1
        uint32_t x0[4], x1[4];
        const uint32_t w0r = wd == 0 ? kd[0].x : wd == 1 ? kd[0].y
                             : wd == 2 ? kd[0].z : kd[0].w;
        const uint32_t w1r = wd == 0 ? kd[1].x : wd == 1 ? kd[1].y
                             : wd == 2 ? kd[1].z : kd[1].w;
        if (wd < 2) {
          dequant_word<0>(w0r, sfw[0], x0);
          dequant_word<0>(w1r, sfw[1], x1);
        } else {
          dequant_word<1>(w0r, sfw[0], x0);
          dequant_word<1>(w1r, sfw[1], x1);
        }
#pragma unroll
        for (int n = 0; n < NB; ++n) {
          const uint4 q4 = lds128(qbase + (n * 128 + wd * 32 + lane) * 16);
          mma16816(sacc[h][n], x0[0], x1[0], x0[1], x1[1], q4.x, q4.y);
          mma16816(e2[n], x0[2], x1[2], x0[3], x1[3], q4.z, q4.w);
        }
      }
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int r = 0; r < 4; ++r) sacc[h][n][r] += e2[n][r];
    }

    // ---- online softmax over the 32 tokens --------------------------------
    // The weights are exp2 of the scaled logits minus a reference m_run that
    // moves only when a step's maximum exceeds it by more than kLazy (then
    // every accumulator of the warp is rescaled at once); in between the
    // weights stay below 2^kLazy.  v holds the unscaled logits; c2 > 0 is
    // applied to their maxima and inside each weight's exponent (one FMA).
    float v[NB][2][4];
    float bmu[NB][2];  // this lane's maximum unscaled logit of head 8n+2t+c
    bool grow = false;
#pragma unroll
    for (int n = 0; n < NB; ++n) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if constexpr (kMasked) {
            const bool ok = (kvalid >> (2 * h + (r >> 1))) & 1u;
            v[n][h][r] = ok ? sacc[h][n][r] : -INFINITY;
          } else {
            v[n][h][r] = sacc[h][n][r];
          }
        }
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // head 8n + 2t + c: this lane's tokens
        bmu[n][c] = fmaxf(fmaxf(v[n][0][c], v[n][0][2 + c]),
                          fmaxf(v[n][1][c], v[n][1][2 + c]));
        grow |= bmu[n][c] > m_thr[n][c];  // false while both -inf
      }
    }
    // the step's maximum over all its tokens exceeds the reference by more
    // than kLazy exactly when some lane's does; only then is it formed
    if (__any_sync(0xFFFFFFFFu, grow)) {  // rare after the first step
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float bm = bmu[n][c] * c2;
          bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, 4));
          bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, 8));
          bm = fmaxf(bm, __shfl_xor_sync(0xFFFFFFFFu, bm, 16));
          const float mnew = fmaxf(m_run[n][c], bm);
          if (mnew > m_run[n][c]) {
            const float alpha = ex2(m_run[n][c] - mnew);  // 0 from -inf
            m_run[n][c] = mnew;
            m_neg[n][c] = -mnew;
            m_thr[n][c] = (mnew + kLazy) / c2;
            lacc[n][c] *= alpha;
#pragma unroll
            for (int mb = 0; mb < 4; ++mb)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                o[mb][e][n][c] *= alpha;
                o[mb][e][n][2 + c] *= alpha;
              }
          }
        }
    }
    uint32_t pb[2][NB][2];  // B fragments of P^T: [half][n][tokens 2t | 2t+8]
#pragma unroll
    for (int n = 0; n < NB; ++n)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // an unusable token's -inf gives 0 (m_neg is finite)
        auto wgt = [&](int r) {
          return ex2(fmaf(v[n][h][r], c2, m_neg[n][r & 1]));
        };
        const uint32_t pl = pack_f16x2(wgt(0), wgt(1));
        const uint32_t ph = pack_f16x2(wgt(2), wgt(3));
        pb[h][n][0] = transpose8x8(pl);  // tokens 16h + 2t, 16h + 2t + 1
        pb[h][n][1] = transpose8x8(ph);  // tokens 16h + 8 + 2t, + 1
      }

    // ---- O^T += V'^T P^T per 8-token block -------------------------------
    // The contraction index of a block runs over (token, e) pairs: A holds
    // the block's V bytes as they are -- one byte = dims 2p, 2p+1 of a token
    // = one f16x2 register after conversion, no nibble shuffling -- with
    // rows = dim pairs p, and two products share it: one whose B is the
    // token's weight at e = 0 and 0 at e = 1 (it sums the even dims of each
    // pair), one the other way round (the odd dims).  Lane (g, t): columns
    // 2t, 2t+1 = token 2t of the block, 2t+8, 2t+9 = token 2t+1; rows g and
    // g+8 of m-block mb = bytes 2mb and 2mb+1 of the token's group g.
    int vleft = 0;
    if constexpr (kMasked) vleft = w1 - T0 - 2 * t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint2 vd0, vd1;  // group g's bytes of tokens 2t and 2t+1
        uint16_t pair;
        if constexpr (kContig) {
          const uint32_t piece = st + kVdOff + (2 * h + q) * 512;
          vd0 = lds64(piece + v_rd0);
          vd1 = lds64(piece + v_rd1);
          pair = lds16(st + kKsOff + 256 * h + 64 * q + vs_rd16);
        } else {
          vd0 = lds64(st + kVdOff + (4 * h + 2 * q) * 256 + lane * 8);
          vd1 = lds64(st + kVdOff + (4 * h + 2 * q + 1) * 256 + lane * 8);
          pair = static_cast<uint16_t>(
              prmt(lds32(st + SL::kVsOff + (2 * h + q) * 128 + lane * 4), 0u,
                   vsel));
        }
        if constexpr (kMasked) {
          // a token past the range may share the word: zero its scale (its
          // data may hold anything), so no stray NaN meets a zero weight;
          // left = tokens of the range from this pair's first one on
          const int left = vleft - 16 * h - 8 * q;
          if (left < 2) pair &= left == 1 ? 0x00FF : 0;
        }
        const uint32_t sfp = e4m3x2_f16x2(pair);  // {sf(2t), sf(2t+1)}
        uint32_t bw[NB][4];  // even: {P(2t), 0}, {P(2t+1), 0}; odd: swapped
#pragma unroll
        for (int n = 0; n < NB; ++n) split_weights(pb[h][n][q], bw[n]);
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {  // bytes 0..3, then 4..7
          uint32_t x0[4], x1[4];
          dequant_word<0>(wi == 0 ? vd0.x : vd0.y, sfp, x0);
          dequant_word<1>(wi == 0 ? vd1.x : vd1.y, sfp, x1);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int mb = 2 * wi + k;
#pragma unroll
            for (int n = 0; n < NB; ++n) {
              mma16816(o[mb][0][n], x0[2 * k], x0[2 * k + 1], x1[2 * k],
                       x1[2 * k + 1], bw[n][0], bw[n][1]);
              mma16816(o[mb][1][n], x0[2 * k], x0[2 * k + 1], x1[2 * k],
                       x1[2 * k + 1], bw[n][2], bw[n][3]);
            }
          }
        }
      }
      // the denominators: an all-ones A times P^T sums the half's 16
      // rounded weights of each head (every row holds the sum)
#pragma unroll
      for (int n = 0; n < NB; ++n)
        mma16816(lacc[n], kOnes2, kOnes2, kOnes2, kOnes2, pb[h][n][0],
                 pb[h][n][1]);
    }
  };

#pragma unroll
  for (int i = 0; i < kDepth - 1; ++i) issue(i, std::false_type{});
#pragma unroll
  for (int n = 0; n < NB; ++n) {
    uint4 v = qv[n];
    if (8 * n + g < p.G) {
      if constexpr (!kF16) {
        v.x = bf16x2_f16x2(v.x);
        v.y = bf16x2_f16x2(v.y);
        v.z = bf16x2_f16x2(v.z);
        v.w = bf16x2_f16x2(v.w);
      }
      v.x ^= qflip; v.y ^= qflip; v.z ^= qflip; v.w ^= qflip;
      if (qzero) v = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                     qbase + (tid + kThreads * n) * 16),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
  }
  if (tid == 0)
    *reinterpret_cast<float*>(smem + SL::kVsc(NB)) = v_scale_in;
  __syncthreads();  // the query is staged
  // the steps with no token to leave out come first; the warp's last
  // (partial) step, and every step when a block of its range has a bad id,
  // take the masked form
  const int nfast = bad_block ? 0 : (w1 - w0) / kStep;
  int i = 0;
  for (; i < nfast; ++i) step(i, std::false_type{});
  for (; i < nsteps; ++i) step(i, std::true_type{});
  cp_async_wait<0>();  // nothing may land after the slots are reused

  // ---- merge the 4 warps' partial results in shared memory ----------------
  // Each warp writes its own into its copy slots (all its copies have
  // landed; no other warp uses them), so one barrier suffices.
  float* const wO = reinterpret_cast<float*>(smem + warp * SL::kWarp);
#pragma unroll
  for (int n = 0; n < NB; ++n)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int hh = 8 * n + 2 * t + c;
      float* row = wO + hh * kMergeRow;
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
        *reinterpret_cast<float2*>(row + merge_col(16 * g + 4 * mb)) =
            make_float2(o[mb][0][n][c], o[mb][1][n][c]);
        *reinterpret_cast<float2*>(row + merge_col(16 * g + 4 * mb + 2)) =
            make_float2(o[mb][0][n][2 + c], o[mb][1][n][2 + c]);
      }
      if (g == 0) {
        wO[16 * kMergeRow + hh] =
            m_run[n][c] == -INFINITY ? kNoLogit : m_run[n][c];
        wO[16 * kMergeRow + 16 + hh] = lacc[n][c];
      }
    }
  __syncthreads();
  // The output, 8 dims of one head per thread: physical columns 4k .. 4k+3
  // and 64 + 4k .. 67 + 4k of the head's rows (a quarter-warp reads 128
  // contiguous bytes), which by merge_col hold head dims 4k .. 4k+3 and
  // 64 + 4(k^1) .. +3, their two pairs swapped when k >= 8.  Per dim the
  // sum runs over the warps in order.
  const float v_scale = *reinterpret_cast<const float*>(smem + SL::kVsc(NB));
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    const int u = tid + kThreads * r;
    const int hh = u >> 4, k = u & 15;
    if (hh >= p.G) break;
    // the head's maximum M over the warps, their factors exp2(m_w - M) and
    // the denominator
    const float* wbuf[kWarps];
    float mw[kWarps];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      wbuf[w] = reinterpret_cast<const float*>(smem + w * SL::kWarp);
      mw[w] = wbuf[w][16 * kMergeRow + hh];
    }
    float M = mw[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, mw[w]);
    float fw[kWarps], den = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      fw[w] = ex2(mw[w] - M);
      den += wbuf[w][16 * kMergeRow + 16 + hh] * fw[w];
    }
    const float inv = den > 0.f ? 1.0f / den : 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* row = wbuf[w] + hh * kMergeRow;
      const float4 x = *reinterpret_cast<const float4*>(row + 4 * k);
      const float4 y = *reinterpret_cast<const float4*>(row + 64 + 4 * k);
      a.x += x.x * fw[w]; a.y += x.y * fw[w];
      a.z += x.z * fw[w]; a.w += x.w * fw[w];
      c.x += y.x * fw[w]; c.y += y.y * fw[w];
      c.z += y.z * fw[w]; c.w += y.w * fw[w];
    }
    if (k >= 8) {
      a = make_float4(a.z, a.w, a.x, a.y);
      c = make_float4(c.z, c.w, c.x, c.y);
    }
    const int da = 4 * k, dc = 64 + 4 * (k ^ 1);
    if (nparts == 1) {
      auto pack = [&](float lo, float hi) -> uint32_t {
        const float ylo = den > 0.f ? lo * inv * v_scale : 0.f;
        const float yhi = den > 0.f ? hi * inv * v_scale : 0.f;
        return static_cast<uint32_t>(float_to_out<kF16>(ylo)) |
               (static_cast<uint32_t>(float_to_out<kF16>(yhi)) << 16);
      };
      uint16_t* orow = p.out + b * p.out_stride0 + (kh * p.G + hh) * kD;
      *reinterpret_cast<uint2*>(orow + da) =
          make_uint2(pack(a.x, a.y), pack(a.z, a.w));
      *reinterpret_cast<uint2*>(orow + dc) =
          make_uint2(pack(c.x, c.y), pack(c.z, c.w));
    } else {
      const int64_t rr =
          (static_cast<int64_t>(b) * p.Hq + kh * p.G + hh) * p.max_parts +
          part;
      const float s = den > 0.f ? inv : 0.f;
      const bool live = den > 0.f;
      float* trow = p.tmp_out + rr * kD;
      *reinterpret_cast<float4*>(trow + da) =
          live ? make_float4(a.x * s, a.y * s, a.z * s, a.w * s)
               : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(trow + dc) =
          live ? make_float4(c.x * s, c.y * s, c.z * s, c.w * s)
               : make_float4(0.f, 0.f, 0.f, 0.f);
      if (k == 0) {
        p.max_logits[rr] = M;
        p.exp_sums[rr] = den;
      }
    }
  }
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

template <int NG, bool kF16, int kPages>
cudaError_t launch_mma(const AttnParams& caller, cudaStream_t stream) {
  constexpr bool kContig = kPages != 0;
  auto kernel = paged_attention_mma_kernel<NG, kF16, kPages>;
  // A CTA may cover a longer partition than the caller's (fewer, longer
  // warp ranges; the scratch rows keep the caller's max_parts stride and
  // need fewer entries).  A warp range spans at most 64 blocks on
  // contiguous pages, 32 elsewhere.
  AttnParams p = caller;
  // (the caller's partitions are at most 512 tokens)
  if (kContig) p.part = kPages >= 9 ? kPartB8 : KVQ_ATTN_MMA_PART;
  const int parts =
      static_cast<int>((static_cast<int64_t>(p.len_cap) + p.part - 1) / p.part);
  static bool configured[64] = {false};  // per instantiation and device
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (!configured[dev & 63]) {
    err = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        Slots<kContig>::template smem<NG / 8>());
    if (err != cudaSuccess) return err;
    configured[dev & 63] = true;
  }
  // one CTA per (stretch, sequence, KV head), stretch-major (the checks
  // keep the count below 2^31)
  const int64_t ctas =
      static_cast<int64_t>(parts > 0 ? parts : 1) * p.num_seqs * p.Hkv;
  const dim3 grid(static_cast<unsigned>(ctas));
  err = launch_kernel(kernel, grid, kThreads,
                      Slots<kContig>::template smem<NG / 8>(), stream, p.pdl,
                      p);
  if (err != cudaSuccess || parts <= 1) return err;
  return launch_attention_merge(p, stream);
}

template <int NG, bool kF16, int kSwz>
cudaError_t launch_form(const AttnParams& p, cudaStream_t stream) {
  // block sizes: powers of two from 16 up (block index and offset by
  // shifts and masks); others take the per-fragment path
  const bool pow2 = p.B >= 16 && p.b_shift >= 0;
  const bool contig = p.dts == kD / 2 && p.sts == kD / 16 && pow2;
  // token rows: NHD pages (a head's rows H rows apart)
  const bool rows = p.dhs == kD / 2 && p.dts == p.Hkv * (kD / 2) &&
                    p.shs == kD / 16 && p.sts == p.Hkv * (kD / 16) && pow2;
  if (contig)
    return p.B == 16 ? launch_mma<NG, kF16, 2 + kSwz>(p, stream)
                     : launch_mma<NG, kF16, 1 + kSwz>(p, stream);
  if (rows)
    return p.B == 16 ? launch_mma<NG, kF16, 4 + kSwz>(p, stream)
                     : launch_mma<NG, kF16, 3 + kSwz>(p, stream);
  // block_size 8 with linear K scales: two blocks per 16-token half
  if (kSwz == 0 && p.B == 8 && p.dhs == 8 * (kD / 2) && p.dts == kD / 2 &&
      p.shs == 8 * (kD / 16) && p.sts == kD / 16)
    return launch_mma<NG, kF16, 9>(p, stream);
  if (kSwz == 0 && p.B == 8 && p.dhs == kD / 2 &&
      p.dts == p.Hkv * (kD / 2) && p.shs == kD / 16 &&
      p.sts == p.Hkv * (kD / 16))
    return launch_mma<NG, kF16, 10>(p, stream);
  return launch_mma<NG, kF16, 0>(p, stream);
}

template <int NG, bool kF16>
cudaError_t launch_layout(const AttnParams& p, cudaStream_t stream) {
  return p.swizzle_k ? launch_form<NG, kF16, 4>(p, stream)
                     : launch_form<NG, kF16, 0>(p, stream);
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

cudaError_t launch_paged_attention_mma(const AttnParams& p,
                                       cudaStream_t stream) {
  if (p.G <= 8)
    return p.f16 ? launch_layout<8, true>(p, stream)
                 : launch_layout<8, false>(p, stream);
  return p.f16 ? launch_layout<16, true>(p, stream)
               : launch_layout<16, false>(p, stream);
}

}  // namespace kvq
