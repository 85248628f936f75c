/*
 * kvq.h -- C ABI of libkvq: GB300 (sm_103a) kernels for the write and read
 * hot path of a paged quantized KV cache.
 *
 * Two operations:
 *
 *   kvq_store_nvfp4       bf16 K/V -> NVFP4, scattered into paged cache pages
 *                         (vLLM csrc/libtorch_stable/nvfp4_kv_cache_kernels.cu,
 *                         commit 7ce4c8e: reshape_and_cache_nvfp4_kernel and
 *                         reshape_and_cache_nvfp4_dispatch).
 *   kvq_load_nvfp4        the read side of the store: NVFP4 pages named by a
 *                         block table -> bf16 K/V rows.
 *   kvq_store_indexer_k   the write side of the indexer cache: bf16 K rows ->
 *                         fp8 e4m3 + per-token fp32 scale, by slot.
 *   kvq_gather_indexer_k  fp8 indexer-K rows and per-token fp32 scales
 *                         gathered out of a paged cache (vLLM PR #25931 "Add
 *                         gather_indexer_k_quant_cache kernel"; PR #26456
 *                         "[Deepseek-V3.2][Kernel] Integrate cuda indexer k
 *                         cache gather").
 *   kvq_paged_attention_nvfp4  decode attention (one query token per
 *                         sequence) over the NVFP4 pages (vLLM PR #12348
 *                         "[ROCm] Faster Custom Paged Attention kernels":
 *                         the paged_attention op).
 *
 * Conventions shared by every entry point:
 *   - Every buffer pointer is DEVICE memory owned by the caller, on the
 *     calling thread's current CUDA device.  The library never allocates,
 *     frees or synchronises.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  A KVQ_OK return means the work was enqueued.
 *   - Arguments are validated on the host without touching device memory;
 *     a failed check returns an error code and launches nothing.  Nothing
 *     throws across this boundary and no kernel traps.
 *   - `dev_error` (nullable, device int32): kernels OR KVQ_DEVERR_* bits into
 *     it when they meet an out-of-range slot, block id or sequence position;
 *     the offending token is skipped, never written out of bounds.  The
 *     caller zeroes it beforehand and reads it after synchronising.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_NULL = -1,    /* a required pointer is NULL */
  KVQ_ERR_SHAPE = -2,   /* a size is negative, zero where it cannot be, or
                           breaks a divisibility rule */
  KVQ_ERR_ALIGN = -3,   /* a pointer or stride breaks the 16-byte rule */
  KVQ_ERR_DTYPE = -4,   /* unsupported input element type */
  KVQ_ERR_LAYOUT = -5,  /* layout is neither HND nor NHD */
  KVQ_ERR_CUDA = -6,    /* the CUDA runtime reported an error at launch */
  KVQ_ERR_ARG = -7,     /* unknown flag bits or inconsistent arguments */
  KVQ_ERR_SCRATCH = -8  /* kvq_paged_attention_nvfp4_noalloc: the call needs
                           more scratch than the built-in array holds */
} kvq_status;

/* Size of the scratch array built into the library for
   kvq_paged_attention_nvfp4_noalloc (held on every GPU that loads the
   library until the process exits). */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Physical layout of one side (K or V) of a cache page. */
enum {
  KVQ_LAYOUT_HND = 0, /* data [H][B][D/2], scales [H][B][S]: per-head tiles */
  KVQ_LAYOUT_NHD = 1  /* data [B][H][D/2], scales [B][H][S] */
};

/* Input element types (the page's dispatch takes both half types). */
enum { KVQ_DTYPE_BF16 = 0, KVQ_DTYPE_FP16 = 1 };

/* Flags. */
enum {
  /* kvq_store_nvfp4 only: also write K scales in the swizzled tile order (by
     default K scales are linear and only V scales are swizzled, as the
     page's kernel does). */
  KVQ_F_SWIZZLE_K_SCALE = 1u << 0,
  /* Every call: launch with programmatic dependent launch.  The kernel may
     become resident while the previous kernel on the stream is finishing;
     it waits (griddepcontrol.wait, in hardware) for that kernel to complete
     and its writes to be visible before it touches any memory, so the
     result is the same as a plain launch -- only the launch latency between
     the two kernels is hidden.  Each kernel also allows the next
     PDL-launched kernel to do the same.  Useful when these calls run back
     to back with other kernels on one stream. */
  KVQ_F_PDL = 1u << 1,
  /* kvq_gather_indexer_k, kvq_load_nvfp4 and kvq_paged_attention_nvfp4;
     implies KVQ_F_PDL.  The caller promises that block_table and
     cu_seq_lens (attention: query, block_table, context_lens, k_scale and
     v_scale) are not written by the kernel that runs just before this call
     on the stream (they are ready before it starts), so the kernel stages
     them while that kernel finishes and waits only before it reads the
     cache or the scales (attention: the pages), or writes anything. */
  KVQ_F_PDL_EARLY_META = 1u << 2,
  /* kvq_gather_indexer_k (implies KVQ_F_PDL_EARLY_META), kvq_store_nvfp4
     and kvq_store_indexer_k (imply KVQ_F_PDL).  The caller promises that the
     kernel that runs just before this call on the stream writes none of
     this call's inputs (gather: kv_cache, block_table, cu_seq_lens;
     store_nvfp4: key, value, slot_mapping, k_scale, v_scale;
     store_indexer_k: k, slot_mapping): the kernel then also issues its
     first reads while that kernel finishes and waits for it only before its
     first write (its outputs and dev_error are still written strictly after
     it). */
  KVQ_F_PDL_EARLY_READ = 1u << 4
  /* (bits 3 and 5 are not used) */
};

/* Bits OR-ed into *dev_error by the kernels. */
enum {
  KVQ_DEVERR_SLOT = 1 << 0,  /* slot >= num_blocks * block_size */
  KVQ_DEVERR_BLOCK = 1 << 1, /* block-table entry outside [0, num_blocks) */
  KVQ_DEVERR_SEQ = 1 << 2,   /* position beyond max_blocks_per_seq * B, or an
                                output row that no sequence covers, or
                                cu_seq_lens[num_seqs] != total_tokens */
  KVQ_DEVERR_TIMEOUT = 1 << 3 /* a bounded wait for an asynchronous copy
                                 gave up; the affected rows were not
                                 written */
};

/*
 * kvq_store_nvfp4 -- quantise bf16 K and V to NVFP4 and scatter them into
 * paged cache pages by slot.  (vLLM nvfp4_kv_cache_kernels.cu, commit
 * 7ce4c8e: reshape_and_cache_nvfp4_kernel, reshape_and_cache_nvfp4_dispatch.)
 *
 * For token t with s = slot_mapping[t] >= 0 (s < 0: the token is skipped and
 * nothing of it is written), blk = s / block_size, off = s % block_size, for
 * each side (K with g = 1/k_scale[0], V with g = 1/v_scale[0]), head h and
 * 16-element group j of the head:
 *   amax = max |x_i|;  sf = e4m3_rn_satfinite((amax / 6) * g)
 *   q_i  = sf == 0 ? 0 : e2m1_rn_satfinite(x_i * (g / float(sf)))
 * (fp32 IEEE divisions and products, no fused multiply-add), packed two codes
 * per byte, element 2k in the low nibble of byte k.
 *
 * Page layout (side = key_cache or value_cache, i.e. kv_cache[:, 0] and
 * kv_cache[:, 1]; page p of a side starts at side + p * page_stride):
 *   [data: H*B*D/2 bytes | scales: H*B*S bytes], S = head_size / 16,
 *   HND: data (h, off) row at h*B*D/2 + off*D/2, scale tile of head h at
 *        D/2*H*B + h*B*S;  NHD: data row at off*H*D/2 + h*D/2, scale tile
 *        of head h at D/2*H*B + h*S with rows H*S apart.
 *   The 8 data bytes of group j sit at +8*j of the row.  Inside the head's
 *   [B, S] scale tile, K scales are linear (row off, column j) unless
 *   KVQ_F_SWIZZLE_K_SCALE; V scales are swizzled: row (off/4)*4 + j/(S/4),
 *   column (j % (S/4))*4 + off % 4.
 *   Bytes that no stored token owns are left unchanged.
 *
 * key, value      bf16 or fp16 [num_tokens, num_heads, head_size]; heads and
 *                 elements contiguous, rows key_stride0 / value_stride0
 *                 ELEMENTS apart (>= 0, multiple of 8); 16-byte aligned.
 * dtype           KVQ_DTYPE_BF16 or KVQ_DTYPE_FP16 (both widen to fp32
 *                 exactly; the arithmetic is the same).
 * key_cache, value_cache  page 0 of the K side and of the V side;
 *                 16-byte aligned; page_stride multiple of 16 and
 *                 >= H*B*(D/2 + S).
 * block_size      multiple of 4;  head_size multiple of 64;
 * num_blocks      pages in the cache (bounds check for slots).
 * slot_mapping    int64 [num_tokens]; distinct non-negative slots
 *                 (duplicates race; the result is then unspecified).
 * k_scale, v_scale  device fp32 scalars, finite and > 0.
 * flags           KVQ_F_SWIZZLE_K_SCALE, KVQ_F_PDL or KVQ_F_PDL_EARLY_READ,
 *                 or 0.
 * dev_error       nullable device int32 (KVQ_DEVERR_SLOT).
 * stream          cudaStream_t.
 * num_tokens == 0 returns KVQ_OK without launching.
 */
kvq_status kvq_store_nvfp4(const void* key, int64_t key_stride0,
                           const void* value, int64_t value_stride0,
                           int32_t dtype, int32_t num_tokens,
                           int32_t num_heads, int32_t head_size,
                           uint8_t* key_cache, uint8_t* value_cache,
                           int64_t page_stride, int32_t block_size,
                           int64_t num_blocks, int32_t layout,
                           const int64_t* slot_mapping, const float* k_scale,
                           const float* v_scale, uint32_t flags,
                           int32_t* dev_error, void* stream);

/*
 * kvq_gather_indexer_k -- gather fp8 indexer-K rows and their fp32 scales out
 * of a paged cache into contiguous outputs.  (vLLM PR #25931
 * cp_gather_indexer_k_quant_cache(kv_cache, k_fp8, k_scale, block_table,
 * cu_seq_lens); PR #26456: k_scale is a byte buffer the consumer views as
 * float32.)
 *
 * Block layout: [block_size*head_dim fp8 K | block_size * 4 scale bytes],
 * blocks block_stride bytes apart.  For sequence b (0 <= b < num_seqs) and
 * position p in [0, cu_seq_lens[b+1] - cu_seq_lens[b]), output row
 * i = cu_seq_lens[b] + p receives, from blk = block_table[b *
 * block_table_stride + p / block_size], off = p % block_size:
 *   k_fp8[i*head_dim .. +head_dim) = K bytes of (blk, off)
 *   k_scale[4*i .. +4)             = the 4 scale bytes of (blk, off)
 * Rows are written for i < total_tokens only; scale bytes are copied raw.
 *
 * kv_cache        16-byte aligned; block_stride multiple of 16 and
 *                 >= block_size * (head_dim + 4).
 * head_dim        multiple of 16.   block_size > 0.
 * block_table     int32, rows block_table_stride entries apart, first
 *                 max_blocks_per_seq entries of each row used.
 * cu_seq_lens     int32 [num_seqs + 1], non-decreasing, cu_seq_lens[0] == 0.
 * total_tokens    cu_seq_lens[num_seqs], as known on the host (the kernel
 *                 flags KVQ_DEVERR_SEQ if the two disagree).
 * k_fp8           [total_tokens, head_dim] bytes, 16-byte aligned.
 * k_scale         [total_tokens * 4] bytes, 4-byte aligned.
 * flags           KVQ_F_PDL, KVQ_F_PDL_EARLY_META, KVQ_F_PDL_EARLY_READ, or 0.
 * dev_error       nullable device int32 (KVQ_DEVERR_BLOCK | KVQ_DEVERR_SEQ |
 *                 KVQ_DEVERR_TIMEOUT).
 * total_tokens == 0 returns KVQ_OK without launching.
 */
kvq_status kvq_gather_indexer_k(const uint8_t* kv_cache, int64_t block_stride,
                                int64_t num_blocks, int32_t block_size,
                                int32_t head_dim, const int32_t* block_table,
                                int64_t block_table_stride,
                                int32_t max_blocks_per_seq,
                                const int32_t* cu_seq_lens, int32_t num_seqs,
                                int64_t total_tokens, uint8_t* k_fp8,
                                uint8_t* k_scale, uint32_t flags,
                                int32_t* dev_error, void* stream);

/*
 * kvq_load_nvfp4 -- the read side of kvq_store_nvfp4: gather the tokens a
 * block table names out of NVFP4 pages and dequantise them to bf16 rows.
 * (Page layout, strides and scale swizzle: vLLM nvfp4_kv_cache_kernels.cu,
 * commit 7ce4c8e, as for the store.  The pages state no dequantisation
 * rule; this is the plain inverse of the store's.)
 *
 * For sequence b and position p in [0, cu_seq_lens[b+1] - cu_seq_lens[b]),
 * output row i = cu_seq_lens[b] + p reads page blk = block_table[b *
 * block_table_stride + p / block_size], offset off = p % block_size; for
 * each side, head h and group j, with s = float(scale byte) (linear or
 * swizzled position as the store wrote it) and c = s * k_scale[0] (or
 * v_scale[0]) in fp32:
 *   out[i, h, 16j + k] = bf16_rn(e2m1(q_k) * c)   (fp32 product, then
 *                                                   round to nearest even)
 *
 * key_cache, value_cache, page_stride, block_size, num_blocks, layout,
 * num_heads, head_size   as for kvq_store_nvfp4.
 * block_table, block_table_stride, max_blocks_per_seq, cu_seq_lens,
 * num_seqs, total_tokens   as for kvq_gather_indexer_k.
 * k_scale, v_scale  device fp32 scalars (the store's).
 * out_dtype       KVQ_DTYPE_BF16.
 * key_out, value_out  [total_tokens, num_heads, head_size] rows,
 *                 out_stride0 elements apart (>= H*D, multiple of 8);
 *                 16-byte aligned.
 * flags           KVQ_F_SWIZZLE_K_SCALE (the pages were stored with it),
 *                 KVQ_F_PDL, KVQ_F_PDL_EARLY_META, or 0.
 * dev_error       nullable (KVQ_DEVERR_BLOCK | KVQ_DEVERR_SEQ |
 *                 KVQ_DEVERR_TIMEOUT); rows it names are left unwritten.
 * total_tokens == 0 returns KVQ_OK without launching.
 */
kvq_status kvq_load_nvfp4(const uint8_t* key_cache, const uint8_t* value_cache,
                          int64_t page_stride, int32_t block_size,
                          int64_t num_blocks, int32_t layout,
                          int32_t num_heads, int32_t head_size,
                          const int32_t* block_table,
                          int64_t block_table_stride,
                          int32_t max_blocks_per_seq,
                          const int32_t* cu_seq_lens, int32_t num_seqs,
                          int64_t total_tokens, const float* k_scale,
                          const float* v_scale, int32_t out_dtype,
                          void* key_out, void* value_out, int64_t out_stride0,
                          uint32_t flags, int32_t* dev_error, void* stream);

/*
 * kvq_store_indexer_k -- the write side of the indexer cache that
 * kvq_gather_indexer_k reads: quantise each token's K row to fp8 e4m3 with
 * one fp32 scale and store both into the token's block slot.  (vLLM PR
 * #25931: "quantized k/k_scale" in the indexer k cache.  The pages give no
 * quantisation rule; per-token absmax scaling is taken.)
 *
 * For token t with s = slot_mapping[t] >= 0 (s < 0: skipped),
 * blk = s / block_size, off = s % block_size:
 *   amax  = max |k[t, d]|;  scale = amax / 448   (fp32 IEEE division)
 *   q[d]  = amax == 0 ? 0 : e4m3_rn_satfinite(k[t, d] / scale)  (IEEE div)
 *   block blk bytes [off*head_dim, +head_dim) = q;
 *   bytes [block_size*head_dim + 4*off, +4)   = scale (fp32).
 *
 * k             bf16 or fp16 [num_tokens, head_dim], rows k_stride0
 *               elements apart (multiple of 8); 16-byte aligned.
 * head_dim      16, 32, 64, 128 or 256.
 * kv_cache      block 0 of [block_size*head_dim | block_size*4] blocks,
 *               block_stride bytes apart (multiple of 16, >= block_size *
 *               (head_dim + 4)); 16-byte aligned.
 * slot_mapping  int64 [num_tokens], distinct slots (duplicates race).
 * flags         KVQ_F_PDL, KVQ_F_PDL_EARLY_READ, or 0.
 * dev_error     nullable (KVQ_DEVERR_SLOT for slots >= num_blocks *
 *               block_size, which are skipped).
 * num_tokens == 0 returns KVQ_OK without launching.
 */
kvq_status kvq_store_indexer_k(const void* k, int64_t k_stride0,
                               int32_t dtype, int32_t num_tokens,
                               int32_t head_dim, uint8_t* kv_cache,
                               int64_t block_stride, int32_t block_size,
                               int64_t num_blocks,
                               const int64_t* slot_mapping, uint32_t flags,
                               int32_t* dev_error, void* stream);

/*
 * kvq_paged_attention_nvfp4 -- paged decode attention over the NVFP4 cache
 * that kvq_store_nvfp4 writes.  (vLLM PR #12348 "[ROCm] Faster Custom Paged
 * Attention kernels": paged_attention(out, exp_sums, max_logits, tmp_out,
 * query, key_cache, value_cache, num_kv_heads, scale, block_tables,
 * context_lens, block_size, max_context_len, alibi_slopes, kv_cache_dtype,
 * k_scale, v_scale, partition_size).  The page shows the signature only;
 * the computation is plain softmax attention on the dequantised cache.)
 *
 * For sequence b (one query token) with L = context_lens[b] and query head
 * h, reading KV head h / (num_q_heads / num_kv_heads):
 *   K^[t, d] = e2m1(q) * float(sf) * k_scale[0]   (V^ with v_scale[0]; sf at
 *              its stored position: K linear unless KVQ_F_SWIZZLE_K_SCALE,
 *              V swizzled), token t of page block_table[b*stride + t/B],
 *              offset t % B, for t < L;
 *   s_t = scale * sum_d q[b, h, d] K^[t, d];  out[b, h, :] =
 *   sum_t softmax(s)_t V^[t, :];  L == 0 gives zeros.
 * Arithmetic (the tolerance of any comparison follows from it): the query
 * is rounded to fp16, e2m1 * sf is exact in fp16, q . (e2m1 * sf) and
 * P . V' accumulate in fp32 on the tensor cores, P = exp2 of the scaled
 * logits minus a reference value of the stretch of context being
 * accumulated (a logit maximum; the kernel moves it only when a logit
 * exceeds it by more than 8, so P < 2^8) is rounded to fp16 and the
 * denominator sums the rounded values; stretches merge in fp32 (rescaled
 * by exp2 of the difference of their references); out is rounded once.
 *
 * query          bf16 / fp16 (dtype) [num_seqs, num_q_heads, 128], rows
 *                query_stride0 elements apart (multiple of 8), 16-byte
 *                aligned; |q| < 65504 (fp16 range).
 * head_size      128.   num_q_heads / num_kv_heads <= 16 (and divides).
 * key_cache, value_cache, page_stride, block_size, num_blocks, layout
 *                as for kvq_store_nvfp4 (num_kv_heads heads per page).
 * block_table    int32, rows block_table_stride apart, first
 *                max_blocks_per_seq entries used.
 * context_lens   int32 [num_seqs]; values above min(max_context_len,
 *                max_blocks_per_seq * block_size) are clamped to it and
 *                flagged (KVQ_DEVERR_SEQ).
 * max_context_len  also sizes the launch (one CTA per stretch a context
 *                of that length would have, for every sequence and KV
 *                head): pass the batch's longest context, not a loose
 *                bound (on a batch of 512..2560-token contexts, 8192
 *                costs 0.5 % and 32768 costs 33 %, in CTAs that find no
 *                work).
 * k_scale, v_scale  device fp32 scalars (the store's).
 * scale          softmax scale, finite.
 * partition_size 128, 256, 384 or 512 tokens.
 * exp_sums, max_logits  fp32 [num_seqs, num_q_heads, max_parts] scratch,
 * tmp_out        fp32 [num_seqs, num_q_heads, max_parts, 128] scratch, with
 *                max_parts = ceil(max_context_len / partition_size); needed
 *                (non-NULL) only when max_parts > 1.  Nothing in them has to
 *                be initialised; their contents afterwards are unspecified.
 * out            dtype [num_seqs, num_q_heads, 128], rows out_stride0
 *                elements apart (multiple of 8), 16-byte aligned.
 * flags          KVQ_F_SWIZZLE_K_SCALE, KVQ_F_PDL, KVQ_F_PDL_EARLY_META
 *                (e.g. after kvq_store_nvfp4, which writes only the pages),
 *                or 0.
 * dev_error      nullable (KVQ_DEVERR_BLOCK: the token is left out;
 *                KVQ_DEVERR_SEQ).
 * num_seqs == 0 returns KVQ_OK without launching.
 */
kvq_status kvq_paged_attention_nvfp4(
    const void* query, int64_t query_stride0, int32_t dtype, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    const uint8_t* key_cache, const uint8_t* value_cache, int64_t page_stride,
    int32_t block_size, int64_t num_blocks, int32_t layout,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const float* k_scale, const float* v_scale,
    float scale, int32_t partition_size, float* exp_sums, float* max_logits,
    float* tmp_out, void* out, int64_t out_stride0, uint32_t flags,
    int32_t* dev_error, void* stream);

/*
 * kvq_paged_attention_nvfp4_noalloc -- kvq_paged_attention_nvfp4 for callers
 * that cannot allocate device memory.  The source material has no
 * counterpart; this entry point is an addition of this library.
 *
 * Who needs it: the attention needs fp32 scratch whenever a context spans
 * more than one partition, and the plain entry point takes it from the
 * caller.  A caller that runs after an engine has reserved all device
 * memory for itself, or inside a runtime that forbids device allocation
 * once it is serving, has no way to provide it.  This entry point takes no
 * scratch arguments and allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine): it uses an array of
 * KVQ_NOALLOC_SCRATCH_BYTES (32 MiB) built into the library, which every
 * GPU that loads the library holds until the process exits.
 *
 * Arguments, result and errors: as kvq_paged_attention_nvfp4 without
 * exp_sums, max_logits and tmp_out (its argument checks run first, so a
 * call it would reject gets the same code).  A call that needs more than
 * the array holds -- num_seqs * num_q_heads * ceil(max_context_len /
 * partition_size) * (head_size + 2) * 4 bytes, when that ceiling is above
 * 1 -- returns KVQ_ERR_SCRATCH and launches nothing.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it; make that first call outside any stream
 * capture.  All calls share the one array, which keeps whatever the last
 * call left in it; nothing in it needs to start at zero, since every entry
 * a call reads it has written first.  Calls whose kernels can overlap on
 * the GPU (other streams, other host threads) race on the array and must be
 * ordered by the caller.
 */
kvq_status kvq_paged_attention_nvfp4_noalloc(
    const void* query, int64_t query_stride0, int32_t dtype, int32_t num_seqs,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    const uint8_t* key_cache, const uint8_t* value_cache, int64_t page_stride,
    int32_t block_size, int64_t num_blocks, int32_t layout,
    const int32_t* block_table, int64_t block_table_stride,
    int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const float* k_scale, const float* v_scale,
    float scale, int32_t partition_size, void* out, int64_t out_stride0,
    uint32_t flags, int32_t* dev_error, void* stream);

/* Static text for a status code. */
const char* kvq_status_string(kvq_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
