/*
 * pagedkv.h -- C ABI of the GB300 paged KV-cache library (libpagedkv.so).
 *
 * Two operations on a paged KV cache, as the pages describe them:
 *
 *  - the KV write ("reshape_and_cache"): each new token's key and value are
 *    scattered into fixed-size physical blocks at the flat slot index the
 *    scheduler assigned ("TGI PagedAttention deep-dive" (lpnh.cn) sec. 4.1,
 *    the write side "writes new key/value into the block cache by slots, with
 *    FP8 KV-cache quantised writes");
 *
 *  - the decode step ("paged_attention"): for each sequence and query head,
 *    walk the sequence's block table to gather K/V scattered across the block
 *    pool, and compute softmax(scale * q K^T) V over the sequence's
 *    context_len tokens ("Lecture 3: PagedAttention and vLLM", section "the
 *    paged implementation of attention": logical block -> physical block, then
 *    softmax and the weighted sum; TGI deep-dive sec. 4.3, block_tables passed
 *    to the kernel). Long contexts are split into partitions (512 tokens on the
 *    pages) computed in parallel and merged by a max / sum-exp reduction (TGI
 *    deep-dive sec. 4.1, PagedAttention V2 and _PARTITION_SIZE 512).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Pointers.   Every tensor pointer is a DEVICE pointer owned by the caller.
 *              The library allocates nothing and keeps no state between calls.
 *              Data arrays (query, out, key, value, the caches, the
 *              workspace) must be 16-byte aligned, index arrays (block
 *              tables, lengths, query starts: 4 bytes; slots, block pairs:
 *              8 bytes) naturally aligned; otherwise PA_ERR_INVALID_ARG.
 *  Streams.    `stream` is a cudaStream_t (NULL = the legacy default stream).
 *              Every call only enqueues work on it and returns; nothing
 *              synchronises the host.
 *  Errors.     Argument errors are found on the host before anything is
 *              launched and returned as PA_ERR_INVALID_ARG or
 *              PA_ERR_UNSUPPORTED; a failed launch returns PA_ERR_CUDA.
 *              Errors found by a kernel in the data (a block id outside the
 *              pool, a slot outside the pool, a bad context length) set bits
 *              in *dev_status with an atomic OR; the kernel skips the bad
 *              access and carries on, and the outputs that depended on it are
 *              unspecified. dev_status is a device uint32 the caller zeroes
 *              and reads back after synchronising; it may be NULL.
 *              No kernel traps or asserts; every wait in a kernel is bounded
 *              in time and reports PA_DEV_TIMEOUT when it runs out.
 *  Types.      Element types are given by pa_dtype. The query and the output
 *              share one type. A cache holds the query type, or OCP E4M3 codes
 *              for a binary16 / bfloat16 query.
 *
 * Cache layout declared by this library
 * -------------------------------------
 *  k_cache and v_cache are separate tensors, each
 *      [num_blocks][num_kv_heads][block_size][head_size]
 *  contiguous, element = cache dtype. One (block, KV head) pair is a
 *  contiguous slab of block_size * head_size elements, so a block's tokens for
 *  one head are read in one bulk copy. (The pages show other layouts, e.g.
 *  [num_blocks, num_heads, head_size, BLOCK_SIZE] in the TGI deep-dive
 *  sec. 4.2; results do not depend on the layout.)
 *
 *  A token at logical position t of sequence s lives in physical block
 *  block_tables[s * max_blocks_per_seq + t / block_size], slot t % block_size.
 *  Its flat slot index is block * block_size + t % block_size.
 *
 * Decode arithmetic
 * -----------------
 *  G = num_q_heads / num_kv_heads (an integer); query head h reads KV head
 *  h / G. For a sequence of length L the output of head h is
 *      out = sum_i softmax_i(scale * <q_h, k_i>) v_i,  i < L,
 *  accumulated in float32. An E4M3 cache is read as code_value * k_scale
 *  (keys) and code_value * v_scale (values). A sequence with L == 0 gets a
 *  zero output. The output is rounded to its type to nearest even.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* a NULL pointer, a negative size, inconsistent shapes */
    PA_ERR_UNSUPPORTED = 2,   /* a valid request this library does not implement */
    PA_ERR_WORKSPACE = 3,     /* the workspace is NULL, misaligned or too small */
    PA_ERR_CUDA = 4,          /* a CUDA call or launch failed */
    PA_ERR_NO_BLOCKS = 5      /* the block allocator has too few free blocks */
} pa_status;

typedef enum pa_dtype {
    PA_F32 = 0,               /* IEEE binary32 */
    PA_F16 = 1,               /* IEEE binary16 */
    PA_BF16 = 2,              /* bfloat16 */
    PA_FP8_E4M3 = 3           /* OCP E4M3 (bias 7, max 448, no infinities) */
} pa_dtype;

/* Bits a kernel ORs into *dev_status. */
#define PA_DEV_BAD_BLOCK_ID 1u  /* a block_tables entry it needed is outside [0, num_blocks) */
#define PA_DEV_BAD_SLOT     2u  /* a slot_mapping entry is >= num_blocks * block_size */
#define PA_DEV_BAD_LEN      4u  /* a context length is < 0, above max_context_len,
                                   or needs more than max_blocks_per_seq blocks */
#define PA_DEV_TIMEOUT      8u  /* a bounded wait inside a kernel ran out */
#define PA_DEV_SLOT_MISMATCH 16u /* a fused write's slot is not the newest position of its
                                    sequence (the token is stored; the decode may miss it) */
#define PA_DEV_BAD_ORDER    32u /* a seq_order entry is outside [0, num_seqs) (the work
                                   it names is skipped) */
#define PA_DEV_BAD_PREFIX   64u /* a shared-prefix unit member whose context does not extend
                                   past the unit's shared partitions, whose skip count differs
                                   from the unit's, or whose block table differs from the
                                   unit's first member's over a shared partition */

/* Supported shapes: head_size in {64, 128, 256}; block_size in [1, 1024];
 * partition_size a positive multiple of 32 (512 on the pages). */

/*
 * pa_reshape_and_cache -- the KV write (TGI deep-dive sec. 4.1, the write
 * side; "vLLM Page Attention Continuous Batching" (lbrq.cn), "KV Block": a
 * block holds block_size tokens of every head of a layer).
 *
 *  key, value     [num_tokens][num_kv_heads][head_size], type in_dtype.
 *  k_cache,
 *  v_cache        the block pool (layout above), type cache_dtype; written in
 *                 place.
 *  slot_mapping   [num_tokens] int64. slot >= 0: the token goes to block
 *                 slot / block_size, position slot % block_size. slot < 0: a
 *                 padding token, skipped. slot >= num_blocks * block_size:
 *                 skipped and PA_DEV_BAD_SLOT is set.
 *  cache_dtype == in_dtype: the element bits are copied.
 *  cache_dtype == PA_FP8_E4M3 (in_dtype F32, F16 or BF16): each element x is
 *                 stored as E4M3(x / scale), the quotient an IEEE binary32
 *                 division, the conversion rounding to nearest even and
 *                 saturating to +-448 (NaN stays NaN). k_scale applies to
 *                 keys, v_scale to values; both must be finite and > 0.
 *  Two tokens that name the same slot race; the result is one of them.
 *  num_tokens == 0 launches nothing and returns PA_OK.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                               int head_size, int block_size, int64_t num_blocks,
                               pa_dtype in_dtype, pa_dtype cache_dtype, float k_scale,
                               float v_scale, uint32_t* dev_status, void* stream);

/*
 * pa_decode -- single-pass decode (PagedAttention "V1" on the pages: one
 * pass per sequence, no reduction). One work unit per (sequence, KV head
 * group); suits short contexts or many sequences.
 *
 *  out            [num_seqs][num_q_heads][head_size], type q_dtype.
 *  query          [num_seqs][num_q_heads][head_size], type q_dtype.
 *  k_cache,
 *  v_cache        the block pool, type cache_dtype, num_blocks blocks.
 *  block_tables   [num_seqs][max_blocks_per_seq] int32. Entries at or past
 *                 ceil(context_lens[s] / block_size) are never read.
 *  context_lens   [num_seqs] int32, 0 <= L <= max_context_len and
 *                 ceil(L / block_size) <= max_blocks_per_seq.
 *  max_context_len  an upper bound on context_lens the caller knows without
 *                 reading the device (no device-to-host copy is made).
 *  scale          the softmax scale (1/sqrt(head_size) is usual).
 *  k_scale,
 *  v_scale        E4M3 dequantisation scales (ignored for other caches).
 *  num_seqs == 0 launches nothing.
 */
pa_status pa_decode(void* out, const void* query, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                    int head_size, int block_size, int64_t num_blocks, int max_context_len,
                    float scale, pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                    float v_scale, uint32_t* dev_status, void* stream);

/*
 * Workspace of the partitioned decode (caller-allocated, 256-byte aligned):
 *      tmp_out     float32 [num_seqs][num_q_heads][max_partitions][head_size]
 *      max_logits  float32 [num_seqs][num_q_heads][max_partitions]
 *      exp_sums    float32 [num_seqs][num_q_heads][max_partitions]
 *  in that order, each region starting on a 256-byte boundary, with
 *  max_partitions = ceil(max_context_len / partition_size) (at least 1).
 *  For partition p of sequence s and head h (tokens [p*P, min((p+1)*P, L))):
 *  max_logits = max_i scale*<q, k_i>, exp_sums = sum_i exp(s_i - max_logits),
 *  tmp_out = sum_i exp(s_i - max_logits) v_i / exp_sums.
 *  pa_decode_workspace_layout gives the three byte offsets and the total.
 */
size_t pa_decode_partitioned_workspace_bytes(int num_seqs, int num_q_heads, int head_size,
                                             int max_context_len, int partition_size);
pa_status pa_decode_workspace_layout(int num_seqs, int num_q_heads, int head_size,
                                     int max_context_len, int partition_size,
                                     size_t* tmp_out_offset, size_t* max_logits_offset,
                                     size_t* exp_sums_offset, size_t* total_bytes);

/*
 * pa_decode_partitions -- the partition kernel of the split decode (the
 * pages' "V2"): writes every partition's (tmp_out, max_logits, exp_sums) into
 * the workspace and nothing else. Arguments as pa_decode, plus the partition
 * size and the workspace. Partitions past a sequence's length are not
 * written.
 */
pa_status pa_decode_partitions(const void* query, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_size, int block_size,
                               int64_t num_blocks, int max_context_len, float scale,
                               pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                               float v_scale, int partition_size, void* workspace,
                               size_t workspace_bytes, uint32_t* dev_status, void* stream);

/*
 * pa_merge -- the reduction of the split decode (TGI deep-dive sec. 4.1:
 * partitions "computed in parallel, then merged"). For each (s, h) with
 * n = ceil(context_lens[s] / partition_size) partitions:
 *      M = max_p max_logits[p],  w_p = exp_sums[p] * exp(max_logits[p] - M),
 *      out = sum_p w_p tmp_out[p] / sum_p w_p
 *  (zero when n == 0). tmp_out, max_logits, exp_sums are the three workspace
 *  regions (any float32 device arrays of those shapes); max_partitions is
 *  their partition extent. out has type out_dtype (F32, F16 or BF16).
 */
pa_status pa_merge(void* out, const float* tmp_out, const float* max_logits, const float* exp_sums,
                   const int32_t* context_lens, int num_seqs, int num_q_heads, int head_size,
                   int partition_size, int max_partitions, pa_dtype out_dtype,
                   uint32_t* dev_status, void* stream);

/* pa_decode_partitioned -- pa_decode_partitions followed by pa_merge on the
 * same stream (two kernels). */
pa_status pa_decode_partitioned(void* out, const void* query, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_size, int block_size,
                                int64_t num_blocks, int max_context_len, float scale,
                                pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                                float v_scale, int partition_size, void* workspace,
                                size_t workspace_bytes, uint32_t* dev_status, void* stream);

/*
 * pa_write_decode -- the KV write and the single-pass decode of one step in
 * ONE launch (the TGI deep-dive, sec. 4.1, runs paged_reshape_and_cache and
 * then paged_attention every decode step; here the write is folded into the
 * decode kernel). Each sequence s brings one new token: key[s], value[s]
 * ([num_seqs][num_kv_heads][head_size], of the query type) stored at
 * slot_mapping[s] exactly as pa_reshape_and_cache stores it (bit copy, or E4M3
 * with k_scale / v_scale), and that token is position context_lens[s] - 1 of
 * the decode. The kernel that loads the stage holding that position stores the
 * token first and then reads it back through its bulk copy, so the slot must be
 * that position of the sequence's own block table (else PA_DEV_SLOT_MISMATCH;
 * a token written elsewhere is not ordered with the reads of other sequences).
 * A negative slot stores nothing (the decode still covers the context). A
 * sequence with context_len 0 stores nothing and gets a zero output.
 * Other arguments as pa_decode; k_cache / v_cache are written.
 */
pa_status pa_write_decode(void* out, const void* query, const void* key, const void* value,
                          const int64_t* slot_mapping, void* k_cache, void* v_cache,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                          int max_context_len, float scale, pa_dtype q_dtype,
                          pa_dtype cache_dtype, float k_scale, float v_scale,
                          uint32_t* dev_status, void* stream);

/* pa_write_decode_partitions -- the partition kernel of the split decode
 * with the new tokens' write folded in (pa_decode_partitions + the write):
 * stores the tokens and every partition's partials in the workspace. */
pa_status pa_write_decode_partitions(const void* query, const void* key, const void* value,
                                     const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_size, int block_size,
                                     int64_t num_blocks, int max_context_len, float scale,
                                     pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                                     float v_scale, int partition_size, void* workspace,
                                     size_t workspace_bytes, uint32_t* dev_status, void* stream);

/* pa_write_decode_partitioned -- pa_write_decode_partitions, then pa_merge on
 * the same stream: two launches for the whole step instead of three. */
pa_status pa_write_decode_partitioned(void* out, const void* query, const void* key,
                                      const void* value, const int64_t* slot_mapping,
                                      void* k_cache, void* v_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_size, int block_size, int64_t num_blocks,
                                      int max_context_len, float scale, pa_dtype q_dtype,
                                      pa_dtype cache_dtype, float k_scale, float v_scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      uint32_t* dev_status, void* stream);

/*
 * Shared-prefix decode. Requests with a common prompt prefix share its cached
 * KV blocks ("TGI PagedAttention deep-dive" (lpnh.cn) sec. 5, prefix reuse;
 * "Lecture 3: PagedAttention and vLLM", "shared prefix": several block tables
 * point at the same physical blocks). The partitioned decode then reads those
 * blocks once per sequence. Here sequences whose tables agree over their
 * first partitions are put in units of up to PA_SHARED_UNIT_MEMBERS, and a
 * unit reads each shared partition's K/V once for all its members; the
 * result is the partitioned decode's, up to floating-point rounding order.
 *
 * pa_shared_prefix_plan -- host only: the units for a batch, from the host
 * copies of block_tables [num_seqs, max_blocks_per_seq] and context_lens
 * [num_seqs]. A sequence can share partition j (tokens [j P, (j+1) P), P =
 * partition_size, a multiple of 32 and of block_size) only if its table
 * names the same blocks there as its unit's other members, and only
 * partitions wholly before its newest token (at most (L - 1) / P).
 * Outputs (host memory, caller-owned):
 *   seq_shared_parts [num_seqs]   leading partitions each sequence shares (0: none)
 *   unit_seqs [max_units * PA_SHARED_UNIT_MEMBERS]  each unit's sequences, -1 padded
 *   unit_parts [max_units]        partitions each unit's members share (>= 1)
 *   *num_units, *max_unit_parts   units formed, and the largest unit_parts
 * Units stop at max_units (the remaining sequences share nothing). Argument
 * errors -> PA_ERR_INVALID_ARG.
 */
#define PA_SHARED_UNIT_MEMBERS 4
pa_status pa_shared_prefix_plan(const int32_t* block_tables, const int32_t* context_lens,
                                int num_seqs, int max_blocks_per_seq, int block_size,
                                int partition_size, int32_t* seq_shared_parts,
                                int32_t* unit_seqs, int32_t* unit_parts, int max_units,
                                int* num_units, int* max_unit_parts);

/*
 * pa_write_decode_shared_prefix -- one decode step with shared-prefix units:
 * one launch of the partition kernel whose first CTAs compute each unit's
 * shared partitions (every stage read once for all members) and whose other
 * CTAs compute every other partition (with the step's KV write folded in when
 * key/value/slot_mapping are given, as in pa_write_decode_partitions), then
 * pa_merge into out. Two launches on `stream`. Arguments are pa_write_decode_partitioned's plus the plan of
 * pa_shared_prefix_plan, copied to the device by the caller:
 *   seq_shared_parts [num_seqs], unit_seqs [num_units, PA_SHARED_UNIT_MEMBERS],
 *   unit_parts [num_units] int32 (device); max_unit_parts (the plan's largest
 *   unit_parts) <= the partitions of max_context_len; num_seqs + num_units <=
 *   65535. num_units == 0: the plain partitioned step.
 * key, value and slot_mapping are all null (decode only) or all given.
 * The workspace is pa_decode_partitioned_workspace_bytes(num_seqs,
 * num_q_heads, head_size, max_context_len, partition_size), as for the
 * partitioned decode. Shapes: those of the tensor-core decode (a 16-bit
 * query with a cache of its type or E4M3, an even group or none, rows of
 * 128/256/512 bytes, block size 8, 16 or a multiple of 32) and
 * partition_size a multiple of block_size; otherwise PA_ERR_UNSUPPORTED.
 * Device checks: a member whose context does not extend past its unit's
 * partitions (or exceeds the bounds) is computed by the partition kernel
 * instead, and PA_DEV_BAD_PREFIX is set; so is it for a member whose skip
 * count or block table over a shared partition differs from the unit's (its
 * output is then unspecified). A sequence with a skip count that belongs to
 * no unit is not detected: the plan must come from pa_shared_prefix_plan or
 * hold the same rules.
 */
pa_status pa_write_decode_shared_prefix(
    void* out, const void* query, const void* key, const void* value, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, int max_context_len, float scale, pa_dtype q_dtype,
    pa_dtype cache_dtype, float k_scale, float v_scale, const int32_t* seq_shared_parts,
    const int32_t* unit_seqs, const int32_t* unit_parts, int num_units, int max_unit_parts,
    int partition_size, void* workspace, size_t workspace_bytes, uint32_t* dev_status,
    void* stream);

/*
 * pa_decode_partitioned_static -- pa_decode_partitioned for callers that
 * cannot allocate device memory. The pages have no counterpart: this is a
 * convenience of this library. A serving loop that has given all device memory
 * to a fixed pool, or a plugin whose host program owns every allocation,
 * cannot call cudaMalloc for the workspace (and cudaMalloc / cudaFree may
 * synchronise the device). This call allocates nothing: it uses a fixed
 * workspace of PA_STATIC_WORKSPACE_BYTES that lives in the library's own device
 * memory, held by every GPU that loads the library until the process exits.
 *
 *  Arguments and results are those of pa_decode_partitioned without
 *  `workspace` / `workspace_bytes`.
 *  Size limit: a problem whose pa_decode_partitioned_workspace_bytes exceeds
 *  PA_STATIC_WORKSPACE_BYTES is rejected with PA_ERR_WORKSPACE before any
 *  launch. 64 MiB holds, e.g., 256 sequences x 32 query heads at head size 128
 *  with max_context_len up to 7,680 tokens at 512-token partitions (15
 *  partitions: 63,897,600 bytes) or up to 15,360 at 1024-token partitions;
 *  8,192 tokens at 512 (68,157,440 bytes) does not fit.
 *  Address lookup: the first call on a device looks up the device address of
 *  the array (cudaGetSymbolAddress, with that device current) and caches it
 *  against the id of the device's current context; make that first call
 *  before any stream capture. If the context is later replaced (a
 *  cudaDeviceReset, or another driver context made current), the next call
 *  sees a new context id and looks the address up again, so it is also a
 *  first call in this sense. A failed lookup returns PA_ERR_CUDA.
 *  Sharing: every call, on every stream, uses the same array, which keeps the
 *  previous call's contents (nothing in it needs to start at zero). Calls whose
 *  kernels overlap on the GPU race on it and give unspecified results:
 *  serialise them, e.g. on one stream.
 */
#define PA_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)
pa_status pa_decode_partitioned_static(void* out, const void* query, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_size, int block_size, int64_t num_blocks,
                                       int max_context_len, float scale, pa_dtype q_dtype,
                                       pa_dtype cache_dtype, float k_scale, float v_scale,
                                       int partition_size, uint32_t* dev_status, void* stream);

/*
 * pa_paged_prefill -- multi-query paged attention: several query tokens per
 * sequence against the paged cache, for a prefill chunk (TGI deep-dive sec.
 * 6.2, PREFILL_CHUNKING: a long prefill is cut into chunks) or the draft
 * tokens of a speculative-decoding verification ("vLLM Page Attention
 * Continuous Batching" (lbrq.cn), "vLLM 主要能力"). The paged attention of
 * "Lecture 3: PagedAttention and vLLM" ("the paged implementation of
 * attention") already takes queries [num_queries, num_heads, head_dim]; the
 * pages give no mask, and this call reads it causally: the Q_s query tokens
 * of sequence s are the last Q_s of its L_s = context_lens[s] tokens (their
 * K/V already written), and query token i (0-based within s) attends to keys
 * 0 .. L_s - Q_s + i. With Q_s = 1 this is the decode.
 *
 *  out, query     [num_queries][num_q_heads][head_size], type q_dtype; the
 *                 tokens of sequence s are rows query_start[s] ..
 *                 query_start[s+1] - 1. 16-byte aligned.
 *  query_start    [num_seqs + 1] int32, device, non-decreasing,
 *                 query_start[0] = 0, query_start[num_seqs] = num_queries.
 *  max_queries_per_seq  an upper bound on Q_s known on the host (sizes the
 *                 grid); 0 <= Q_s <= max_queries_per_seq and Q_s <= L_s.
 *  seq_order      null, or [num_seqs] int32, device, 4-byte aligned: a
 *                 permutation of 0..num_seqs-1, the order in which the
 *                 sequences' work is started (a scheduling hint: the
 *                 outputs do not depend on it). The GPU starts work in launch
 *                 order and cannot see the lengths before it starts, so a
 *                 caller that knows them on the host (a serving scheduler
 *                 does) passes the longest contexts first, and the last CTAs
 *                 to start are short ones. An entry outside [0, num_seqs)
 *                 sets PA_DEV_BAD_ORDER and its work is skipped; sequences a
 *                 non-permutation omits have unspecified rows. The CUDA-core
 *                 path (one query token per work unit) ignores it.
 *  Other arguments as pa_decode; scale must be > 0.
 *  Kernel selection, by the arguments alone: with max_queries_per_seq *
 *  (num_q_heads / num_kv_heads) query rows per sequence and KV head at most
 *  32 (head_size <= 128) or 16 (head_size 256; also 16 where the tcgen05
 *  kernels below take the E4M3 products), a 16-bit query with a cache
 *  of its type or of E4M3 codes, on the shapes of the TMA decode
 *  (rows of 128, 256 or 512 bytes, block_size 8, 16 or a multiple of 32),
 *  the warp-level MMA kernels run, reading each sequence's K/V once for all
 *  its rows (speculative verification). Else a
 *  16-bit query with a cache of the same type (head_size 64/128/256) or an
 *  E4M3 cache (head_size 64/128), a block_size that is a power of two in
 *  [8, 256] and a group of at most 128 heads runs on the tcgen05 tensor
 *  cores (with an E4M3 cache, a bf16 query and head_size 128, both products
 *  take E4M3 operands -- the E4M3 products: the query as two E4M3 terms of
 *  each row times a power of two, exact for bf16 values in E4M3's normal
 *  range, and the softmax weights as two E4M3 terms, relative error at most
 *  about 2^-8; else the E4M3 tiles are widened to binary16); other
 *  supported combinations run one query token per work unit on the CUDA
 *  cores. A sequence whose lengths
 *  break the rules above sets PA_DEV_BAD_LEN and its rows are unspecified.
 *  num_queries == 0 launches nothing.
 */
/* The kernel pa_paged_prefill selects for a shape (16-byte-aligned pointers
 * assumed; the selection depends on nothing else). */
typedef enum {
    PA_PREFILL_CUDA_CORES = 0,     /* one query token per work unit (the decode kernel) */
    PA_PREFILL_MMA = 1,            /* warp-level MMA, up to 16 rows per (sequence, KV head) */
    PA_PREFILL_MMA_TWO_TILES = 2,  /* warp-level MMA, 17-32 rows, two n-tiles per warp */
    PA_PREFILL_TC = 3,             /* tcgen05, one 128-row query tile per CTA */
    PA_PREFILL_TC_TWO_TILES = 4    /* tcgen05, two query tiles per CTA */
} pa_prefill_kernel;

/* Host only (no launch, no GPU needed): the pa_prefill_kernel value for
 * these arguments of pa_paged_prefill, or -1 where pa_paged_prefill would
 * reject them (max_queries_per_seq < 1, a group that is not an integer, an
 * unsupported type pair, head size or block size). */
int pa_paged_prefill_kernel(int max_queries_per_seq, int num_q_heads, int num_kv_heads,
                            int head_size, int block_size, int64_t num_blocks, pa_dtype q_dtype,
                            pa_dtype cache_dtype);

pa_status pa_paged_prefill(void* out, const void* query, const int32_t* query_start,
                           int num_queries, int max_queries_per_seq, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_size, int block_size,
                           int64_t num_blocks, int max_context_len, float scale,
                           pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale, float v_scale,
                           const int32_t* seq_order, uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Block management: the host-side allocator and the copy-on-write copy.
 * ------------------------------------------------------------------------ */

/*
 * pa_copy_blocks -- copy whole physical blocks (every KV head of K and of V)
 * for each (src, dst) pair of block_pairs ([num_pairs][2] int64, device), the
 * copy of copy-on-write ("vLLM Page Attention Continuous Batching" (lbrq.cn),
 * "Sharing KV Cache-COW"). A pair naming a block outside [0, num_blocks) is
 * skipped and sets PA_DEV_BAD_BLOCK_ID. Pairs must not write the same dst, or
 * read a block another pair writes, in one call (they run concurrently).
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_pairs,
                         int64_t num_pairs, int num_kv_heads, int head_size, int block_size,
                         int64_t num_blocks, pa_dtype cache_dtype, uint32_t* dev_status,
                         void* stream);

/*
 * pa_block_allocator -- host-side free list of physical block ids with
 * reference counts (TGI deep-dive sec. 4.3 SimpleAllocator: div_ceil(tokens,
 * block_size) blocks taken from the end of the free list, block 0 reserved;
 * "Continuous Batching and PagedAttention" sec. 3.2: fork shares blocks by
 * reference, free returns a block when its count reaches zero). Host memory
 * only; every call validates first and changes nothing when it fails; calls
 * are serialised by an internal mutex.
 *
 *  create      num_blocks ids, block 0 kept out of the free list if
 *              reserve_block0 (NULL on bad arguments or no memory).
 *  allocate    ceil(num_tokens / block_size) blocks into blocks[], reference
 *              count 1; PA_ERR_NO_BLOCKS (nothing taken) when short.
 *  fork        one more reference to each listed block (all must be held).
 *  free        one reference less for each listed entry; a block returns to
 *              the free list at zero. Listing a block more often than it is
 *              referenced is PA_ERR_INVALID_ARG.
 *  append_slot the slot of a sequence's token at `position` given its block
 *              table (table_len entries, room for capacity): a token starting
 *              a new block gets a fresh block appended; a token in a block
 *              referenced by others (count > 1) triggers copy-on-write: a fresh
 *              block replaces it in the table, the old one loses a reference,
 *              and (*copy_src, *copy_dst) name the copy the caller must make
 *              (pa_copy_blocks) before writing; otherwise both are -1.
 */
typedef struct pa_block_allocator pa_block_allocator;
pa_block_allocator* pa_allocator_create(int64_t num_blocks, int block_size, int reserve_block0);
void pa_allocator_destroy(pa_block_allocator* allocator);
int64_t pa_allocator_num_free(pa_block_allocator* allocator);
int32_t pa_allocator_refcount(pa_block_allocator* allocator, int32_t block);
pa_status pa_allocator_allocate(pa_block_allocator* allocator, int64_t num_tokens, int32_t* blocks,
                                int64_t capacity, int64_t* num_allocated);
pa_status pa_allocator_fork(pa_block_allocator* allocator, const int32_t* blocks, int64_t n);
pa_status pa_allocator_free(pa_block_allocator* allocator, const int32_t* blocks, int64_t n);
pa_status pa_allocator_append_slot(pa_block_allocator* allocator, int32_t* table,
                                   int64_t* table_len, int64_t capacity, int64_t position,
                                   int64_t* slot, int32_t* copy_src, int32_t* copy_dst);

/*
 * pa_radix_allocator -- prefix caching: a radix trie from token sequences to
 * the physical blocks holding their K/V, so that requests sharing a prompt
 * prefix share its blocks (TGI deep-dive sec. 5.2-5.3, RadixAllocator). Host
 * memory only; calls are serialised by an internal mutex; each validates
 * first and changes nothing when it fails.
 *
 *  create      num_blocks ids, block 0 kept out if reserve_block0 (NULL on
 *              bad arguments or no memory).
 *  allocate    blocks for a request whose prompt is tokens[0, num_tokens) and
 *              which may grow to total_tokens (>= num_tokens): the longest
 *              cached block-aligned prefix of the prompt (*prefix_len tokens,
 *              a multiple of block_size) is shared -- its blocks come first in
 *              blocks[] -- and ceil(total_tokens / block_size) blocks are
 *              returned in all (*num_allocated <= capacity). Missing blocks
 *              come from the free list, evicting cached sequences nobody uses,
 *              least recently used first. PA_ERR_NO_BLOCKS (nothing changed)
 *              when even eviction cannot supply them. *allocation_id names the
 *              request for pa_radix_free.
 *  free        ends a request. tokens[0, num_tokens) are the tokens its blocks
 *              now hold (prompt and generated tokens; they must start with the
 *              shared prefix): their whole blocks are inserted into the trie
 *              for later requests, a node that only partly matches is split,
 *              and blocks the trie does not take return to the free list.
 *  num_free    blocks on the free list; num_cached: blocks held by the trie;
 *              num_evictable: blocks of trie leaves no request uses.
 */
typedef struct pa_radix_allocator pa_radix_allocator;
pa_radix_allocator* pa_radix_create(int64_t num_blocks, int block_size, int reserve_block0);
void pa_radix_destroy(pa_radix_allocator* allocator);
pa_status pa_radix_allocate(pa_radix_allocator* allocator, const int32_t* tokens,
                            int64_t num_tokens, int64_t total_tokens, int32_t* blocks,
                            int64_t capacity, int64_t* num_allocated, int64_t* prefix_len,
                            int64_t* allocation_id);
pa_status pa_radix_free(pa_radix_allocator* allocator, int64_t allocation_id,
                        const int32_t* tokens, int64_t num_tokens);
int64_t pa_radix_num_free(pa_radix_allocator* allocator);
int64_t pa_radix_num_cached(pa_radix_allocator* allocator);
int64_t pa_radix_num_evictable(pa_radix_allocator* allocator);

/*
 * pa_decode_choose -- which decode to run: 0 = single pass (pa_decode),
 * 1 = partitioned (pa_decode_partitioned). The pages' rule (TGI deep-dive
 * sec. 4.1) picks V1 when there is one partition or when num_seqs x num_heads
 * is large; this library decides from the current device's SM count and the
 * number of work units each form would launch. Never fails; a non-positive
 * argument gives 0.
 */
int pa_decode_choose(int num_seqs, int num_q_heads, int num_kv_heads, int max_context_len,
                     int partition_size);

/*
 * pa_decode_partition_size -- a partition size for this device: 512 (the
 * pages' _PARTITION_SIZE) doubled (up to 4096) while the longest context
 * still spans three or more partitions and the launch keeps about two waves of
 * work units. Longer partitions mean fewer CTA start-ups and fewer partials to
 * merge. Never fails.
 */
int pa_decode_partition_size(int num_seqs, int num_kv_heads, int max_context_len);

/*
 * pa_selftest_wait -- a device check of the kernels' bounded waits (see
 * "Errors" above). Launches one CTA in which two threads wait on mbarriers
 * expecting one arrival each, one through the wait of the TMA pipelines and
 * one through the wait of the tensor-core pipelines. arrive = 1: the
 * arrivals are made first; both waits return at once and nothing is set.
 * arrive = 0: nothing arrives; each wait runs out after its limit (about a
 * second of SM clocks), sets PA_DEV_TIMEOUT in *dev_status and returns, and
 * the kernel ends, the context still usable. A wait that returned without an
 * arrival sets PA_DEV_BAD_LEN. dev_status (device, 4-byte aligned) is
 * required; arrive must be 0 or 1 (else PA_ERR_INVALID_ARG).
 */
pa_status pa_selftest_wait(int arrive, uint32_t* dev_status, void* stream);

/* Human-readable name of a status code (a static string). */
const char* pa_status_string(pa_status status);

/* Library ABI version: 100 * major + minor. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
