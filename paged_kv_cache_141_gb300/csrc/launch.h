// launch.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units. Arguments have been validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pagedkv {

struct DecodeParams {
    void* out;                    // single pass: [S, Hq, D] of the query type
    const void* query;            // [S, Hq, D]
    const void* k_cache;          // [num_blocks, Hkv, B, D]
    const void* v_cache;
    const int32_t* block_tables;  // [S, max_blocks]
    const int32_t* context_lens;  // [S]
    float* tmp_out;               // split: [S, Hq, max_parts, D]
    float* max_logits;            // split: [S, Hq, max_parts]
    float* exp_sums;              // split: [S, Hq, max_parts]
    uint32_t* status;             // may be null
    int64_t num_blocks;
    int max_blocks;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int max_context_len;
    int partition_size;           // split only
    int max_parts;                // split only
    int group;                    // Hq / Hkv
    int sub_groups;               // group / heads per work unit
    float q_mul;                  // scale * log2(e) * (E4M3 cache ? k_scale : 1)
    float v_mul;                  // E4M3 cache ? v_scale : 1
    // fused KV write (all null for a plain decode): each sequence's newest
    // key/value [S, Hkv, D] of the query type, stored at new_slots[s]
    const void* new_key;
    const void* new_value;
    const int64_t* new_slots;
    void* wk_cache;               // the caches, writable (same addresses as k_cache / v_cache)
    void* wv_cache;
    float k_scale_w;              // E4M3 quantisation scales of the write
    float v_scale_w;
    // multi-query attention on the CUDA cores (null for the decode): the
    // rows of query/out are query tokens; token t of sequence s (query_start[s]
    // <= t < query_start[s+1]) attends to the first L_s - Q_s + (t -
    // query_start[s]) + 1 keys. Single pass only, no fused write.
    const int32_t* query_start;   // [S + 1]
    int num_queries;              // rows of query / out
    int max_queries;              // max over s of Q_s (sizes the tensor-core multi-query grid)
    const int32_t* seq_order;     // null or [S]: launch position -> sequence (longest first)
    // shared-prefix partitions (tensor-core decode, split only; all null / 0
    // otherwise): skip_parts[s] leading partitions of sequence s are computed
    // by the CTAs of the unit holding s (grid z < num_units, in the same
    // launch), whose members are unit_seqs[u * 4 .. u * 4 + 3] (-1 = none)
    // sharing unit_parts[u] partitions
    const int32_t* skip_parts;    // [S]
    const int32_t* unit_seqs;     // [num_units, 4]
    const int32_t* unit_parts;    // [num_units]
    int num_units;
};

// Generic CUDA-core decode; one launcher per (query type, cache type).
// head_size in {64, 128, 256}; heads_per_unit in {1, 2, 4, 8}.
cudaError_t launch_decode_simt_f32(const DecodeParams& p, int head_size, int heads_per_unit,
                                   bool split, cudaStream_t stream);
cudaError_t launch_decode_simt_f16(const DecodeParams& p, int head_size, int heads_per_unit,
                                   bool split, cudaStream_t stream);
cudaError_t launch_decode_simt_bf16(const DecodeParams& p, int head_size, int heads_per_unit,
                                    bool split, cudaStream_t stream);
cudaError_t launch_decode_simt_f16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                        bool split, cudaStream_t stream);
cudaError_t launch_decode_simt_bf16_e4m3(const DecodeParams& p, int head_size,
                                         int heads_per_unit, bool split, cudaStream_t stream);

// Tensor-TMA decode (rows of 128/256/512 bytes, block size 8, 16 or a
// multiple of 32); heads_per_unit <= 32 / (head_size / 32).
cudaError_t launch_decode_tma_f32(const DecodeParams& p, int head_size, int heads_per_unit,
                                  bool split, cudaStream_t stream);
cudaError_t launch_decode_tma_f16(const DecodeParams& p, int head_size, int heads_per_unit,
                                  bool split, cudaStream_t stream);
cudaError_t launch_decode_tma_bf16(const DecodeParams& p, int head_size, int heads_per_unit,
                                   bool split, cudaStream_t stream);
cudaError_t launch_decode_tma_f16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                       bool split, cudaStream_t stream);
cudaError_t launch_decode_tma_bf16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                        bool split, cudaStream_t stream);

// Tensor-core decode for 16-bit caches (query type = cache type), TMA-eligible
// shapes, heads_per_unit in {1, 2, 4, 8}.
cudaError_t launch_decode_mma_f16(const DecodeParams& p, int head_size, int heads_per_unit,
                                  bool split, cudaStream_t stream);
cudaError_t launch_decode_mma_bf16(const DecodeParams& p, int head_size, int heads_per_unit,
                                   bool split, cudaStream_t stream);
// E4M3 caches (rows of 128 or 256 bytes) with a 16-bit query, MMAs in f16.
cudaError_t launch_decode_mma_f16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                       bool split, cudaStream_t stream);
cudaError_t launch_decode_mma_bf16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                        bool split, cudaStream_t stream);
// Multi-query paged attention for a few query rows per (sequence, KV head)
// (max_queries * group <= 32 at head_size <= 128, <= 16 at 256) on
// warp-level MMA: 16-bit query with a cache of
// the same type (head_size 64/128/256) or E4M3 (128/256), TMA-eligible shapes.
// Uses the multi-query fields of DecodeParams; single pass.
cudaError_t launch_prefill_mma_f16(const DecodeParams& p, int head_size, cudaStream_t stream);
cudaError_t launch_prefill_mma_bf16(const DecodeParams& p, int head_size, cudaStream_t stream);
cudaError_t launch_prefill_mma_f16_e4m3(const DecodeParams& p, int head_size, cudaStream_t stream);
cudaError_t launch_prefill_mma_bf16_e4m3(const DecodeParams& p, int head_size, cudaStream_t stream);

// Multi-query paged attention on the tensor cores (tcgen05): 16-bit query and
// cache of the same type (head_size in {64, 128, 256}) or E4M3 (64, 128),
// block size a power of two in [8, 256], group <= 128.
struct PrefillParams {
    void* out;                    // [T, Hq, D], query type
    const void* query;            // [T, Hq, D]
    const int32_t* query_start;   // [S + 1]
    const void* k_cache;          // [num_blocks, Hkv, B, D]
    const void* v_cache;
    const int32_t* block_tables;  // [S, max_blocks]
    const int32_t* context_lens;  // [S]
    uint32_t* status;             // may be null
    int64_t num_blocks;
    int max_blocks;
    int num_seqs;
    int num_q_heads;
    int num_kv_heads;
    int block_size;
    int group;                    // Hq / Hkv
    int max_context_len;
    int max_queries;              // max over s of Q_s (sizes the grid)
    int tokens_per_tile;          // floor(128 / G)
    int q_tiles;                  // ceil(max_queries / tokens_per_tile)
    float q_mul;                  // scale * log2(e) * (E4M3 cache ? k_scale : 1)
    float v_mul;                  // E4M3 cache ? v_scale : 1
    const int32_t* seq_order;     // null or [S]: launch position -> sequence (longest first)
};

cudaError_t launch_prefill_tc_f16(const PrefillParams& p, int head_size, cudaStream_t stream);
cudaError_t launch_prefill_tc_bf16(const PrefillParams& p, int head_size, cudaStream_t stream);
// E4M3 caches with a 16-bit query, head_size 64 or 128 (MMAs in binary16).
cudaError_t launch_prefill_tc_f16_e4m3(const PrefillParams& p, int head_size, cudaStream_t stream);
cudaError_t launch_prefill_tc_bf16_e4m3(const PrefillParams& p, int head_size, cudaStream_t stream);

// len_cap: context lengths above it are clamped to it (and flagged
// PA_DEV_BAD_LEN), the clamp the partition kernel applied, so that only
// partitions it wrote are merged.
cudaError_t launch_merge(void* out, const float* tmp_out, const float* max_logits,
                         const float* exp_sums, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int head_size, int partition_size, int max_parts,
                         long long len_cap, pa_dtype out_dtype, uint32_t* status,
                         cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs,
                               int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                               uint32_t* status, cudaStream_t stream);

cudaError_t launch_wait_selftest(int arrive, uint32_t* status, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                     void* v_cache, const int64_t* slots, int64_t num_tokens,
                                     int num_kv_heads, int head_size, int block_size,
                                     int64_t num_blocks, pa_dtype in_dtype, pa_dtype cache_dtype,
                                     float k_scale, float v_scale, uint32_t* status,
                                     cudaStream_t stream);

}  // namespace pagedkv
