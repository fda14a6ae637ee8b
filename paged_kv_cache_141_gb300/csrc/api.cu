// api.cu -- the C ABI (include/pagedkv.h): argument validation on the host,
// then kernel launches on the caller's stream. Nothing here allocates memory
// or synchronises.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "launch.h"
#include "pagedkv.h"

using namespace pagedkv;

namespace {

bool is_compute_type(pa_dtype t) { return t == PA_F32 || t == PA_F16 || t == PA_BF16; }

bool supported_head_size(int d) { return d == 64 || d == 128 || d == 256; }

// (query type, cache type) pairs the decode implements.
bool supported_pair(pa_dtype q, pa_dtype c) {
    if (q == c) return is_compute_type(q);
    return c == PA_FP8_E4M3 && (q == PA_F16 || q == PA_BF16);
}

int elem_bytes(pa_dtype t) { return t == PA_F32 ? 4 : (t == PA_FP8_E4M3 ? 1 : 2); }

// The tensor-TMA kernel takes rows of 128, 256 or 512 bytes (whole 128-byte
// swizzle spans) and block sizes 8, 16 or a multiple of 32 (so every box lands
// on a 1 KB-aligned row group), with row coordinates below 2^31.
bool tma_eligible(int head_size, pa_dtype cache_dtype, int block_size, int64_t num_blocks,
                  int num_kv_heads) {
    const int row = head_size * elem_bytes(cache_dtype);
    if (row != 128 && row != 256 && row != 512) return false;
    if (!(block_size == 8 || block_size == 16 || (block_size >= 32 && block_size % 32 == 0)))
        return false;
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    return rows > 0 && rows < (1ll << 31);
}

// Query heads per work unit: the largest power of two dividing the group, up
// to a cap that bounds the per-lane accumulators.
int heads_per_unit(int group, int head_size, bool tma) {
    const int cap = tma ? (head_size <= 64 ? 16 : (head_size <= 128 ? 8 : 4))
                        : (head_size >= 256 ? 4 : 8);
    for (int g = cap; g > 1; g >>= 1)
        if (group % g == 0) return g;
    return 1;
}

// The tensor-core decode: a 16-bit query with a cache of the same type or of
// E4M3 codes, and an even group or none (multi-head attention, one head per
// unit in the MMA tile's 8 columns); other odd groups stay on the CUDA cores.
bool mma_eligible(pa_dtype q_dtype, pa_dtype cache_dtype, int group) {
    if ((group % 2 != 0 && group != 1) || !(q_dtype == PA_F16 || q_dtype == PA_BF16)) return false;
    return cache_dtype == q_dtype || cache_dtype == PA_FP8_E4M3;
}

int mma_heads_per_unit(int group) {
    return group % 8 == 0 ? 8 : (group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Data arrays move as 16-byte vectors and bulk copies: their addresses must
// be 16-byte aligned; index arrays need their element's alignment.
bool aligned(const void* p, uintptr_t bytes) {
    return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}
bool aligned16(const void* a, const void* b = nullptr, const void* c = nullptr,
               const void* d = nullptr) {
    return aligned(a, 16) && aligned(b, 16) && aligned(c, 16) && aligned(d, 16);
}

int max_partitions(int max_context_len, int partition_size) {
    const int n = (max_context_len + partition_size - 1) / partition_size;
    return n < 1 ? 1 : n;
}

struct Layout {
    size_t tmp_out, max_logits, exp_sums, total;
};

Layout workspace_layout(int num_seqs, int num_q_heads, int head_size, int max_context_len,
                        int partition_size) {
    const size_t parts = (size_t)num_seqs * num_q_heads * max_partitions(max_context_len, partition_size);
    Layout l;
    l.tmp_out = 0;
    l.max_logits = align256(parts * head_size * sizeof(float));
    l.exp_sums = l.max_logits + align256(parts * sizeof(float));
    l.total = l.exp_sums + align256(parts * sizeof(float));
    return l;
}

pa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// Shared validation of the decode arguments. Fills `p` on success.
pa_status check_decode(const void* query, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                       int max_context_len, float scale, pa_dtype q_dtype, pa_dtype cache_dtype,
                       float k_scale, float v_scale, uint32_t* dev_status, DecodeParams& p) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
        block_size <= 0 || num_blocks < 0 || max_blocks_per_seq < 0 || max_context_len < 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (cache_dtype == PA_FP8_E4M3 &&
        (!isfinite(k_scale) || !isfinite(v_scale) || k_scale <= 0.f || v_scale <= 0.f))
        return PA_ERR_INVALID_ARG;
    if ((int)q_dtype < 0 || (int)q_dtype > 3 || (int)cache_dtype < 0 || (int)cache_dtype > 3)
        return PA_ERR_INVALID_ARG;
    if (!supported_pair(q_dtype, cache_dtype) || !supported_head_size(head_size) ||
        block_size > 1024)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || (long long)num_kv_heads * (num_q_heads / num_kv_heads) > 65535)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs > 0 &&
        (!query || !k_cache || !v_cache || !block_tables || !context_lens || max_blocks_per_seq == 0))
        return PA_ERR_INVALID_ARG;
    if (!aligned16(query, k_cache, v_cache) || !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    p = DecodeParams{};
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.status = dev_status;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size = block_size;
    p.max_context_len = max_context_len;
    p.group = num_q_heads / num_kv_heads;
    const bool tma = tma_eligible(head_size, cache_dtype, block_size, num_blocks, num_kv_heads);
    const bool mma = tma && mma_eligible(q_dtype, cache_dtype, p.group);
    p.sub_groups = p.group / (mma ? mma_heads_per_unit(p.group)
                                  : heads_per_unit(p.group, head_size, tma));
    const bool fp8 = cache_dtype == PA_FP8_E4M3;
    p.q_mul = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);
    p.v_mul = fp8 ? v_scale : 1.f;
    return PA_OK;
}

cudaError_t run_decode_kernel(const DecodeParams& p, int head_size, pa_dtype q_dtype,
                              pa_dtype cache_dtype, bool split, cudaStream_t stream) {
    const int gs = p.group / p.sub_groups;
    if (tma_eligible(head_size, cache_dtype, p.block_size, p.num_blocks, p.num_kv_heads)) {
        if (mma_eligible(q_dtype, cache_dtype, p.group)) {
            if (cache_dtype == PA_FP8_E4M3) {
                if (q_dtype == PA_F16) return launch_decode_mma_f16_e4m3(p, head_size, gs, split, stream);
                return launch_decode_mma_bf16_e4m3(p, head_size, gs, split, stream);
            }
            if (q_dtype == PA_F16) return launch_decode_mma_f16(p, head_size, gs, split, stream);
            return launch_decode_mma_bf16(p, head_size, gs, split, stream);
        }
        if (cache_dtype == PA_FP8_E4M3) {
            if (q_dtype == PA_F16) return launch_decode_tma_f16_e4m3(p, head_size, gs, split, stream);
            return launch_decode_tma_bf16_e4m3(p, head_size, gs, split, stream);
        }
        switch (q_dtype) {
        case PA_F32: return launch_decode_tma_f32(p, head_size, gs, split, stream);
        case PA_F16: return launch_decode_tma_f16(p, head_size, gs, split, stream);
        default: return launch_decode_tma_bf16(p, head_size, gs, split, stream);
        }
    }
    if (cache_dtype == PA_FP8_E4M3) {
        if (q_dtype == PA_F16) return launch_decode_simt_f16_e4m3(p, head_size, gs, split, stream);
        return launch_decode_simt_bf16_e4m3(p, head_size, gs, split, stream);
    }
    switch (q_dtype) {
    case PA_F32: return launch_decode_simt_f32(p, head_size, gs, split, stream);
    case PA_F16: return launch_decode_simt_f16(p, head_size, gs, split, stream);
    default: return launch_decode_simt_bf16(p, head_size, gs, split, stream);
    }
}

// The CUDA-core decode alone (the multi-query fallback).
cudaError_t run_simt_decode_kernel(DecodeParams p, int head_size, pa_dtype q_dtype,
                                   pa_dtype cache_dtype, cudaStream_t stream) {
    p.sub_groups = p.group / heads_per_unit(p.group, head_size, false);
    const int gs = p.group / p.sub_groups;
    if (cache_dtype == PA_FP8_E4M3) {
        if (q_dtype == PA_F16) return launch_decode_simt_f16_e4m3(p, head_size, gs, false, stream);
        return launch_decode_simt_bf16_e4m3(p, head_size, gs, false, stream);
    }
    switch (q_dtype) {
    case PA_F32: return launch_decode_simt_f32(p, head_size, gs, false, stream);
    case PA_F16: return launch_decode_simt_f16(p, head_size, gs, false, stream);
    default: return launch_decode_simt_bf16(p, head_size, gs, false, stream);
    }
}

pa_status check_partition_size(int partition_size) {
    if (partition_size <= 0 || partition_size % 32 != 0) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa_status bind_workspace(DecodeParams& p, int num_seqs, int num_q_heads, int head_size,
                         int max_context_len, int partition_size, void* workspace,
                         size_t workspace_bytes) {
    const Layout l = workspace_layout(num_seqs, num_q_heads, head_size, max_context_len, partition_size);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < l.total)
        return PA_ERR_WORKSPACE;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    p.tmp_out = reinterpret_cast<float*>(w + l.tmp_out);
    p.max_logits = reinterpret_cast<float*>(w + l.max_logits);
    p.exp_sums = reinterpret_cast<float*>(w + l.exp_sums);
    p.partition_size = partition_size;
    p.max_parts = max_partitions(max_context_len, partition_size);
    return PA_OK;
}

void bind_fused_write(DecodeParams& p, const void* key, const void* value,
                      const int64_t* slot_mapping, void* k_cache, void* v_cache, float k_scale,
                      float v_scale) {
    p.new_key = key;
    p.new_value = value;
    p.new_slots = slot_mapping;
    p.wk_cache = k_cache;
    p.wv_cache = v_cache;
    p.k_scale_w = k_scale;
    p.v_scale_w = v_scale;
}

// The warp-level MMA multi-query kernel (a few query rows per sequence and KV
// head): 16-bit query and a cache of the same type or of E4M3 codes, on the
// shapes of the TMA decode.
// Rows per (sequence, KV head) it takes: 32 at head size <= 128 (two n-tiles
// per warp), 16 at head size 256.
long long prefill_mma_max_rows(int head_size) {
    return head_size <= 128 ? 32 : 16;
}

bool prefill_mma_eligible(pa_dtype q_dtype, pa_dtype cache_dtype, int head_size, int block_size,
                          int64_t num_blocks, int num_kv_heads) {
    if (!(q_dtype == PA_F16 || q_dtype == PA_BF16)) return false;
    if (!(cache_dtype == q_dtype || cache_dtype == PA_FP8_E4M3)) return false;
    return tma_eligible(head_size, cache_dtype, block_size, num_blocks, num_kv_heads);
}

// The tcgen05 multi-query kernel: 16-bit query and a cache of the same type
// or of E4M3 codes (head size 64 or 128), whole 128-byte column spans, block sizes that are powers of two in [8, 256] (every
// TMA box then starts on a swizzle-atom boundary), groups that fit the
// 128-row tile, 16-byte-aligned rows, row coordinates below 2^31.
bool prefill_tc_eligible(pa_dtype q_dtype, pa_dtype cache_dtype, int head_size, int block_size,
                         int group, int64_t num_blocks, int num_kv_heads) {
    if (!(q_dtype == PA_F16 || q_dtype == PA_BF16)) return false;
    if (cache_dtype == PA_FP8_E4M3) {
        if (head_size != 64 && head_size != 128) return false;      // E4M3 staging fits
    } else if (cache_dtype != q_dtype || !supported_head_size(head_size)) {
        return false;
    }
    if (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)) != 0) return false;
    if (group < 1 || group > 128) return false;
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    return rows > 0 && rows < (1ll << 31);
}

// The kernel pa_paged_prefill runs: the warp-level MMA kernels for up to 32
// rows per (sequence, KV head) (16 at head size 256, and 16 where the tcgen05
// kernels take the E4M3 products: E4M3 cache, bf16 query, head size 128),
// else the tcgen05 ones (two query tiles per CTA at head size <= 128 with at
// least two tiles per sequence), else one query token per work unit on the
// CUDA cores. `aligned`: out, query and the caches are 16-byte aligned (the
// tcgen05 rows). With the E4M3 products the one-tile tcgen05 kernel beats the
// two-n-tile warp-level one from 17 rows on (shared-prefix E4M3 pool at
// G = 8: 24 rows 2.75 against 2.47 TB/s of logical bytes, 32 rows 2.78
// against 2.43; at 16 rows the warp-level kernel, 3.26 against 2.75).
pa_prefill_kernel prefill_kernel(pa_dtype q_dtype, pa_dtype cache_dtype, int head_size,
                                 int block_size, int group, int64_t num_blocks, int num_kv_heads,
                                 int max_queries, bool aligned) {
    const long long rows = (long long)max_queries * group;
    const bool tc = aligned && prefill_tc_eligible(q_dtype, cache_dtype, head_size, block_size,
                                                   group, num_blocks, num_kv_heads);
    const bool e4m3_products = tc && cache_dtype == PA_FP8_E4M3 && q_dtype == PA_BF16 &&
                               head_size == 128;
    const long long mma_rows = e4m3_products ? 16 : prefill_mma_max_rows(head_size);
    if (rows <= mma_rows &&
        prefill_mma_eligible(q_dtype, cache_dtype, head_size, block_size, num_blocks, num_kv_heads))
        return rows <= 16 ? PA_PREFILL_MMA : PA_PREFILL_MMA_TWO_TILES;
    if (tc) {
        const int per_tile = 128 / group;
        const int tiles = (max_queries + per_tile - 1) / per_tile;
        const bool two = head_size <= 128 && tiles >= 2;
        return two ? PA_PREFILL_TC_TWO_TILES : PA_PREFILL_TC;
    }
    return PA_PREFILL_CUDA_CORES;
}

// pa_merge's validation and launch; len_cap is the context-length clamp of
// the partition kernel whose partials are merged.
pa_status merge_checked(void* out, const float* tmp_out, const float* max_logits,
                        const float* exp_sums, const int32_t* context_lens, int num_seqs,
                        int num_q_heads, int head_size, int partition_size, int max_partitions,
                        long long len_cap, pa_dtype out_dtype, uint32_t* dev_status,
                        void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || max_partitions <= 0)
        return PA_ERR_INVALID_ARG;
    pa_status st = check_partition_size(partition_size);
    if (st != PA_OK) return st;
    if ((int)out_dtype < 0 || (int)out_dtype > 3) return PA_ERR_INVALID_ARG;
    if (!is_compute_type(out_dtype) || !supported_head_size(head_size)) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_q_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !tmp_out || !max_logits || !exp_sums || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out, tmp_out) || !aligned(max_logits, 4) || !aligned(exp_sums, 4) ||
        !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    const long long parts_cap = (long long)max_partitions * partition_size;
    return from_cuda(launch_merge(out, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                  num_q_heads, head_size, partition_size, max_partitions,
                                  len_cap < parts_cap ? len_cap : parts_cap, out_dtype, dev_status,
                                  static_cast<cudaStream_t>(stream)));
}

// The context-length clamp of the decode kernels: min(max_context_len,
// max_blocks_per_seq * block_size).
long long decode_len_cap(int max_context_len, int max_blocks_per_seq, int block_size) {
    const long long tab = (long long)max_blocks_per_seq * block_size;
    return tab < max_context_len ? tab : (long long)max_context_len;
}

}  // namespace

extern "C" {

pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                               int head_size, int block_size, int64_t num_blocks,
                               pa_dtype in_dtype, pa_dtype cache_dtype, float k_scale,
                               float v_scale, uint32_t* dev_status, void* stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if ((int)in_dtype < 0 || (int)in_dtype > 3 || (int)cache_dtype < 0 || (int)cache_dtype > 3)
        return PA_ERR_INVALID_ARG;
    if (!is_compute_type(in_dtype)) return PA_ERR_UNSUPPORTED;
    if (cache_dtype != in_dtype && cache_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
    if (cache_dtype == PA_FP8_E4M3 &&
        (!isfinite(k_scale) || !isfinite(v_scale) || k_scale <= 0.f || v_scale <= 0.f))
        return PA_ERR_INVALID_ARG;
    // rows move as 16-byte vectors
    const int in_bytes = in_dtype == PA_F32 ? 4 : 2;
    if ((head_size * in_bytes) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key, value, k_cache, v_cache) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    return from_cuda(launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                              num_kv_heads, head_size, block_size, num_blocks,
                                              in_dtype, cache_dtype, k_scale, v_scale, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode(void* out, const void* query, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                    int head_size, int block_size, int64_t num_blocks, int max_context_len,
                    float scale, pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                    float v_scale, uint32_t* dev_status, void* stream) {
    DecodeParams p;
    pa_status st = check_decode(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                block_size, num_blocks, max_context_len, scale, q_dtype,
                                cache_dtype, k_scale, v_scale, dev_status, p);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !aligned16(out)) return PA_ERR_INVALID_ARG;
    p.out = out;
    return from_cuda(run_decode_kernel(p, head_size, q_dtype, cache_dtype, false,
                                       static_cast<cudaStream_t>(stream)));
}

pa_status pa_write_decode(void* out, const void* query, const void* key, const void* value,
                          const int64_t* slot_mapping, void* k_cache, void* v_cache,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int num_q_heads,
                          int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
                          int max_context_len, float scale, pa_dtype q_dtype,
                          pa_dtype cache_dtype, float k_scale, float v_scale,
                          uint32_t* dev_status, void* stream) {
    DecodeParams p;
    pa_status st = check_decode(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                block_size, num_blocks, max_context_len, scale, q_dtype,
                                cache_dtype, k_scale, v_scale, dev_status, p);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(out, key, value) || !aligned(slot_mapping, 8)) return PA_ERR_INVALID_ARG;
    bind_fused_write(p, key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale);
    p.out = out;
    return from_cuda(run_decode_kernel(p, head_size, q_dtype, cache_dtype, false,
                                       static_cast<cudaStream_t>(stream)));
}

pa_status pa_write_decode_partitions(const void* query, const void* key, const void* value,
                                     const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_size, int block_size,
                                     int64_t num_blocks, int max_context_len, float scale,
                                     pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                                     float v_scale, int partition_size, void* workspace,
                                     size_t workspace_bytes, uint32_t* dev_status, void* stream) {
    DecodeParams p;
    pa_status st = check_decode(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                block_size, num_blocks, max_context_len, scale, q_dtype,
                                cache_dtype, k_scale, v_scale, dev_status, p);
    if (st != PA_OK) return st;
    if ((st = check_partition_size(partition_size)) != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key, value) || !aligned(slot_mapping, 8)) return PA_ERR_INVALID_ARG;
    if ((st = bind_workspace(p, num_seqs, num_q_heads, head_size, max_context_len, partition_size,
                             workspace, workspace_bytes)) != PA_OK)
        return st;
    bind_fused_write(p, key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale);
    return from_cuda(run_decode_kernel(p, head_size, q_dtype, cache_dtype, true,
                                       static_cast<cudaStream_t>(stream)));
}

pa_status pa_write_decode_partitioned(void* out, const void* query, const void* key,
                                      const void* value, const int64_t* slot_mapping,
                                      void* k_cache, void* v_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_size, int block_size, int64_t num_blocks,
                                      int max_context_len, float scale, pa_dtype q_dtype,
                                      pa_dtype cache_dtype, float k_scale, float v_scale,
                                      int partition_size, void* workspace, size_t workspace_bytes,
                                      uint32_t* dev_status, void* stream) {
    if (num_seqs > 0 && !out) return PA_ERR_INVALID_ARG;
    pa_status st = pa_write_decode_partitions(query, key, value, slot_mapping, k_cache, v_cache,
                                              block_tables, max_blocks_per_seq, context_lens,
                                              num_seqs, num_q_heads, num_kv_heads, head_size,
                                              block_size, num_blocks, max_context_len, scale,
                                              q_dtype, cache_dtype, k_scale, v_scale,
                                              partition_size, workspace, workspace_bytes,
                                              dev_status, stream);
    if (st != PA_OK || num_seqs == 0) return st;
    const Layout l = workspace_layout(num_seqs, num_q_heads, head_size, max_context_len, partition_size);
    const uint8_t* w = static_cast<const uint8_t*>(workspace);
    return merge_checked(out, reinterpret_cast<const float*>(w + l.tmp_out),
                         reinterpret_cast<const float*>(w + l.max_logits),
                         reinterpret_cast<const float*>(w + l.exp_sums), context_lens, num_seqs,
                         num_q_heads, head_size, partition_size,
                         max_partitions(max_context_len, partition_size),
                         decode_len_cap(max_context_len, max_blocks_per_seq, block_size), q_dtype,
                         dev_status, stream);
}

pa_status pa_write_decode_shared_prefix(
    void* out, const void* query, const void* key, const void* value, const int64_t* slot_mapping,
    void* k_cache, void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, int max_context_len, float scale, pa_dtype q_dtype,
    pa_dtype cache_dtype, float k_scale, float v_scale, const int32_t* seq_shared_parts,
    const int32_t* unit_seqs, const int32_t* unit_parts, int num_units, int max_unit_parts,
    int partition_size, void* workspace, size_t workspace_bytes, uint32_t* dev_status,
    void* stream) {
    DecodeParams p;
    pa_status st = check_decode(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                block_size, num_blocks, max_context_len, scale, q_dtype,
                                cache_dtype, k_scale, v_scale, dev_status, p);
    if (st != PA_OK) return st;
    if ((st = check_partition_size(partition_size)) != PA_OK) return st;
    if (num_units < 0 || max_unit_parts < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !aligned16(out)) return PA_ERR_INVALID_ARG;
    const bool write = key || value || slot_mapping;
    if (write && (!key || !value || !slot_mapping || !aligned16(key, value) || !aligned(slot_mapping, 8)))
        return PA_ERR_INVALID_ARG;
    const bool shared = num_units > 0 && max_unit_parts > 0;
    if (shared) {
        if (!seq_shared_parts || !unit_seqs || !unit_parts || !aligned(seq_shared_parts, 4) ||
            !aligned(unit_seqs, 4) || !aligned(unit_parts, 4))
            return PA_ERR_INVALID_ARG;
        if (max_unit_parts > max_partitions(max_context_len, partition_size)) return PA_ERR_INVALID_ARG;
        // the tensor-core decode's shapes; whole blocks per partition, so that
        // a sequence's newest token never lies in a shared block
        if (!tma_eligible(head_size, cache_dtype, block_size, num_blocks, num_kv_heads) ||
            !mma_eligible(q_dtype, cache_dtype, p.group) || partition_size % block_size != 0 ||
            num_seqs + num_units > 65535)
            return PA_ERR_UNSUPPORTED;
    }
    if ((st = bind_workspace(p, num_seqs, num_q_heads, head_size, max_context_len, partition_size,
                             workspace, workspace_bytes)) != PA_OK)
        return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (shared) {
        p.skip_parts = seq_shared_parts;
        p.unit_seqs = unit_seqs;
        p.unit_parts = unit_parts;
        p.num_units = num_units;
    }
    if (write) bind_fused_write(p, key, value, slot_mapping, k_cache, v_cache, k_scale, v_scale);
    cudaError_t e = run_decode_kernel(p, head_size, q_dtype, cache_dtype, true, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    return merge_checked(out, p.tmp_out, p.max_logits, p.exp_sums, context_lens, num_seqs,
                         num_q_heads, head_size, partition_size, p.max_parts,
                         decode_len_cap(max_context_len, max_blocks_per_seq, block_size), q_dtype,
                         dev_status, stream);
}

size_t pa_decode_partitioned_workspace_bytes(int num_seqs, int num_q_heads, int head_size,
                                             int max_context_len, int partition_size) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || max_context_len < 0 ||
        partition_size <= 0)
        return 0;
    return workspace_layout(num_seqs, num_q_heads, head_size, max_context_len, partition_size).total;
}

pa_status pa_decode_workspace_layout(int num_seqs, int num_q_heads, int head_size,
                                     int max_context_len, int partition_size,
                                     size_t* tmp_out_offset, size_t* max_logits_offset,
                                     size_t* exp_sums_offset, size_t* total_bytes) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || max_context_len < 0 ||
        partition_size <= 0)
        return PA_ERR_INVALID_ARG;
    const Layout l = workspace_layout(num_seqs, num_q_heads, head_size, max_context_len, partition_size);
    if (tmp_out_offset) *tmp_out_offset = l.tmp_out;
    if (max_logits_offset) *max_logits_offset = l.max_logits;
    if (exp_sums_offset) *exp_sums_offset = l.exp_sums;
    if (total_bytes) *total_bytes = l.total;
    return PA_OK;
}

pa_status pa_decode_partitions(const void* query, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_size, int block_size,
                               int64_t num_blocks, int max_context_len, float scale,
                               pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                               float v_scale, int partition_size, void* workspace,
                               size_t workspace_bytes, uint32_t* dev_status, void* stream) {
    DecodeParams p;
    pa_status st = check_decode(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                block_size, num_blocks, max_context_len, scale, q_dtype,
                                cache_dtype, k_scale, v_scale, dev_status, p);
    if (st != PA_OK) return st;
    if ((st = check_partition_size(partition_size)) != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if ((st = bind_workspace(p, num_seqs, num_q_heads, head_size, max_context_len, partition_size,
                             workspace, workspace_bytes)) != PA_OK)
        return st;
    return from_cuda(run_decode_kernel(p, head_size, q_dtype, cache_dtype, true,
                                       static_cast<cudaStream_t>(stream)));
}

pa_status pa_merge(void* out, const float* tmp_out, const float* max_logits, const float* exp_sums,
                   const int32_t* context_lens, int num_seqs, int num_q_heads, int head_size,
                   int partition_size, int max_partitions, pa_dtype out_dtype,
                   uint32_t* dev_status, void* stream) {
    return merge_checked(out, tmp_out, max_logits, exp_sums, context_lens, num_seqs, num_q_heads,
                         head_size, partition_size, max_partitions,
                         (long long)max_partitions * partition_size, out_dtype, dev_status,
                         stream);
}

pa_status pa_decode_partitioned(void* out, const void* query, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_size, int block_size,
                                int64_t num_blocks, int max_context_len, float scale,
                                pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
                                float v_scale, int partition_size, void* workspace,
                                size_t workspace_bytes, uint32_t* dev_status, void* stream) {
    if (num_seqs > 0 && !out) return PA_ERR_INVALID_ARG;
    pa_status st = pa_decode_partitions(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                        context_lens, num_seqs, num_q_heads, num_kv_heads,
                                        head_size, block_size, num_blocks, max_context_len, scale,
                                        q_dtype, cache_dtype, k_scale, v_scale, partition_size,
                                        workspace, workspace_bytes, dev_status, stream);
    if (st != PA_OK || num_seqs == 0) return st;
    const Layout l = workspace_layout(num_seqs, num_q_heads, head_size, max_context_len, partition_size);
    const uint8_t* w = static_cast<const uint8_t*>(workspace);
    return merge_checked(out, reinterpret_cast<const float*>(w + l.tmp_out),
                         reinterpret_cast<const float*>(w + l.max_logits),
                         reinterpret_cast<const float*>(w + l.exp_sums), context_lens, num_seqs,
                         num_q_heads, head_size, partition_size,
                         max_partitions(max_context_len, partition_size),
                         decode_len_cap(max_context_len, max_blocks_per_seq, block_size), q_dtype,
                         dev_status, stream);
}

int pa_decode_partition_size(int num_seqs, int num_kv_heads, int max_context_len) {
    if (num_seqs <= 0 || num_kv_heads <= 0 || max_context_len <= 0) return 512;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        sms = 148;
    }
    // Longer partitions mean fewer CTA start-ups and fewer partials, while the
    // longest context still spans three or more of them (balance) and the launch
    // keeps about two waves of work units (3 CTAs per SM), estimating a
    // context's length at half the maximum. Measured on 8 contexts of 32k-131k
    // tokens (32/8 heads): steps of 0.399, 0.392 and 0.477 ms at 2048, 4096 and
    // 8192 tokens (the last 1.4 waves); shorter pools stop at the three-partition rule.
    const long long want = 2ll * 3 * sms;
    int P = 512;
    while (P < 4096) {
        const int next = 2 * P;
        const long long units = (long long)num_seqs * num_kv_heads *
                                ((max_context_len / 2 + next - 1) / next);
        if (max_context_len < 3 * next || units < want) break;
        P = next;
    }
    return P;
}

int pa_decode_choose(int num_seqs, int num_q_heads, int num_kv_heads, int max_context_len,
                     int partition_size) {
    if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len <= 0 ||
        partition_size <= 0)
        return 0;
    const int parts = max_partitions(max_context_len, partition_size);
    if (parts <= 1) return 0;                    // one partition: the merge would only copy
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        sms = 148;
    }
    // Single pass launches one unit per (sequence, KV head); with ragged
    // lengths the longest unit sets the finish time, so it only pays when
    // the units fill many waves and no context spans many partitions.
    const long long units = (long long)num_seqs * num_kv_heads;
    const long long slots = (long long)sms * 3;
    if (units >= 8 * slots && parts <= 2) return 0;
    return 1;
}

pa_status pa_paged_prefill(void* out, const void* query, const int32_t* query_start,
                           int num_queries, int max_queries_per_seq, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_size, int block_size,
                           int64_t num_blocks, int max_context_len, float scale,
                           pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale, float v_scale,
                           const int32_t* seq_order, uint32_t* dev_status, void* stream) {
    if (num_queries < 0 || max_queries_per_seq < 0 || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
    if (!aligned(seq_order, 4)) return PA_ERR_INVALID_ARG;
    // with no query tokens the data pointers may be null: validate the shape only
    const int seqs_with_work = num_queries == 0 ? 0 : num_seqs;
    DecodeParams p;
    pa_status st = check_decode(query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, seqs_with_work, num_q_heads, num_kv_heads,
                                head_size, block_size, num_blocks, max_context_len, scale,
                                q_dtype, cache_dtype, k_scale, v_scale, dev_status, p);
    if (st != PA_OK) return st;
    if (num_queries == 0) return PA_OK;
    if (num_seqs == 0) return PA_ERR_INVALID_ARG;        // query tokens need a sequence
    if (!out || !query_start || max_queries_per_seq == 0) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned(query_start, 4)) return PA_ERR_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    p.out = out;
    p.query_start = query_start;
    p.num_queries = num_queries;
    p.max_queries = max_queries_per_seq;
    p.seq_order = seq_order;
    const pa_prefill_kernel kind =
        prefill_kernel(q_dtype, cache_dtype, head_size, block_size, p.group, num_blocks,
                       num_kv_heads, max_queries_per_seq, aligned16(out, query, k_cache, v_cache));
    if (kind == PA_PREFILL_MMA || kind == PA_PREFILL_MMA_TWO_TILES) {
        // one pass over each sequence's K/V for all of its query rows
        if (cache_dtype == PA_FP8_E4M3)
            return from_cuda(q_dtype == PA_F16 ? launch_prefill_mma_f16_e4m3(p, head_size, s)
                                               : launch_prefill_mma_bf16_e4m3(p, head_size, s));
        return from_cuda(q_dtype == PA_F16 ? launch_prefill_mma_f16(p, head_size, s)
                                           : launch_prefill_mma_bf16(p, head_size, s));
    }
    if (kind == PA_PREFILL_TC || kind == PA_PREFILL_TC_TWO_TILES) {
        PrefillParams pp{};
        pp.out = out;
        pp.query = query;
        pp.query_start = query_start;
        pp.k_cache = k_cache;
        pp.v_cache = v_cache;
        pp.block_tables = block_tables;
        pp.context_lens = context_lens;
        pp.status = dev_status;
        pp.num_blocks = num_blocks;
        pp.max_blocks = max_blocks_per_seq;
        pp.num_seqs = num_seqs;
        pp.num_q_heads = num_q_heads;
        pp.num_kv_heads = num_kv_heads;
        pp.block_size = block_size;
        pp.group = p.group;
        pp.max_context_len = max_context_len;
        pp.max_queries = max_queries_per_seq;
        pp.tokens_per_tile = 128 / p.group;
        pp.q_tiles = (max_queries_per_seq + pp.tokens_per_tile - 1) / pp.tokens_per_tile;
        const bool fp8 = cache_dtype == PA_FP8_E4M3;
        pp.q_mul = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);
        pp.v_mul = fp8 ? v_scale : 1.f;
        pp.seq_order = seq_order;
        if (fp8)
            return from_cuda(q_dtype == PA_F16 ? launch_prefill_tc_f16_e4m3(pp, head_size, s)
                                               : launch_prefill_tc_bf16_e4m3(pp, head_size, s));
        return from_cuda(q_dtype == PA_F16 ? launch_prefill_tc_f16(pp, head_size, s)
                                           : launch_prefill_tc_bf16(pp, head_size, s));
    }
    // CUDA cores: one query token per work unit, the decode kernel over the
    // token's causal prefix (the work is per token: no sequence order)
    p.seq_order = nullptr;
    return from_cuda(run_simt_decode_kernel(p, head_size, q_dtype, cache_dtype, s));
}

int pa_paged_prefill_kernel(int max_queries_per_seq, int num_q_heads, int num_kv_heads,
                            int head_size, int block_size, int64_t num_blocks, pa_dtype q_dtype,
                            pa_dtype cache_dtype) {
    if (max_queries_per_seq < 1 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
        num_blocks < 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    if ((int)q_dtype < 0 || (int)q_dtype > 3 || (int)cache_dtype < 0 || (int)cache_dtype > 3)
        return -1;
    if (!supported_pair(q_dtype, cache_dtype) || !supported_head_size(head_size) ||
        block_size > 1024)
        return -1;
    return prefill_kernel(q_dtype, cache_dtype, head_size, block_size, num_q_heads / num_kv_heads,
                          num_blocks, num_kv_heads, max_queries_per_seq, true);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_pairs,
                         int64_t num_pairs, int num_kv_heads, int head_size, int block_size,
                         int64_t num_blocks, pa_dtype cache_dtype, uint32_t* dev_status,
                         void* stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if ((int)cache_dtype < 0 || (int)cache_dtype > 3) return PA_ERR_INVALID_ARG;
    const int64_t block_bytes = (int64_t)num_kv_heads * block_size * head_size * elem_bytes(cache_dtype);
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !block_pairs) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache, v_cache) || !aligned(block_pairs, 8)) return PA_ERR_INVALID_ARG;
    return from_cuda(launch_copy_blocks(k_cache, v_cache, block_pairs, num_pairs, num_blocks,
                                        block_bytes, dev_status, static_cast<cudaStream_t>(stream)));
}

pa_status pa_selftest_wait(int arrive, uint32_t* dev_status, void* stream) {
    if (!dev_status || (arrive != 0 && arrive != 1)) return PA_ERR_INVALID_ARG;
    if (!aligned(dev_status, 4)) return PA_ERR_INVALID_ARG;
    return from_cuda(launch_wait_selftest(arrive, dev_status, static_cast<cudaStream_t>(stream)));
}

const char* pa_status_string(pa_status status) {
    switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_NO_BLOCKS: return "not enough free blocks";
    }
    return "unknown status";
}

int pa_version(void) { return 100; }

}  // extern "C"
