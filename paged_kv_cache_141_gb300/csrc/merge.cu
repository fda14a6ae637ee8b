// merge.cu -- the reduction of the split decode ("TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 4.1: long sequences are cut into partitions that
// are computed in parallel and then merged). For each (sequence, query head):
//   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// One warp per (sequence, head), eight per CTA: the lanes take partitions for
// the maximum and the weights (warp shuffles, no block barriers), then every
// lane accumulates head_size/32 components of each partition's output, the
// weight broadcast by shuffle, reading each partition's row as coalesced
// vectors. One partition is copied; none gives zeros.
#include "device_common.cuh"
#include "launch.h"

namespace pagedkv {

constexpr int kMergeWarps = 8;

template <int D, typename OT>
__global__ void __launch_bounds__(kMergeWarps * 32)
paged_merge_kernel(OT* __restrict__ out, const float* __restrict__ tmp_out,
                   const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
                   const int32_t* __restrict__ context_lens, int num_seqs, int num_q_heads,
                   int partition_size, int max_parts, uint32_t* status) {
    constexpr int EPL = D / 32;                // components per lane
    const int lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (item >= (long long)num_seqs * num_q_heads) return;
    const int s = (int)(item / num_q_heads);
    const int h = (int)(item - (long long)s * num_q_heads);
    const size_t row = (size_t)s * num_q_heads + h;
    OT* o = out + row * D;

    int L = context_lens[s];
    const long long cap = (long long)max_parts * partition_size;
    if (L < 0 || L > cap) {
        if (lane == 0 && h == 0 && status) atomicOr(status, PA_DEV_BAD_LEN);
        L = L < 0 ? 0 : (int)cap;
    }
    const int n = (L + partition_size - 1) / partition_size;
    const float* ml = max_logits + row * max_parts;
    const float* es = exp_sums + row * max_parts;
    const float* to = tmp_out + row * max_parts * D;

    float acc[EPL];
    if (n <= 1) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = n == 1 ? to[lane * EPL + e] : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[lane * EPL + e] = from_float<OT>(acc[e]);
        return;
    }

    float M = -INFINITY;
    for (int i = lane; i < n; i += 32) M = fmaxf(M, ml[i]);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));

#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int i = c0 + lane;
        const float w = i < n ? es[i] * fast_exp2((ml[i] - M) * kLog2e) : 0.f;
        wsum += w;
        const int cn = min(32, n - c0);
#pragma unroll 4
        for (int j = 0; j < cn; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
            const float* tp = to + (size_t)(c0 + j) * D + lane * EPL;
            if constexpr (EPL == 2) {
                const float2 v = *reinterpret_cast<const float2*>(tp);
                acc[0] = fmaf(wj, v.x, acc[0]);
                acc[1] = fmaf(wj, v.y, acc[1]);
            } else {
#pragma unroll
                for (int e = 0; e < EPL; e += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(tp + e);
                    acc[e] = fmaf(wj, v.x, acc[e]);
                    acc[e + 1] = fmaf(wj, v.y, acc[e + 1]);
                    acc[e + 2] = fmaf(wj, v.z, acc[e + 2]);
                    acc[e + 3] = fmaf(wj, v.w, acc[e + 3]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, m);
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[lane * EPL + e] = from_float<OT>(__fdiv_rn(acc[e], wsum));
}

template <int D, typename OT>
static cudaError_t launch_merge_t(OT* out, const float* tmp_out, const float* max_logits,
                                  const float* exp_sums, const int32_t* context_lens, int num_seqs,
                                  int num_q_heads, int partition_size, int max_parts,
                                  uint32_t* status, cudaStream_t stream) {
    const long long items = (long long)num_seqs * num_q_heads;
    const unsigned grid = (unsigned)((items + kMergeWarps - 1) / kMergeWarps);
    paged_merge_kernel<D, OT><<<grid, kMergeWarps * 32, 0, stream>>>(
        out, tmp_out, max_logits, exp_sums, context_lens, num_seqs, num_q_heads, partition_size,
        max_parts, status);
    return cudaGetLastError();
}

template <typename OT>
static cudaError_t launch_merge_o(void* out, const float* tmp_out, const float* max_logits,
                                  const float* exp_sums, const int32_t* context_lens, int num_seqs,
                                  int num_q_heads, int head_size, int partition_size, int max_parts,
                                  uint32_t* status, cudaStream_t stream) {
    OT* o = static_cast<OT*>(out);
    switch (head_size) {
    case 64:
        return launch_merge_t<64>(o, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                  num_q_heads, partition_size, max_parts, status, stream);
    case 128:
        return launch_merge_t<128>(o, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                   num_q_heads, partition_size, max_parts, status, stream);
    case 256:
        return launch_merge_t<256>(o, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                   num_q_heads, partition_size, max_parts, status, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge(void* out, const float* tmp_out, const float* max_logits,
                         const float* exp_sums, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int head_size, int partition_size, int max_parts,
                         pa_dtype out_dtype, uint32_t* status, cudaStream_t stream) {
    switch (out_dtype) {
    case PA_F32:
        return launch_merge_o<float>(out, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                     num_q_heads, head_size, partition_size, max_parts, status,
                                     stream);
    case PA_F16:
        return launch_merge_o<__half>(out, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                      num_q_heads, head_size, partition_size, max_parts, status,
                                      stream);
    case PA_BF16:
        return launch_merge_o<__nv_bfloat16>(out, tmp_out, max_logits, exp_sums, context_lens,
                                             num_seqs, num_q_heads, head_size, partition_size,
                                             max_parts, status, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace pagedkv
