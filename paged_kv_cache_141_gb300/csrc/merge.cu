// merge.cu -- the reduction of the split decode ("TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 4.1: long sequences are cut into partitions that
// are computed in parallel and then merged). For each (sequence, query head):
//   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// One CTA per (head, sequence); 128 threads stride over the head components.
// Partition weights are staged through shared memory in chunks, so any number
// of partitions fits.
#include "device_common.cuh"
#include "launch.h"

namespace pagedkv {

constexpr int kMergeThreads = 128;
constexpr int kMergeChunk = 1024;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) r = fmaxf(r, red[w]);
    return r;
}

template <typename OT>
__global__ void __launch_bounds__(kMergeThreads)
paged_merge_kernel(OT* __restrict__ out, const float* __restrict__ tmp_out,
                   const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
                   const int32_t* __restrict__ context_lens, int num_q_heads, int D,
                   int partition_size, int max_parts, uint32_t* status) {
    __shared__ float w_s[kMergeChunk];
    __shared__ float red[kMergeThreads / 32];
    const int h = blockIdx.x;
    const int s = blockIdx.y;
    const size_t row = (size_t)s * num_q_heads + h;
    OT* o = out + row * D;

    int L = context_lens[s];
    const long long cap = (long long)max_parts * partition_size;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && h == 0 && status) atomicOr(status, PA_DEV_BAD_LEN);
        L = L < 0 ? 0 : (int)cap;
    }
    const int n = (L + partition_size - 1) / partition_size;
    const float* ml = max_logits + row * max_parts;
    const float* es = exp_sums + row * max_parts;
    const float* to = tmp_out + row * max_parts * D;

    if (n == 0) {
        for (int e = threadIdx.x; e < D; e += kMergeThreads) o[e] = from_float<OT>(0.f);
        return;
    }
    if (n == 1) {  // one partition: its normalised output is the answer
        for (int e = threadIdx.x; e < D; e += kMergeThreads) o[e] = from_float<OT>(to[e]);
        return;
    }

    float M = -INFINITY;
    for (int i = threadIdx.x; i < n; i += kMergeThreads) M = fmaxf(M, ml[i]);
    M = block_max(M, red);

    // each thread keeps up to two components (head_size <= 256)
    float acc0 = 0.f, acc1 = 0.f, wsum = 0.f;
    const int e0 = threadIdx.x, e1 = threadIdx.x + kMergeThreads;
    for (int c0 = 0; c0 < n; c0 += kMergeChunk) {
        const int cn = min(kMergeChunk, n - c0);
        __syncthreads();
        for (int i = threadIdx.x; i < cn; i += kMergeThreads)
            w_s[i] = es[c0 + i] * fast_exp2((ml[c0 + i] - M) * kLog2e);
        __syncthreads();
        for (int i = 0; i < cn; ++i) {
            const float w = w_s[i];
            wsum += w;
            const float* tp = to + (size_t)(c0 + i) * D;
            if (e0 < D) acc0 = fmaf(w, tp[e0], acc0);
            if (e1 < D) acc1 = fmaf(w, tp[e1], acc1);
        }
    }
    if (e0 < D) o[e0] = from_float<OT>(__fdiv_rn(acc0, wsum));
    if (e1 < D) o[e1] = from_float<OT>(__fdiv_rn(acc1, wsum));
}

cudaError_t launch_merge(void* out, const float* tmp_out, const float* max_logits,
                         const float* exp_sums, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int head_size, int partition_size, int max_parts,
                         pa_dtype out_dtype, uint32_t* status, cudaStream_t stream) {
    dim3 grid(num_q_heads, num_seqs);
    switch (out_dtype) {
    case PA_F32:
        paged_merge_kernel<float><<<grid, kMergeThreads, 0, stream>>>(
            static_cast<float*>(out), tmp_out, max_logits, exp_sums, context_lens, num_q_heads,
            head_size, partition_size, max_parts, status);
        break;
    case PA_F16:
        paged_merge_kernel<__half><<<grid, kMergeThreads, 0, stream>>>(
            static_cast<__half*>(out), tmp_out, max_logits, exp_sums, context_lens, num_q_heads,
            head_size, partition_size, max_parts, status);
        break;
    case PA_BF16:
        paged_merge_kernel<__nv_bfloat16><<<grid, kMergeThreads, 0, stream>>>(
            static_cast<__nv_bfloat16*>(out), tmp_out, max_logits, exp_sums, context_lens,
            num_q_heads, head_size, partition_size, max_parts, status);
        break;
    default:
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pagedkv
