// merge.cu -- the reduction of the split decode ("TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 4.1: long sequences are cut into partitions that
// are computed in parallel and then merged). For each (sequence, query head):
//   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// One warp per (sequence, head), eight per CTA (merge_common.cuh). One
// partition is copied; none gives zeros.
#include "device_common.cuh"
#include "launch.h"
#include "merge_common.cuh"

namespace pagedkv {

constexpr int kMergeWarps = 8;

// Four CTAs (32 warps) per SM at least: the merge is a latency-bound pass
// over L2-resident partials, so occupancy is what hides its loads.
template <int D, typename OT>
__global__ void __launch_bounds__(kMergeWarps * 32, 4)
paged_merge_kernel(OT* __restrict__ out, const float* __restrict__ tmp_out,
                   const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
                   const int32_t* __restrict__ context_lens, int num_seqs, int num_q_heads,
                   int partition_size, int max_parts, long long len_cap, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const long long item = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
    if (item >= (long long)num_seqs * num_q_heads) return;
    const int s = (int)(item / num_q_heads);
    const int h = (int)(item - (long long)s * num_q_heads);
    const size_t row = (size_t)s * num_q_heads + h;
    // launched as a programmatic dependent of the partition kernel: nothing
    // the previous kernels wrote is read before they have completed
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the partition kernel's clamp (len_cap): only partitions it wrote are read
    int L = context_lens[s];
    const long long cap = len_cap;
    if (L < 0 || L > cap) {
        if (lane == 0 && h == 0 && status) atomicOr(status, PA_DEV_BAD_LEN);
        L = L < 0 ? 0 : (int)cap;
    }
    const int n = (L + partition_size - 1) / partition_size;
    merge_one_head<D, OT, false>(out + row * D, tmp_out + row * max_parts * D,
                                 max_logits + row * max_parts, exp_sums + row * max_parts, n,
                                 lane);
}

template <int D, typename OT>
static cudaError_t launch_merge_t(OT* out, const float* tmp_out, const float* max_logits,
                                  const float* exp_sums, const int32_t* context_lens, int num_seqs,
                                  int num_q_heads, int partition_size, int max_parts,
                                  long long len_cap, uint32_t* status, cudaStream_t stream) {
    const long long items = (long long)num_seqs * num_q_heads;
    const unsigned grid = (unsigned)((items + kMergeWarps - 1) / kMergeWarps);
    // programmatic dependent launch: the merge's CTAs may be scheduled while
    // the previous kernel drains; each waits (griddepcontrol.wait) for it to
    // complete before reading anything, so stream order is kept
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, paged_merge_kernel<D, OT>, out, tmp_out, max_logits, exp_sums,
                              context_lens, num_seqs, num_q_heads, partition_size, max_parts,
                              len_cap, status);
}

template <typename OT>
static cudaError_t launch_merge_o(void* out, const float* tmp_out, const float* max_logits,
                                  const float* exp_sums, const int32_t* context_lens, int num_seqs,
                                  int num_q_heads, int head_size, int partition_size, int max_parts,
                                  long long len_cap, uint32_t* status, cudaStream_t stream) {
    OT* o = static_cast<OT*>(out);
    switch (head_size) {
    case 64:
        return launch_merge_t<64>(o, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                  num_q_heads, partition_size, max_parts, len_cap, status, stream);
    case 128:
        return launch_merge_t<128>(o, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                   num_q_heads, partition_size, max_parts, len_cap, status, stream);
    case 256:
        return launch_merge_t<256>(o, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                   num_q_heads, partition_size, max_parts, len_cap, status, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge(void* out, const float* tmp_out, const float* max_logits,
                         const float* exp_sums, const int32_t* context_lens, int num_seqs,
                         int num_q_heads, int head_size, int partition_size, int max_parts,
                         long long len_cap, pa_dtype out_dtype, uint32_t* status,
                         cudaStream_t stream) {
    switch (out_dtype) {
    case PA_F32:
        return launch_merge_o<float>(out, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                     num_q_heads, head_size, partition_size, max_parts, len_cap,
                                     status, stream);
    case PA_F16:
        return launch_merge_o<__half>(out, tmp_out, max_logits, exp_sums, context_lens, num_seqs,
                                      num_q_heads, head_size, partition_size, max_parts, len_cap,
                                      status, stream);
    case PA_BF16:
        return launch_merge_o<__nv_bfloat16>(out, tmp_out, max_logits, exp_sums, context_lens,
                                             num_seqs, num_q_heads, head_size, partition_size,
                                             max_parts, len_cap, status, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace pagedkv
