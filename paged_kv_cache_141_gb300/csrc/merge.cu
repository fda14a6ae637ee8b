// merge.cu -- the reduction of the split decode ("TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 4.1: long sequences are cut into partitions that
// are computed in parallel and then merged). For each (sequence, query head):
//   M = max_p m_p,  w_p = l_p * exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// Up to 15 partitions: one warp per (sequence, head), eight per CTA
// (merge_common.cuh). 16 or more (long contexts): one CTA of 16 warps per
// (sequence, head), each warp reducing its own slice of the partitions, so
// that a few long sequences do not leave the GPU waiting on one warp's chain
// of loads. One partition is copied; none gives zeros.
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


// ---------------------------------------------------------------- wide merge

constexpr int kWideWarps = 16;
constexpr int kWideFrom = 16;          // partitions at which the wide merge is used

template <int D, typename OT>
__global__ void __launch_bounds__(kWideWarps * 32)
paged_merge_wide_kernel(OT* __restrict__ out, const float* __restrict__ tmp_out,
                        const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
                        const int32_t* __restrict__ context_lens, int num_seqs, int num_q_heads,
                        int partition_size, int max_parts, long long len_cap, uint32_t* status) {
    constexpr int EPL = D / 32;
    constexpr int kGroup = EPL >= 8 ? 4 : 8;     // partitions' outputs in flight per warp
    __shared__ float red_m[kWideWarps];
    __shared__ float red_w[kWideWarps];
    __shared__ __align__(16) float red_o[kWideWarps][D];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = (int)(blockIdx.x / num_q_heads);
    const int h = (int)(blockIdx.x - (long long)s * num_q_heads);
    const size_t row = (size_t)s * num_q_heads + h;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int L = context_lens[s];
    if (L < 0 || L > len_cap) {
        if (threadIdx.x == 0 && h == 0 && status) atomicOr(status, PA_DEV_BAD_LEN);
        L = L < 0 ? 0 : (int)len_cap;
    }
    const int n = (L + partition_size - 1) / partition_size;
    const float* to = tmp_out + row * max_parts * D;
    const float* ml = max_logits + row * max_parts;
    const float* es = exp_sums + row * max_parts;
    OT* o = out + row * D;
    if (n <= 1) {
        for (int e = threadIdx.x; e < D; e += blockDim.x)
            o[e] = from_float<OT>(n == 1 ? __ldg(to + e) : 0.f);
        return;
    }
    // the maximum over all partitions, across the CTA
    float M = -INFINITY;
    for (int i = threadIdx.x; i < n; i += blockDim.x) M = fmaxf(M, __ldg(ml + i));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    if (lane == 0) red_m[warp] = M;
    __syncthreads();
    M = red_m[0];
#pragma unroll
    for (int w = 1; w < kWideWarps; ++w) M = fmaxf(M, red_m[w]);

    // this warp's contiguous slice of the partitions
    const int per = (n + kWideWarps - 1) / kWideWarps;
    const int first = warp * per;
    const int last = min(n, first + per);
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int c0 = first; c0 < last; c0 += 32) {
        const int i = c0 + lane;
        const float w = i < last ? __ldg(es + i) * fast_exp2((__ldg(ml + i) - M) * kLog2e) : 0.f;
        wsum += w;
        const int cn = min(32, last - c0);
        for (int j0 = 0; j0 < cn; j0 += kGroup) {
            float v[kGroup][EPL];
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                if (j0 + j < cn) {
                    // this lane's EPL components: 2 (8-byte aligned), 4 or 8
                    const float* tp = to + (size_t)(c0 + j0 + j) * D + lane * EPL;
                    if constexpr (EPL == 2) {
                        const float2 x = __ldg(reinterpret_cast<const float2*>(tp));
                        v[j][0] = x.x; v[j][1] = x.y;
                    } else {
#pragma unroll
                        for (int e = 0; e < EPL; e += 4) {
                            const float4 x = __ldg(reinterpret_cast<const float4*>(tp + e));
                            v[j][e] = x.x; v[j][e + 1] = x.y; v[j][e + 2] = x.z; v[j][e + 3] = x.w;
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                const float wj = __shfl_sync(0xffffffffu, w, (j0 + j) & 31);
                if (j0 + j < cn) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wj, v[j][e], acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, m);
#pragma unroll
    for (int e = 0; e < EPL; ++e) red_o[warp][lane * EPL + e] = acc[e];
    if (lane == 0) red_w[warp] = wsum;
    __syncthreads();
    float W = 0.f;
#pragma unroll
    for (int w = 0; w < kWideWarps; ++w) W += red_w[w];
    for (int e = threadIdx.x; e < D; e += blockDim.x) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kWideWarps; ++w) a += red_o[w][e];
        o[e] = from_float<OT>(__fdiv_rn(a, W));
    }
}

template <int D, typename OT>
static cudaError_t launch_merge_t(OT* out, const float* tmp_out, const float* max_logits,
                                  const float* exp_sums, const int32_t* context_lens, int num_seqs,
                                  int num_q_heads, int partition_size, int max_parts,
                                  long long len_cap, uint32_t* status, cudaStream_t stream) {
    const long long items = (long long)num_seqs * num_q_heads;
    const bool wide = max_parts >= kWideFrom;
    const unsigned grid = wide ? (unsigned)items
                               : (unsigned)((items + kMergeWarps - 1) / kMergeWarps);
    // programmatic dependent launch: the merge's CTAs may be scheduled while
    // the previous kernel drains; each waits (griddepcontrol.wait) for it to
    // complete before reading anything, so stream order is kept
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((wide ? kWideWarps : kMergeWarps) * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (wide)
        return cudaLaunchKernelEx(&cfg, paged_merge_wide_kernel<D, OT>, out, tmp_out, max_logits,
                                  exp_sums, context_lens, num_seqs, num_q_heads, partition_size,
                                  max_parts, len_cap, status);
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
