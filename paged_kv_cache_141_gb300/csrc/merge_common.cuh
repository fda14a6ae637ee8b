// merge_common.cuh -- the partition merge for one (sequence, query head),
// run by one warp: M = max_p m_p, w_p = l_p * exp(m_p - M),
// out = sum_p w_p o_p / sum_p w_p ("TGI PagedAttention deep-dive" (lpnh.cn)
// sec. 4.1: partitions computed in parallel, then reduced). Used by the merge
// kernel. The lanes take
// partitions for the maximum and the weights; every lane then accumulates
// head_size/32 components of a group of partitions' outputs at a time, all
// loads of a group issued before their use, the first group together with
// the maxima and sums.
#pragma once

#include "device_common.cuh"

namespace pagedkv {

// Loads of partials written by other CTAs of the same launch go through L2
// (ld.global.cg), never a possibly stale L1 line.
template <int D, typename OT, bool kFromOtherCtas>
__device__ __forceinline__ void merge_one_head(OT* __restrict__ o, const float* __restrict__ to,
                                               const float* __restrict__ ml,
                                               const float* __restrict__ es, int n, int lane) {
    constexpr int EPL = D / 32;
    // partitions per load group: few registers, so that many warps fit
    constexpr int kGroup = EPL >= 4 ? 4 : 8;
    auto ld = [](const float* q) { return kFromOtherCtas ? __ldcg(q) : __ldg(q); };
    auto ld4 = [](const float* q) {
        return kFromOtherCtas ? __ldcg(reinterpret_cast<const float4*>(q))
                              : __ldg(reinterpret_cast<const float4*>(q));
    };
    float acc[EPL];
    if (n <= 1) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = n == 1 ? ld(to + lane * EPL + e) : 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[lane * EPL + e] = from_float<OT>(acc[e]);
        return;
    }
    // One round trip to L2 for the common case (n <= 32 partitions): the
    // first 32 maxima and sums and the first group of partial outputs are all
    // in flight before the maximum is reduced.
    const float m0 = lane < n ? ld(ml + lane) : -INFINITY;
    const float s0 = lane < n ? ld(es + lane) : 0.f;
    float v[kGroup][EPL];
    auto load_group = [&](float (&v)[kGroup][EPL], int first, int count) {
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            if (j < count) {
                const float* tp = to + (size_t)(first + j) * D + lane * EPL;
                if constexpr (EPL == 2) {
                    v[j][0] = ld(tp);
                    v[j][1] = ld(tp + 1);
                } else {
#pragma unroll
                    for (int e = 0; e < EPL; e += 4) {
                        const float4 x = ld4(tp + e);
                        v[j][e] = x.x; v[j][e + 1] = x.y; v[j][e + 2] = x.z; v[j][e + 3] = x.w;
                    }
                }
            }
        }
    };
    load_group(v, 0, min(kGroup, n));
    float M = m0;
    for (int i = lane + 32; i < n; i += 32) M = fmaxf(M, ld(ml + i));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int i = c0 + lane;
        float w;
        if (c0 == 0) w = lane < n ? s0 * fast_exp2((m0 - M) * kLog2e) : 0.f;
        else w = i < n ? ld(es + i) * fast_exp2((ld(ml + i) - M) * kLog2e) : 0.f;
        wsum += w;
        const int cn = min(32, n - c0);
        for (int j0 = 0; j0 < cn; j0 += kGroup) {
            // up to kGroup partitions' loads in flight, then their use (the
            // first group is already loaded)
            if (c0 != 0 || j0 != 0) load_group(v, c0 + j0, cn - j0);
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
    for (int e = 0; e < EPL; ++e) o[lane * EPL + e] = from_float<OT>(__fdiv_rn(acc[e], wsum));
}

}  // namespace pagedkv
