// kv_store.cuh -- storing one 16-byte vector of new key/value elements into
// the cache: a bit copy for the same type, or E4M3 quantisation (IEEE binary32
// division by the per-tensor scale, then CUDA's saturating E4M3 converter).
// Shared by the KV write kernel and the decode kernels' fused write, so both
// store identical bits.
#pragma once

#include "device_common.cuh"
#include "launch.h"

namespace pagedkv {

template <typename TI>
struct Vec16 {
    static constexpr int n = 16 / (int)sizeof(TI);
};

template <typename TI>
__device__ __forceinline__ void widen16(const uint4& w, float (&x)[Vec16<TI>::n]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    if constexpr (std::is_same<TI, float>::value) {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(ws[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f;
            if constexpr (std::is_same<TI, __half>::value)
                f = __half22float2(*reinterpret_cast<const __half2*>(&ws[i]));
            else
                f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
}

template <typename TI>
__device__ __forceinline__ void store_e4m3(uint8_t* dst, const uint4& w, float scale) {
    constexpr int N = Vec16<TI>::n;   // 4 (binary32) or 8 (16-bit types)
    float x[N];
    widen16<TI>(w, x);
    uint32_t packed[N / 4];
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const float2 q = make_float2(__fdiv_rn(x[i], scale), __fdiv_rn(x[i + 1], scale));
        const uint32_t two = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
        if ((i & 2) == 0) packed[i / 4] = two;
        else packed[i / 4] |= two << 16;
    }
    if constexpr (N == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    else *reinterpret_cast<uint32_t*>(dst) = packed[0];
}

// Store one 16-byte vector of new elements (type TI) at cache element offset
// `dst` (units of the cache type): a bit copy, or E4M3 codes.
template <typename TI, bool kE4M3>
__device__ __forceinline__ void store_kv_vector(void* cache, size_t dst, const uint4& w, float scale) {
    if constexpr (kE4M3) {
        store_e4m3<TI>(static_cast<uint8_t*>(cache) + dst, w, scale);
    } else {
        *reinterpret_cast<uint4*>(static_cast<TI*>(cache) + dst) = w;
    }
}


// Fused KV write, run by a decode kernel's producer warp (all 32 lanes) before
// it loads the stage that holds position L-1 of sequence s: store the
// sequence's newest key and value (KV head kvh) at slot_mapping[s]
// (fused_store_token), then fence the generic-proxy stores against the
// bulk-copy (async-proxy) reads that follow (fused_write_token does both; a
// producer may issue the stores earlier and fence right before that stage's
// copy). A negative slot stores nothing; a slot outside the pool sets
// PA_DEV_BAD_SLOT; a slot that is not position L-1 of the sequence's table
// sets PA_DEV_SLOT_MISMATCH (the token is still stored, the decode may not see
// it).
template <typename QT, typename CT, int D>
__device__ __forceinline__ void fused_store_token(const DecodeParams& p, int s, int kvh, int L,
                                                  int lane) {
    constexpr bool kE4M3 = std::is_same<CT, e4m3_t>::value;
    constexpr int VEC = 16 / (int)sizeof(QT);
    constexpr int NVEC = D / VEC;
    const int64_t slot = p.new_slots[s];
    if (slot >= 0) {
        const int B = p.block_size;
        if (slot >= p.num_blocks * (int64_t)B) {
            if (lane == 0 && p.status) atomicOr(p.status, PA_DEV_BAD_SLOT);
        } else {
            const int pos = L - 1;
            const int64_t expect = (int64_t)p.block_tables[(size_t)s * p.max_blocks + pos / B] * B + pos % B;
            if (slot != expect && lane == 0 && p.status) atomicOr(p.status, PA_DEV_SLOT_MISMATCH);
            const int64_t blk = slot / B;
            const int off = (int)(slot - blk * B);
            const size_t src0 = ((size_t)s * p.num_kv_heads + kvh) * D;
            const size_t dst0 = (((size_t)blk * p.num_kv_heads + kvh) * B + off) * D;
            for (int i = lane; i < 2 * NVEC; i += 32) {
                const bool is_v = i >= NVEC;
                const int c = is_v ? i - NVEC : i;
                const QT* src = static_cast<const QT*>(is_v ? p.new_value : p.new_key) + src0 + c * VEC;
                const uint4 w = *reinterpret_cast<const uint4*>(src);
                store_kv_vector<QT, kE4M3>(is_v ? p.wv_cache : p.wk_cache, dst0 + (size_t)c * VEC, w,
                                           is_v ? p.v_scale_w : p.k_scale_w);
            }
        }
    }
}

// The stores' fence against the async proxy, by the lanes that stored.
__device__ __forceinline__ void fused_write_fence() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
}

template <typename QT, typename CT, int D>
__device__ __forceinline__ void fused_write_token(const DecodeParams& p, int s, int kvh, int L,
                                                  int lane) {
    fused_store_token<QT, CT, D>(p, s, kvh, L, lane);
    fused_write_fence();
}

}  // namespace pagedkv
