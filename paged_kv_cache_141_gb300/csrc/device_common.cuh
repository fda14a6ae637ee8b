// device_common.cuh -- device helpers shared by the library's kernels:
// element types, bulk-copy (TMA) and mbarrier wrappers in inline PTX, bounded
// waits, and vector loads that widen cache elements to float.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "pagedkv.h"

namespace pagedkv {

// ------------------------------------------------------------------ types

struct e4m3_t {  // one OCP E4M3 code
    uint8_t bits;
};

template <typename T> struct TypeInfo;
template <> struct TypeInfo<float> { static constexpr int bytes = 4; };
template <> struct TypeInfo<__half> { static constexpr int bytes = 2; };
template <> struct TypeInfo<__nv_bfloat16> { static constexpr int bytes = 2; };
template <> struct TypeInfo<e4m3_t> { static constexpr int bytes = 1; };

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Widen N consecutive stored elements (read as one aligned vector) to float.
// N * sizeof(T) is 2, 4, 8, 16 or 32 bytes.
template <typename T, int N> struct RowLoader;

template <int N> struct RowLoader<float, N> {
    __device__ __forceinline__ static void load(const float* p, float (&x)[N]) {
        if constexpr (N == 2) {
            float2 v = *reinterpret_cast<const float2*>(p);
            x[0] = v.x; x[1] = v.y;
        } else {
#pragma unroll
            for (int i = 0; i < N; i += 4) {
                float4 v = *reinterpret_cast<const float4*>(p + i);
                x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
            }
        }
    }
};

template <typename H2, typename H, int N>
__device__ __forceinline__ void load_half_like(const H* p, float (&x)[N]) {
    static_assert(N % 2 == 0, "pairs");
    if constexpr (N == 2) {
        uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        H2 h = *reinterpret_cast<H2*>(&w);
        float2 f;
        if constexpr (sizeof(H) == 2 && std::is_same<H, __half>::value) f = __half22float2(h);
        else f = __bfloat1622float2(h);
        x[0] = f.x; x[1] = f.y;
    } else if constexpr (N == 4) {
        uint2 w = *reinterpret_cast<const uint2*>(p);
        uint32_t ws[2] = {w.x, w.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            H2 h = *reinterpret_cast<H2*>(&ws[i]);
            float2 f;
            if constexpr (std::is_same<H, __half>::value) f = __half22float2(h);
            else f = __bfloat1622float2(h);
            x[2 * i] = f.x; x[2 * i + 1] = f.y;
        }
    } else {
#pragma unroll
        for (int c = 0; c < N; c += 8) {
            uint4 w = *reinterpret_cast<const uint4*>(p + c);
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                H2 h = *reinterpret_cast<H2*>(&ws[i]);
                float2 f;
                if constexpr (std::is_same<H, __half>::value) f = __half22float2(h);
                else f = __bfloat1622float2(h);
                x[c + 2 * i] = f.x; x[c + 2 * i + 1] = f.y;
            }
        }
    }
}

template <int N> struct RowLoader<__half, N> {
    __device__ __forceinline__ static void load(const __half* p, float (&x)[N]) {
        load_half_like<__half2, __half, N>(p, x);
    }
};
template <int N> struct RowLoader<__nv_bfloat16, N> {
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&x)[N]) {
        load_half_like<__nv_bfloat162, __nv_bfloat16, N>(p, x);
    }
};

// E4M3 pairs widen exactly to binary16 with one conversion each, then to float.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

template <int N> struct RowLoader<e4m3_t, N> {
    __device__ __forceinline__ static void load(const e4m3_t* p, float (&x)[N]) {
        static_assert(N % 2 == 0, "pairs");
        if constexpr (N == 2) {
            float2 f = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
            x[0] = f.x; x[1] = f.y;
        } else if constexpr (N == 4) {
            uint32_t w = *reinterpret_cast<const uint32_t*>(p);
            float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w & 0xffffu));
            float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w >> 16));
            x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
        } else {
#pragma unroll
            for (int c = 0; c < N; c += 8) {
                uint2 w = *reinterpret_cast<const uint2*>(p + c);
                uint32_t ws[2] = {w.x, w.y};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    float2 a = e4m3x2_to_float2(static_cast<uint16_t>(ws[i] & 0xffffu));
                    float2 b = e4m3x2_to_float2(static_cast<uint16_t>(ws[i] >> 16));
                    x[c + 4 * i] = a.x; x[c + 4 * i + 1] = a.y;
                    x[c + 4 * i + 2] = b.x; x[c + 4 * i + 3] = b.y;
                }
            }
        }
    }
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// A wait gives up after about a second of SM clocks (GB300 runs near 2 GHz)
// and reports PA_DEV_TIMEOUT; no pipeline in this library legitimately waits
// anywhere near that long.
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            if (status) atomicOr(status, PA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// 1-D bulk copy global -> shared (the TMA engine), completing on an mbarrier.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                                   uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads.
__device__ __forceinline__ bool named_barrier_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// 2^x on the special-function unit (PTX ex2.approx: relative error about 2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Host: raise a kernel's dynamic shared-memory limit once per device.
// `key` identifies the kernel (its address); the table is small and
// append-only, and a race only repeats the (idempotent) attribute call.
inline cudaError_t ensure_smem_attribute(const void* key, int bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    constexpr int kSlots = 512;
    static std::atomic<const void*> keys[kSlots];
    static std::atomic<uint64_t> masks[kSlots];
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    int slot = -1;
    for (int i = 0; i < kSlots; ++i) {
        const void* k = keys[i].load(std::memory_order_acquire);
        if (k == key) { slot = i; break; }
        if (k == nullptr) {
            const void* expected = nullptr;
            if (keys[i].compare_exchange_strong(expected, key) || expected == key) { slot = i; break; }
        }
    }
    if (slot >= 0 && bit && (masks[slot].load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(key, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && slot >= 0 && bit) masks[slot].fetch_or(bit);
    return e;
}

constexpr float kLog2e = 1.4426950408889634f;   // log2(e)
constexpr float kLn2 = 0.6931471805599453f;     // ln(2)

}  // namespace pagedkv
