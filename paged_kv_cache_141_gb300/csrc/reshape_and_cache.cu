// reshape_and_cache.cu -- the KV write ("TGI PagedAttention deep-dive"
// (lpnh.cn) sec. 4.1, the write side: new keys/values go into the block cache
// at their `slots`, optionally quantised to FP8).
//
// Each thread moves one 16-byte vector of the input for both K and V: it reads
// the token's slot, splits it into (block, offset) and stores the vector into
// [block][head][offset][:] of each cache. Same-type writes copy bits; E4M3
// writes divide by the per-tensor scale in IEEE binary32 and convert with
// round-to-nearest-even and saturation to +-448 (CUDA's E4M3 converter).
// A grid-stride loop keeps the grid at a multiple of the SM count.
#include "device_common.cuh"
#include "kv_store.cuh"
#include "launch.h"

namespace pagedkv {

constexpr int kWriteThreads = 256;

template <typename TI, bool kE4M3>
__global__ void __launch_bounds__(kWriteThreads)
reshape_and_cache_kernel(const TI* __restrict__ key, const TI* __restrict__ value,
                         void* __restrict__ k_cache, void* __restrict__ v_cache,
                         const int64_t* __restrict__ slots, int64_t num_tokens, int H, int D,
                         int B, int64_t num_blocks, float k_scale, float v_scale,
                         uint32_t* status) {
    constexpr int VEC = Vec16<TI>::n;
    const int vec_per_row = D / VEC;
    const int64_t per_token = (int64_t)H * vec_per_row;
    const int64_t total = num_tokens * per_token;
    const int64_t limit = num_blocks * B;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_token;
        const int r = (int)(i - t * per_token);
        const int h = r / vec_per_row;
        const int c = r - h * vec_per_row;
        const int64_t slot = slots[t];
        if (slot < 0) continue;                                   // padding token
        if (slot >= limit) {
            if (r == 0 && status) atomicOr(status, PA_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / B;
        const int off = (int)(slot - blk * B);
        const size_t src = ((size_t)t * H + h) * D + (size_t)c * VEC;
        const size_t dst = (((size_t)blk * H + h) * B + off) * D + (size_t)c * VEC;
        const uint4 kw = *reinterpret_cast<const uint4*>(key + src);
        const uint4 vw = *reinterpret_cast<const uint4*>(value + src);
        if constexpr (kE4M3) {
            store_e4m3<TI>(static_cast<uint8_t*>(k_cache) + dst, kw, k_scale);
            store_e4m3<TI>(static_cast<uint8_t*>(v_cache) + dst, vw, v_scale);
        } else {
            *reinterpret_cast<uint4*>(static_cast<TI*>(k_cache) + dst) = kw;
            *reinterpret_cast<uint4*>(static_cast<TI*>(v_cache) + dst) = vw;
        }
    }
}

template <typename TI, bool kE4M3>
static cudaError_t launch_write(const void* key, const void* value, void* k_cache, void* v_cache,
                                const int64_t* slots, int64_t num_tokens, int H, int D, int B,
                                int64_t num_blocks, float k_scale, float v_scale,
                                uint32_t* status, cudaStream_t stream) {
    const int64_t total = num_tokens * H * (D / Vec16<TI>::n);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (total + kWriteThreads - 1) / kWriteThreads;
    const int64_t cap = (int64_t)sms * 8;                         // 8 resident CTAs per SM
    const int grid = (int)(want < cap ? want : cap);
    reshape_and_cache_kernel<TI, kE4M3><<<grid, kWriteThreads, 0, stream>>>(
        static_cast<const TI*>(key), static_cast<const TI*>(value), k_cache, v_cache, slots,
        num_tokens, H, D, B, num_blocks, k_scale, v_scale, status);
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache,
                                     void* v_cache, const int64_t* slots, int64_t num_tokens,
                                     int num_kv_heads, int head_size, int block_size,
                                     int64_t num_blocks, pa_dtype in_dtype, pa_dtype cache_dtype,
                                     float k_scale, float v_scale, uint32_t* status,
                                     cudaStream_t stream) {
    const bool fp8 = cache_dtype == PA_FP8_E4M3;
#define PA_WRITE(T, F) launch_write<T, F>(key, value, k_cache, v_cache, slots, num_tokens, \
    num_kv_heads, head_size, block_size, num_blocks, k_scale, v_scale, status, stream)
    switch (in_dtype) {
    case PA_F32: return fp8 ? PA_WRITE(float, true) : PA_WRITE(float, false);
    case PA_F16: return fp8 ? PA_WRITE(__half, true) : PA_WRITE(__half, false);
    case PA_BF16: return fp8 ? PA_WRITE(__nv_bfloat16, true) : PA_WRITE(__nv_bfloat16, false);
    default: return cudaErrorInvalidValue;
    }
#undef PA_WRITE
}

}  // namespace pagedkv
