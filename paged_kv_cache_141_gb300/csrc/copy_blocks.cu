// copy_blocks.cu -- the copy of copy-on-write: whole physical blocks (every
// KV head of K and of V) copied from src to dst for each (src, dst) pair, so
// that a sequence diverging from a shared block continues in a private copy
// ("vLLM Page Attention Continuous Batching" (lbrq.cn), "Sharing KV Cache-COW";
// "Lecture 3: PagedAttention and vLLM", "shared prefix").
// One CTA column per pair; threads move 16-byte vectors of the block slab
// (Hkv * B * d elements, contiguous in the declared layout).
#include "device_common.cuh"
#include "launch.h"

namespace pagedkv {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                   const int64_t* __restrict__ pairs, int64_t num_pairs, int64_t num_blocks,
                   int64_t block_bytes, uint32_t* status) {
    const int64_t i = blockIdx.y;
    if (i >= num_pairs) return;
    const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && status) atomicOr(status, PA_DEV_BAD_BLOCK_ID);
        return;
    }
    const int64_t nvec = block_bytes / 16;
    const uint4* ks = reinterpret_cast<const uint4*>(k_cache + src * block_bytes);
    const uint4* vs = reinterpret_cast<const uint4*>(v_cache + src * block_bytes);
    uint4* kd = reinterpret_cast<uint4*>(k_cache + dst * block_bytes);
    uint4* vd = reinterpret_cast<uint4*>(v_cache + dst * block_bytes);
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (int64_t)gridDim.x * blockDim.x) {
        kd[v] = ks[v];
        vd[v] = vs[v];
    }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs,
                               int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                               uint32_t* status, cudaStream_t stream) {
    const int64_t nvec = block_bytes / 16;
    int64_t cols = (nvec + kCopyThreads - 1) / kCopyThreads;
    if (cols > 64) cols = 64;
    for (int64_t first = 0; first < num_pairs; first += 65535) {
        const int64_t n = num_pairs - first < 65535 ? num_pairs - first : 65535;
        dim3 grid((unsigned)cols, (unsigned)n);
        copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(
            static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), pairs + 2 * first, n,
            num_blocks, block_bytes, status);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pagedkv
