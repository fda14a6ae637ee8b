// decode_static_workspace.cu -- the partitioned decode for callers that
// cannot allocate device memory.
//
// pa_decode_partitioned needs a workspace for the per-partition partials,
// which its caller normally allocates. Some callers cannot: a serving loop that
// has handed all device memory to a fixed, pre-sized pool, a plugin embedded
// in a host program that owns every allocation, or a step that must not risk
// the device-wide synchronisation cudaMalloc and cudaFree may cause. This entry
// point takes its workspace from a fixed array in this library's device
// memory instead. The array is PA_STATIC_WORKSPACE_BYTES long; every GPU that
// loads the library holds it until the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "pagedkv.h"

namespace {

// The workspace itself. In host code the name below is a host-side stand-in,
// never a device address; the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_workspace_address[kMaxDevices];

// Device address of the array on the current device, looked up once per
// device (the first call on a device does the lookup).
cudaError_t static_workspace_address(void** address) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* p = g_workspace_address[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess) return e;
        g_workspace_address[dev].store(p, std::memory_order_release);
    }
    *address = p;
    return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_partitioned_static(
    void* out, const void* query, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
    int max_context_len, float scale, pa_dtype q_dtype, pa_dtype cache_dtype, float k_scale,
    float v_scale, int partition_size, uint32_t* dev_status, void* stream) {
    const size_t need = pa_decode_partitioned_workspace_bytes(num_seqs, num_q_heads, head_size,
                                                              max_context_len, partition_size);
    if (need > (size_t)PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
    void* workspace = nullptr;
    if (static_workspace_address(&workspace) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return pa_decode_partitioned(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size,
                                 block_size, num_blocks, max_context_len, scale, q_dtype,
                                 cache_dtype, k_scale, v_scale, partition_size, workspace,
                                 (size_t)PA_STATIC_WORKSPACE_BYTES, dev_status, stream);
}
