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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv.h"

namespace {

// The workspace itself. In host code the name below is a host-side stand-in,
// never a device address; the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// Per device: the id of the context the address was looked up in, and the
// address. A context id is unique for the life of the process, so a device
// whose context was destroyed and created again (cudaDeviceReset, or the
// caller's own driver context) gets a fresh lookup instead of a stale address.
struct Entry {
    unsigned long long ctx_id;    // 0: not looked up yet
    void* address;
};
std::mutex g_lock;
Entry g_entries[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The id of the calling thread's current context, 0 if there is none yet.
// Driver calls are reached through the runtime's entry-point query, so the
// library does not link the driver library. Called with g_lock held.
cudaError_t current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000,
                                                         cudaEnableDefault, &qa);
        if (e != cudaSuccess || qa != cudaDriverEntryPointSuccess || !a) return cudaErrorUnknown;
        e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb);
        if (e != cudaSuccess || qb != cudaDriverEntryPointSuccess || !b) return cudaErrorUnknown;
        get_current = reinterpret_cast<CtxGetCurrentFn>(a);
        get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
    *id = 0;
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorUnknown;
    return cudaSuccess;
}

// Device address of the array in the current device's context, looked up
// with that device current the first time the context is seen (the first call
// on a device, and the first after its context was replaced).
cudaError_t static_workspace_address(void** address) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> hold(g_lock);
    unsigned long long id = 0;
    if ((e = current_context_id(&id)) != cudaSuccess) return e;
    Entry& entry = g_entries[dev];
    if (id != 0 && entry.ctx_id == id) {
        *address = entry.address;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);       // makes the context current if needed
    if (e != cudaSuccess) return e;
    if ((e = current_context_id(&id)) != cudaSuccess) return e;
    if (id == 0) return cudaErrorInvalidDevice;
    entry.ctx_id = id;
    entry.address = p;
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
