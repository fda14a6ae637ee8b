// prefill_mma_bf16.cu -- instantiates the warp-level MMA multi-query kernel
// for a query of type __nv_bfloat16 and a cache of type __nv_bfloat16.
#include "prefill_mma.cuh"

namespace pagedkv {

cudaError_t launch_prefill_mma_bf16(const DecodeParams& p, int head_size, cudaStream_t stream) {
    return launch_prefill_mma<__nv_bfloat16, __nv_bfloat16>(p, head_size, stream);
}

}  // namespace pagedkv
