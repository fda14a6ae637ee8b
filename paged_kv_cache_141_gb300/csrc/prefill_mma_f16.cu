// prefill_mma_f16.cu -- instantiates the warp-level MMA multi-query kernel
// for a query of type __half and a cache of type __half.
#include "prefill_mma.cuh"

namespace pagedkv {

cudaError_t launch_prefill_mma_f16(const DecodeParams& p, int head_size, cudaStream_t stream) {
    return launch_prefill_mma<__half, __half>(p, head_size, stream);
}

}  // namespace pagedkv
