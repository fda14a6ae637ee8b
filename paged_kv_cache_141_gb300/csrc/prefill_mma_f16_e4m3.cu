// prefill_mma_f16_e4m3.cu -- instantiates the warp-level MMA multi-query kernel
// for a query of type __half and a cache of type e4m3_t.
#include "prefill_mma.cuh"

namespace pagedkv {

cudaError_t launch_prefill_mma_f16_e4m3(const DecodeParams& p, int head_size, cudaStream_t stream) {
    return launch_prefill_mma<__half, e4m3_t>(p, head_size, stream);
}

}  // namespace pagedkv
