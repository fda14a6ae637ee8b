// decode_mma_bf16_e4m3.cu -- instantiates the tensor-core decode kernel for a
// query of type __nv_bfloat16 and a cache of type e4m3_t.
#include "decode_mma.cuh"

namespace pagedkv {

cudaError_t launch_decode_mma_bf16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                      bool split, cudaStream_t stream) {
    return launch_mma<__nv_bfloat16, e4m3_t>(p, head_size, heads_per_unit, split, stream);
}

}  // namespace pagedkv
