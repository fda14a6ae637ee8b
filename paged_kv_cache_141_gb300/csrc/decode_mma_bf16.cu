// decode_mma_bf16.cu -- instantiates the tensor-core decode kernel for a
// query of type __nv_bfloat16 and a cache of type __nv_bfloat16.
#include "decode_mma.cuh"

namespace pagedkv {

cudaError_t launch_decode_mma_bf16(const DecodeParams& p, int head_size, int heads_per_unit,
                                 bool split, cudaStream_t stream) {
    return launch_mma<__nv_bfloat16, __nv_bfloat16>(p, head_size, heads_per_unit, split, stream);
}

}  // namespace pagedkv
