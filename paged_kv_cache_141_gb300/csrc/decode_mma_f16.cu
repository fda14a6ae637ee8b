// decode_mma_f16.cu -- instantiates the tensor-core decode kernel for a
// query of type __half and a cache of type __half.
#include "decode_mma.cuh"

namespace pagedkv {

cudaError_t launch_decode_mma_f16(const DecodeParams& p, int head_size, int heads_per_unit,
                                bool split, cudaStream_t stream) {
    return launch_mma<__half, __half>(p, head_size, heads_per_unit, split, stream);
}

}  // namespace pagedkv
