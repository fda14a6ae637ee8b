// decode_tma_f32.cu -- instantiates the tensor-TMA decode kernel for a
// query of type float and a cache of type float.
#include "decode_tma.cuh"

namespace pagedkv {

cudaError_t launch_decode_tma_f32(const DecodeParams& p, int head_size, int heads_per_unit,
                                bool split, cudaStream_t stream) {
    return launch_tma<float, float>(p, head_size, heads_per_unit, split, stream);
}

}  // namespace pagedkv
