// decode_tma_bf16_e4m3.cu -- instantiates the tensor-TMA decode kernel for a
// query of type __nv_bfloat16 and a cache of type e4m3_t.
#include "decode_tma.cuh"

namespace pagedkv {

cudaError_t launch_decode_tma_bf16_e4m3(const DecodeParams& p, int head_size, int heads_per_unit,
                                      bool split, cudaStream_t stream) {
    return launch_tma<__nv_bfloat16, e4m3_t>(p, head_size, heads_per_unit, split, stream);
}

}  // namespace pagedkv
