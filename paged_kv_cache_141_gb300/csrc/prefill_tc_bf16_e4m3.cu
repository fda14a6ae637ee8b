// prefill_tc_bf16_e4m3.cu -- instantiation of the tcgen05 multi-query kernel
// for bf16 queries and E4M3 caches.
#include "prefill_tc.cuh"

namespace pagedkv {

cudaError_t launch_prefill_tc_bf16_e4m3(const PrefillParams& p, int head_size, cudaStream_t stream) {
    return launch_prefill_tc_e4m3<__nv_bfloat16>(p, head_size, stream);
}

}  // namespace pagedkv
