// gq_fused_f16.cu -- the cluster kernel k_fused (gq_fused.cuh) for fp16 gradients.
#include "gq_fused.cuh"

namespace gq {

static fused::DeviceInit g_init_f16[64];

cudaError_t launch_fused_f16(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales,
                             cudaStream_t stream) {
    return fused::launch<1>(g_init_f16, a, order, out, codes, scales, stream);
}

cudaError_t fused_f16_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

cudaError_t fused_f16_set_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    return fused::set_stall(extra_bytes, limit_ns);
}

}  // namespace gq
