// gq_fused_f16.cu -- the fused kernel for fp16 gradients: the persistent kernel for W = 8
// (gq_reg_f16.cu) when it applies, else the staged / re-read cluster kernel k_fused (gq_fused.cuh).
#include "gq_fused.cuh"

namespace gq {

static fused::DeviceInit g_init_f16[64];

cudaError_t launch_fused_f16(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales,
                             cudaStream_t stream) {
#ifndef GQ_NO_REG_KERNEL
    bool launched = false;
    const cudaError_t e = launch_reg_f16(a, order, out, codes, scales, stream, &launched);
    if (launched || e != cudaSuccess) return e;
#endif
    return fused::launch<1>(g_init_f16, a, order, out, codes, scales, stream);
}

cudaError_t fused_f16_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

cudaError_t fused_f16_set_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    return fused::set_stall(extra_bytes, limit_ns);
}

}  // namespace gq
