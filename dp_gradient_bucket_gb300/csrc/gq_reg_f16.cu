// gq_reg_f16.cu -- the persistent register-staged fused kernel k_fused_pipe for fp16 gradients,
// W = 8 (gq_fused.cuh), in a translation unit of its own so it compiles in parallel with the rest.
#include "gq_fused.cuh"

namespace gq {

static fused::RegInit g_reg_init_f16[64];

cudaError_t launch_reg_f16(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales,
                          cudaStream_t stream, bool* launched) {
    return fused::launch_reg_dt<1>(g_reg_init_f16, a, order, out, codes, scales, stream, launched);
}

cudaError_t reg_f16_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

}  // namespace gq
