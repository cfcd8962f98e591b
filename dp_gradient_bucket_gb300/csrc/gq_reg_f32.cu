// gq_reg_f32.cu -- the persistent register-staged fused kernel k_fused_pipe for fp32 gradients,
// W = 8 (gq_fused.cuh), in a translation unit of its own so it compiles in parallel with the rest.
#include "gq_fused.cuh"

namespace gq {

static fused::RegInit g_reg_init_f32[64];

cudaError_t launch_reg_f32(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales,
                          cudaStream_t stream, bool* launched) {
    return fused::launch_reg_dt<0>(g_reg_init_f32, a, order, out, codes, scales, stream, launched);
}

cudaError_t reg_f32_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

}  // namespace gq
