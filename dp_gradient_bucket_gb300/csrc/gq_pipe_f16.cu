// gq_pipe_f16.cu -- the pipelined fused kernel k_pipe for fp16 gradients (gq_pipe.cuh).
#include "gq_pipe.cuh"

namespace gq {

static pipe::PipeInit g_pipe_init_f16[64];

cudaError_t launch_pipe_f16(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales, void* workspace,
                            int max_ctas, cudaStream_t stream) {
    return pipe::launch_pipe_dt<1>(g_pipe_init_f16, a, order, out, codes, scales, workspace, max_ctas, stream);
}

cudaError_t pipe_f16_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

cudaError_t pipe_f16_set_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    return fused::set_stall(extra_bytes, limit_ns);
}

}  // namespace gq
