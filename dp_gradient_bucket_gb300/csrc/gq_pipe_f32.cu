// gq_pipe_f32.cu -- the pipelined fused kernel k_pipe for fp32 gradients (gq_pipe.cuh).
#include "gq_pipe.cuh"

namespace gq {

static pipe::PipeInit g_pipe_init_f32[64];

size_t pipe_workspace_bytes(int W, int64_t rank_stride, int64_t num_chunks) {
    return pipe::workspace_bytes(W, rank_stride, num_chunks);
}

cudaError_t launch_pipe_f32(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales, void* workspace,
                            int max_ctas, cudaStream_t stream) {
    return pipe::launch_pipe_dt<0>(g_pipe_init_f32, a, order, out, codes, scales, workspace, max_ctas, stream);
}

cudaError_t pipe_f32_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

cudaError_t pipe_f32_set_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    return fused::set_stall(extra_bytes, limit_ns);
}

}  // namespace gq
