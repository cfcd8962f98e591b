// gq_queue_f16.cu -- the work-queue fused kernel k_queue for fp16 gradients, W = 8 (gq_queue.cuh).
#include "gq_queue.cuh"

namespace gq {

static fused::QueueInit g_queue_init_f16[64];

cudaError_t launch_queue_f16(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales,
                             uint32_t* workspace, size_t workspace_bytes, cudaStream_t stream,
                             bool* launched) {
    return fused::launch_queue_dt<1>(g_queue_init_f16, a, order, out, codes, scales, workspace, workspace_bytes,
                                     stream, launched);
}

cudaError_t queue_f16_read_clear_error(unsigned* word) { return fused::read_clear_error(word); }

cudaError_t queue_f16_set_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    return fused::set_stall(extra_bytes, limit_ns);
}

}  // namespace gq
