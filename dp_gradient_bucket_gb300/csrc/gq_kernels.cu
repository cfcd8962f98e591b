// gq_kernels.cu -- sm_103a kernels of the int8 gradient-bucket path and their launchers.
//
//   k_plan      chunk table of dynamic_chunk ("pipelined HCCL AllReduce" article, §2.1)
//   k_quantize  per-(rank, chunk) absmax scale + int8 codes (§2.2.1 quantize_gradient)
//   k_reduce    W-way dequantise-sum in a fixed order + mean (§2.2.1 INT8_ALLREDUCE,
//               §3.1 per-chunk SUM all_reduce; mean as in the "torchtitan-npu 3D parallel"
//               article, AMP + 3D section)
//   k_fused     all of the above in one pass over the gradients
//
// Rows are read in 16-byte groups on the global 16-byte grid (4 fp32 or 8 fp16 elements);
// groups that stick out of a chunk are masked element by element.  A row starts on a
// 16-byte boundary, so a whole group never leaves the caller's buffer.
#include <cuda_runtime.h>

#include <climits>
#include <mutex>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {

__device__ unsigned g_error_word;

__device__ __forceinline__ void raise_error(unsigned bit) { atomicOr(&g_error_word, bit); }

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s for a bulk copy that takes microseconds

// Bulk-copy wait settings; changed only by the fault-injection hook of the tests.
__device__ uint64_t g_wait_limit_ns = kWaitLimitNs;
__device__ uint32_t g_stall_extra_tx = 0;
constexpr int kThreads = 256;

// Chunk j is used only if 0 <= lo <= hi <= min(rank_stride, offsets[num_chunks]): then every
// row access stays inside its row and every output index inside out[0, offsets[num_chunks]),
// whatever the rest of the table holds.
__device__ __forceinline__ bool chunk_bounds(const int64_t* offsets, int64_t j, int64_t num_chunks,
                                             int64_t rank_stride, int64_t* lo, int64_t* hi) {
    *lo = __ldg(offsets + j);
    *hi = __ldg(offsets + j + 1);
    const int64_t end = __ldg(offsets + num_chunks);
    return *lo >= 0 && *lo <= *hi && *hi <= rank_stride && *hi <= end && (*hi - *lo) <= INT_MAX;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* scratch) {
    v = __reduce_max_sync(0xffffffffu, v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    uint32_t r = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) r = max(r, scratch[w]);
    return r;
}

template <int DT>
__device__ __forceinline__ float raw_abs_to_float(uint32_t bits) {
    if (DT == 0) return __uint_as_float(bits);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

template <int DT>
__device__ __forceinline__ bool raw_abs_nonfinite(uint32_t bits) {
    return DT == 0 ? bits >= 0x7f800000u : bits >= 0x7c00u;
}

// Absmax of g = x * inv over a chunk from the absmax of |x|: rounding is monotone and odd,
// so max |fl(x * inv)| = fl(max|x| * inv).
template <int DT>
__device__ __forceinline__ float chunk_absmax(uint32_t raw_bits, const QuantArgs& a, bool* nonfinite) {
    float m = raw_abs_to_float<DT>(raw_bits);
    if (a.scaled) m = __fmul_rn(m, a.inv);
    *nonfinite = raw_abs_nonfinite<DT>(raw_bits) || !(fabsf(m) <= 3.40282347e38f);
    return m;
}

__device__ __forceinline__ float mean_of(float acc, int W, float invW, bool pow2) {
    // For W a power of two, acc * (1/W) and acc / W round the same exact value.
    return pow2 ? __fmul_rn(acc, invW) : __fdiv_rn(acc, static_cast<float>(W));
}

// ===================================================================== chunk plan

struct PlanArgs {
    PlanBucket b[kPlanBucketsPerLaunch];
    int nb;
    int64_t* offsets;
    int64_t total_chunks;
    int64_t end_elem;
};

__global__ void k_plan(const PlanArgs a) {
    if (static_cast<int>(blockIdx.x) < a.nb) {
        const PlanBucket pb = a.b[blockIdx.x];
        for (int64_t j = threadIdx.x; j < pb.count; j += blockDim.x)
            a.offsets[pb.chunk_start + j] = pb.elem_start + j * pb.piece;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.total_chunks >= 0) a.offsets[a.total_chunks] = a.end_elem;
}

cudaError_t launch_plan(const PlanBucket* buckets, int nb, int64_t* d_offsets, int64_t total_chunks,
                        int64_t end_elem, cudaStream_t stream) {
    PlanArgs a;
    for (int i = 0; i < nb; ++i) a.b[i] = buckets[i];
    a.nb = nb;
    a.offsets = d_offsets;
    a.total_chunks = total_chunks;
    a.end_elem = end_elem;
    k_plan<<<nb > 0 ? nb : 1, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

// ===================================================================== unfused quantise

// One CTA per (chunk, rank).  Pass 1 reads the chunk for its absmax; pass 2 reads it again
// (from L2: a chunk is at most a few hundred KB) and writes the codes.
template <int DT>
__global__ void __launch_bounds__(kThreads) k_quantize(const QuantArgs a, int8_t* codes, float* scales) {
    constexpr int VEC = DT == 0 ? 4 : 8;
    constexpr int EB = DT == 0 ? 4 : 2;
    __shared__ uint32_t red[kThreads / 32];
    const int64_t j = blockIdx.x;
    const int r = blockIdx.y;
    int64_t lo, hi;
    if (!chunk_bounds(a.offsets, j, a.num_chunks, a.rank_stride, &lo, &hi)) {
        if (threadIdx.x == 0 && r == 0) raise_error(kErrBadTable);
        return;
    }
    const char* row = static_cast<const char*>(a.grads) + static_cast<int64_t>(r) * a.rank_stride * EB;
    const int64_t g0 = lo / VEC, g1 = hi > lo ? (hi + VEC - 1) / VEC : g0;

    uint32_t mx = 0;
    for (int64_t g = g0 + threadIdx.x; g < g1; g += blockDim.x) {
        const V16 v = ld_global_nc_v16(row + g * 16);
        const int64_t e0 = g * VEC;
        if (e0 >= lo && e0 + VEC <= hi) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) mx = max(mx, group_abs_bits<DT>(v, e));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (e0 + e >= lo && e0 + e < hi) mx = max(mx, group_abs_bits<DT>(v, e));
        }
    }
    mx = block_max_u32(mx, red);
    bool nonfinite;
    const float m = chunk_absmax<DT>(mx, a, &nonfinite);
    const ScaleQ sq = make_scale(m);
    if (threadIdx.x == 0) {
        scales[static_cast<int64_t>(r) * a.num_chunks + j] = sq.s;
        if (nonfinite) raise_error(kErrNonfinite);
    }

    int8_t* crow = codes + static_cast<int64_t>(r) * a.rank_stride;
    for (int64_t g = g0 + threadIdx.x; g < g1; g += blockDim.x) {
        const V16 v = ld_global_nc_v16(row + g * 16);
        const int64_t e0 = g * VEC;
        uint32_t packed[VEC / 4];
#pragma unroll
        for (int k = 0; k < VEC / 4; ++k) packed[k] = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float x = group_elem<DT>(v, e);
            if (a.scaled) x = __fmul_rn(x, a.inv);
            packed[e >> 2] |= code_byte(quant_u(x, sq)) << (8 * (e & 3));
        }
        if (e0 >= lo && e0 + VEC <= hi) {
            if (VEC == 4) {
                *reinterpret_cast<uint32_t*>(crow + e0) = packed[0];
            } else {
                *reinterpret_cast<uint2*>(crow + e0) = make_uint2(packed[0], packed[VEC / 4 - 1]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (e0 + e >= lo && e0 + e < hi)
                    crow[e0 + e] = static_cast<int8_t>((packed[e >> 2] >> (8 * (e & 3))) & 0xffu);
        }
    }
}

cudaError_t launch_quantize(const QuantArgs& a, int8_t* codes, float* scales, cudaStream_t stream) {
    if (a.num_chunks > INT_MAX) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(a.num_chunks), static_cast<unsigned>(a.W));
    if (a.dt == 0)
        k_quantize<0><<<grid, kThreads, 0, stream>>>(a, codes, scales);
    else
        k_quantize<1><<<grid, kThreads, 0, stream>>>(a, codes, scales);
    return cudaGetLastError();
}

// ===================================================================== unfused reduce

// Index of element i's segment in torch.chunk(chunk, W): pieces of seg = ceil(len / W).
__device__ __forceinline__ int segment_of(int64_t i, int64_t lo, uint32_t seg) {
    return static_cast<int>(static_cast<uint32_t>(i - lo) / seg);
}

__device__ __forceinline__ float code_to_float(uint32_t word, int e) {
    return static_cast<float>(static_cast<int8_t>((word >> (8 * e)) & 0xffu));
}

constexpr int kReducePieces = 8;

// One CTA per (chunk, piece of the chunk); a thread sums 4 consecutive elements.
__global__ void __launch_bounds__(kThreads) k_reduce(const int8_t* codes, const float* scales, int W,
                                                     int64_t rank_stride, const int64_t* offsets,
                                                     int64_t num_chunks, int order, float* out, float invW,
                                                     int w_pow2) {
    __shared__ float s_scale[kMaxRanks];
    const int64_t j = blockIdx.x;
    int64_t lo, hi;
    if (!chunk_bounds(offsets, j, num_chunks, rank_stride, &lo, &hi)) {
        if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(kErrBadTable);
        return;
    }
    if (threadIdx.x < W) s_scale[threadIdx.x] = scales[static_cast<int64_t>(threadIdx.x) * num_chunks + j];
    __syncthreads();
    if (hi == lo) return;
    const uint32_t seg = static_cast<uint32_t>((hi - lo + W - 1) / W);
    const int64_t g0 = lo / 4, g1 = (hi + 3) / 4, ng = g1 - g0;
    const int64_t per = (ng + gridDim.y - 1) / gridDim.y;
    const int64_t pg0 = g0 + min(ng, per * blockIdx.y), pg1 = g0 + min(ng, per * (blockIdx.y + 1));
    const bool pow2 = w_pow2 != 0;

    for (int64_t g = pg0 + threadIdx.x; g < pg1; g += blockDim.x) {
        const int64_t e0 = g * 4;
        const int64_t first = max(e0, lo), last = min(e0 + 3, hi - 1);
        float acc[4];
        auto deq = [&](int r, float* d) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(codes + static_cast<int64_t>(r) * rank_stride + e0);
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] = __fmul_rn(code_to_float(w, e), s_scale[r]);
        };
        const int t0 = segment_of(first, lo, seg), t1 = segment_of(last, lo, seg);
        if (order == 2) {
            TreeAcc tr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) tr[e].init();
            for (int r = 0; r < W; ++r) {
                float d[4];
                deq(r, d);
#pragma unroll
                for (int e = 0; e < 4; ++e) tr[e].push(d[e]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = tr[e].result();
        } else if (order == 0 || t0 == t1) {
            int r = order == 0 ? 0 : (t0 + 1 == W ? 0 : t0 + 1);
            deq(r, acc);
            for (int k = 1; k < W; ++k) {
                r = (r + 1 == W) ? 0 : r + 1;
                float d[4];
                deq(r, d);
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[e] = __fadd_rn(acc[e], d[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t i = e0 + e;
                if (i < lo || i >= hi) continue;
                const int t = segment_of(i, lo, seg);
                int r = (t + 1 == W) ? 0 : t + 1;
                float d[4];
                deq(r, d);
                float s = d[e];
                for (int k = 1; k < W; ++k) {
                    r = (r + 1 == W) ? 0 : r + 1;
                    deq(r, d);
                    s = __fadd_rn(s, d[e]);
                }
                acc[e] = s;
            }
        }
        if (e0 >= lo && e0 + 4 <= hi) {
            *reinterpret_cast<float4*>(out + e0) =
                make_float4(mean_of(acc[0], W, invW, pow2), mean_of(acc[1], W, invW, pow2),
                            mean_of(acc[2], W, invW, pow2), mean_of(acc[3], W, invW, pow2));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e0 + e >= lo && e0 + e < hi) out[e0 + e] = mean_of(acc[e], W, invW, pow2);
        }
    }
}

static bool is_pow2(int w) { return (w & (w - 1)) == 0; }

cudaError_t launch_reduce(const int8_t* codes, const float* scales, int W, int64_t rank_stride,
                          const int64_t* offsets, int64_t num_chunks, int order, float* out,
                          cudaStream_t stream) {
    if (num_chunks > INT_MAX) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(num_chunks), kReducePieces);
    k_reduce<<<grid, kThreads, 0, stream>>>(codes, scales, W, rank_stride, offsets, num_chunks, order, out,
                                            1.0f / static_cast<float>(W), is_pow2(W) ? 1 : 0);
    return cudaGetLastError();
}

// ===================================================================== fused kernel

struct FusedArgs {
    QuantArgs q;
    int order;
    float* out;
    int8_t* codes;     // may be null
    float* scales;     // may be null
    uint32_t row_cap;  // shared staging bytes per rank row (0: never stage)
    uint32_t P;        // CTAs per cluster (one cluster per chunk)
    float invW;
    int w_pow2;
};

// A cluster of P CTAs owns one chunk; CTA p owns slice p of it (P near-equal runs of
// 16-byte groups) for all W ranks.
//   1. The slice of every rank row is bulk-copied (TMA, one cp.async.bulk per row) into
//      shared memory, or, if it does not fit the staging rows, read from global twice.
//   2. Each CTA reduces the absmax of its slice per rank; the P partial maxima of a rank are
//      combined through distributed shared memory after a cluster barrier, so every CTA
//      holds the chunk's W scales.
//   3. Each thread takes 16-byte groups, quantises every rank's values, dequantises and sums
//      them in the requested order, and writes the mean (and, if asked, codes and scales).
template <int DT>
__global__ void __launch_bounds__(kThreads, 1) k_fused(const FusedArgs A) {
    constexpr int VEC = DT == 0 ? 4 : 8;
    constexpr int EB = DT == 0 ? 4 : 2;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ uint64_t bar;
    __shared__ uint32_t part[kMaxRanks];
    __shared__ ScaleQ sq[kMaxRanks];

    const int tid = threadIdx.x;
    const int W = A.q.W;
    const uint32_t P = A.P;
    const uint32_t crank = cluster_ctarank();
    const int64_t j = blockIdx.x / P;
    int64_t lo, hi;
    // The table entry is the same for every CTA of the cluster, so a bad chunk makes the
    // whole cluster leave here, before any cluster barrier.
    if (!chunk_bounds(A.q.offsets, j, A.q.num_chunks, A.q.rank_stride, &lo, &hi)) {
        if (tid == 0 && crank == 0) raise_error(kErrBadTable);
        return;
    }
    const int64_t ng = hi > lo ? (hi + VEC - 1) / VEC - lo / VEC : 0;
    const int64_t gs = (ng + P - 1) / P;
    const int64_t sg0 = lo / VEC + min(ng, gs * crank);
    const int64_t sg1 = lo / VEC + min(ng, gs * (crank + 1));
    const int64_t slo = max(lo, sg0 * VEC), shi = min(hi, sg1 * VEC);
    const uint32_t slice_bytes = static_cast<uint32_t>((sg1 - sg0) * 16);
    const bool staged = sg1 > sg0 && A.row_cap != 0 && slice_bytes <= A.row_cap;
    const char* grads = static_cast<const char*>(A.q.grads);
    const int64_t row_bytes = A.q.rank_stride * EB;

    if (tid < W) part[tid] = 0;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    const uint64_t wait_limit = g_wait_limit_ns;
    if (staged && tid == 0) {
        mbar_arrive_expect_tx(&bar, slice_bytes * static_cast<uint32_t>(W) + g_stall_extra_tx);
        for (int r = 0; r < W; ++r)
            bulk_copy_g2s(stage + static_cast<uint32_t>(r) * A.row_cap, grads + r * row_bytes + sg0 * 16, slice_bytes,
                          &bar);
    }
    bool copied = true;
    if (staged) {
        copied = mbar_wait_bounded(&bar, 0, wait_limit);
        if (!copied) raise_error(kErrTimeout);
    }
    auto load_group = [&](int r, int64_t g) -> V16 {
        if (staged) return ld_shared_v16(stage + static_cast<uint32_t>(r) * A.row_cap + (g - sg0) * 16);
        return ld_global_nc_v16(grads + r * row_bytes + g * 16);
    };

    // ---- absmax of the slice, per rank
    for (int r = 0; r < W; ++r) {
        uint32_t mx = 0;
        for (int64_t g = sg0 + tid; g < sg1; g += kThreads) {
            const V16 v = load_group(r, g);
            const int64_t e0 = g * VEC;
            if (e0 >= slo && e0 + VEC <= shi) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) mx = max(mx, group_abs_bits<DT>(v, e));
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (e0 + e >= slo && e0 + e < shi) mx = max(mx, group_abs_bits<DT>(v, e));
            }
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        if ((tid & 31) == 0 && mx != 0) atomicMax(&part[r], mx);
    }

    // ---- combine the P partial maxima through distributed shared memory
    cluster_arrive_release();
    cluster_wait_acquire();
    if (tid < W) {
        uint32_t mraw = 0;
        for (uint32_t c = 0; c < P; ++c) mraw = max(mraw, dsmem_load_u32(&part[tid], c));
        bool nonfinite;
        const float m = chunk_absmax<DT>(mraw, A.q, &nonfinite);
        sq[tid] = make_scale(m);
        if (crank == 0) {
            if (nonfinite) raise_error(kErrNonfinite);
            if (A.scales) A.scales[static_cast<int64_t>(tid) * A.q.num_chunks + j] = sq[tid].s;
        }
    }
    __syncthreads();
    cluster_arrive_release();  // this CTA is done reading its peers' partial maxima

    // ---- quantise, dequantise, sum over ranks, mean
    const uint32_t seg = hi > lo ? static_cast<uint32_t>((hi - lo + W - 1) / W) : 1u;
    const bool pow2 = A.w_pow2 != 0;
    const float inv = A.q.inv;
    const bool scaled = A.q.scaled != 0;
    for (int64_t g = sg0 + tid; g < sg1; g += kThreads) {
        const int64_t e0 = g * VEC;
        const bool full = e0 >= slo && e0 + VEC <= shi;
        // Dequantised values of rank r for this group; writes rank r's codes when asked.
        auto deq = [&](int r, float* d, bool write_codes) {
            const V16 v = load_group(r, g);
            const ScaleQ s = sq[r];
            uint32_t packed[VEC / 4];
#pragma unroll
            for (int k = 0; k < VEC / 4; ++k) packed[k] = 0;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float x = group_elem<DT>(v, e);
                if (scaled) x = __fmul_rn(x, inv);
                const float u = quant_u(x, s);
                packed[e >> 2] |= code_byte(u) << (8 * (e & 3));
                d[e] = __fmul_rn(code_value(u), s.s);
            }
            if (write_codes && A.codes) {
                int8_t* crow = A.codes + static_cast<int64_t>(r) * A.q.rank_stride;
                if (full) {
                    if (VEC == 4) {
                        *reinterpret_cast<uint32_t*>(crow + e0) = packed[0];
                    } else {
                        *reinterpret_cast<uint2*>(crow + e0) = make_uint2(packed[0], packed[VEC / 4 - 1]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if (e0 + e >= slo && e0 + e < shi)
                            crow[e0 + e] = static_cast<int8_t>((packed[e >> 2] >> (8 * (e & 3))) & 0xffu);
                }
            }
        };
        float acc[VEC];
        const int64_t first = max(e0, slo), last = min(e0 + VEC - 1, shi - 1);
        const int t0 = segment_of(first, lo, seg), t1 = segment_of(last, lo, seg);
        if (A.order == 2) {
            TreeAcc tr[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) tr[e].init();
            for (int r = 0; r < W; ++r) {
                float d[VEC];
                deq(r, d, true);
#pragma unroll
                for (int e = 0; e < VEC; ++e) tr[e].push(d[e]);
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = tr[e].result();
        } else if (A.order == 0 || t0 == t1) {
            int r = A.order == 0 ? 0 : (t0 + 1 == W ? 0 : t0 + 1);
            deq(r, acc, true);
            for (int k = 1; k < W; ++k) {
                r = (r + 1 == W) ? 0 : r + 1;
                float d[VEC];
                deq(r, d, true);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], d[e]);
            }
        } else {
            // The group straddles a ring-segment boundary: each element has its own order.
            bool codes_done = false;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int64_t i = e0 + e;
                acc[e] = 0.0f;
                if (i < slo || i >= shi) continue;
                const int t = segment_of(i, lo, seg);
                int r = (t + 1 == W) ? 0 : t + 1;
                float d[VEC];
                deq(r, d, !codes_done);
                float s = d[e];
                for (int k = 1; k < W; ++k) {
                    r = (r + 1 == W) ? 0 : r + 1;
                    deq(r, d, !codes_done);
                    s = __fadd_rn(s, d[e]);
                }
                codes_done = true;
                acc[e] = s;
            }
        }
        if (full) {
#pragma unroll
            for (int k = 0; k < VEC / 4; ++k)
                *reinterpret_cast<float4*>(A.out + e0 + 4 * k) = make_float4(
                    mean_of(acc[4 * k + 0], W, A.invW, pow2), mean_of(acc[4 * k + 1], W, A.invW, pow2),
                    mean_of(acc[4 * k + 2], W, A.invW, pow2), mean_of(acc[4 * k + 3], W, A.invW, pow2));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (e0 + e >= slo && e0 + e < shi) A.out[e0 + e] = mean_of(acc[e], W, A.invW, pow2);
        }
    }

    cluster_wait_acquire();  // no CTA leaves while a peer may still read its partial maxima
    if (staged && !copied) mbar_wait_bounded(&bar, 0, wait_limit);  // let late copies land
}

// Per-rank staging capacity for a cluster of P: chunks up to 144 KiB per rank (dynamic_chunk
// pieces are 128 KiB plus a remainder share; buckets of 1 MiB and more stay within 144 KiB),
// split into P slices, plus one group for a slice that starts mid-group.
static uint32_t staging_row_cap(uint32_t P) {
    const uint32_t groups = (147456u / 16u + 2u + P - 1u) / P;
    return groups * 16u;
}

static constexpr size_t kMaxStagingBytes = 200 * 1024;

struct DeviceInit {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    bool cluster16 = false;
};
static DeviceInit g_dev_init[64];

template <int DT>
static cudaError_t init_fused_kernel(bool* cluster16) {
    cudaError_t e = cudaFuncSetAttribute(k_fused<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMaxStagingBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_fused<DT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *cluster16 = false;
        return cudaSuccess;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 8 * staging_row_cap(16);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k_fused<DT>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    *cluster16 = n > 0;
    return cudaSuccess;
}

cudaError_t launch_fused(const QuantArgs& a, int order, float* out, int8_t* codes, float* scales,
                         cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInit& di = g_dev_init[dev];
    std::call_once(di.once, [&] {
        bool c16a = false, c16b = false;
        di.err = init_fused_kernel<0>(&c16a);
        if (di.err == cudaSuccess) di.err = init_fused_kernel<1>(&c16b);
        di.cluster16 = c16a && c16b;
    });
    if (di.err != cudaSuccess) return di.err;

    const uint32_t pmax = di.cluster16 ? 16u : 8u;
    uint32_t P = 2;
    while (P < pmax && P < 2u * static_cast<uint32_t>(a.W)) P *= 2;
    uint32_t row_cap = staging_row_cap(P);
    size_t smem = static_cast<size_t>(a.W) * row_cap;
    if (smem > kMaxStagingBytes) {
        row_cap = 0;
        smem = 0;
    }
    const int64_t grid = a.num_chunks * P;
    if (grid > INT_MAX) return cudaErrorInvalidValue;

    FusedArgs A;
    A.q = a;
    A.order = order;
    A.out = out;
    A.codes = codes;
    A.scales = scales;
    A.row_cap = row_cap;
    A.P = P;
    A.invW = 1.0f / static_cast<float>(a.W);
    A.w_pow2 = is_pow2(a.W) ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.dt == 0) return cudaLaunchKernelEx(&cfg, k_fused<0>, A);
    return cudaLaunchKernelEx(&cfg, k_fused<1>, A);
}

// ===================================================================== error word

cudaError_t set_copy_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    cudaError_t e = cudaMemcpyToSymbol(g_stall_extra_tx, &extra_bytes, sizeof(extra_bytes));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_wait_limit_ns, &limit_ns, sizeof(limit_ns));
}

cudaError_t read_and_clear_error_word(unsigned* word, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned w = 0;
    e = cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    *word = w;
    return cudaSuccess;
}

}  // namespace gq
