// gq_fused.cuh -- the fused quantise + W-way reduce kernels (one cluster of CTAs per chunk).
//
// Included by gq_fused_f32.cu / gq_fused_f16.cu (and by gq_stream.cuh for shared helpers).
// Each including translation unit gets its own device error word and wait settings (the
// library is linked without relocatable device code); gq_get_error reads all of them.
//
// Method: "pipelined HCCL AllReduce" article (bjdmk.com.cn/news/6235379), §2.1 chunks,
// §2.2.1 quantize_gradient and INT8_ALLREDUCE, §3.1 one SUM all_reduce per chunk, §6.1
// unscale before quantising; mean over the group as in the "torchtitan-npu 3D parallel"
// article (framerc.cn/news/2545645), AMP + 3D section.
//
// k_fused: one chunk per thread-block cluster, CTA p of the cluster owning slice p.  For W other
// than 8 the slice is bulk-copied into shared memory (TMA) when it fits; for W = 8 (compiled for
// that W), and for slices that do not fit, it is read twice from global memory, the second time
// from L2, with one CTA per ring segment: on GB300 that form ran the 25 MiB W = 8 bucket in
// 92 us, against 164 us staged (clusters of 16), its CTAs being small enough for three to share
// an SM.
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <mutex>

#include "gq_device.cuh"
#include "gq_internal.h"

namespace gq {
namespace fused {

static __device__ unsigned g_error_word;
static __device__ uint64_t g_wait_limit_ns = 2000000000ull;  // 2 s for copies that take microseconds
static __device__ uint32_t g_stall_extra_tx = 0;              // set only by the fault-injection hook

__device__ __forceinline__ void raise_error(unsigned bit) { atomicOr(&g_error_word, bit); }

__device__ __forceinline__ int ld_volatile_shared_int(const int* p) { return *static_cast<const volatile int*>(p); }
__device__ __forceinline__ void st_volatile_shared_int(int* p, int v) { *static_cast<volatile int*>(p) = v; }

constexpr int kThreads = 256;     // k_fused
constexpr int kOrderSeq = 0, kOrderRing = 1, kOrderTree = 2;

struct Args {
    QuantArgs q;
    int order;
    float* out;
    int8_t* codes;         // may be null
    float* scales;         // may be null
    uint32_t row_cap;      // shared staging bytes per rank row (0: never stage)
    uint32_t P;            // CTAs per cluster (one cluster per chunk)
    float invW;
    int w_pow2;
    int ring_split;        // RING order and P a multiple of W: slices follow ring segments
};

// Chunk j is used only if 0 <= lo <= hi <= min(rank_stride, offsets[num_chunks]): then every row
// access stays inside its row and every output index inside out[0, offsets[num_chunks]).
__device__ __forceinline__ bool chunk_bounds(const int64_t* offsets, int64_t j, int64_t num_chunks,
                                             int64_t rank_stride, int64_t* lo, int64_t* hi) {
    *lo = __ldg(offsets + j);
    *hi = __ldg(offsets + j + 1);
    const int64_t end = __ldg(offsets + num_chunks);
    return *lo >= 0 && *lo <= *hi && *hi <= rank_stride && *hi <= end && (*hi - *lo) <= INT_MAX;
}

__device__ __forceinline__ float mean_of(float acc, int W, float invW, bool pow2) {
    // For W a power of two, acc * (1/W) and acc / W round the same exact value.
    return pow2 ? __fmul_rn(acc, invW) : __fdiv_rn(acc, static_cast<float>(W));
}

// Index of element i's piece in torch.chunk(chunk, W): pieces of seg = ceil(len / W).
__device__ __forceinline__ int segment_of(int64_t i, int64_t lo, uint32_t seg) {
    return static_cast<int>(static_cast<uint32_t>(i - lo) / seg);
}

struct Slice {
    int64_t g0, g1;    // 16-byte groups [g0, g1) on the global grid
    int64_t lo, hi;    // elements [lo, hi) this CTA owns
};

// CTA `c` of P takes a near-equal run of the groups of [a, b).
template <int VEC>
__device__ __forceinline__ Slice split_range(int64_t a, int64_t b, uint32_t c, uint32_t P) {
    Slice s;
    if (b <= a) {
        s.g0 = s.g1 = a / VEC;
        s.lo = s.hi = a;
        return s;
    }
    const int64_t G0 = a / VEC, ng = (b + VEC - 1) / VEC - G0;
    const int64_t gs = (ng + P - 1) / P;
    s.g0 = G0 + min(ng, gs * c);
    s.g1 = G0 + min(ng, gs * (c + 1));
    s.lo = max(a, s.g0 * VEC);
    s.hi = min(b, s.g1 * VEC);
    if (s.hi < s.lo) s.hi = s.lo;
    return s;
}

// The slice of CTA `crank` in chunk [lo, hi): with ring_split, P / W CTAs share each ring segment.
template <int VEC>
__device__ __forceinline__ Slice cta_slice(const Args& A, int W, int64_t lo, int64_t hi, uint32_t seg,
                                           uint32_t crank) {
    if (A.ring_split) {
        const uint32_t sub = A.P / static_cast<uint32_t>(W);
        const int64_t t = crank / sub;
        const int64_t a = min(hi, lo + t * seg), b = min(hi, lo + (t + 1) * seg);
        return split_range<VEC>(a, b, crank % sub, sub);
    }
    return split_range<VEC>(lo, hi, crank, A.P);
}

// One element-rank of the fast path: c = inv * rcp(s) folded, so t = x * c is within 2^-15 of
// g / s (g = fl(x * inv)); when t is not within 2^-14 of a half-integer, rne(t) = rne(fl(g / s)).
// Returns u = M + rne(t); sets `near` when the exact division must decide.
__device__ __forceinline__ float fast_u(float x, float c, bool& near) {
    const float t = __fmul_rn(x, c);
    const float u = __fadd_rn(t, kMagic);
    const float d = __fsub_rn(t, __fsub_rn(u, kMagic));
    near |= fabsf(d) > kNearTie;
    return u;
}

// The exact decision for one element-rank (any scale mode).
__device__ __forceinline__ float exact_u(float x, float inv, bool scaled, const ScaleQ& sq) {
    const float g = scaled ? __fmul_rn(x, inv) : x;
    return quant_u(g, sq);
}

template <int VEC>
__device__ __forceinline__ void store_codes(int8_t* crow, int64_t e0, bool full, int64_t lo, int64_t hi,
                                            const uint32_t (&packed)[VEC / 4]) {
    if (full) {
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

template <int VEC>
__device__ __forceinline__ void store_out(float* out, int64_t e0, bool full, int64_t lo, int64_t hi,
                                          const float (&v)[VEC]) {
    if (full) {
#pragma unroll
        for (int k = 0; k < VEC / 4; ++k)
            *reinterpret_cast<float4*>(out + e0 + 4 * k) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (e0 + e >= lo && e0 + e < hi) out[e0 + e] = v[e];
    }
}

// Per-CTA scale tables, indexed by the row that holds a rank (row k holds rank (k + rot) % W).
struct RowScales {
    const float* s;       // scale
    const float* c;       // inv * rcp(scale), 0 for a zero scale
    const int* rank;      // rank held in row k
    const ScaleQ* sq;     // scales by rank (exact path)
};

// Fast path for one 16-byte group: every scale normal or zero and every element of the group
// starting its sum at the rank in row 0.  Per element-rank: t = x * c, u = t + M, the near-tie
// test, dq = (u - M) * s, one addition.  If any quotient lay within 2^-14 of a half-integer the
// group is redone with the exact IEEE division deciding every element-rank.
// load(k) returns the group of row k.
template <int DT, int WC, bool CODES, bool TREE, class Load>
__device__ __forceinline__ void fast_group(Load load, int W, const RowScales& rs, int64_t e0, bool full,
                                           int64_t slo, int64_t shi, const Args& A, bool pow2) {
    constexpr int VEC = DT == 0 ? 4 : 8;
    const float inv = A.q.inv;
    const bool scaled = A.q.scaled != 0;
    const int64_t cstride = A.q.rank_stride;
    float acc[VEC];
    TreeAcc tr[TREE ? VEC : 1];
    bool near = false;
    const int KW = WC ? WC : W;
#pragma unroll
    for (int redo = 0; redo < 2; ++redo) {
        if (TREE) {
#pragma unroll
            for (int e = 0; e < (TREE ? VEC : 1); ++e) tr[e].init();
        }
#pragma unroll
        for (int k = 0; k < KW; ++k) {
            const V16 v = load(k);
            uint32_t packed[VEC / 4];
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) packed[q] = 0;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float x = group_elem<DT>(v, e);
                const float u = redo == 0 ? fast_u(x, rs.c[k], near) : exact_u(x, inv, scaled, rs.sq[rs.rank[k]]);
                const float dq = __fmul_rn(code_value(u), rs.s[k]);
                if (TREE) {
                    tr[e % (TREE ? VEC : 1)].push(dq);
                } else {
                    acc[e] = k == 0 ? dq : __fadd_rn(acc[e], dq);
                }
                if (CODES) packed[e >> 2] |= code_byte(u) << (8 * (e & 3));
            }
            if (CODES && A.codes)
                store_codes<VEC>(A.codes + static_cast<int64_t>(rs.rank[k]) * cstride, e0, full, slo, shi, packed);
        }
        if (!near) break;
    }
    float o[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[e] = mean_of(TREE ? tr[e % (TREE ? VEC : 1)].result() : acc[e], W, A.invW, pow2);
    store_out<VEC>(A.out, e0, full, slo, shi, o);
}

// General path for one group: any scale (subnormal scales divide and clamp everywhere), and a
// ring group that spans two segments (each element gets its own start rank).
// load_rank(r) returns the group of rank r.
template <int DT, bool CODES, class LoadRank>
__device__ __forceinline__ void general_group(LoadRank load_rank, int W, const ScaleQ* sq, int64_t lo, uint32_t seg,
                                              int64_t e0, bool full, int64_t slo, int64_t shi, const Args& A,
                                              bool pow2) {
    constexpr int VEC = DT == 0 ? 4 : 8;
    const float inv = A.q.inv;
    const bool scaled = A.q.scaled != 0;
    const int64_t cstride = A.q.rank_stride;
    auto deq = [&](int r, float* d, bool write_codes) {
        const V16 v = load_rank(r);
        const ScaleQ s = sq[r];
        uint32_t packed[VEC / 4];
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) packed[q] = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float u = exact_u(group_elem<DT>(v, e), inv, scaled, s);
            packed[e >> 2] |= code_byte(u) << (8 * (e & 3));
            d[e] = __fmul_rn(code_value(u), s.s);
        }
        if (CODES && write_codes && A.codes)
            store_codes<VEC>(A.codes + static_cast<int64_t>(r) * cstride, e0, full, slo, shi, packed);
    };
    float acc[VEC];
    const int64_t first = max(e0, slo), last = min(e0 + VEC - 1, shi - 1);
    const int t0 = segment_of(first, lo, seg), t1 = segment_of(last, lo, seg);
    if (A.order == kOrderTree) {
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
    } else if (A.order == kOrderSeq || t0 == t1) {
        int r = A.order == kOrderSeq ? 0 : (t0 + 1 == W ? 0 : t0 + 1);
        deq(r, acc, true);
        for (int k = 1; k < W; ++k) {
            r = (r + 1 == W) ? 0 : r + 1;
            float d[VEC];
            deq(r, d, true);
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = __fadd_rn(acc[e], d[e]);
        }
    } else {
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
    float o[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) o[e] = mean_of(acc[e], W, A.invW, pow2);
    store_out<VEC>(A.out, e0, full, slo, shi, o);
}

// Absmax over the elements of group v that lie in [slo, shi), as a |x| bit pattern (integer
// order equals float order for non-negative values; NaN orders above +Inf).
template <int DT>
__device__ __forceinline__ uint32_t group_absmax(const V16& v, int64_t e0, bool full, int64_t slo, int64_t shi,
                                                 uint32_t m) {
    constexpr int VEC = DT == 0 ? 4 : 8;
#ifdef GQ_NO_FMAX_ABSMAX
    if (false) {
#else
    if (DT == 0 && full) {
#endif
        float f = __uint_as_float(m);
#pragma unroll
        for (int e = 0; e < 4; ++e) f = absmax_acc(f, __uint_as_float(v.w[e]));
        return __float_as_uint(f) & 0x7fffffffu;
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        if (full || (e0 + e >= slo && e0 + e < shi)) m = max(m, group_abs_bits<DT>(v, e));
    return m;
}

// Cluster-wide absmax exchange and scale setup, shared by both kernels.  On entry lmax[k] holds
// this CTA's partial max of the rank in row k and part[] is zero in every CTA (guaranteed by a
// cluster barrier the caller arrived at after zeroing and waits on here).  On exit every CTA
// holds the chunk's W scales; returns whether all of them are normal or zero.
template <int DT>
__device__ __forceinline__ bool exchange_scales(const Args& A, int W, uint32_t P, uint32_t crank, int64_t j,
                                                uint32_t* part, const uint32_t* lmax, const int* row_rank,
                                                ScaleQ* sq, float* row_s, float* row_c) {
    const int tid = threadIdx.x;
    __syncthreads();
    cluster_wait_acquire();  // every peer's part[] is zeroed
    // this CTA's partials into every peer: one remote atomic max per thread
    for (int t = tid; t < W * static_cast<int>(P); t += blockDim.x) {
        const int k = t % W;
        const uint32_t m = lmax[k];
        if (m != 0) dsmem_red_max_u32(&part[row_rank[k]], static_cast<uint32_t>(t / W), m);
    }
    cluster_arrive_release();
    cluster_wait_acquire();  // every CTA's part[r] is the chunk max; no peer touches this CTA again

    const float inv = A.q.inv;
    const bool scaled = A.q.scaled != 0;
    bool not_subnormal = true;
    if (tid < W) {
        const uint32_t mraw = part[tid];
        float m = DT == 0 ? __uint_as_float(mraw) : __half2float(__ushort_as_half(static_cast<unsigned short>(mraw)));
        if (scaled) m = __fmul_rn(m, inv);  // max|fl(x*inv)| = fl(max|x| * inv): rounding is monotone
        const bool nonfinite = (DT == 0 ? mraw >= 0x7f800000u : mraw >= 0x7c00u) || !(fabsf(m) <= 3.40282347e38f);
        const ScaleQ s = make_scale(m);
        sq[tid] = s;
        not_subnormal = s.mode != 2;
        if (crank == 0) {
            if (nonfinite) {
                raise_error(kErrNonfinite);
                if (A.q.found_inf) *A.q.found_inf = 1.0f;
            }
            if (A.scales) A.scales[static_cast<int64_t>(tid) * A.q.num_chunks + j] = s.s;
        }
    }
    const bool fast = __syncthreads_and(not_subnormal) != 0;
    if (tid < W) {
        const ScaleQ s = sq[row_rank[tid]];
        row_s[tid] = s.s;
        row_c[tid] = s.mode == 1 ? (scaled ? __fmul_rn(inv, s.rcp) : s.rcp) : 0.0f;
    }
    __syncthreads();
    return fast;
}

#ifndef GQ_FUSED_MIN_CTAS_F32
#define GQ_FUSED_MIN_CTAS_F32 3
#endif
#ifndef GQ_FUSED_MIN_CTAS_F16
#define GQ_FUSED_MIN_CTAS_F16 1
#endif

// ---------------------------------------------------------------------------------- k_fused
// Staged (TMA bulk copies into shared memory) or, for slices that do not fit, read twice from
// global memory.
//   1. One thread bulk-copies each rank's slice into a shared-memory row (cp.async.bulk, mbarrier
//      transaction count, bounded wait); row k holds rank (k + rot) % W, rot being the CTA's ring
//      start, so the sum runs over rows 0..W-1.
//   2. Per-rank absmax of the slice, combined across the cluster (exchange_scales).
//   3. Each thread takes 16-byte groups: quantise, dequantise, sum, store the mean.
template <int DT, int WC, bool CODES>
__global__ void __launch_bounds__(kThreads, DT == 0 ? GQ_FUSED_MIN_CTAS_F32 : GQ_FUSED_MIN_CTAS_F16)
    k_fused(const Args A) {
    constexpr int VEC = DT == 0 ? 4 : 8;
    constexpr int EB = DT == 0 ? 4 : 2;
    extern __shared__ __align__(128) unsigned char stage[];
    __shared__ uint64_t bar;
    __shared__ uint32_t part[kMaxRanks];      // absmax partials, by rank
    __shared__ uint32_t lmax[kMaxRanks];      // this CTA's absmax partial of the rank in row k
    __shared__ ScaleQ sq[kMaxRanks];          // scales, by rank
    __shared__ float row_s[kMaxRanks];
    __shared__ float row_c[kMaxRanks];
    __shared__ int row_rank[kMaxRanks];

    const int tid = threadIdx.x;
    const int W = WC ? WC : A.q.W;
    const uint32_t P = A.P;
    const uint32_t crank = cluster_ctarank();
    const int64_t j = blockIdx.x / P;
    int64_t lo, hi;
    // The table entry is the same for every CTA of the cluster, so a bad chunk makes the whole
    // cluster leave here, before any cluster barrier.
    if (!chunk_bounds(A.q.offsets, j, A.q.num_chunks, A.q.rank_stride, &lo, &hi)) {
        if (tid == 0 && crank == 0) raise_error(kErrBadTable);
        return;
    }
    const uint32_t seg = hi > lo ? static_cast<uint32_t>((hi - lo + W - 1) / W) : 1u;
    const Slice sl = cta_slice<VEC>(A, W, lo, hi, seg, crank);
    bool uniform = true;  // every element of the slice starts its ring sum at the same rank
    int rot = 0;
    if (A.order == kOrderRing && sl.hi > sl.lo) {
        const int t0 = segment_of(sl.lo, lo, seg), t1 = segment_of(sl.hi - 1, lo, seg);
        uniform = t0 == t1;
        if (uniform) rot = (t0 + 1 == W) ? 0 : t0 + 1;
    }
    const uint32_t slice_bytes = static_cast<uint32_t>((sl.g1 - sl.g0) * 16);
    const bool staged = sl.g1 > sl.g0 && A.row_cap != 0 && slice_bytes <= A.row_cap;
    const char* grads = static_cast<const char*>(A.q.grads);
    const int64_t row_bytes = A.q.rank_stride * EB;
    const uint64_t wait_limit = g_wait_limit_ns;

    if (tid < W) {
        part[tid] = 0;
        lmax[tid] = 0;
        row_rank[tid] = (tid + rot) % W;
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // Peers will max their partials into part[]: it must be zero in every CTA before any of them
    // does.  This barrier's wait (in exchange_scales) comes after the copy wait.
    cluster_arrive_release();
    if (staged && tid == 0) {
        mbar_arrive_expect_tx(&bar, slice_bytes * static_cast<uint32_t>(W) + g_stall_extra_tx);
        for (int k = 0; k < W; ++k)
            bulk_copy_g2s(stage + static_cast<uint32_t>(k) * A.row_cap, grads + row_rank[k] * row_bytes + sl.g0 * 16,
                          slice_bytes, &bar);
    }
    bool copied = true;
    if (staged) {
        copied = mbar_wait_bounded(&bar, 0, wait_limit);
        if (!copied) raise_error(kErrTimeout);
    }
    auto load_row = [&](int k, int64_t g) -> V16 {
        if (staged) return ld_shared_v16(stage + static_cast<uint32_t>(k) * A.row_cap + (g - sl.g0) * 16);
        return ld_global_nc_v16(grads + row_rank[k] * row_bytes + g * 16);
    };

    // ---- absmax of the slice per rank (integer max of |x| bit patterns)
    if (WC) {
        constexpr int NR = WC ? WC : 1;
        uint32_t mx[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) mx[k] = 0;
        for (int64_t g = sl.g0 + tid; g < sl.g1; g += kThreads) {
            const int64_t e0 = g * VEC;
            const bool full = e0 >= sl.lo && e0 + VEC <= sl.hi;
            V16 v[NR];
#pragma unroll
            for (int k = 0; k < NR; ++k) v[k] = load_row(k, g);
#pragma unroll
            for (int k = 0; k < NR; ++k) mx[k] = group_absmax<DT>(v[k], e0, full, sl.lo, sl.hi, mx[k]);
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, mx[k]);
            if ((tid & 31) == 0 && m != 0) atomicMax(&lmax[k], m);
        }
    } else {
        for (int k = 0; k < W; ++k) {
            uint32_t mx = 0;
            for (int64_t g = sl.g0 + tid; g < sl.g1; g += kThreads) {
                const int64_t e0 = g * VEC;
                mx = group_absmax<DT>(load_row(k, g), e0, e0 >= sl.lo && e0 + VEC <= sl.hi, sl.lo, sl.hi, mx);
            }
            mx = __reduce_max_sync(0xffffffffu, mx);
            if ((tid & 31) == 0 && mx != 0) atomicMax(&lmax[k], mx);
        }
    }

    const bool fast = exchange_scales<DT>(A, W, P, crank, j, part, lmax, row_rank, sq, row_s, row_c);
    const RowScales rs{row_s, row_c, row_rank, sq};

    // ---- quantise, dequantise, sum over ranks, mean
    const bool pow2 = A.w_pow2 != 0;
    for (int64_t g = sl.g0 + tid; g < sl.g1; g += kThreads) {
        const int64_t e0 = g * VEC;
        const bool full = e0 >= sl.lo && e0 + VEC <= sl.hi;
        if (fast && uniform) {
            auto ld = [&](int k) { return load_row(k, g); };
            if (A.order == kOrderTree)
                fast_group<DT, WC, CODES, true>(ld, W, rs, e0, full, sl.lo, sl.hi, A, pow2);
            else
                fast_group<DT, WC, CODES, false>(ld, W, rs, e0, full, sl.lo, sl.hi, A, pow2);
        } else {
            auto ldr = [&](int r) { return load_row(r >= rot ? r - rot : r - rot + W, g); };
            general_group<DT, CODES>(ldr, W, sq, lo, seg, e0, full, sl.lo, sl.hi, A, pow2);
        }
    }
    if (staged && !copied) mbar_wait_bounded(&bar, 0, wait_limit);  // let late copies land
}

// Per-rank staging capacity for a cluster of P: chunks up to 144 KiB per rank (dynamic_chunk
// pieces are 128 KiB plus a share of the remainder, within 144 KiB for buckets of 1 MiB and
// more), split P ways, plus room for slices that start and end mid-group.
inline uint32_t staging_row_cap(uint32_t P) { return 16u * ((147456u / 16u + P - 1u) / P + 3u); }

#ifndef GQ_FUSED_MAX_STAGING_BYTES
#define GQ_FUSED_MAX_STAGING_BYTES (200 * 1024)
#endif
// Shared memory a CTA may use for staging rows; above it (or at 0) every chunk is read twice
// from global memory instead.
constexpr size_t kMaxStagingBytes = GQ_FUSED_MAX_STAGING_BYTES;

template <int DT, int WC, bool CODES>
inline cudaError_t set_attrs() {
    cudaError_t e = cudaFuncSetAttribute(k_fused<DT, WC, CODES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMaxStagingBytes > 0 ? kMaxStagingBytes : 1024));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_fused<DT, WC, CODES>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) cudaGetLastError();  // cluster size 16 then stays unavailable
    return cudaSuccess;
}

template <int DT, int WC>
inline cudaError_t set_attrs_wc() {
    cudaError_t e = set_attrs<DT, WC, false>();
    return e != cudaSuccess ? e : set_attrs<DT, WC, true>();
}

template <int DT>
inline cudaError_t init_device(bool* cluster16) {
    cudaError_t e;
    if ((e = set_attrs_wc<DT, 0>()) != cudaSuccess) return e;
    if ((e = set_attrs_wc<DT, 8>()) != cudaSuccess) return e;
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
    if (cudaOccupancyMaxActiveClusters(&n, k_fused<DT, 0, false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    *cluster16 = n > 0;
    return cudaSuccess;
}

struct DeviceInit {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    bool cluster16 = false;
};

// Cluster size: about 64 KiB of staged gradients per CTA for 128 KiB chunks, and a multiple
// of W (up to 16) so that ring segments map onto whole CTAs.
inline uint32_t cluster_size(int W, bool cluster16) {
    const uint32_t pmax = cluster16 ? 16u : 8u;
    const uint32_t w = static_cast<uint32_t>(W);
    if (2 * w <= pmax) return 2 * w;
    if (w <= pmax) return w;
    return pmax;
}

template <int DT, int WC, bool CODES>
inline cudaError_t launch_wc(cudaLaunchConfig_t* cfg, const Args& A) {
    return cudaLaunchKernelEx(cfg, k_fused<DT, WC, CODES>, A);
}

template <int DT, bool CODES>
inline cudaError_t launch_codes(cudaLaunchConfig_t* cfg, const Args& A) {
    if (A.q.W == 8) return cudaLaunchKernelEx(cfg, k_fused<DT, 8, CODES>, A);
    return cudaLaunchKernelEx(cfg, k_fused<DT, 0, CODES>, A);
}

template <int DT>
inline cudaError_t launch(DeviceInit* table, const QuantArgs& a, int order, float* out, int8_t* codes,
                          float* scales, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInit& di = table[dev];
    std::call_once(di.once, [&] { di.err = init_device<DT>(&di.cluster16); });
    if (di.err != cudaSuccess) return di.err;

    uint32_t P = cluster_size(a.W, di.cluster16);
    uint32_t row_cap = staging_row_cap(P);
    size_t smem = static_cast<size_t>(a.W) * row_cap;
    if (smem > kMaxStagingBytes || kMaxStagingBytes == 0 || a.W == 8) {
        row_cap = 0;
        smem = 0;
        // Re-read form: one CTA per ring segment (its clusters are half the size, and on GB300 the
        // W = 8 bucket ran in 92 us with clusters of 8 against 131 us with clusters of 16).
        if (static_cast<uint32_t>(a.W) <= (di.cluster16 ? 16u : 8u)) P = static_cast<uint32_t>(a.W);
    }
    const int64_t grid = a.num_chunks * P;
    if (grid > INT_MAX) return cudaErrorInvalidValue;

    Args A;
    A.q = a;
    A.order = order;
    A.out = out;
    A.codes = codes;
    A.scales = scales;
    A.row_cap = row_cap;
    A.P = P;
    A.invW = 1.0f / static_cast<float>(a.W);
    A.w_pow2 = (a.W & (a.W - 1)) == 0 ? 1 : 0;
    A.ring_split = (order == kOrderRing && P % static_cast<uint32_t>(a.W) == 0) ? 1 : 0;

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
    return codes ? launch_codes<DT, true>(&cfg, A) : launch_codes<DT, false>(&cfg, A);
}

inline cudaError_t read_clear_error(unsigned* word) {
    unsigned w = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (e == cudaSuccess) *word |= w;
    return e;
}

inline cudaError_t set_stall(uint32_t extra_bytes, uint64_t limit_ns) {
    cudaError_t e = cudaMemcpyToSymbol(g_stall_extra_tx, &extra_bytes, sizeof(extra_bytes));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_wait_limit_ns, &limit_ns, sizeof(limit_ns));
}

}  // namespace fused
}  // namespace gq
