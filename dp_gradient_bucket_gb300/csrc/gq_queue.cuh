// gq_queue.cuh -- the fused quantise + W-way reduce as a dependency-ordered work queue.
//
// Same arithmetic as gq_fused.cuh ("pipelined HCCL AllReduce" article, bjdmk.com.cn/news/6235379,
// §2.1 chunks, §2.2.1 quantize_gradient + INT8_ALLREDUCE, §3.1 one SUM per chunk, §6.1 unscale;
// mean as in the "torchtitan-npu 3D parallel" article, AMP + 3D section), scheduled so that HBM
// streams without waiting for any chunk's absmax:
//
//   - Each chunk is cut into S slices (S a multiple of W under the ring order, so a slice lies in
//     one ring segment).  Work items are (pass, chunk, slice).
//   - Pass 1 of a slice reads its W rank rows from HBM (L2 policy evict_last: the bytes are read
//     again soon), reduces the per-rank absmax, folds it into a per-(chunk, rank) word with
//     atomicMax, and counts the slice done for its chunk.
//   - Pass 2 of a slice waits (bounded) until all S slices of its chunk finished pass 1, reads the W
//     scales, reads the rows again (from L2, evict_first), quantises, dequantises, sums and stores.
//   - Items are handed out in one global order by atomicAdd on a queue head: pass 1 of chunk k,
//     then pass 2 of chunk k - L (L chunks of lag).  An item's dependencies are always handed out
//     before it, to CTAs that are already running and wait on nothing, so the queue makes progress
//     whatever the number of resident CTAs.  The lag keeps about L chunks of re-read data in L2 and
//     hides the absmax hand-off.
//   - The workspace (queue head, exit count, per-chunk counters, per-(chunk, rank) absmax words)
//     must be zero when a launch starts; the last pass 2 of each chunk and the last CTA to leave
//     zero it again, so consecutive launches need no clearing in between.
#pragma once

#include "gq_fused.cuh"

namespace gq {
namespace fused {

constexpr int kQueueThreads = 256;
constexpr int kQueueSlices = 32;  // per chunk (a multiple of W = 8)
constexpr int kQueueLag = 24;     // chunks between pass 1 and pass 2 of a chunk

// Workspace words: [0] queue head, [1] CTAs done, [2 + j] chunk j's counter (pass-1 slices done,
// then pass-2 slices done on top), [2 + num_chunks + j * W + r] absmax bits of rank r in chunk j.
inline size_t queue_workspace_words(int64_t num_chunks, int W) {
    return 2 + static_cast<size_t>(num_chunks) + static_cast<size_t>(num_chunks) * W;
}

struct QueueArgs {
    Args f;
    uint32_t* ws;
    int64_t total_items;
    int lag;
};

// Item i -> (pass, chunk, slice).  Steps k = 0, 1, ...: pass 1 of chunk k (if k < n), then pass 2 of
// chunk k - L (if k >= L); S items each.
__device__ __forceinline__ void queue_item(int64_t i, int64_t n, int L, int* pass, int64_t* chunk, int* slice) {
    const int64_t S = kQueueSlices;
    const int64_t head = S * (static_cast<int64_t>(L) < n ? static_cast<int64_t>(L) : n);  // steps k < L: pass 1 only
    *slice = static_cast<int>(i % S);
    if (i < head) {
        *pass = 0;
        *chunk = i / S;
        return;
    }
    const int64_t i2 = i - head;
    const int64_t both = n > L ? n - L : 0;  // steps L .. n-1 hold pass 1 then pass 2
    if (i2 < 2 * S * both) {
        const int64_t k = L + i2 / (2 * S);
        const bool second = (i2 % (2 * S)) >= S;
        *pass = second ? 1 : 0;
        *chunk = second ? k - L : k;
        return;
    }
    // steps n .. n+L-1: pass 2 only
    const int64_t i3 = i2 - 2 * S * both;
    *pass = 1;
    *chunk = (n > L ? n - L : 0) + i3 / S;
}

__device__ __forceinline__ V16 ld_global_hint_v16(const void* p, uint64_t policy) {
    V16 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <int DT, int WC, bool CODES>
__global__ void __launch_bounds__(kQueueThreads, 3) k_queue(const QueueArgs Q) {
    constexpr int VEC = DT == 0 ? 4 : 8;
    constexpr int EB = DT == 0 ? 4 : 2;
    constexpr int W = WC;
    constexpr int NWARP = kQueueThreads / 32;
    constexpr int S = kQueueSlices;
    const Args& A = Q.f;
    __shared__ int64_t s_item;
    __shared__ uint32_t wmax[NWARP][W];
    __shared__ ScaleQ sq[W];
    __shared__ float row_s[W], row_c[W];
    __shared__ int row_rank[W];
    __shared__ int s_ok;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n = A.q.num_chunks;
    uint32_t* head = Q.ws;
    uint32_t* done = Q.ws + 1;
    uint32_t* counter = Q.ws + 2;
    uint32_t* amax = Q.ws + 2 + n;
    const char* grads = static_cast<const char*>(A.q.grads);
    const int64_t row_bytes = A.q.rank_stride * EB;
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    const uint64_t wait_limit = g_wait_limit_ns;
    const bool pow2 = (W & (W - 1)) == 0;
    const float inv = A.q.inv;
    const bool scaled = A.q.scaled != 0;

    for (;;) {
        if (tid == 0) s_item = static_cast<int64_t>(atomicAdd(head, 1u));
        __syncthreads();
        const int64_t item = s_item;
        __syncthreads();  // s_item is read by everyone before thread 0 may overwrite it
        if (item >= Q.total_items) break;
        int pass, slice;
        int64_t j;
        queue_item(item, n, Q.lag, &pass, &j, &slice);
        int64_t lo, hi;
        if (!chunk_bounds(A.q.offsets, j, n, A.q.rank_stride, &lo, &hi)) {
            if (tid == 0 && pass == 0 && slice == 0) raise_error(kErrBadTable);
            continue;
        }
        const uint32_t seg = hi > lo ? static_cast<uint32_t>((hi - lo + W - 1) / W) : 1u;
        // slice `slice` of S: S / W slices per ring segment under the ring order, else S equal runs
        Slice sl;
        if (A.ring_split) {
            const int sub = S / W;
            const int64_t t = slice / sub;
            const int64_t a = min(hi, lo + t * seg), b = min(hi, lo + (t + 1) * seg);
            sl = split_range<VEC>(a, b, static_cast<uint32_t>(slice % sub), static_cast<uint32_t>(sub));
        } else {
            sl = split_range<VEC>(lo, hi, static_cast<uint32_t>(slice), static_cast<uint32_t>(S));
        }
        int rot = 0;
        bool uniform = true;
        if (A.order == kOrderRing && sl.hi > sl.lo) {
            const int t0 = segment_of(sl.lo, lo, seg), t1 = segment_of(sl.hi - 1, lo, seg);
            uniform = t0 == t1;
            if (uniform) rot = (t0 + 1 == W) ? 0 : t0 + 1;
        }

        if (pass == 0) {
            // ---------------------------------------------------------------- pass 1: absmax
            uint32_t mx[W];
#pragma unroll
            for (int k = 0; k < W; ++k) mx[k] = 0;
            for (int64_t g = sl.g0 + tid; g < sl.g1; g += kQueueThreads) {
                const int64_t e0 = g * VEC;
                const bool full = e0 >= sl.lo && e0 + VEC <= sl.hi;
                V16 v[W];
#pragma unroll
                for (int k = 0; k < W; ++k) v[k] = ld_global_hint_v16(grads + k * row_bytes + g * 16, keep);
#pragma unroll
                for (int k = 0; k < W; ++k) mx[k] = group_absmax<DT>(v[k], e0, full, sl.lo, sl.hi, mx[k]);
            }
#pragma unroll
            for (int k = 0; k < W; ++k) {
                const uint32_t m = __reduce_max_sync(0xffffffffu, mx[k]);
                if (lane == 0) wmax[warp][k] = m;
            }
            __syncthreads();
            if (tid < W) {
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < NWARP; ++w) m = max(m, wmax[w][tid]);
                if (m != 0) atomicMax(amax + j * W + tid, m);
                __threadfence();  // this thread's absmax update before the count below
            }
            __syncthreads();
            if (tid == 0) {
                __threadfence();  // the absmax words before the count that publishes them
                atomicAdd(counter + j, 1u);
            }
        } else {
            // ---------------------------------------------------------------- pass 2: reduce
            if (tid == 0) {
                int ok = 1;
                if (ld_acquire_gpu_u32(counter + j) < static_cast<uint32_t>(S)) {
                    const uint64_t t0 = global_timer_ns();
                    while (ld_acquire_gpu_u32(counter + j) < static_cast<uint32_t>(S)) {
                        if (global_timer_ns() - t0 > wait_limit) {
                            raise_error(kErrTimeout);
                            ok = 0;
                            break;
                        }
                        __nanosleep(200);
                    }
                }
                s_ok = ok;
                // the thread that acquired the count reads the chunk's absmax words for everyone
#pragma unroll
                for (int r = 0; r < W; ++r) wmax[0][r] = ld_acquire_gpu_u32(amax + j * W + r);
            }
            __syncthreads();
            bool not_subnormal = true;
            if (tid < W) {
                const uint32_t mraw = wmax[0][tid];
                float m = DT == 0 ? __uint_as_float(mraw)
                                  : __half2float(__ushort_as_half(static_cast<unsigned short>(mraw)));
                if (scaled) m = __fmul_rn(m, inv);  // max|fl(x*inv)| = fl(max|x| * inv)
                const bool nonfinite = (DT == 0 ? mraw >= 0x7f800000u : mraw >= 0x7c00u) || !(fabsf(m) <= 3.40282347e38f);
                const ScaleQ s = make_scale(m);
                sq[tid] = s;
                not_subnormal = s.mode != 2;
                if (slice == 0) {
                    if (nonfinite) raise_error(kErrNonfinite);
                    if (A.scales) A.scales[static_cast<int64_t>(tid) * n + j] = s.s;
                }
            }
            const bool fast = __syncthreads_and(not_subnormal) != 0;
            if (tid < W) {
                const int r = (tid + rot) % W;
                row_rank[tid] = r;
                const ScaleQ s = sq[r];
                row_s[tid] = s.s;
                row_c[tid] = s.mode == 1 ? (scaled ? __fmul_rn(inv, s.rcp) : s.rcp) : 0.0f;
            }
            __syncthreads();
            const RowScales rs{row_s, row_c, row_rank, sq};
            for (int64_t g = sl.g0 + tid; g < sl.g1; g += kQueueThreads) {
                const int64_t e0 = g * VEC;
                const bool full = e0 >= sl.lo && e0 + VEC <= sl.hi;
                if (fast && uniform) {
                    V16 v[W];
#pragma unroll
                    for (int k = 0; k < W; ++k)
                        v[k] = ld_global_hint_v16(grads + static_cast<int64_t>((k + rot) % W) * row_bytes + g * 16, drop);
                    auto ld = [&](int k) { return v[k]; };
                    if (A.order == kOrderTree)
                        fast_group<DT, WC, CODES, true>(ld, W, rs, e0, full, sl.lo, sl.hi, A, pow2);
                    else if (DT == 0)
                        fast_group_f32x2<WC, CODES>(ld, W, rs, e0, full, sl.lo, sl.hi, A, pow2);
                    else
                        fast_group<DT, WC, CODES, false>(ld, W, rs, e0, full, sl.lo, sl.hi, A, pow2);
                } else {
                    auto ldr = [&](int r) { return ld_global_nc_v16(grads + static_cast<int64_t>(r) * row_bytes + g * 16); };
                    general_group<DT, CODES>(ldr, W, sq, lo, seg, e0, full, sl.lo, sl.hi, A, pow2);
                }
            }
            __syncthreads();
            if (tid == 0) {
                // the last pass-2 slice of the chunk clears its counter and absmax words for the next launch
                if (atomicAdd(counter + j, 1u) == static_cast<uint32_t>(2 * S - 1)) {
                    for (int r = 0; r < W; ++r) amax[j * W + r] = 0;
                    counter[j] = 0;
                }
            }
        }
    }
    // the last CTA out resets the queue for the next launch: nobody takes items any more
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(done, 1u) == gridDim.x - 1) {
            *head = 0;
            *done = 0;
            __threadfence();
        }
    }
}

struct QueueInit {
    std::once_flag once;
    int ctas = 0;  // resident CTAs of k_queue<DT, 8, false> on this device
};

template <int DT>
inline void init_queue(QueueInit* qi) {
    int per_sm = 0, sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_queue<DT, 8, false>, kQueueThreads, 0) !=
            cudaSuccess) {
        cudaGetLastError();
        qi->ctas = 0;
        return;
    }
    qi->ctas = per_sm * sms;
}

// Launches k_queue for W = 8 on a zero-filled workspace of queue_workspace_words(num_chunks, 8)
// words; *launched = false when W != 8.
template <int DT>
inline cudaError_t launch_queue_dt(QueueInit* table, const QuantArgs& a, int order, float* out, int8_t* codes,
                                   float* scales, uint32_t* ws, cudaStream_t stream, bool* launched) {
    *launched = false;
    if (a.W != 8) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    QueueInit& qi = table[dev];
    std::call_once(qi.once, [&] { init_queue<DT>(&qi); });
    if (qi.ctas <= 0) return cudaSuccess;
    QueueArgs Q;
    Q.f.q = a;
    Q.f.order = order;
    Q.f.out = out;
    Q.f.codes = codes;
    Q.f.scales = scales;
    Q.f.row_cap = 0;
    Q.f.P = kQueueSlices;
    Q.f.invW = 0.125f;
    Q.f.w_pow2 = 1;
    Q.f.ring_split = order == kOrderRing ? 1 : 0;
    Q.ws = ws;
    Q.total_items = 2 * static_cast<int64_t>(kQueueSlices) * a.num_chunks;
#ifdef GQ_QUEUE_LAG
    Q.lag = GQ_QUEUE_LAG;
#else
    Q.lag = kQueueLag;
#endif
    const int64_t want = Q.total_items < qi.ctas ? Q.total_items : qi.ctas;
    *launched = true;
    if (codes) k_queue<DT, 8, true><<<static_cast<unsigned>(want), kQueueThreads, 0, stream>>>(Q);
    else k_queue<DT, 8, false><<<static_cast<unsigned>(want), kQueueThreads, 0, stream>>>(Q);
    return cudaGetLastError();
}

}  // namespace fused
}  // namespace gq
