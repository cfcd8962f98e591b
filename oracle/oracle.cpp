/*
 * oracle.cpp -- CPU oracle (TEST INFRASTRUCTURE ONLY; see oracle.h for the rules on
 * who may load it and for the page names cited below).
 *
 * Single-threaded, scalar, binary32 with round-to-nearest-even.  Build with
 * -O2 -ffp-contract=off and without -ffast-math (oracle/build.py does).
 */
#include "oracle.h"

#include <cfenv>
#include <cmath>
#include <cstdint>
#include <vector>

namespace {

// [HCCL-PIPE] §2.1 dynamic_chunk: base chunk size 128 KB, HCCS alignment 64 B.
const int64_t kChunkSize = 128 * 1024;
const int64_t kAlignment = 64;

bool round_to_nearest_mode() { return std::fegetround() == FE_TONEAREST; }

// One gradient value after the optional unscale: float(x) * inv.
float load_grad(const void* grads, int dt, int64_t index, float inv) {
    float x;
    if (dt == ORACLE_F16) {
        const uint16_t* h = static_cast<const uint16_t*>(grads);
        x = oracle_half_to_float(h[index]);
    } else {
        const float* f = static_cast<const float*>(grads);
        x = f[index];
    }
    return x * inv;
}

}  // namespace

extern "C" {

float oracle_half_to_float(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = std::ldexp(static_cast<double>(f), -24);          // subnormal: f * 2^-24
    } else if (e == 31) {
        v = (f != 0) ? NAN : INFINITY;
    } else {
        v = std::ldexp(static_cast<double>(1024 + f), e - 25);  // (1 + f/1024) * 2^(e-15)
    }
    return static_cast<float>(sign ? -v : v);  // exact: every binary16 value is a binary32 value
}

int64_t oracle_bucket_chunks_sized(int64_t n, int64_t eb, int64_t chunk_size, int64_t* chunk_elems) {
    const int64_t nbytes = n * eb;
    int64_t k = nbytes / (chunk_size - chunk_size % kAlignment);  // num_chunks before max(1, .)
    if (k < 1) k = 1;
    if (n == 0) {                       // torch.chunk of an empty tensor: one empty piece
        if (chunk_elems) *chunk_elems = 0;
        return 1;
    }
    const int64_t c = (n + k - 1) / k;  // torch.chunk piece length: ceil(n / k)
    if (chunk_elems) *chunk_elems = c;
    return (n + c - 1) / c;             // pieces actually returned: ceil(n / c)
}

int64_t oracle_bucket_chunks(int64_t n, int64_t eb, int64_t* chunk_elems) {
    return oracle_bucket_chunks_sized(n, eb, kChunkSize, chunk_elems);
}

// Chunks of one entry of a plan: dynamic_chunk pieces, or the whole entry as one chunk.
static int64_t entry_chunks(int64_t n, int64_t eb, int scope, int64_t chunk_size, int64_t* chunk_elems) {
    if (scope == ORACLE_SCOPE_CHUNK) return oracle_bucket_chunks_sized(n, eb, chunk_size, chunk_elems);
    if (chunk_elems) *chunk_elems = n;  // one scale over the whole bucket or tensor
    return 1;
}

int64_t oracle_plan_chunks_ex(const int64_t* elems, int64_t count, int64_t eb, int scope, int64_t chunk_size,
                              int64_t* offsets, int64_t capacity) {
    if (scope != ORACLE_SCOPE_CHUNK && scope != ORACLE_SCOPE_BUCKET && scope != ORACLE_SCOPE_TENSOR) return -1;
    if (scope == ORACLE_SCOPE_CHUNK && chunk_size - chunk_size % kAlignment <= 0) return -1;
    int64_t total = 0;
    for (int64_t b = 0; b < count; ++b) {
        if (elems[b] < 0) return -1;
        total += entry_chunks(elems[b], eb, scope, chunk_size, nullptr);
    }
    if (offsets == nullptr || capacity < total + 1) return total;
    int64_t pos = 0;       // next table slot
    int64_t start = 0;     // element offset of the current entry
    for (int64_t b = 0; b < count; ++b) {
        const int64_t n = elems[b];
        int64_t c = 0;
        const int64_t pieces = entry_chunks(n, eb, scope, chunk_size, &c);
        for (int64_t j = 0; j < pieces; ++j) offsets[pos++] = start + j * c;
        start += n;
    }
    offsets[pos] = start;
    return total;
}

int64_t oracle_plan_chunks(const int64_t* bucket_elems, int64_t num_buckets, int64_t eb,
                           int64_t* offsets, int64_t capacity) {
    return oracle_plan_chunks_ex(bucket_elems, num_buckets, eb, ORACLE_SCOPE_CHUNK, kChunkSize, offsets, capacity);
}

int64_t oracle_assign_buckets(const int64_t* tensor_elems, int64_t num_tensors, int64_t eb,
                              int64_t cap_bytes, int64_t* bucket_of_tensor,
                              int64_t* bucket_elems, int64_t max_buckets) {
    int64_t nb = 0;
    int64_t open_bytes = 0;
    for (int64_t t = 0; t < num_tensors; ++t) {
        const int64_t bytes = tensor_elems[t] * eb;
        if (nb == 0 || (open_bytes > 0 && open_bytes + bytes > cap_bytes)) {
            if (nb == max_buckets) return -1;
            bucket_elems[nb] = 0;
            ++nb;
            open_bytes = 0;
        }
        bucket_of_tensor[t] = nb - 1;
        bucket_elems[nb - 1] += tensor_elems[t];
        open_bytes += bytes;
    }
    return nb;
}

int64_t oracle_quantize(const void* grads, int dt, int W, int64_t rank_stride,
                        const int64_t* offsets, int64_t num_chunks, float loss_scale,
                        int8_t* codes, float* scales) {
    if (!round_to_nearest_mode()) std::fesetround(FE_TONEAREST);
    const float inv = static_cast<float>(1.0 / static_cast<double>(loss_scale));
    int64_t nonfinite = 0;
    for (int r = 0; r < W; ++r) {
        const int64_t row = static_cast<int64_t>(r) * rank_stride;
        for (int64_t j = 0; j < num_chunks; ++j) {
            const int64_t lo = offsets[j], hi = offsets[j + 1];
            // scale = max|g| / 127.0
            float m = 0.0f;
            bool finite = true;
            for (int64_t i = lo; i < hi; ++i) {
                const float g = load_grad(grads, dt, row + i, inv);
                if (!std::isfinite(g)) finite = false;
                const float a = std::fabs(g);
                if (a > m) m = a;
            }
            const float s = m / 127.0f;
            scales[static_cast<int64_t>(r) * num_chunks + j] = s;
            if (!finite) ++nonfinite;
            // quantized = clamp(round(g / scale), -128, 127) as int8; all-zero scale -> 0
            for (int64_t i = lo; i < hi; ++i) {
                int8_t q = 0;
                if (finite && s != 0.0f) {
                    const float g = load_grad(grads, dt, row + i, inv);
                    float y = std::nearbyint(g / s);   // ties to even in FE_TONEAREST
                    if (y < -128.0f) y = -128.0f;
                    if (y > 127.0f) y = 127.0f;
                    q = static_cast<int8_t>(y);
                }
                codes[row + i] = q;
            }
        }
    }
    return nonfinite;
}

void oracle_reduce(const int8_t* codes, const float* scales, int W, int64_t rank_stride,
                   const int64_t* offsets, int64_t num_chunks, int order, float* out) {
    if (!round_to_nearest_mode()) std::fesetround(FE_TONEAREST);
    std::vector<float> d(W);
    for (int64_t j = 0; j < num_chunks; ++j) {
        const int64_t lo = offsets[j], hi = offsets[j + 1];
        const int64_t len = hi - lo;
        const int64_t seg = (len + W - 1) / W;  // torch.chunk(chunk, W) piece length
        for (int64_t i = lo; i < hi; ++i) {
            // dequantise every rank's code: d_r = q_r * s_r
            for (int r = 0; r < W; ++r) {
                const float q = static_cast<float>(codes[static_cast<int64_t>(r) * rank_stride + i]);
                d[r] = q * scales[static_cast<int64_t>(r) * num_chunks + j];
            }
            float acc;
            if (order == ORACLE_RING) {
                const int t = static_cast<int>((i - lo) / seg);  // segment of this element
                acc = d[(t + 1) % W];
                for (int k = 2; k <= W; ++k) acc = acc + d[(t + k) % W];
            } else if (order == ORACLE_TREE) {
                std::vector<float> level(d);
                while (level.size() > 1) {
                    std::vector<float> next;
                    for (size_t p = 0; p + 1 < level.size(); p += 2) next.push_back(level[p] + level[p + 1]);
                    if (level.size() % 2 == 1) next.push_back(level.back());
                    level.swap(next);
                }
                acc = level[0];
            } else {
                acc = d[0];
                for (int r = 1; r < W; ++r) acc = acc + d[r];
            }
            out[i] = acc / static_cast<float>(W);  // mean over the data-parallel group
        }
    }
}

int oracle_reduce_hier(const int8_t* codes, const float* scales, int W, int64_t rank_stride,
                       const int64_t* offsets, int64_t num_chunks, int L, float* out) {
    if (L < 1 || W % L != 0) return -1;
    if (!round_to_nearest_mode()) std::fesetround(FE_TONEAREST);
    const int nodes = W / L;
    std::vector<float> d(W);
    for (int64_t j = 0; j < num_chunks; ++j) {
        const int64_t lo = offsets[j], hi = offsets[j + 1];
        const int64_t len = hi - lo;
        const int64_t seg = (len + L - 1) / L;  // torch.chunk(chunk, L) piece length
        for (int64_t i = lo; i < hi; ++i) {
            for (int r = 0; r < W; ++r) {
                const float q = static_cast<float>(codes[static_cast<int64_t>(r) * rank_stride + i]);
                d[r] = q * scales[static_cast<int64_t>(r) * num_chunks + j];
            }
            // stage 1: ring inside each node over the node's own segment schedule
            const int t = static_cast<int>((i - lo) / seg);
            std::vector<float> level(nodes);
            for (int n = 0; n < nodes; ++n) {
                float node_sum = d[n * L + (t + 1) % L];
                for (int k = 2; k <= L; ++k) node_sum = node_sum + d[n * L + (t + k) % L];
                level[n] = node_sum;
            }
            // stage 2: aggregation tree over the node sums
            while (level.size() > 1) {
                std::vector<float> next;
                for (size_t p = 0; p + 1 < level.size(); p += 2) next.push_back(level[p] + level[p + 1]);
                if (level.size() % 2 == 1) next.push_back(level.back());
                level.swap(next);
            }
            out[i] = level[0] / static_cast<float>(W);
        }
    }
    return 0;
}

void oracle_amp_update_scale(float* scale, int32_t* tracker, float found_inf, float growth, float backoff,
                             int32_t interval) {
    if (found_inf != 0.0f) {  // true for NaN as well
        const float backed = *scale * backoff;
        *scale = backed;
        *tracker = 0;
        return;
    }
    const int32_t t = *tracker + 1;
    if (t == interval) {
        const float grown = *scale * growth;
        if (std::isfinite(grown)) *scale = grown;
        *tracker = 0;
    } else {
        *tracker = t;
    }
}

}  // extern "C"
