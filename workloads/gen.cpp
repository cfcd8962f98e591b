/*
 * gen.cpp -- seeded synthetic gradient generators for the five workloads.
 *
 * This module only draws input values; it holds none of the quantise / reduce
 * arithmetic, and neither the CUDA library nor the CPU oracle includes it.  Tests
 * and the benchmark fill host buffers with it and hand the same bytes to both.
 *
 * Randomness: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014) used as a counter-based generator: draw k of stream S at
 * counter i is mix(S + (i + 1) * 0x9E3779B97F4A7C15), with stream keys derived from
 * (seed, rank, k) through the same mixer.  Every element is a pure function of
 * (seed, rank, index), so any sub-range can be regenerated and thread count does not
 * change the bytes.  Transcendentals come from the host libm; buffers are consumed in
 * the process that made them, never stored.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

const uint64_t kGamma = 0x9E3779B97F4A7C15ull;

uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t stream_key(uint64_t seed, uint64_t a, uint64_t b) {
    return mix(seed + kGamma * (mix(a * 0x100000001B3ull + 0x1234567ull) ^ (b + 1)));
}

uint64_t draw(uint64_t key, uint64_t i) { return mix(key + (i + 1) * kGamma); }

// uniform in the open interval (0, 1)
double unif(uint64_t u) { return (static_cast<double>(u >> 11) + 0.5) * 0x1.0p-53; }

double gauss(uint64_t k1, uint64_t k2, uint64_t i) {
    const double u1 = unif(draw(k1, i)), u2 = unif(draw(k2, i));
    return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
}

const uint64_t kLayoutStream = 0xFFFFull;

struct Layout {
    std::vector<int64_t> start;   // element offset of each tensor (size + 1 entries)
    std::vector<double> sigma;    // per-tensor standard deviation
};

// Workload 3: ResNet-152-sized gradient list.  Sizes round(exp(U(ln 64, ln 2359296))) drawn
// until the total reaches 60,192,808 (the last one trimmed); sigma log-uniform in 1e-6..1e-2.
void layout_resnet(uint64_t seed, Layout* L) {
    const int64_t target = 60192808;
    const uint64_t k = stream_key(seed, kLayoutStream, 0);
    L->start.assign(1, 0);
    L->sigma.clear();
    int64_t total = 0;
    for (uint64_t t = 0; total < target; ++t) {
        const double ls = std::log(64.0) + unif(draw(k, 2 * t)) * (std::log(2359296.0) - std::log(64.0));
        int64_t n = std::llround(std::exp(ls));
        if (total + n > target) n = target - total;
        total += n;
        L->start.push_back(total);
        L->sigma.push_back(std::exp(std::log(1e-6) + unif(draw(k, 2 * t + 1)) * (std::log(1e-2) - std::log(1e-6))));
    }
}

// Workload 4: BERT-Large parameter shapes in model order (embeddings, 24 encoder layers,
// pooler); 335,141,888 elements.  Sigma log-uniform in 1e-6..1e-2 per tensor.
void layout_bert(uint64_t seed, Layout* L) {
    std::vector<int64_t> sizes = {30522LL * 1024, 512LL * 1024, 2LL * 1024, 1024, 1024};
    for (int layer = 0; layer < 24; ++layer) {
        for (int p = 0; p < 4; ++p) { sizes.push_back(1024LL * 1024); sizes.push_back(1024); }  // Q K V O
        sizes.push_back(1024); sizes.push_back(1024);                                          // attention LayerNorm
        sizes.push_back(4096LL * 1024); sizes.push_back(4096);                                 // FFN in
        sizes.push_back(1024LL * 4096); sizes.push_back(1024);                                 // FFN out
        sizes.push_back(1024); sizes.push_back(1024);                                          // output LayerNorm
    }
    sizes.push_back(1024LL * 1024); sizes.push_back(1024);                                     // pooler
    const uint64_t k = stream_key(seed, kLayoutStream, 1);
    L->start.assign(1, 0);
    L->sigma.clear();
    for (size_t t = 0; t < sizes.size(); ++t) {
        L->start.push_back(L->start.back() + sizes[t]);
        L->sigma.push_back(std::exp(std::log(1e-6) + unif(draw(k, t)) * (std::log(1e-2) - std::log(1e-6))));
    }
}

bool get_layout(int cfg, uint64_t seed, Layout* L) {
    if (cfg == 3) { layout_resnet(seed, L); return true; }
    if (cfg == 4) { layout_bert(seed, L); return true; }
    return false;
}

template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
    if (nthreads <= 1 || n < (1 << 16)) { f(int64_t(0), n); return; }
    std::vector<std::thread> th;
    const int64_t per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        const int64_t a = t * per, b = std::min(n, a + per);
        if (a < b) th.emplace_back(f, a, b);
    }
    for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

/* Tensor list of workload 3 or 4: returns the tensor count and writes up to cap sizes
 * and sigmas; -1 for a workload without a tensor list. */
int64_t wl_tensor_layout(int cfg, uint64_t seed, int64_t* sizes, double* sigmas, int64_t cap) {
    Layout L;
    if (!get_layout(cfg, seed, &L)) return -1;
    const int64_t nt = static_cast<int64_t>(L.sigma.size());
    for (int64_t t = 0; t < nt && t < cap; ++t) {
        if (sizes) sizes[t] = L.start[t + 1] - L.start[t];
        if (sigmas) sigmas[t] = L.sigma[t];
    }
    return nt;
}

/* Fill out[0 .. i1-i0) with elements [i0, i1) of virtual rank `rank`.
 *   cfg 1, 5: N(0, 1e-3)                                   -> float
 *   cfg 2:    Laplace(0, 1e-4); 30% exact zeros; 0.1% x100 -> float
 *   cfg 3:    per-tensor N(0, sigma_t)                     -> float
 *   cfg 4:    per-tensor N(0, sigma_t) * 65536, to fp16    -> uint16 bit patterns
 * Returns 0, or -1 for an unknown workload. */
int wl_fill(int cfg, uint64_t seed, int rank, int64_t i0, int64_t i1, void* out, int nthreads) {
    const uint64_t k0 = stream_key(seed, static_cast<uint64_t>(rank), 0);
    const uint64_t k1 = stream_key(seed, static_cast<uint64_t>(rank), 1);
    const uint64_t k2 = stream_key(seed, static_cast<uint64_t>(rank), 2);
    const uint64_t k3 = stream_key(seed, static_cast<uint64_t>(rank), 3);
    const int64_t n = i1 - i0;
    if (cfg == 1 || cfg == 5) {
        float* o = static_cast<float*>(out);
        parallel_for(n, nthreads, [&](int64_t a, int64_t b) {
            for (int64_t e = a; e < b; ++e) o[e] = static_cast<float>(1e-3 * gauss(k0, k1, i0 + e));
        });
        return 0;
    }
    if (cfg == 2) {
        float* o = static_cast<float*>(out);
        parallel_for(n, nthreads, [&](int64_t a, int64_t b) {
            for (int64_t e = a; e < b; ++e) {
                const uint64_t i = i0 + e;
                double v = unif(draw(k0, i)) - 0.5;
                double x = -1e-4 * (v < 0 ? -1.0 : 1.0) * std::log(1.0 - 2.0 * std::fabs(v));
                if (unif(draw(k1, i)) < 0.3) x = 0.0;
                else if (unif(draw(k2, i)) < 0.001) x *= 100.0;
                o[e] = static_cast<float>(x);
            }
        });
        return 0;
    }
    if (cfg == 3 || cfg == 4) {
        Layout L;
        get_layout(cfg, seed, &L);
        parallel_for(n, nthreads, [&](int64_t a, int64_t b) {
            int64_t t = std::upper_bound(L.start.begin(), L.start.end(), i0 + a) - L.start.begin() - 1;
            for (int64_t e = a; e < b; ++e) {
                const int64_t i = i0 + e;
                while (t + 1 < static_cast<int64_t>(L.start.size()) - 1 && i >= L.start[t + 1]) ++t;
                const double x = L.sigma[t] * gauss(k0, k1, static_cast<uint64_t>(i));
                if (cfg == 3) {
                    static_cast<float*>(out)[e] = static_cast<float>(x);
                } else {
                    const _Float16 h = static_cast<_Float16>(x * 65536.0);
                    std::memcpy(static_cast<uint16_t*>(out) + e, &h, 2);
                }
            }
        });
        (void)k2; (void)k3;
        return 0;
    }
    return -1;
}

/* Workload 5's adversarial chunks, written over rows already filled by wl_fill.  For a
 * table with at least five chunks, in every rank r:
 *   chunk 0: all zero                                  (scale 0)
 *   chunk 1: zero but one seeded element               (single nonzero)
 *   chunk 2: subnormals in +-[2^-149, 2^-126); rank 1 peaks at 190 * 2^-149, rank 2 at
 *            most 63 * 2^-149 in magnitude
 *   chunk 3: (k + 0.5) * 2^e with one element +-127 * 2^e, e = -20 - r (exact ties)
 *   chunk 4: the N(0, 1e-3) values with every third element set to -0.0
 * rows: W rows of rank_stride floats.  Returns 0, or -1 if the table has < 5 chunks. */
int wl_adversarial(uint64_t seed, int W, int64_t rank_stride, const int64_t* offsets,
                   int64_t num_chunks, float* rows) {
    if (num_chunks < 5) return -1;
    for (int r = 0; r < W; ++r) {
        float* g = rows + static_cast<int64_t>(r) * rank_stride;
        const uint64_t k = stream_key(seed, 0x10000ull + static_cast<uint64_t>(r), 7);
        for (int64_t i = offsets[0]; i < offsets[1]; ++i) g[i] = 0.0f;
        {
            const int64_t lo = offsets[1], len = offsets[2] - lo;
            for (int64_t i = 0; i < len; ++i) g[lo + i] = 0.0f;
            if (len > 0) g[lo + static_cast<int64_t>(draw(k, 0) % static_cast<uint64_t>(len))] =
                static_cast<float>((unif(draw(k, 1)) - 0.5) * 1e-2);
        }
        {
            const int64_t lo = offsets[2], len = offsets[3] - lo;
            const uint32_t cap = (r == 2) ? 63u : (1u << 23) - 1u;
            for (int64_t i = 0; i < len; ++i) {
                uint32_t m = static_cast<uint32_t>(draw(k, 100 + i) % cap) + 1u;
                if (r == 1) m = static_cast<uint32_t>(draw(k, 100 + i) % 190u) + 1u;
                const uint32_t bits = m | ((draw(k, 200000000 + i) & 1u) ? 0x80000000u : 0u);
                std::memcpy(g + lo + i, &bits, 4);
            }
            if (r == 1 && len > 0) { const uint32_t b = 190u; std::memcpy(g + lo, &b, 4); }
        }
        {
            const int64_t lo = offsets[3], len = offsets[4] - lo;
            const double p = std::ldexp(1.0, -20 - r);
            for (int64_t i = 0; i < len; ++i) {
                const double kk = static_cast<double>(static_cast<int64_t>(draw(k, 300000000 + i) % 254u) - 127) + 0.5;
                g[lo + i] = static_cast<float>(kk * p);
            }
            if (len > 0) g[lo + len / 2] = static_cast<float>((r % 2 ? -127.0 : 127.0) * p);
        }
        for (int64_t i = offsets[4]; i < offsets[5]; i += 3) g[i] = -0.0f;
    }
    return 0;
}

}  // extern "C"
