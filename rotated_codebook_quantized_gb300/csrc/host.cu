// Host-side entry points: status names, format sizes, the Gaussian Lloyd-Max
// codebook, the seeded rotation signs and the device error word.
#include <atomic>
#include <math.h>
#include <string.h>

#include "common.cuh"

using namespace tq;

extern "C" const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported combination";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_TIMEOUT: return "device wait timed out";
        case TQ_ERR_DEVICE: return "device reported bad input";
    }
    return "unknown status";
}

extern "C" int32_t tq_codes_per_word(int32_t levels) { return host_codes_per_word(levels); }

extern "C" int64_t tq_row_words(int32_t levels, int32_t cols) {
    const int cw = host_codes_per_word(levels);
    if (cw == 0 || cols < 0) return 0;
    return ((int64_t)cols + cw - 1) / cw;
}

extern "C" int64_t tq_row_stride_words(int32_t levels, int32_t cols) {
    return (tq_row_words(levels, cols) + 3) / 4 * 4;
}

// ---------------------------------------------------------------- codebook

namespace {

const double kInvSqrt2Pi = 0.39894228040143267794;

double npdf(double x) { return isinf(x) ? 0.0 : kInvSqrt2Pi * exp(-0.5 * x * x); }

// Probability of (a, b] under N(0,1), taken from the tail that keeps digits.
double nmass(double a, double b) {
    if (a >= 0.0) return 0.5 * erfc(a / sqrt(2.0)) - 0.5 * erfc(b / sqrt(2.0));
    if (b <= 0.0) return 0.5 * erfc(-b / sqrt(2.0)) - 0.5 * erfc(-a / sqrt(2.0));
    return 1.0 - 0.5 * erfc(b / sqrt(2.0)) - 0.5 * erfc(-a / sqrt(2.0));
}

double ncdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

// Cell edge i of a book with L centroids: -inf, midpoints, +inf.
double edge(const double* c, int L, int i) {
    if (i == 0) return -INFINITY;
    if (i == L) return INFINITY;
    return 0.5 * (c[i - 1] + c[i]);
}

// Truncated-normal mean of cell i, (phi(a) - phi(b)) / P(a < X <= b).
double cell_mean(const double* c, int L, int i, double* mass) {
    const double a = edge(c, L, i), b = edge(c, L, i + 1);
    const double m = nmass(a, b);
    if (mass) *mass = m;
    return (npdf(a) - npdf(b)) / m;
}

void symmetrize(double* c, int L) {
    for (int i = 0; i < L / 2; ++i) {
        const double m = 0.5 * (c[L - 1 - i] - c[i]);
        c[i] = -m;
        c[L - 1 - i] = m;
    }
    if (L & 1) c[L / 2] = 0.0;
}

}  // namespace

// The Gaussian Lloyd-Max quantizer: the fixed point of "centroid = mean of its
// cell" and "threshold = midpoint of neighbours".  Start from equiprobable
// cells, run the Lloyd map, then solve the fixed-point equation by Newton's
// method with the tridiagonal Jacobian (Thomas algorithm).
extern "C" tq_status tq_codebook(int32_t levels, double* centroids, double* thresholds) {
    const int L = levels;
    if (!(L == 2 || L == 3 || L == 4 || L == 8 || L == 16 || L == 256) || !centroids || !thresholds)
        return TQ_ERR_INVALID;
    double c[256], m[256], P[256], lo[256], di[256], up[256], r[256];
    // Equiprobable quantiles by bisection on the CDF, then cell means.
    double q[257];
    q[0] = -INFINITY;
    q[L] = INFINITY;
    for (int i = 1; i < L; ++i) {
        double a = -40, b = 40, p = (double)i / L;
        for (int it = 0; it < 200; ++it) {
            const double mid = 0.5 * (a + b);
            if (ncdf(mid) < p) a = mid; else b = mid;
        }
        q[i] = 0.5 * (a + b);
    }
    for (int i = 0; i < L; ++i) c[i] = (npdf(q[i]) - npdf(q[i + 1])) / nmass(q[i], q[i + 1]);
    for (int it = 0; it < 200; ++it) {
        for (int i = 0; i < L; ++i) m[i] = cell_mean(c, L, i, nullptr);
        memcpy(c, m, sizeof(double) * L);
    }
    symmetrize(c, L);
    for (int it = 0; it < 100; ++it) {
        double worst = 0.0;
        for (int i = 0; i < L; ++i) {
            m[i] = cell_mean(c, L, i, &P[i]);
            r[i] = m[i] - c[i];
            worst = fmax(worst, fabs(r[i]));
        }
        if (worst <= 1e-15) break;
        // Jacobian J of the map c -> m, then solve (J - I) dc = -r.
        for (int i = 0; i < L; ++i) {
            lo[i] = di[i] = up[i] = 0.0;
            if (i < L - 1) {
                const double b = edge(c, L, i + 1);
                const double d = npdf(b) * (b - m[i]) / P[i];
                di[i] += 0.5 * d;
                up[i] += 0.5 * d;
            }
            if (i > 0) {
                const double a = edge(c, L, i);
                const double d = npdf(a) * (m[i] - a) / P[i];
                lo[i] += 0.5 * d;
                di[i] += 0.5 * d;
            }
            di[i] -= 1.0;
            r[i] = -r[i];
        }
        for (int i = 1; i < L; ++i) {  // forward elimination
            const double f = lo[i] / di[i - 1];
            di[i] -= f * up[i - 1];
            r[i] -= f * r[i - 1];
        }
        r[L - 1] /= di[L - 1];
        for (int i = L - 2; i >= 0; --i) r[i] = (r[i] - up[i] * r[i + 1]) / di[i];
        for (int i = 0; i < L; ++i) c[i] += r[i];
        symmetrize(c, L);
    }
    for (int i = 0; i < L; ++i) centroids[i] = c[i];
    for (int i = 0; i + 1 < L; ++i) thresholds[i] = 0.5 * (c[i] + c[i + 1]);
    return TQ_OK;
}

// ---------------------------------------------------------------- signs

extern "C" tq_status tq_rotation_signs(uint64_t seed, int32_t dim, int8_t* signs) {
    if (dim < 0 || (dim > 0 && !signs)) return TQ_ERR_INVALID;
    uint64_t state = seed;
    for (int32_t i = 0; i < dim; ++i) {
        // SplitMix64 (Steele, Lea & Flood 2014): golden-gamma increment, then mix.
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        signs[i] = (z >> 63) ? (int8_t)-1 : (int8_t)1;
    }
    return TQ_OK;
}

// ---------------------------------------------------------------- bounded-wait budget

namespace {
constexpr long long kDefaultWaitCycles = 1ll << 31;  // about a second at GB300 clocks
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};
}  // namespace

namespace tq {
long long wait_budget() { return g_wait_cycles.load(std::memory_order_relaxed); }
}  // namespace tq

extern "C" tq_status tq_set_wait_budget(int64_t cycles) {
    g_wait_cycles.store(cycles < 0 ? kDefaultWaitCycles : (long long)cycles, std::memory_order_relaxed);
    return TQ_OK;
}

// ---------------------------------------------------------------- error word

extern "C" tq_status tq_check_error(uint32_t* err, uint32_t* bits, void* stream) {
    if (!err) return TQ_ERR_INVALID;
    uint32_t h = 0;
    if (cudaMemcpyAsync(&h, err, sizeof(h), cudaMemcpyDeviceToHost, as_stream(stream)) != cudaSuccess)
        return TQ_ERR_CUDA;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return TQ_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof(uint32_t), as_stream(stream)) != cudaSuccess) return TQ_ERR_CUDA;
    if (bits) *bits = h;
    if (h == 0) return TQ_OK;
    return (h & TQ_DEVERR_TIMEOUT) ? TQ_ERR_TIMEOUT : TQ_ERR_DEVICE;
}

// ---------------------------------------------------------------- trit decoder self-check

namespace {

__global__ void selftest_trit_kernel(uint32_t first, uint32_t count, unsigned long long* mismatches) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    unsigned long long bad = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
        const uint32_t w = first + (uint32_t)i;
        TritHalves f = trit_split(w);
        uint32_t ref = w;
        uint32_t dig_ref[20];
#pragma unroll
        for (int j = 0; j < 20; ++j) {
            dig_ref[j] = ref % 3u;
            ref /= 3u;
        }
        bool ok = true;
        uint32_t F = f.hi;
#pragma unroll
        for (int t = 0; t < 10; ++t) {
            const float d = trit_next(F);
            ok &= (d == (float)dig_ref[19 - t]);
        }
        F = f.lo;
#pragma unroll
        for (int t = 0; t < 10; ++t) {
            const float d = trit_next(F);
            ok &= (d == (float)dig_ref[9 - t]);
        }
        bad += ok ? 0 : 1;
    }
    if (bad) atomicAdd(mismatches, bad);
}

}  // namespace

extern "C" tq_status tq_selftest_trit_decode(uint32_t first, uint32_t count, unsigned long long* mismatches,
                                             void* stream) {
    if (!mismatches || (uint64_t)first + count > 3486784401ull) return TQ_ERR_INVALID;
    if (count == 0) return TQ_OK;
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int blocks = sms > 0 ? sms * 8 : 1024;
    selftest_trit_kernel<<<blocks, 256, 0, as_stream(stream)>>>(first, count, mismatches);
    return launch_status();
}
