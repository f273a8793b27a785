// Dense rotation for input dimensions the block Hadamard transform mixes too
// little (the QR fallback), and its application to rows on the GPU.
//
// Weight-reservoir page: a layer whose input dimension the fast transform
// cannot take gets a rotation derived from its seed by a QR decomposition of a
// random matrix; the rotation is dense (d^2 numbers), orthonormal, and the
// layer multiplies its input by it exactly as a Hadamard layer does ("How it
// works", "Running a quantized layer": rotate the input, not the weights).
//
// Host: G[i][j] = the (i*d + j)-th standard normal draw of the seed's SplitMix64
// stream through the Box-Muller transform (draws 2p and 2p+1 from outputs 2p
// and 2p+1, u = (output >> 11) / 2^53); G = QU by Householder reflections in
// fp64, with the sign of each column of Q chosen so that U has a positive
// diagonal (the unique factorisation, which makes Q Haar-distributed).  R = Q.
//
// Device: y[r, i] = sum_j R[i, j] x[r, j], a register-tiled GEMM on the CUDA
// cores (64 x 64 outputs per CTA, 4 x 4 per thread), or for up to 8 rows a
// matvec that streams R once (one warp per output dimension), accumulating in
// fp64 for encodes (the code decision must not move by more than the rounding
// of the rotated value) or in fp32 for a decode input.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <thread>
#include <vector>

#include "common.cuh"

using namespace tq;

namespace {

// The SplitMix64 stream of `seed` (Steele, Lea & Flood 2014): output k mixes seed + (k+1) gamma.
uint64_t splitmix_at(uint64_t seed, uint64_t k) {
    uint64_t z = seed + (k + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Standard normal draw n of the seed (Box & Muller 1958 on the pair of outputs 2p, 2p+1).
double gaussian_at(uint64_t seed, uint64_t n) {
    const uint64_t p = n / 2;
    const double u1 = (double)(splitmix_at(seed, 2 * p) >> 11) * (1.0 / 9007199254740992.0);
    const double u2 = (double)(splitmix_at(seed, 2 * p + 1) >> 11) * (1.0 / 9007199254740992.0);
    const double r = sqrt(-2.0 * log1p(-u1));
    const double a = 2.0 * M_PI * u2;
    return (n & 1) ? r * sin(a) : r * cos(a);
}

// Runs fn(lo, hi) over [0, n) split across the host's threads (serially for small n).
template <class Fn>
void parallel_cols(int n, int64_t work_per_col, Fn fn) {
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    const int nt = (int)std::min<int64_t>(hw, std::max<int64_t>(1, (int64_t)n * work_per_col / (1 << 18)));
    if (nt <= 1) {
        fn(0, n);
        return;
    }
    std::vector<std::thread> th;
    for (int t = 0; t < nt; ++t) {
        const int lo = (int)((int64_t)n * t / nt), hi = (int)((int64_t)n * (t + 1) / nt);
        th.emplace_back([=] { fn(lo, hi); });
    }
    for (auto& x : th) x.join();
}

}  // namespace

extern "C" tq_status tq_rotation_dense(uint64_t seed, int32_t dim, double* R) {
    if (dim <= 0 || dim > 16384 || !R) return TQ_ERR_INVALID;
    const int n = dim;
    // A column-major: A[j * n + i] = G[i][j]
    std::vector<double> A((size_t)n * n), V((size_t)n * n, 0.0), beta(n, 0.0);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) A[(size_t)j * n + i] = gaussian_at(seed, (uint64_t)i * n + j);
    std::vector<double> diag(n);
    // Householder: reflector k maps A[k:, k] to (alpha, 0, ..., 0), alpha = -sign(a_kk) ||A[k:, k]||.
    for (int k = 0; k < n; ++k) {
        double* a = &A[(size_t)k * n];
        double nrm = 0.0;
        for (int i = k; i < n; ++i) nrm += a[i] * a[i];
        nrm = sqrt(nrm);
        const double alpha = a[k] >= 0.0 ? -nrm : nrm;
        double* v = &V[(size_t)k * n];
        for (int i = k; i < n; ++i) v[i] = a[i];
        v[k] -= alpha;
        double vv = 0.0;
        for (int i = k; i < n; ++i) vv += v[i] * v[i];
        beta[k] = vv > 0.0 ? 2.0 / vv : 0.0;
        diag[k] = vv > 0.0 ? alpha : a[k];
        const double b = beta[k];
        parallel_cols(n - k - 1, n - k, [&, k, b](int lo, int hi) {
            for (int j = k + 1 + lo; j < k + 1 + hi; ++j) {
                double* c = &A[(size_t)j * n];
                double d = 0.0;
                for (int i = k; i < n; ++i) d += v[i] * c[i];
                d *= b;
                for (int i = k; i < n; ++i) c[i] -= d * v[i];
            }
        });
    }
    // Q = H_0 H_1 ... H_{n-1} I, accumulated backwards into Qc (column-major)
    std::vector<double> Qc((size_t)n * n, 0.0);
    for (int i = 0; i < n; ++i) Qc[(size_t)i * n + i] = 1.0;
    for (int k = n - 1; k >= 0; --k) {
        const double* v = &V[(size_t)k * n];
        const double b = beta[k];
        if (b == 0.0) continue;
        parallel_cols(n - k, n - k, [&, k, b, v](int lo, int hi) {
            for (int j = k + lo; j < k + hi; ++j) {
                double* c = &Qc[(size_t)j * n];
                double d = 0.0;
                for (int i = k; i < n; ++i) d += v[i] * c[i];
                d *= b;
                for (int i = k; i < n; ++i) c[i] -= d * v[i];
            }
        });
    }
    // column k of Q times the sign of U's diagonal entry k; R row-major: R[i * n + j] = Q[i][j]
    for (int j = 0; j < n; ++j) {
        const double sg = diag[j] < 0.0 ? -1.0 : 1.0;
        for (int i = 0; i < n; ++i) R[(size_t)i * n + j] = sg * Qc[(size_t)j * n + i];
    }
    return TQ_OK;
}

namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16;  // outputs per CTA (dims i x rows r) and the j step

template <class ACC>
__global__ void __launch_bounds__(256) rotate_dense_kernel(const float* __restrict__ R, int dim,
                                                           const void* __restrict__ x, int xdt, int64_t rows,
                                                           float* __restrict__ y) {
    __shared__ float Rs[kTK][kTM + 4];  // R[i0 + m][j0 + k] at Rs[k][m]
    __shared__ float Xs[kTK][kTN + 4];  // x[r0 + n][j0 + k] at Xs[k][n]
    const int tid = threadIdx.x, tm = tid % 16, tn = tid / 16;  // thread owns outputs (4 tm + a, 4 tn + b)
    const int i0 = blockIdx.x * kTM;
    const int64_t r0 = (int64_t)blockIdx.y * kTN;
    ACC acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0;
    for (int j0 = 0; j0 < dim; j0 += kTK) {
        // 64 x 16 elements of each operand, 4 per thread
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid + 256 * q, m = e / kTK, k = e % kTK;
            const int i = i0 + m, j = j0 + k;
            Rs[k][m] = i < dim && j < dim ? R[(size_t)i * dim + j] : 0.f;
            const int64_t r = r0 + m;
            Xs[k][m] = r < rows && j < dim ? load_as_float(x, r * dim + j, xdt) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTK; ++k) {
            float ra[4], xb[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) ra[a] = Rs[k][4 * tm + a];
#pragma unroll
            for (int b = 0; b < 4; ++b) xb[b] = Xs[k][4 * tn + b];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fma((ACC)ra[a], (ACC)xb[b], acc[a][b]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int64_t r = r0 + 4 * tn + b;
        if (r >= rows) continue;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = i0 + 4 * tm + a;
            if (i < dim) y[r * dim + i] = (float)acc[a][b];
        }
    }
}

// Few rows (a decode input): one warp per output dimension i streams row i of R once with
// 16-byte loads (dim % 4 == 0) and dots it with every input row held in shared memory.
constexpr int kGvRows = 8, kGvWarps = 8;

template <class ACC>
__global__ void __launch_bounds__(256) rotate_dense_gemv_kernel(const float* __restrict__ R, int dim,
                                                                const void* __restrict__ x, int xdt, int rows,
                                                                float* __restrict__ y) {
    extern __shared__ __align__(16) float xs[];  // [rows][dim]
    for (int e = threadIdx.x; e < rows * dim; e += blockDim.x) xs[e] = load_as_float(x, e, xdt);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kGvWarps + (threadIdx.x >> 5);
    if (i >= dim) return;
    const float4* r4 = reinterpret_cast<const float4*>(R + (size_t)i * dim);
    const int n4 = dim / 4;
    ACC acc[kGvRows];
#pragma unroll
    for (int r = 0; r < kGvRows; ++r) acc[r] = 0;
    constexpr int U = 8;  // loads in flight per lane
    for (int b = 0; b < n4; b += 32 * U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = b + u * 32 + lane;
            v[u] = q < n4 ? __ldg(r4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = b + u * 32 + lane;
            if (q >= n4) break;
#pragma unroll
            for (int r = 0; r < kGvRows; ++r) {
                if (r >= rows) break;
                const float4 xv = reinterpret_cast<const float4*>(xs + (size_t)r * dim)[q];
                acc[r] = fma((ACC)v[u].x, (ACC)xv.x, acc[r]);
                acc[r] = fma((ACC)v[u].y, (ACC)xv.y, acc[r]);
                acc[r] = fma((ACC)v[u].z, (ACC)xv.z, acc[r]);
                acc[r] = fma((ACC)v[u].w, (ACC)xv.w, acc[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kGvRows; ++r) {
        if (r >= rows) break;
        ACC a = acc[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) y[(size_t)r * dim + i] = (float)a;
    }
}

}  // namespace

extern "C" tq_status tq_rotate_dense(const float* R, int32_t dim, const void* x, tq_dtype xdt, int64_t rows, float* y,
                                     int32_t precise, void* stream) {
    if (!R || dim <= 0 || rows < 0 || (xdt != TQ_F32 && xdt != TQ_BF16 && xdt != TQ_F16)) return TQ_ERR_INVALID;
    if (rows == 0) return TQ_OK;
    if (!x || !y || (const void*)y == x) return TQ_ERR_INVALID;
    cudaStream_t st = as_stream(stream);
    const size_t xs_bytes = (size_t)rows * dim * 4;
    if (rows <= kGvRows && dim % 4 == 0 && aligned(R, 16) && xs_bytes <= 48 * 1024) {
        const unsigned g = (unsigned)((dim + kGvWarps - 1) / kGvWarps);
        if (precise)
            rotate_dense_gemv_kernel<double><<<g, 32 * kGvWarps, xs_bytes, st>>>(R, dim, x, xdt, (int)rows, y);
        else
            rotate_dense_gemv_kernel<float><<<g, 32 * kGvWarps, xs_bytes, st>>>(R, dim, x, xdt, (int)rows, y);
        return launch_status();
    }
    const int64_t gy = (rows + kTN - 1) / kTN;
    if (gy > 65535) return TQ_ERR_UNSUPPORTED;
    const dim3 grid((dim + kTM - 1) / kTM, (unsigned)gy);
    if (precise)
        rotate_dense_kernel<double><<<grid, 256, 0, st>>>(R, dim, x, xdt, rows, y);
    else
        rotate_dense_kernel<float><<<grid, 256, 0, st>>>(R, dim, x, xdt, rows, y);
    return launch_status();
}
