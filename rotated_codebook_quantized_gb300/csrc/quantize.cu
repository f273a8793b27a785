// Fused encode: rotate, per-group RMS scale, snap to the codebook, pack.
// tq_quantize (weight rows) and tq_kv_quantize (KV-cache vectors).
//
// "How it works", "Quantizing a weight, with no data": randomized Hadamard
// rotation along the input dimension, groups divided by their RMS, each value
// replaced by its nearest Lloyd-Max centroid, indices packed into 32-bit words
// (20 base-3 trits per word for the three-level book, "The ternary tier").
#include <math.h>

#include "common.cuh"

using namespace tq;

namespace {

// Number of thresholds strictly below u (the nearest centroid's index; a tie
// goes to the lower cell).  Linear scan for small books, lower bound otherwise.
TQ_DEVFN int snap_code(float u, const float* t, int nthr) {
    if (nthr <= 15) {
        int c = 0;
        for (int i = 0; i < nthr; ++i) c += (t[i] < u) ? 1 : 0;
        return c;
    }
    int lo = 0, hi = nthr;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (t[mid] < u) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Word j of a packed row from codes held in shared memory (0 beyond `n`).
TQ_DEVFN uint32_t pack_word(const uint8_t* codes, int n, int j, int levels, int cw, int bits) {
    uint32_t w = 0;
    if (levels == 3) {
        for (int i = cw - 1; i >= 0; --i) {
            const int k = j * cw + i;
            w = w * 3u + (k < n ? codes[k] : 0u);
        }
    } else {
        for (int i = 0; i < cw; ++i) {
            const int k = j * cw + i;
            w |= (uint32_t)(k < n ? codes[k] : 0u) << (bits * i);
        }
    }
    return w;
}

template <int E>
__global__ void __launch_bounds__(1024) quantize_rows_kernel(const void* __restrict__ W, int wdt, int cols, int group,
                                                             int block, float rscale, const int8_t* __restrict__ signs,
                                                             const float* __restrict__ thresholds, int levels,
                                                             uint32_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                                             int64_t row_stride) {
    extern __shared__ float smem[];
    float* fw = smem;                                           // cols floats (FWHT exchange)
    float* thr = smem + cols;                                   // levels-1 thresholds
    uint8_t* cd = reinterpret_cast<uint8_t*>(thr + 256);        // cols codes
    const int64_t row = blockIdx.x;
    const int base = threadIdx.x * E;
    const int lane = threadIdx.x & 31;
    const int nthr = levels - 1;
    for (int i = threadIdx.x; i < nthr; i += blockDim.x) thr[i] = thresholds[i];

    float v[E];
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = load_as_float(W, row * cols + base + i, wdt) * (float)signs[base + i];
    fwht_cta<E>(v, fw, block);  // ends with a barrier when it used shared memory
    __syncthreads();
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] *= rscale;

    const float inv_g = 1.0f / (float)group;
    const int ngroups = cols / group;
    if (E >= group) {
        for (int g0 = 0; g0 < E; g0 += group) {
            float ss = 0.f;
            for (int i = g0; i < g0 + group; ++i) ss += v[i] * v[i];
            const float s = sqrtf(ss * inv_g);
            scales[row * ngroups + (base + g0) / group] = __half_as_ushort(__float2half_rn(s));
            for (int i = g0; i < g0 + group; ++i) {
                const float u = s > 0.f ? __fdiv_rn(v[i], s) : 0.f;
                cd[base + i] = (uint8_t)snap_code(u, thr, nthr);
            }
        }
    } else {
        const int lpg = group / E;  // lanes per group, 2..32
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) ss += v[i] * v[i];
        for (int m = 1; m < lpg; m <<= 1) ss += __shfl_xor_sync(kFull, ss, m);
        const float s = sqrtf(ss * inv_g);
        if ((lane & (lpg - 1)) == 0) scales[row * ngroups + base / group] = __half_as_ushort(__float2half_rn(s));
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const float u = s > 0.f ? __fdiv_rn(v[i], s) : 0.f;
            cd[base + i] = (uint8_t)snap_code(u, thr, nthr);
        }
    }
    __syncthreads();
    const int cw = levels == 3 ? 20 : (levels == 8 ? 10 : 32 / (31 - __clz(levels)));
    const int bits = 31 - __clz(levels);
    for (int64_t j = threadIdx.x; j < row_stride; j += blockDim.x)
        codes[row * row_stride + j] = pack_word(cd, cols, (int)j, levels, cw, bits);
}

// One warp encodes one D = 128 vector (4 values per lane), used for K and V.
TQ_DEVFN void encode_vec128(float (&v)[4], int group, const float* thr, int nthr, int levels,
                            uint32_t* codes_out, uint16_t* scales_out) {
    const int lane = threadIdx.x & 31;
    const float inv_g = 1.0f / (float)group;
    const int lpg = group / 4;
    float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
    for (int m = 1; m < lpg; m <<= 1) ss += __shfl_xor_sync(kFull, ss, m);
    const float s = sqrtf(ss * inv_g);
    if ((lane & (lpg - 1)) == 0) scales_out[(lane * 4) / group] = __half_as_ushort(__float2half_rn(s));
    uint32_t pk = 0;  // the lane's four codes, one byte each
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float u = s > 0.f ? __fdiv_rn(v[i], s) : 0.f;
        pk |= (uint32_t)snap_code(u, thr, nthr) << (8 * i);
    }
    const int bits = 31 - __clz(levels);
    const int cw = levels == 3 ? 20 : (levels == 8 ? 10 : 32 / bits);
    const int nw = (128 + cw - 1) / cw;
    uint32_t w = 0;
    // Lane j builds word j by gathering its codes from the lanes that hold them.
    for (int i = 0; i < cw; ++i) {
        const int idx = (levels == 3) ? (cw - 1 - i) : i;
        const int k = lane * cw + idx;
        const int src = k < 128 ? (k >> 2) : 0;
        const uint32_t got = __shfl_sync(kFull, pk, src);
        const uint32_t c = k < 128 ? ((got >> (8 * (k & 3))) & 0xffu) : 0u;
        if (levels == 3) w = w * 3u + c;
        else w |= c << (bits * idx);
    }
    if (lane < nw) codes_out[lane] = w;
}

__global__ void __launch_bounds__(256) kv_quantize_kernel(const void* __restrict__ k, const void* __restrict__ v, int dt,
                                                          int T, int Hkv, int64_t pos, int64_t capacity, float rscale,
                                                          const int8_t* __restrict__ signs,
                                                          const float* __restrict__ kthr, int klevels,
                                                          const float* __restrict__ vthr, int vlevels, int group,
                                                          uint32_t* kcodes, uint16_t* kscales, uint32_t* vcodes,
                                                          uint16_t* vscales, int kw, int vw) {
    __shared__ float st_k[256];
    __shared__ float st_v[256];
    for (int i = threadIdx.x; i < klevels - 1; i += blockDim.x) st_k[i] = kthr[i];
    for (int i = threadIdx.x; i < vlevels - 1; i += blockDim.x) st_v[i] = vthr[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t vec = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;  // (token, head) index
    if (vec >= (int64_t)T * Hkv) return;
    const int64_t t = vec / Hkv;
    const int h = (int)(vec - t * Hkv);
    const int64_t slot = (int64_t)h * capacity + pos + t;
    const int ng = 128 / group;
    for (int which = 0; which < 2; ++which) {
        const void* src = which ? v : k;
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = load_as_float(src, vec * 128 + lane * 4 + i, dt) * (float)signs[lane * 4 + i];
        fwht_warp128(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] *= rscale;
        if (which == 0)
            encode_vec128(x, group, st_k, klevels - 1, klevels, kcodes + slot * kw, kscales + slot * ng);
        else
            encode_vec128(x, group, st_v, vlevels - 1, vlevels, vcodes + slot * vw, vscales + slot * ng);
    }
}

// Elements per thread: smallest power of two E with whole warps (dim % 32E == 0),
// at most 1024 threads, E <= block, and a group spread over at most one warp
// (group / E <= 32) so the group's sum of squares is a warp-shuffle reduction.
int pick_e(int dim, int block, int group) {
    for (int e = 1; e <= 16; e <<= 1)
        if (e <= block && dim % (32 * e) == 0 && dim / e <= 1024 && group <= 32 * e) return e;
    return 0;
}

bool book_ok(const tq_codebook_t* cb) {
    return cb && cb->thresholds && host_codes_per_word(cb->levels) != 0;
}

}  // namespace

extern "C" tq_status tq_quantize(const void* W, tq_dtype wdt, int64_t rows, int32_t cols, int32_t group,
                                 const tq_rotation_t* rot, const tq_codebook_t* cb, uint32_t* codes, uint16_t* scales,
                                 int64_t row_stride_words, void* stream) {
    if (!rot || !rot->signs || !book_ok(cb) || rows < 0 || rows > 0x7fffffffll || cols <= 0) return TQ_ERR_INVALID;
    if (wdt != TQ_F32 && wdt != TQ_BF16) return TQ_ERR_INVALID;
    if (rot->dim != cols || !is_pow2(rot->block) || rot->block > 8192 || cols % rot->block) return TQ_ERR_INVALID;
    if (!(group == 16 || group == 32 || group == 64 || group == 128) || cols % group) return TQ_ERR_INVALID;
    if (row_stride_words < tq_row_words(cb->levels, cols)) return TQ_ERR_INVALID;
    if (!(cb->levels == 3 || cb->levels == 4 || cb->levels == 8 || cb->levels == 16)) return TQ_ERR_UNSUPPORTED;
    if (rows == 0) return TQ_OK;
    if (!W || !codes || !scales) return TQ_ERR_INVALID;
    const int e = pick_e(cols, rot->block, group);
    if (e == 0 || cols > 16384) return TQ_ERR_UNSUPPORTED;
    const int threads = cols / e;
    const size_t smem = (size_t)cols * 4 + 256 * 4 + (size_t)cols;
    const float rscale = (float)(1.0 / sqrt((double)rot->block));
    cudaStream_t st = as_stream(stream);
    switch (e) {
#define TQ_Q_CASE(EE)                                                                                           \
    case EE:                                                                                                    \
        if (ensure_smem((const void*)quantize_rows_kernel<EE>, smem) != cudaSuccess) return TQ_ERR_CUDA;     \
        quantize_rows_kernel<EE><<<(unsigned)rows, threads, smem, st>>>(W, wdt, cols, group, rot->block, rscale, \
                                                                        rot->signs, cb->thresholds, cb->levels, \
                                                                        codes, scales, row_stride_words);       \
        break;
        TQ_Q_CASE(1)
        TQ_Q_CASE(2)
        TQ_Q_CASE(4)
        TQ_Q_CASE(8)
        TQ_Q_CASE(16)
#undef TQ_Q_CASE
        default: return TQ_ERR_UNSUPPORTED;
    }
    return launch_status();
}

extern "C" tq_status tq_kv_quantize(const void* k, const void* v, tq_dtype dt, int32_t T, int32_t Hkv, int32_t D,
                                    int64_t pos, int64_t capacity, const tq_rotation_t* rot, const tq_codebook_t* kcb,
                                    const tq_codebook_t* vcb, int32_t group, uint32_t* kcodes, uint16_t* kscales,
                                    uint32_t* vcodes, uint16_t* vscales, void* stream) {
    if (D != 128) return TQ_ERR_UNSUPPORTED;
    if (!rot || !rot->signs || rot->dim != D || rot->block != D) return TQ_ERR_INVALID;
    if (!book_ok(kcb) || !book_ok(vcb) || T < 0 || Hkv <= 0 || pos < 0 || pos + T > capacity) return TQ_ERR_INVALID;
    if (!(group == 16 || group == 32 || group == 64 || group == 128)) return TQ_ERR_INVALID;
    if (dt != TQ_F32 && dt != TQ_BF16) return TQ_ERR_INVALID;
    if (kcb->levels == 2 || vcb->levels == 2) return TQ_ERR_UNSUPPORTED;
    if (T == 0) return TQ_OK;
    if (!k || !v || !kcodes || !kscales || !vcodes || !vscales) return TQ_ERR_INVALID;
    const int kw = (int)tq_row_words(kcb->levels, D), vw = (int)tq_row_words(vcb->levels, D);
    const int64_t nvec = (int64_t)T * Hkv;
    const int warps = 8;
    const int64_t blocks = (nvec + warps - 1) / warps;
    if (blocks > 0x7fffffffll) return TQ_ERR_INVALID;
    kv_quantize_kernel<<<(unsigned)blocks, warps * 32, 0, as_stream(stream)>>>(
        k, v, dt, T, Hkv, pos, capacity, (float)(1.0 / sqrt((double)D)), rot->signs, kcb->thresholds, kcb->levels,
        vcb->thresholds, vcb->levels, group, kcodes, kscales, vcodes, vscales, kw, vw);
    return launch_status();
}
