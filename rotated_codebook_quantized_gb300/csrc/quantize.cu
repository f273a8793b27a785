// Fused encode: rotate, per-group RMS scale, snap to the codebook, pack.
// tq_quantize (weight rows) and tq_kv_quantize (KV-cache vectors).
//
// "How it works", "Quantizing a weight, with no data": randomized Hadamard
// rotation along the input dimension, groups divided by their RMS, each value
// replaced by its nearest Lloyd-Max centroid, indices packed into 32-bit words
// (20 base-3 trits per word for the three-level book, "The ternary tier").
#include <math.h>

#include <algorithm>
#include <type_traits>

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

// Number of thresholds strictly below u, the book's thresholds in registers (unrolled).
template <int NT>
TQ_DEVFN uint32_t snap_reg(float u, const float (&t)[NT]) {
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < NT; ++i) c += (t[i] < u) ? 1u : 0u;
    return c;
}

// Word j of a packed row of a book of LEVELS codes from the codes in shared memory (0 beyond n).
template <int LEVELS>
TQ_DEVFN uint32_t pack_word_l(const uint8_t* codes, int n, int j) {
    constexpr int kCW = LEVELS == 3 ? 20 : (LEVELS == 8 ? 10 : (LEVELS == 4 ? 16 : 8));
    constexpr int kBits = LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4);
    uint32_t w = 0;
    const int k0 = j * kCW;
    if (k0 + kCW <= n) {
#pragma unroll
        for (int i = kCW - 1; i >= 0; --i) {
            const uint32_t c = codes[k0 + i];
            if constexpr (LEVELS == 3) w = w * 3u + c;
            else w |= c << (kBits * i);
        }
    } else {
#pragma unroll
        for (int i = kCW - 1; i >= 0; --i) {
            const uint32_t c = k0 + i < n ? codes[k0 + i] : 0u;
            if constexpr (LEVELS == 3) w = w * 3u + c;
            else w |= c << (kBits * i);
        }
    }
    return w;
}

// One CTA per row of cols = threads * E values: rotate (signs, FWHT blocks, 1/sqrt(block)), group
// RMS, snap each u = v / RMS (through one reciprocal per group) to the book of LEVELS codes,
// pack.  The thresholds sit in registers and every loop over codes is unrolled.
template <int E, int LEVELS>
__global__ void __launch_bounds__(1024) quantize_rows_kernel(const void* __restrict__ W, int wdt, int cols, int group,
                                                             int block, float rscale, const int8_t* __restrict__ signs,
                                                             const float* __restrict__ thresholds,
                                                             uint32_t* __restrict__ codes, uint16_t* __restrict__ scales,
                                                             int64_t row_stride) {
    constexpr int NT = LEVELS - 1;
    extern __shared__ float smem[];
    float* fw = smem;                                           // fwht_pad_floats(cols) (FWHT exchange)
    uint8_t* cd = reinterpret_cast<uint8_t*>(smem + fwht_pad_floats(cols) + 256);  // cols codes
    const int64_t row = blockIdx.x;
    const int base = threadIdx.x * E;
    const int lane = threadIdx.x & 31;
    float thr[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) thr[i] = __ldg(thresholds + i);

    float v[E];
    const int64_t off = row * cols + base;
    if (E >= 8 && wdt == TQ_BF16 && (reinterpret_cast<uintptr_t>(W) & 15) == 0 && (cols & 7) == 0 &&
        (reinterpret_cast<uintptr_t>(signs) & 7) == 0) {
        // 8 values and 8 signs per 16-byte / 8-byte load
#pragma unroll
        for (int c = 0; c < E; c += 8) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(W) + off + c));
            const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + base + c));
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
            const uint32_t s2[2] = {sg.x, sg.y};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t bits = k & 1 ? (w4[k >> 1] & 0xffff0000u) : (w4[k >> 1] << 16);
                const int sgn = (int)(int8_t)(s2[k >> 2] >> (8 * (k & 3)));
                v[c + k] = __uint_as_float(bits) * (float)sgn;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < E; ++i) v[i] = load_as_float(W, off + i, wdt) * (float)signs[base + i];
    }
    fwht_cta<E>(v, fw, block);  // ends with a barrier when it used shared memory
    __syncthreads();
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] *= rscale;

    const float inv_g = 1.0f / (float)group;
    const int ngroups = cols / group;
    uint32_t cpk[(E + 3) / 4];  // the thread's codes, four bytes to a word
#pragma unroll
    for (int q = 0; q < (E + 3) / 4; ++q) cpk[q] = 0u;
    if (E >= 16 && group <= 16) {  // a thread holds whole groups (E = 16, group 16): fixed indices
#pragma unroll
        for (int g0 = 0; g0 < E; g0 += 16) {
            float ss = 0.f;
#pragma unroll
            for (int i = g0; i < g0 + 16; ++i) ss += v[i] * v[i];
            const float s = sqrtf(ss * inv_g);
            scales[row * ngroups + (base + g0) / 16] = __half_as_ushort(__float2half_rn(s));
            const float r = s > 0.f ? 1.0f / s : 0.f;
#pragma unroll
            for (int i = g0; i < g0 + 16; ++i) cpk[i >> 2] |= snap_reg(v[i] * r, thr) << (8 * (i & 3));
        }
    } else {
        const int lpg = group / E;  // lanes per group, 2..32
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) ss += v[i] * v[i];
        for (int m = 1; m < lpg; m <<= 1) ss += __shfl_xor_sync(kFull, ss, m);
        const float s = sqrtf(ss * inv_g);
        if ((lane & (lpg - 1)) == 0) scales[row * ngroups + base / group] = __half_as_ushort(__float2half_rn(s));
        const float r = s > 0.f ? 1.0f / s : 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) cpk[i >> 2] |= snap_reg(v[i] * r, thr) << (8 * (i & 3));
    }
    if constexpr (E >= 4) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) reinterpret_cast<uint32_t*>(cd + base)[q] = cpk[q];
    } else {
#pragma unroll
        for (int i = 0; i < E; ++i) cd[base + i] = (uint8_t)(cpk[0] >> (8 * i));
    }
    __syncthreads();
    for (int64_t j = threadIdx.x; j < row_stride; j += blockDim.x)
        codes[row * row_stride + j] = pack_word_l<LEVELS>(cd, cols, (int)j);
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

// ---------------------------------------------------------------- KV vectors, 8-bit keys, group 32
//
// Persistent warps, one (token, kv head) vector pair (K and V) at a time, the next pair's
// inputs in flight while the current one is encoded.  A lane holds dims 4l .. 4l+3, so an
// 8-bit key word is exactly one lane's four codes.  The 255 key thresholds are looked up in
// a table of 1024 equal bins over [-4.5, 4.5): bin(x) = floor((x + 4.5) * 1024 / 9), the
// same float expression for the thresholds and for a value, so it is monotone in x.  The
// book's thresholds are at least 0.0169 apart, wider than a bin (0.0088), so a bin holds at
// most one; every threshold of a lower bin is below u, every one of a higher bin above, and
// code = (thresholds of lower bins) + (the bin's own threshold < u) is exactly the count of
// thresholds strictly below u.  Values are divided by the group scale through one
// reciprocal per group (a code can differ from a correctly rounded division only at a tie).
constexpr int kKvBins = 1024;
constexpr int kKvVBins = 64;  // value books: 8 or 16 levels, thresholds >= 0.258 apart, bins 0.14 wide
constexpr float kKvVBinScale = (float)kKvVBins / 9.0f;
// vector pairs per warp ring: 8 of bf16 (4 KB), 4 of fp32 (4 KB)
template <bool BF16>
constexpr int kv_ring_len() { return BF16 ? 8 : 4; }

// Pairs gw, gw + nw, ... below nvec.
TQ_DEVFN int64_t vec0_count(int64_t gw, int64_t nw, int64_t nvec) { return gw < nvec ? (nvec - gw + nw - 1) / nw : 0; }
constexpr float kKvLo = -4.5f, kKvBinScale = (float)kKvBins / 9.0f;

template <int VL, bool BF16>
__global__ void __launch_bounds__(256, 4) kv_quantize8_kernel(const void* __restrict__ k, const void* __restrict__ v,
                                                           int64_t nvec, int Hkv, int64_t pos, int64_t capacity,
                                                           float rscale, const int8_t* __restrict__ signs,
                                                           const float* __restrict__ kthr, const float* __restrict__ vthr,
                                                           uint32_t* __restrict__ kcodes, uint16_t* __restrict__ kscales,
                                                           uint32_t* __restrict__ vcodes, uint16_t* __restrict__ vscales) {
    constexpr int VB = VL == 8 ? 3 : 4, VCW = VL == 8 ? 10 : 8, VW = (128 + VCW - 1) / VCW;
    __shared__ float2 bins[kKvBins];  // (count of thresholds of lower bins, the bin's threshold or +inf)
    __shared__ float2 vbins[kKvVBins];
    __shared__ float kt[256];
    __shared__ int kb[256];
    __shared__ float vt[16];
    __shared__ int vb[16];
    constexpr int kRing = kv_ring_len<BF16>();
    __shared__ __align__(16) uint8_t kv_ring[8 * kRing * 2 * 128 * (BF16 ? 2 : 4)];  // [8 warps][kRing][pair]
    auto bin_of = [](float x) { return min(max(__float2int_rd((x - kKvLo) * kKvBinScale), 0), kKvBins - 1); };
    auto vbin_of = [](float x) { return min(max(__float2int_rd((x - kKvLo) * kKvVBinScale), 0), kKvVBins - 1); };
    for (int i = threadIdx.x; i < 255; i += blockDim.x) {
        kt[i] = __ldg(kthr + i);
        kb[i] = bin_of(kt[i]);
    }
    if (threadIdx.x < VL - 1) {
        vt[threadIdx.x] = __ldg(vthr + threadIdx.x);
        vb[threadIdx.x] = vbin_of(vt[threadIdx.x]);
    }
    __syncthreads();
    // bin b: (thresholds whose bin is below b, the one whose bin is b or +inf); the thresholds ascend
    auto fill = [&](float2* tab, int nb, const float* t, const int* tb, int n) {
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            int lo = 0, hi = n;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (tb[mid] < b) lo = mid + 1; else hi = mid;
            }
            tab[b] = make_float2(__int_as_float(lo), lo < n && tb[lo] == b ? t[lo] : INFINITY);
        }
    };
    fill(bins, kKvBins, kt, kb, 255);
    fill(vbins, kKvVBins, vt, vb, VL - 1);
    // A book whose thresholds share a bin (not a Gaussian Lloyd-Max book) is snapped by search.
    const bool kfast = __syncthreads_and(threadIdx.x >= 254 || kb[threadIdx.x] < kb[threadIdx.x + 1]);
    const bool vfast = __syncthreads_and(threadIdx.x >= VL - 2 || vb[threadIdx.x] < vb[threadIdx.x + 1]);
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t sg = __ldg(reinterpret_cast<const uint32_t*>(signs) + lane);  // signs of dims 4l .. 4l+3
    float sgn[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sgn[i] = (float)(int8_t)(sg >> (8 * i));

    // Per-warp ring of kRing vector pairs in shared memory, filled with 16-byte cp.async copies
    // (K then V, 32 lanes x ES / 2 copies per pair): kRing - 1 pairs in flight while one is encoded.
    constexpr int ES = BF16 ? 2 : 4, PAIR = 2 * 128 * ES, CPL = PAIR / (32 * 16);
    uint8_t* ring = kv_ring + (threadIdx.x >> 5) * kRing * PAIR;
    const int64_t nmine = vec0_count(gw, nw, nvec);  // pairs of this warp: gw, gw + nw, ...
    auto issue = [&](int64_t j) {  // pair j of this warp into slot j % kRing
        if (j < nmine) {
            const int64_t vec = gw + j * nw;
            uint8_t* dst = ring + (j % kRing) * PAIR;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int piece = lane + 32 * c;  // 16-byte piece of the pair
                const int half = piece >= (PAIR / 32) ? 1 : 0;
                const int off = piece * 16 - half * (PAIR / 2);
                const uint8_t* src = reinterpret_cast<const uint8_t*>(half ? v : k) + vec * (PAIR / 2) + off;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst + piece * 16)),
                             "l"(src)
                             : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    auto read4 = [&](const uint8_t* src, float (&x)[4]) {  // this lane's dims 4l .. 4l+3
        if (BF16) {
            const uint2 r = *reinterpret_cast<const uint2*>(src + lane * 8);
            x[0] = __uint_as_float(r.x << 16);
            x[1] = __uint_as_float(r.x & 0xffff0000u);
            x[2] = __uint_as_float(r.y << 16);
            x[3] = __uint_as_float(r.y & 0xffff0000u);
        } else {
            const float4 r = *reinterpret_cast<const float4*>(src + lane * 16);
            x[0] = r.x;
            x[1] = r.y;
            x[2] = r.z;
            x[3] = r.w;
        }
    };
    // rotate, then scale by the group RMS (8 lanes per group of 32): returns the fp16 scale bits
    auto prep = [&](float (&x)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] *= sgn[i];
        fwht_warp128(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] *= rscale;
        float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
        ss += __shfl_xor_sync(kFull, ss, 1);
        ss += __shfl_xor_sync(kFull, ss, 2);
        ss += __shfl_xor_sync(kFull, ss, 4);
        const float sc = sqrtf(ss * (1.0f / 32.0f));
        const float inv = sc > 0.f ? 1.0f / sc : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] *= inv;
        return __half_as_ushort(__float2half_rn(sc));
    };

    // the encode loop, once with the bin tables and once (any other book) with searches
    auto run = [&](auto fast_c) {
    constexpr bool FAST = decltype(fast_c)::value;
#pragma unroll 1
    for (int j = 0; j < kRing - 1; ++j) issue(j);
    // (token, head) of this warp's pair j, advanced by nw pairs per step without a division
    int64_t tok = gw / Hkv;
    int hh = (int)(gw - tok * Hkv);
    const int64_t dtok = nw / Hkv;
    const int dhh = (int)(nw - dtok * Hkv);
    for (int64_t j = 0; j < nmine; ++j) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 2) : "memory");  // pair j has landed (this lane's pieces)
        __syncwarp();                                                       // every lane's, and slot j - 1 is free
        issue(j + kRing - 1);
        const uint8_t* pr = ring + (j % kRing) * PAIR;
        float kx[4], vx[4];
        read4(pr, kx);
        read4(pr + PAIR / 2, vx);
        const int64_t slot = (int64_t)hh * capacity + pos + tok;
        tok += dtok;
        hh += dhh;
        if (hh >= Hkv) {
            hh -= Hkv;
            ++tok;
        }
        const uint16_t ks = prep(kx), vs = prep(vx);
        // keys: one word per lane
        uint32_t kw = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float u = kx[i];
            int c;
            if constexpr (FAST) {
                const float2 e = bins[bin_of(u)];
                c = __float_as_int(e.x) + (e.y < u ? 1 : 0);
            } else {
                c = snap_code(u, kt, 255);
            }
            kw |= (uint32_t)c << (8 * i);
        }
        kcodes[slot * 32 + lane] = kw;
        // values: lane's four codes, then word j gathers codes 10j .. 10j+9 (3-bit) or 8j .. 8j+7
        uint32_t vc4 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int c;
            if constexpr (FAST) {
                const float2 e = vbins[vbin_of(vx[i])];
                c = __float_as_int(e.x) + (e.y < vx[i] ? 1 : 0);
            } else {
                c = snap_code(vx[i], vt, VL - 1);
            }
            vc4 |= (uint32_t)c << (VB * i);
        }
        uint32_t vw = 0;
        const int first = lane * VCW;  // first dim of word `lane`
        const int src0 = min(first >> 2, 31);
        const uint32_t a0 = __shfl_sync(kFull, vc4, src0), a1 = __shfl_sync(kFull, vc4, min(src0 + 1, 31)),
                       a2 = __shfl_sync(kFull, vc4, min(src0 + 2, 31));
        // the three lanes' 12 codes as one bit string, then the word's VCW codes from dim `first`
        const uint64_t cat = (uint64_t)a0 | ((uint64_t)a1 << (4 * VB)) | ((uint64_t)a2 << (8 * VB));
        vw = (uint32_t)(cat >> (VB * (first & 3)));
        if (VCW * VB < 32) vw &= (1u << (VCW * VB)) - 1u;
        if (lane == VW - 1 && 128 % VCW) vw &= (1u << (VB * (128 % VCW))) - 1u;  // last word: past dim 127 is 0
        if (lane < VW) vcodes[slot * VW + lane] = vw;
        // scales: lanes 0, 8, 16, 24 hold their group's
        if ((lane & 7) == 0) {
            kscales[slot * 4 + (lane >> 3)] = ks;
            vscales[slot * 4 + (lane >> 3)] = vs;
        }
    }    };
    if (kfast && vfast) run(std::true_type{}); else run(std::false_type{});
}

// Elements per thread: smallest power of two E with whole warps (dim % 32E == 0),
// at most 1024 threads, E <= block, and a group spread over at most one warp
// (group / E <= 32) so the group's sum of squares is a warp-shuffle reduction.
// Values per thread: the most (up to 16) that still give whole warps, so that more of the
// transform runs in registers and shuffles and fewer stages go through shared memory.
// Encode of rows whose rotation is diagonal (block 1: the signs alone), for widths the fused
// kernel's layout does not take (e.g. rows already rotated by a dense rotation): one CTA per row,
// a thread per group for the RMS and the codes, then a thread per word for the packing.
__global__ void __launch_bounds__(256) quantize_diag_kernel(const void* __restrict__ W, int wdt, int cols, int group,
                                                            const int8_t* __restrict__ signs,
                                                            const float* __restrict__ thresholds, int levels,
                                                            uint32_t* __restrict__ codes,
                                                            uint16_t* __restrict__ scales, int64_t row_stride) {
    extern __shared__ float smem[];
    float* thr = smem;                                       // levels-1 thresholds
    uint8_t* cd = reinterpret_cast<uint8_t*>(smem + 256);   // [cols] codes of the row
    const int nthr = levels - 1;
    for (int i = threadIdx.x; i < nthr; i += blockDim.x) thr[i] = thresholds[i];
    __syncthreads();
    const int64_t row = blockIdx.x;
    const int64_t off = row * cols;
    const int ngroups = cols / group;
    for (int g = threadIdx.x; g < ngroups; g += blockDim.x) {
        float ss = 0.f;
        for (int i = 0; i < group; ++i) {
            const int k = g * group + i;
            const float v = load_as_float(W, off + k, wdt) * (float)signs[k];
            ss += v * v;
        }
        const float s = sqrtf(ss * (1.0f / (float)group));
        scales[row * ngroups + g] = __half_as_ushort(__float2half_rn(s));
        for (int i = 0; i < group; ++i) {
            const int k = g * group + i;
            const float v = load_as_float(W, off + k, wdt) * (float)signs[k];
            const float u = s > 0.f ? __fdiv_rn(v, s) : 0.f;
            cd[k] = (uint8_t)snap_code(u, thr, nthr);
        }
    }
    __syncthreads();
    const int cw = levels == 3 ? 20 : (levels == 8 ? 10 : 32 / (31 - __clz(levels)));
    const int bits = 31 - __clz(levels);
    for (int64_t j = threadIdx.x; j < row_stride; j += blockDim.x)
        codes[row * row_stride + j] = pack_word(cd, cols, (int)j, levels, cw, bits);
}

template <int E, int LEVELS>
tq_status quantize_rows_launch(const void* W, tq_dtype wdt, int64_t rows, int32_t cols, int32_t group,
                               const tq_rotation_t* rot, const tq_codebook_t* cb, uint32_t* codes, uint16_t* scales,
                               int64_t row_stride_words, size_t smem, float rscale, cudaStream_t st) {
    if (ensure_smem((const void*)quantize_rows_kernel<E, LEVELS>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    quantize_rows_kernel<E, LEVELS><<<(unsigned)rows, cols / E, smem, st>>>(
        W, wdt, cols, group, rot->block, rscale, rot->signs, cb->thresholds, codes, scales, row_stride_words);
    return launch_status();
}

template <int E>
tq_status quantize_rows_e(const void* W, tq_dtype wdt, int64_t rows, int32_t cols, int32_t group,
                          const tq_rotation_t* rot, const tq_codebook_t* cb, uint32_t* codes, uint16_t* scales,
                          int64_t row_stride_words, size_t smem, float rscale, cudaStream_t st) {
    switch (cb->levels) {
        case 3: return quantize_rows_launch<E, 3>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 4: return quantize_rows_launch<E, 4>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 8: return quantize_rows_launch<E, 8>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 16: return quantize_rows_launch<E, 16>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

int pick_e(int dim, int block, int group) {
    for (int e = 16; e >= 1; e >>= 1)
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
    if ((e == 0 || cols > 16384) && rot->block == 1 && cols <= 65536) {  // a diagonal rotation
        const size_t smem_d = 256 * 4 + (size_t)cols;
        if (ensure_smem((const void*)quantize_diag_kernel, smem_d) != cudaSuccess) return TQ_ERR_CUDA;
        quantize_diag_kernel<<<(unsigned)rows, 256, smem_d, as_stream(stream)>>>(
            W, wdt, cols, group, rot->signs, cb->thresholds, cb->levels, codes, scales, row_stride_words);
        return launch_status();
    }
    if (e == 0 || cols > 16384) return TQ_ERR_UNSUPPORTED;
    const size_t smem = fwht_pad_floats(cols) * 4 + 256 * 4 + (size_t)cols;
    const float rscale = (float)(1.0 / sqrt((double)rot->block));
    cudaStream_t st = as_stream(stream);
    switch (e) {
        case 1: return quantize_rows_e<1>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 2: return quantize_rows_e<2>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 4: return quantize_rows_e<4>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 8: return quantize_rows_e<8>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        case 16: return quantize_rows_e<16>(W, wdt, rows, cols, group, rot, cb, codes, scales, row_stride_words, smem, rscale, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
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
    const float rscale = (float)(1.0 / sqrt((double)D));
    // 8-bit keys, 3- or 4-bit values, groups of 32: the persistent kernel above
    const uintptr_t need = 15;  // 16-byte copies of the inputs
    if (kcb->levels == 256 && (vcb->levels == 8 || vcb->levels == 16) && group == 32 &&
        ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & need) == 0 &&
        (reinterpret_cast<uintptr_t>(rot->signs) & 3) == 0) {
        static int sms = 0;
        if (sms == 0) {
            int dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        }
        const int64_t blocks = std::min<int64_t>((nvec + 7) / 8, (int64_t)sms * 4);
        cudaStream_t st = as_stream(stream);
#define TQ_KV8(VL, BF)                                                                                            \
    kv_quantize8_kernel<VL, BF><<<(unsigned)blocks, 256, 0, st>>>(k, v, nvec, Hkv, pos, capacity, rscale, rot->signs, \
                                                                   kcb->thresholds, vcb->thresholds, kcodes, kscales,  \
                                                                   vcodes, vscales)
        if (vcb->levels == 8) {
            if (dt == TQ_BF16) TQ_KV8(8, true); else TQ_KV8(8, false);
        } else {
            if (dt == TQ_BF16) TQ_KV8(16, true); else TQ_KV8(16, false);
        }
#undef TQ_KV8
        return launch_status();
    }
    const int warps = 8;
    const int64_t blocks = (nvec + warps - 1) / warps;
    if (blocks > 0x7fffffffll) return TQ_ERR_INVALID;
    kv_quantize_kernel<<<(unsigned)blocks, warps * 32, 0, as_stream(stream)>>>(
        k, v, dt, T, Hkv, pos, capacity, (float)(1.0 / sqrt((double)D)), rot->signs, kcb->thresholds, kcb->levels,
        vcb->thresholds, vcb->levels, group, kcodes, kscales, vcodes, vscales, kw, vw);
    return launch_status();
}
