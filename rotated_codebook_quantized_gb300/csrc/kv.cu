// One decode step of attention read straight from the compressed KV cache:
// tq_kv_attend.
//
// "Running a 1T-Parameter Model on a Laptop", update_and_fetch: the cache is
// dequantized and de-rotated, then softmax(q K^T / sqrt(D)) V.  Rotation is
// orthonormal, so q . k = (R q) . (R k): the query is rotated once, scores use
// the rotated, dequantized keys as stored, and the weighted sum of rotated
// values is de-rotated once at the end.  "How it works", "The KV cache": the
// same rotation and codebook as the weights (8-bit keys, 3-bit values).
//
// Split-context (flash-decoding) layout: CTA (kv head, chunk) scores its chunk
// of tokens for the Hq/Hkv query heads that share the kv head, keeps the
// chunk's max and sum, and writes an unnormalised partial output; a second
// kernel merges the chunks and de-rotates.
#include <math.h>

#include <mutex>

#include <cuda.h>

#include "common.cuh"

using namespace tq;

namespace {

constexpr int kD = 128;
constexpr int kChunk = 1024;   // tokens per CTA
constexpr int kThreads = 256;  // 8 warps
constexpr int kMaxGQ = 8;      // query heads per kv head

template <int LEVELS>
struct KvFmt {
    static constexpr int kBits = LEVELS == 256 ? 8 : (LEVELS == 16 ? 4 : (LEVELS == 8 ? 3 : 2));
    static constexpr int kCW = LEVELS == 8 ? 10 : 32 / kBits;
    static constexpr int kWords = (kD + kCW - 1) / kCW;
};

template <int KL, int VL, int GQ>
__global__ void __launch_bounds__(kThreads) kv_partial_kernel(
    const void* __restrict__ q, int qdt, int Hkv, int64_t ctx, int64_t capacity, const int8_t* __restrict__ signs,
    const float* __restrict__ kcent, const float* __restrict__ vcent, int group,
    const uint32_t* __restrict__ kcodes, const uint16_t* __restrict__ kscales, const uint32_t* __restrict__ vcodes,
    const uint16_t* __restrict__ vscales, float* __restrict__ part, int nsplit) {
    using KF = KvFmt<KL>;
    using VF = KvFmt<VL>;
    __shared__ __align__(16) float qs[GQ][kD];  // rotated query / sqrt(D)
    __shared__ float klut[KL];
    __shared__ float vlut[VL];
    __shared__ float sc[GQ][kChunk];           // scores, then probabilities
    __shared__ float obuf[GQ][kD];             // sum over warps of the weighted values
    __shared__ float stat[GQ][2];

    const int h = blockIdx.x, split = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)split * kChunk;
    const int n = (int)min((int64_t)kChunk, ctx - t0);
    const int ng = kD / group;

    for (int i = threadIdx.x; i < KL; i += kThreads) klut[i] = kcent[i];
    for (int i = threadIdx.x; i < GQ * kD; i += kThreads) (&obuf[0][0])[i] = 0.f;
    for (int i = threadIdx.x; i < VL; i += kThreads) vlut[i] = vcent[i];
    // q_rot = H diag(s) q / sqrt(D), and the 1/sqrt(D) of the scores folded in.
    for (int g = warp; g < GQ; g += kThreads / 32) {
        const int hq = h * GQ + g;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = load_as_float(q, (int64_t)hq * kD + lane * 4 + i, qdt) * (float)signs[lane * 4 + i];
        fwht_warp128(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[g][lane * 4 + i] = v[i] * (1.0f / 128.0f);  // (1/sqrt(128))^2
    }
    __syncthreads();

    // Scores: one thread per token; the query is read with broadcast loads.
    const uint32_t* kbase = kcodes + ((int64_t)h * capacity + t0) * KF::kWords;
    const uint16_t* ksbase = kscales + ((int64_t)h * capacity + t0) * ng;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t* kr = kbase + (int64_t)i * KF::kWords;
        const uint16_t* sr = ksbase + (int64_t)i * ng;
        float acc[GQ], tot[GQ];
#pragma unroll
        for (int g = 0; g < GQ; ++g) tot[g] = 0.f;
        for (int g0 = 0; g0 < ng; ++g0) {
#pragma unroll
            for (int g = 0; g < GQ; ++g) acc[g] = 0.f;
            for (int d = g0 * group; d < (g0 + 1) * group; ++d) {
                const uint32_t w = kr[d / KF::kCW];
                const uint32_t c = (w >> (KF::kBits * (d % KF::kCW))) & (KL - 1);
                const float cv = klut[c];
#pragma unroll
                for (int g = 0; g < GQ; ++g) acc[g] = fmaf(cv, qs[g][d], acc[g]);
            }
            const float s = half_bits_to_float(sr[g0]);
#pragma unroll
            for (int g = 0; g < GQ; ++g) tot[g] = fmaf(s, acc[g], tot[g]);
        }
#pragma unroll
        for (int g = 0; g < GQ; ++g) sc[g][i] = tot[g];
    }
    __syncthreads();

    // Chunk max and sum per head (warp g handles head g).
    for (int g = warp; g < GQ; g += kThreads / 32) {
        float m = -INFINITY;
        for (int i = lane; i < n; i += 32) m = fmaxf(m, sc[g][i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float l = 0.f;
        for (int i = lane; i < n; i += 32) {
            const float p = expf(sc[g][i] - m);
            sc[g][i] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
        if (lane == 0) {
            stat[g][0] = m;
            stat[g][1] = l;
        }
    }
    __syncthreads();

    // Weighted sum of rotated values: warp per token, lane owns dims 4l..4l+3.
    float o[GQ][4];
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[g][j] = 0.f;
    const uint32_t* vbase = vcodes + ((int64_t)h * capacity + t0) * VF::kWords;
    const uint16_t* vsbase = vscales + ((int64_t)h * capacity + t0) * ng;
    const int gl = (lane * 4) / group;  // the lane's four dims share one group (group >= 4)
    for (int i = warp; i < n; i += kThreads / 32) {
        const uint32_t* vr = vbase + (int64_t)i * VF::kWords;
        const float s = half_bits_to_float(vsbase[(int64_t)i * ng + gl]);
        float vv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int d = lane * 4 + j;
            const uint32_t w = vr[d / VF::kCW];
            vv[j] = s * vlut[(w >> (VF::kBits * (d % VF::kCW))) & (VL - 1)];
        }
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            const float p = sc[g][i];
#pragma unroll
            for (int j = 0; j < 4; ++j) o[g][j] = fmaf(p, vv[j], o[g][j]);
        }
    }
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int j = 0; j < 4; ++j) atomicAdd(&obuf[g][lane * 4 + j], o[g][j]);
    __syncthreads();
    // part[(split * Hq + hq) * (D + 2)] = {m, l, o[0..D)}
    for (int idx = threadIdx.x; idx < GQ * kD; idx += kThreads) {
        const int g = idx / kD, d = idx % kD;
        const float sum = obuf[g][d];
        const int hq = h * GQ + g;
        float* dst = part + ((int64_t)split * Hkv * GQ + hq) * (kD + 2);
        dst[2 + d] = sum;
        if (d == 0) {
            dst[0] = stat[g][0];
            dst[1] = stat[g][1];
        }
    }
}

// Merge the chunks of one query head and de-rotate: o = diag(s) H o_rot / sqrt(D).
__global__ void __launch_bounds__(32) kv_merge_kernel(const float* __restrict__ part, int Hq, int nsplit,
                                                      const int8_t* __restrict__ signs, float* __restrict__ out) {
    const int hq = blockIdx.x, lane = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part[((int64_t)s * Hq + hq) * (kD + 2)]);
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < nsplit; ++s) {
        const float* src = part + ((int64_t)s * Hq + hq) * (kD + 2);
        const float f = expf(src[0] - M);
        L = fmaf(f, src[1], L);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = fmaf(f, src[2 + lane * 4 + j], acc[j]);
    }
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = acc[j] / L;
    fwht_warp128(v);
    const float r = 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
    for (int j = 0; j < 4; ++j) out[(int64_t)hq * kD + lane * 4 + j] = v[j] * r * (float)signs[lane * 4 + j];
}

// ---------------------------------------------------------------- 8-bit keys, group 32
//
// Same split-context layout, built for the cache the pages describe (8-bit keys
// with a 256-level book, 3- or 4-bit values, groups of 32):
//  * scores: a lane owns two tokens of the chunk and reads their key rows (128
//    bytes each) with 16-byte loads; a code indexes a per-lane copy of the
//    256-entry book in shared memory, and the rotated query of every head is a
//    broadcast load per dimension; a group's partial sums are scaled once;
//  * weighted values: a lane owns 8 dimensions for every token of its half warp,
//    the row's codes arrive with one 64-bit funnel shift (3-bit words hold 10
//    codes in bits 0..29, so word b shifted left by 30 continues word a), and
//    p * s_v is formed once per token and head.
constexpr int kGroupF = 32;

TQ_DEVFN void cp_async16_kv(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
TQ_DEVFN void cp_async4_kv(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}

template <int VL, int GQ>
struct KvFast {
    static constexpr int kVB = VL == 8 ? 3 : 4;        // value bits
    static constexpr int kVCW = VL == 8 ? 10 : 8;      // value codes per word
    static constexpr int kVW = (kD + kVCW - 1) / kVCW;  // value words per token
    static constexpr size_t kVStage = (size_t)kChunk * kVW * 4 + (size_t)kChunk * 4 * 2;  // value codes + scales
    static constexpr size_t kSmem =
        sizeof(float) * (256 * 32 + (size_t)kD * GQ + (size_t)GQ * kChunk + (size_t)GQ * kD + 16 + 2 * GQ) + kVStage;
};

template <int VL, int GQ>
__global__ void __launch_bounds__(kThreads, 2) kv_partial8_kernel(
    const void* __restrict__ q, int qdt, int Hkv, int64_t ctx, int64_t capacity, const int8_t* __restrict__ signs,
    const float* __restrict__ kcent, const float* __restrict__ vcent, const uint32_t* __restrict__ kcodes,
    const uint16_t* __restrict__ kscales, const uint32_t* __restrict__ vcodes, const uint16_t* __restrict__ vscales,
    float* __restrict__ part) {
    using V = KvFast<VL, GQ>;
    constexpr int NG = kD / kGroupF;  // 4 groups per row
    extern __shared__ __align__(16) float smf[];
    float* klut = smf;                   // [256][32]: entry c of lane l at c * 32 + l
    float* qs = klut + 256 * 32;         // [kD][GQ]: rotated query / sqrt(D), per dimension
    float* sc = qs + kD * GQ;            // [GQ][kChunk]: scores, then probabilities
    float* obuf = sc + GQ * kChunk;      // [GQ][kD]
    float* vlut = obuf + GQ * kD;        // [16]
    float* stat = vlut + 16;             // [GQ][2]
    uint32_t* vstage = reinterpret_cast<uint32_t*>(stat + 2 * GQ);                 // [kChunk][kVW] value codes
    uint16_t* vsstage = reinterpret_cast<uint16_t*>(vstage + kChunk * V::kVW);   // [kChunk][4] value scales

    const int h = blockIdx.x, split = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)split * kChunk;
    const int n = (int)min((int64_t)kChunk, ctx - t0);

    {
        // the chunk's value codes and scales stream into shared memory during the scores
        const uint32_t* vsrc = vcodes + ((int64_t)h * capacity + t0) * V::kVW;
        const uint16_t* vssrc = vscales + ((int64_t)h * capacity + t0) * NG;
        const int vwords = n * V::kVW, vsw = n * NG / 2;  // NG = 4 halves per token: whole words
        if (((reinterpret_cast<uintptr_t>(vsrc) | reinterpret_cast<uintptr_t>(vstage)) & 15) == 0) {
            for (int i = threadIdx.x; i < vwords / 4; i += kThreads) cp_async16_kv(vstage + 4 * i, vsrc + 4 * i);
            for (int i = vwords / 4 * 4 + threadIdx.x; i < vwords; i += kThreads) cp_async4_kv(vstage + i, vsrc + i);
        } else {
            for (int i = threadIdx.x; i < vwords; i += kThreads) cp_async4_kv(vstage + i, vsrc + i);
        }
        const uint32_t* vss32 = reinterpret_cast<const uint32_t*>(vssrc);
        for (int i = threadIdx.x; i < vsw; i += kThreads) cp_async4_kv(reinterpret_cast<uint32_t*>(vsstage) + i, vss32 + i);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int i = threadIdx.x; i < 256 * 32; i += kThreads) klut[i] = __ldg(kcent + (i >> 5));
    for (int i = threadIdx.x; i < GQ * kD; i += kThreads) obuf[i] = 0.f;
    if (threadIdx.x < VL) vlut[threadIdx.x] = __ldg(vcent + threadIdx.x);
    // q_rot = H diag(s) q / sqrt(D), and the 1/sqrt(D) of the scores folded in.
    for (int g = warp; g < GQ; g += kThreads / 32) {
        const int hq = h * GQ + g;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = load_as_float(q, (int64_t)hq * kD + lane * 4 + i, qdt) * (float)signs[lane * 4 + i];
        fwht_warp128(v);
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[(lane * 4 + i) * GQ + g] = v[i] * (1.0f / 128.0f);  // (1/sqrt(128))^2
    }
    __syncthreads();

    // ---- scores: lane takes tokens i and i + 32 of each 64-token slice of its warp
    const float* kl = klut + lane;
    const uint4* kbase = reinterpret_cast<const uint4*>(kcodes + ((int64_t)h * capacity + t0) * (kD / 4));
    const uint2* ksbase = reinterpret_cast<const uint2*>(kscales + ((int64_t)h * capacity + t0) * NG);
    for (int i0 = warp * 64; i0 < n; i0 += (kThreads / 32) * 64) {
        const int ia = i0 + lane, ib = i0 + 32 + lane;
        const bool va = ia < n, vb = ib < n;
        const uint4* ra = kbase + (int64_t)(va ? ia : 0) * 8;
        const uint4* rb = kbase + (int64_t)(vb ? ib : 0) * 8;
        const uint2 sa2 = va ? __ldg(ksbase + ia) : make_uint2(0u, 0u);
        const uint2 sb2 = vb ? __ldg(ksbase + ib) : make_uint2(0u, 0u);
        float tota[GQ], totb[GQ];
#pragma unroll
        for (int g = 0; g < GQ; ++g) tota[g] = totb[g] = 0.f;
        // a group's two 16-byte loads per row are in flight while the previous group is decoded
        uint4 na[2], nb[2];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
            na[hc] = va ? __ldg(ra + hc) : make_uint4(0u, 0u, 0u, 0u);
            nb[hc] = vb ? __ldg(rb + hc) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll 1
        for (int grp = 0; grp < NG; ++grp) {
            float pa[GQ], pb[GQ];
#pragma unroll
            for (int g = 0; g < GQ; ++g) pa[g] = pb[g] = 0.f;
            const uint4 ca[2] = {na[0], na[1]}, cb[2] = {nb[0], nb[1]};
            if (grp + 1 < NG) {
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    na[hc] = va ? __ldg(ra + (grp + 1) * 2 + hc) : make_uint4(0u, 0u, 0u, 0u);
                    nb[hc] = vb ? __ldg(rb + (grp + 1) * 2 + hc) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {  // 16 dimensions per 16-byte load
                const int c = grp * 2 + hc;
                const uint4 wa = ca[hc];
                const uint4 wb = cb[hc];
                const uint32_t aw[4] = {wa.x, wa.y, wa.z, wa.w}, bw[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int d = c * 16 + w * 4 + b;
                        const float ka = kl[((aw[w] >> (8 * b)) & 255u) * 32];
                        const float kb = kl[((bw[w] >> (8 * b)) & 255u) * 32];
                        float qd[GQ];
                        if constexpr (GQ % 4 == 0) {
#pragma unroll
                            for (int g = 0; g < GQ; g += 4) {
                                const float4 q4 = *reinterpret_cast<const float4*>(qs + d * GQ + g);
                                qd[g] = q4.x;
                                qd[g + 1] = q4.y;
                                qd[g + 2] = q4.z;
                                qd[g + 3] = q4.w;
                            }
                        } else {
#pragma unroll
                            for (int g = 0; g < GQ; ++g) qd[g] = qs[d * GQ + g];
                        }
#pragma unroll
                        for (int g = 0; g < GQ; ++g) {
                            pa[g] = fmaf(ka, qd[g], pa[g]);
                            pb[g] = fmaf(kb, qd[g], pb[g]);
                        }
                    }
                }
            }
            const uint32_t swa = grp < 2 ? sa2.x : sa2.y, swb = grp < 2 ? sb2.x : sb2.y;
            const float sa = half_bits_to_float((uint16_t)(swa >> (16 * (grp & 1))));
            const float sb = half_bits_to_float((uint16_t)(swb >> (16 * (grp & 1))));
#pragma unroll
            for (int g = 0; g < GQ; ++g) {
                tota[g] = fmaf(sa, pa[g], tota[g]);
                totb[g] = fmaf(sb, pb[g], totb[g]);
            }
        }
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            if (va) sc[g * kChunk + ia] = tota[g];
            if (vb) sc[g * kChunk + ib] = totb[g];
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's value copies
    __syncthreads();                                       // everyone's, and the scores

    // ---- chunk max and sum per head (warp g handles head g)
    for (int g = warp; g < GQ; g += kThreads / 32) {
        float m = -INFINITY;
        for (int i = lane; i < n; i += 32) m = fmaxf(m, sc[g * kChunk + i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float l = 0.f;
        for (int i = lane; i < n; i += 32) {
            const float pr = expf(sc[g * kChunk + i] - m);
            sc[g * kChunk + i] = pr;
            l += pr;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
        if (lane == 0) {
            stat[2 * g] = m;
            stat[2 * g + 1] = l;
        }
    }
    __syncthreads();

    // ---- weighted sum of rotated values: half warp per token, lane owns dims 8 dl .. 8 dl + 7
    const int half = lane >> 4, dl = lane & 15;
    const int vgrp = (8 * dl) / kGroupF;
    const int wlo = (8 * dl) / V::kVCW, whi = (8 * dl + 7) / V::kVCW;
    const int vstart = V::kVB * ((8 * dl) % V::kVCW);
    float o[GQ][8];
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int j = 0; j < 8; ++j) o[g][j] = 0.f;
    for (int i = warp * 2 + half; i < n; i += (kThreads / 32) * 2) {
        const uint32_t* vr = vstage + i * V::kVW;
        uint32_t bits;
        if constexpr (V::kVB == 3) {
            const uint64_t c64 = (uint64_t)vr[wlo] | ((uint64_t)vr[whi] << 30);
            bits = (uint32_t)(c64 >> vstart);
        } else {
            bits = vr[dl];
        }
        const float s = half_bits_to_float(vsstage[i * NG + vgrp]);
        float cv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) cv[j] = vlut[(bits >> (V::kVB * j)) & (VL - 1)];
#pragma unroll
        for (int g = 0; g < GQ; ++g) {
            const float pw = sc[g * kChunk + i] * s;
#pragma unroll
            for (int j = 0; j < 8; ++j) o[g][j] = fmaf(pw, cv[j], o[g][j]);
        }
    }
#pragma unroll
    for (int g = 0; g < GQ; ++g)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float v = o[g][j] + __shfl_xor_sync(kFull, o[g][j], 16);
            if (half == 0) atomicAdd(obuf + g * kD + 8 * dl + j, v);
        }
    __syncthreads();
    // part[(split * Hq + hq) * (D + 2)] = {m, l, o[0..D)}
    for (int idx = threadIdx.x; idx < GQ * kD; idx += kThreads) {
        const int g = idx / kD, d = idx % kD;
        const int hq = h * GQ + g;
        float* dst = part + ((int64_t)split * Hkv * GQ + hq) * (kD + 2);
        dst[2 + d] = obuf[idx];
        if (d == 0) {
            dst[0] = stat[2 * g];
            dst[1] = stat[2 * g + 1];
        }
    }
}

template <int VL>
tq_status launch_kv8(int gq, dim3 grid, cudaStream_t st, const void* q, int qdt, int Hkv, int64_t ctx,
                     int64_t capacity, const int8_t* signs, const float* kc, const float* vc, const uint32_t* kcodes,
                     const uint16_t* kscales, const uint32_t* vcodes, const uint16_t* vscales, float* part) {
#define TQ_KV8_GQ(G)                                                                                           \
    case G: {                                                                                                  \
        const void* fn = (const void*)kv_partial8_kernel<VL, G>;                                              \
        if (ensure_smem(fn, KvFast<VL, G>::kSmem) != cudaSuccess) return TQ_ERR_CUDA;                          \
        kv_partial8_kernel<VL, G><<<grid, kThreads, KvFast<VL, G>::kSmem, st>>>(                               \
            q, qdt, Hkv, ctx, capacity, signs, kc, vc, kcodes, kscales, vcodes, vscales, part);                \
        break;                                                                                                 \
    }
    switch (gq) {
        TQ_KV8_GQ(1)
        TQ_KV8_GQ(2)
        TQ_KV8_GQ(4)
        TQ_KV8_GQ(8)
        default: return TQ_ERR_UNSUPPORTED;
    }
#undef TQ_KV8_GQ
    return launch_status();
}

template <int KL, int VL>
tq_status launch_kv(int gq, dim3 grid, cudaStream_t st, const void* q, int qdt, int Hkv, int64_t ctx, int64_t capacity,
                    const int8_t* signs, const float* kc, const float* vc, int group, const uint32_t* kcodes,
                    const uint16_t* kscales, const uint32_t* vcodes, const uint16_t* vscales, float* part, int nsplit) {
#define TQ_KV_GQ(G)                                                                                                \
    case G:                                                                                                        \
        kv_partial_kernel<KL, VL, G><<<grid, kThreads, 0, st>>>(q, qdt, Hkv, ctx, capacity, signs, kc, vc, group,  \
                                                                kcodes, kscales, vcodes, vscales, part, nsplit);   \
        break;
    switch (gq) {
        TQ_KV_GQ(1)
        TQ_KV_GQ(2)
        TQ_KV_GQ(4)
        TQ_KV_GQ(8)
        default: return TQ_ERR_UNSUPPORTED;
    }
#undef TQ_KV_GQ
    return launch_status();
}

}  // namespace

extern "C" size_t tq_kv_attend_workspace_bytes(int32_t Hq, int32_t D, int64_t ctx) {
    if (Hq <= 0 || D <= 0 || ctx <= 0) return 0;
    const int64_t nsplit = (ctx + kChunk - 1) / kChunk;
    return (size_t)nsplit * Hq * (D + 2) * sizeof(float);
}

extern "C" tq_status tq_kv_attend(const void* q, tq_dtype qdt, int32_t Hq, int32_t Hkv, int32_t D, int64_t ctx,
                                  int64_t capacity, const tq_rotation_t* rot, const tq_codebook_t* kcb,
                                  const tq_codebook_t* vcb, int32_t group, const uint32_t* kcodes,
                                  const uint16_t* kscales, const uint32_t* vcodes, const uint16_t* vscales, float* o,
                                  void* ws, size_t ws_bytes, void* stream) {
    if (D != kD) return TQ_ERR_UNSUPPORTED;
    if (!rot || !rot->signs || rot->dim != D || rot->block != D) return TQ_ERR_INVALID;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || ctx <= 0 || ctx > capacity) return TQ_ERR_INVALID;
    if (!(group == 16 || group == 32 || group == 64 || group == 128)) return TQ_ERR_INVALID;
    if (!kcb || !vcb || !kcb->centroids || !vcb->centroids) return TQ_ERR_INVALID;
    if (qdt != TQ_F32 && qdt != TQ_BF16) return TQ_ERR_INVALID;
    if (!q || !kcodes || !kscales || !vcodes || !vscales || !o || !ws) return TQ_ERR_INVALID;
    if (ws_bytes < tq_kv_attend_workspace_bytes(Hq, D, ctx)) return TQ_ERR_INVALID;
    const int gq = Hq / Hkv;
    if (gq > kMaxGQ || (gq & (gq - 1))) return TQ_ERR_UNSUPPORTED;
    const int64_t nsplit = (ctx + kChunk - 1) / kChunk;
    if (nsplit > 65535 || Hkv > 65535) return TQ_ERR_UNSUPPORTED;
    cudaStream_t st = as_stream(stream);
    float* part = reinterpret_cast<float*>(ws);
    const dim3 grid(Hkv, (unsigned)nsplit);
    tq_status s;
    const int kl = kcb->levels, vl = vcb->levels;
    // 8-bit keys in groups of 32 with 16-byte aligned key rows: the kernel above
    const bool k8 = kl == 256 && (vl == 8 || vl == 16) && group == kGroupF &&
                    (reinterpret_cast<uintptr_t>(kcodes) & 15) == 0 && (reinterpret_cast<uintptr_t>(kscales) & 7) == 0 &&
                    (reinterpret_cast<uintptr_t>(vcodes) & 3) == 0 && (reinterpret_cast<uintptr_t>(vscales) & 3) == 0;
    if (k8)
        s = vl == 8 ? launch_kv8<8>(gq, grid, st, q, qdt, Hkv, ctx, capacity, rot->signs, kcb->centroids,
                                    vcb->centroids, kcodes, kscales, vcodes, vscales, part)
                    : launch_kv8<16>(gq, grid, st, q, qdt, Hkv, ctx, capacity, rot->signs, kcb->centroids,
                                     vcb->centroids, kcodes, kscales, vcodes, vscales, part);
    else if (kl == 256 && vl == 8)
        s = launch_kv<256, 8>(gq, grid, st, q, qdt, Hkv, ctx, capacity, rot->signs, kcb->centroids, vcb->centroids,
                              group, kcodes, kscales, vcodes, vscales, part, (int)nsplit);
    else if (kl == 16 && vl == 16)
        s = launch_kv<16, 16>(gq, grid, st, q, qdt, Hkv, ctx, capacity, rot->signs, kcb->centroids, vcb->centroids,
                              group, kcodes, kscales, vcodes, vscales, part, (int)nsplit);
    else if (kl == 256 && vl == 16)
        s = launch_kv<256, 16>(gq, grid, st, q, qdt, Hkv, ctx, capacity, rot->signs, kcb->centroids, vcb->centroids,
                               group, kcodes, kscales, vcodes, vscales, part, (int)nsplit);
    else
        return TQ_ERR_UNSUPPORTED;
    if (s != TQ_OK) return s;
    kv_merge_kernel<<<Hq, 32, 0, st>>>(part, Hq, (int)nsplit, rot->signs, o);
    return launch_status();
}

// ---------------------------------------------------------------- allocation-free variant

namespace {

// Scratch of the allocation-free entry point: a fixed array in the library's
// device image.  Every GPU that loads the library holds it until the process
// exits; all calls on a device share it.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) float g_kv_attend_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // id of the context the address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the current CUDA context (0 if the driver cannot say).  A context that
// cudaDeviceReset destroyed and the runtime re-created gets a new id, so an address cached for
// the old one is never reused.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked = false;
    if (!looked) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        looked = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array on the current device.  The host-side
// name of a __device__ array is only a stand-in, so the address is looked up
// (with that device current) the first time a device is used in a context and
// cached; a new context on the device (after cudaDeviceReset) looks it up again.
tq_status noalloc_scratch(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TQ_ERR_UNSUPPORTED;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kv_attend_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = static_cast<float*>(g_scratch_addr[dev]);
    return TQ_OK;
}

}  // namespace

extern "C" size_t tq_kv_attend_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" tq_status tq_kv_attend_noalloc(const void* q, tq_dtype qdt, int32_t Hq, int32_t Hkv, int32_t D, int64_t ctx,
                                          int64_t capacity, const tq_rotation_t* rot, const tq_codebook_t* kcb,
                                          const tq_codebook_t* vcb, int32_t group, const uint32_t* kcodes,
                                          const uint16_t* kscales, const uint32_t* vcodes, const uint16_t* vscales,
                                          float* o, void* stream) {
    const size_t need = tq_kv_attend_workspace_bytes(Hq, D, ctx);
    if (need == 0 || need > kNoAllocScratchBytes) return TQ_ERR_INVALID;
    float* ws = nullptr;
    const tq_status s = noalloc_scratch(&ws);
    if (s != TQ_OK) return s;
    return tq_kv_attend(q, qdt, Hq, Hkv, D, ctx, capacity, rot, kcb, vcb, group, kcodes, kscales, vcodes, vscales, o,
                        ws, kNoAllocScratchBytes, stream);
}
