// Expert-sorted batched gather-GEMM on the 5th-generation tensor cores:
// tq_gather_qmm.
//
// "How it works", "Running a quantized layer", row "A large batch sorted by
// expert": polar_gather_qmm, a batched gather-GEMM.  For every expert e and its
// sorted pairs i in [offsets[e], offsets[e+1]): y[i] = W_e x_src(i), with W_e
// decoded from its packed codes inline (the full-precision weights are never
// written to global memory).
//
// GB300 design.  D[128 weight rows, up to 256 pairs] = A . B^T with
//   A = 128 x 64 tile of decoded weights (fp16/bf16, K-major, 128-byte swizzle),
//       written to shared memory by 8 decoder warps from the packed codes;
//   B = the pairs' input rows (gathered token rows of x), copied by 4 producer
//       warps with cp.async into the same swizzled K-major layout;
//   D accumulated in tensor memory (TMEM, fp32) by tcgen05.mma issued from one
//   thread, 4 MMAs of K = 16 per 64-wide stage, 4 stages in flight.
// Each decoded weight is c[code] * (s_group / s_rowmax) so every A element
// stays in [-c_max, c_max] whatever the scales; the epilogue multiplies row m
// by s_rowmax[m].  CTAs are persistent (one per SM) and walk the work items
// (expert, 128-row tile, 256-pair tile) in expert-major order so that CTAs
// running together share the expert's codes in L2.  Every wait on an mbarrier
// is bounded; on expiry the CTA sets TQ_DEVERR_TIMEOUT, drains and frees TMEM.
#include <type_traits>

#include "common.cuh"

using namespace tq;

namespace {

constexpr int kBM = 128;       // weight rows per tile (MMA M)
constexpr int kNT = 256;       // max pairs per tile (MMA N)
constexpr int kBK = 64;        // K per stage (one 128-byte swizzle atom of fp16)
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kNT * kBK * 2;   // 32 KB
constexpr int kProdWarps = 4;            // B producers: warps 1..4
constexpr int kDecWarps = 8;             // decoders / epilogue: warps 5..12
constexpr int kThreads = 32 * (1 + kProdWarps + kDecWarps);
constexpr int kFirstDec = 1 + kProdWarps;
constexpr int kMaxExperts = 1024;
constexpr long long kWaitCycles = 1ll << 31;  // about a second at GB300 clocks

// ---------------------------------------------------------------- PTX wrappers

TQ_DEVFN uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

TQ_DEVFN void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

TQ_DEVFN void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

TQ_DEVFN bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait bounded by time only (used to drain in-flight MMAs before freeing TMEM).
TQ_DEVFN bool mbar_wait_drain(uint64_t* b, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// Bounded wait for the phase of parity `parity` to complete.  Returns false
// (and raises the CTA's abort flag) if it did not within kWaitCycles or if
// another role already aborted.
TQ_DEVFN bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

TQ_DEVFN void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

TQ_DEVFN void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
TQ_DEVFN void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
TQ_DEVFN void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

TQ_DEVFN void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
TQ_DEVFN void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major tile, 128-byte swizzle, 8-row atoms
// 1024 bytes apart (stride byte offset), tile base 1024-byte aligned.
TQ_DEVFN uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: D fp32, A and B fp16 (fmt 0) or bf16
// (fmt 1), both K-major, M = 128, N = n.
TQ_DEVFN uint32_t f16_idesc(int fmt, int n) {
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(kBM >> 4) << 24);
}

TQ_DEVFN void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
        : "memory");
}

TQ_DEVFN void tc_commit(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(b))
                 : "memory");
}

#define TQ_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                 "=r"(v[i + 6]), "=r"(v[i + 7])
TQ_DEVFN void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : TQ_R8(0), TQ_R8(8), TQ_R8(16), TQ_R8(24)
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
#undef TQ_R8

// ---------------------------------------------------------------- codes -> operand

template <int LEVELS>
struct BitFmt {
    static constexpr int kBits = LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4);
    static constexpr int kCW = LEVELS == 8 ? 10 : 32 / kBits;
    static constexpr int kWords = 32 / kCW + (LEVELS == 8 ? 1 : 0);  // words holding 32 consecutive codes
};

template <int XT>
TQ_DEVFN uint32_t pack2(float a, float b) {
    if constexpr (XT == 0) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// 32 consecutive codes starting at slot POS0 of W[0] -> 16 packed operand pairs.
// Pairs never straddle words (code counts per word are even).  r0 applies to
// the first 16 codes, r1 to the next 16 (they differ only for group 16).
template <int LEVELS, int POS0, int XT>
TQ_DEVFN void decode32(const uint32_t* W, float r0, float r1, const float2* lut, uint32_t (&out)[16]) {
    using F = BitFmt<LEVELS>;
    constexpr uint32_t kMask = (1u << (2 * F::kBits)) - 1u;
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const int t = POS0 + 2 * p;
        const uint32_t idx = (W[t / F::kCW] >> (F::kBits * (t % F::kCW))) & kMask;
        const float2 c = lut[idx];
        const float r = p < 8 ? r0 : r1;
        out[p] = pack2<XT>(c.x * r, c.y * r);
    }
}

struct QmmParams {
    const uint32_t* codes;
    const uint16_t* scales;
    int64_t row_stride, esw, ess;
    int rows, cols, experts;
    const float* centroids;
    const void* x;
    const int32_t* perm;
    const int32_t* offsets;
    int P, k, per_pair;
    void* y;
    int ydt;
    uint32_t* err;
};

template <int LEVELS, int G, int XT>
__global__ void __launch_bounds__(kThreads, 1) gather_qmm_kernel(const QmmParams p) {
    using F = BitFmt<LEVELS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = base + kStages * kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tile_full = empty + kStages;
    uint64_t* tile_empty = tile_full + 1;
    uint64_t* drain = tile_empty + 1;
    uint64_t* decbar = drain + 1;  // decoder-only rendezvous (bounded, unlike bar.sync)
    int* ctl = reinterpret_cast<int*>(decbar + 1);                       // 8 ints: tmem slot, abort, item count
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl);
    volatile int* abort_flag = ctl + 1;
    int* total_items = ctl + 2;
    float2* lut = reinterpret_cast<float2*>(ctl + 8);                    // 8-byte aligned
    float* rowscale = reinterpret_cast<float*>(lut + LEVELS * LEVELS);  // [128]
    float* rowmax_part = rowscale + kBM;                                 // [2][128]
    int* cum = reinterpret_cast<int*>(rowmax_part + 2 * kBM);            // [experts + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.experts;
    const int mtiles = p.rows / kBM;
    const int nk = p.cols / kBK;
    const int ngroups = p.cols / G;

    // ---- prologue: offsets -> per-expert work prefix; validation before any TMEM use
    for (int i = tid; i <= E; i += kThreads) cum[i] = p.offsets[i];
    for (int i = tid; i < LEVELS * LEVELS; i += kThreads)
        lut[i] = make_float2(p.centroids[i & (LEVELS - 1)], p.centroids[i / LEVELS]);
    __syncthreads();
    if (tid == 0) {
        bool ok = cum[0] == 0 && cum[E] == p.P;
        int prev = 0, acc = 0;
        for (int e = 0; e <= E; ++e) {
            const int off = cum[e];
            if (e > 0) {
                const int n = off - prev;
                ok = ok && n >= 0;
                const int nt = n > 0 ? (n + kNT - 1) / kNT : 0;
                cum[e - 1] = acc;
                acc += nt * mtiles;
            }
            prev = off;
        }
        cum[E] = acc;
        *total_items = ok ? acc : -1;
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 32 * kDecWarps + 32 * kProdWarps);
            mbar_init(empty + s, 1);
        }
        mbar_init(tile_full, 1);
        mbar_init(tile_empty, 32 * kDecWarps);
        mbar_init(drain, 1);
        mbar_init(decbar, 32 * kDecWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int total = *total_items;
    if (total < 0) {  // uniform: bad offsets, nothing allocated yet
        if (tid == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        return;
    }
    // Per-expert first item index is cum[e]; the pair offsets are read again from global.
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kNT)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto item_coords = [&](int item, int& e, int& mt, int& nt, int& i0, int& nvalid) {
        int lo = 0, hi = E - 1;  // last e with cum[e] <= item
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum[mid] <= item) lo = mid; else hi = mid - 1;
        }
        e = lo;
        const int off0 = p.offsets[e], n = p.offsets[e + 1] - off0;
        const int ntiles = (n + kNT - 1) / kNT;
        const int local = item - cum[e];
        mt = local / ntiles;
        nt = local - mt * ntiles;
        i0 = off0 + nt * kNT;
        nvalid = min(kNT, n - nt * kNT);
    };

    if (warp == 0) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            uint32_t it = 0, tile_it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++tile_it) {
                int e, mt, nt, i0, nvalid;
                item_coords(item, e, mt, nt, i0, nvalid);
                const int ninst = (nvalid + 15) & ~15;
                const uint32_t idesc = f16_idesc(XT, ninst);
                if (!mbar_wait(tile_empty, (tile_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(full + s, (it / kStages) & 1, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(a0 + s * kABytes), bd = sw128_desc(b0 + s * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kc | kk) != 0);
                    tc_commit(empty + s);
                }
                if (!ok) break;
                tc_commit(tile_full);
            }
            tc_commit(drain);  // completes when every MMA issued above has finished
            if (!mbar_wait_drain(drain, 0)) *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp < kFirstDec) {
        // ------------------------------------------------ B producers: gathered input rows
        const int pt = tid - 32;  // 0..127: rows pt and pt + 128
        const uint8_t* xb = reinterpret_cast<const uint8_t*>(p.x);
        const int64_t xrow_bytes = (int64_t)p.cols * 2;
        uint32_t it = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            int e, mt, nt, i0, nvalid;
            item_coords(item, e, mt, nt, i0, nvalid);
            const int ninst = (nvalid + 15) & ~15;
            int64_t src[2];
            uint32_t bytes[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = pt + 128 * h;
                src[h] = 0;
                bytes[h] = 0;
                if (r < nvalid) {
                    int64_t row = p.per_pair ? (int64_t)(i0 + r) : (int64_t)p.perm[i0 + r];
                    if (!p.per_pair) {
                        if (row < 0 || row >= p.P) {
                            if (p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
                            row = -1;
                        } else {
                            row /= p.k;
                        }
                    }
                    if (row >= 0) {
                        src[h] = row * xrow_bytes;
                        bytes[h] = 16;
                    }
                }
            }
            int prev_s = -1;
            for (int kc = 0; kc < nk; ++kc, ++it) {
                const int s = it % kStages;
                if (!mbar_wait(empty + s, ((it / kStages) & 1) ^ 1, abort_flag)) { ok = false; break; }
                const uint32_t dst0 = smem_u32(sB + s * kBBytes);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = pt + 128 * h;
                    if (r < ninst) {
                        const uint8_t* srow = xb + src[h] + (int64_t)kc * kBK * 2;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            cp_async16(dst0 + r * 128 + ((j ^ (r & 7)) << 4), srow + j * 16, bytes[h]);
                    }
                }
                cp_async_commit();
                if (prev_s >= 0) {
                    cp_async_wait<1>();
                    fence_async_smem();
                    mbar_arrive(full + prev_s);
                }
                prev_s = s;
            }
            cp_async_wait<0>();
            fence_async_smem();
            if (ok && prev_s >= 0) mbar_arrive(full + prev_s);
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------ decoders, then epilogue
        const int dw = warp - kFirstDec;      // 0..7
        const int h = dw >> 2;                // which 32 codes of the 64-wide stage
        const int r = (dw & 3) * 32 + lane;   // tile row
        const int quarter = warp & 3;         // TMEM lanes this warp may access
        const int chalf = dw >> 2;            // epilogue: columns [128*chalf, 128*chalf + 128)
        uint32_t it = 0, tile_it = 0, dec_phase = 0;
        bool ok = true;
        // All decoder threads meet here; bounded, so an aborting thread cannot strand the others.
        auto dec_sync = [&]() -> bool {
            mbar_arrive(decbar);
            const bool r = mbar_wait(decbar, dec_phase, abort_flag);
            dec_phase ^= 1;
            return r;
        };
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++tile_it) {
            int e, mt, nt, i0, nvalid;
            item_coords(item, e, mt, nt, i0, nvalid);
            const int m0 = mt * kBM;
            const uint32_t* wrow = p.codes + (int64_t)e * p.esw + (int64_t)(m0 + r) * p.row_stride;
            const uint16_t* srow = p.scales + (int64_t)e * p.ess + (int64_t)(m0 + r) * ngroups;
            // row scale = max group scale of the row (each half of the decoders scans half the groups)
            float mx = 0.f;
            for (int g = h; g < ngroups; g += 2) mx = fmaxf(mx, half_bits_to_float(__ldg(srow + g)));
            rowmax_part[h * kBM + r] = mx;
            if (!dec_sync()) { ok = false; break; }
            float smax = fmaxf(rowmax_part[r], rowmax_part[kBM + r]);
            if (!(smax > 0.f)) smax = 1.f;
            const float inv = 1.0f / smax;
            if (h == 0) rowscale[r] = smax;

            constexpr int PF = 4;
            uint32_t wb[PF][F::kWords];
            float sb[PF][2];
            auto load = [&](int kc, uint32_t (&W)[F::kWords], float (&S)[2]) {
                const int q0 = kc * kBK + 32 * h;
                const uint32_t* wp = wrow + q0 / F::kCW;
#pragma unroll
                for (int j = 0; j < F::kWords; ++j) W[j] = __ldg(wp + j);
                S[0] = half_bits_to_float(__ldg(srow + q0 / G));
                S[1] = G == 16 ? half_bits_to_float(__ldg(srow + q0 / G + 1)) : S[0];
            };
#pragma unroll
            for (int u = 0; u < PF - 1; ++u)
                if (u < nk) load(u, wb[u], sb[u]);
            for (int kc0 = 0; kc0 < nk && ok; kc0 += PF) {
#pragma unroll
                for (int u = 0; u < PF; ++u) {
                    const int kc = kc0 + u;
                    if (kc < nk && ok) {
                        if (kc + PF - 1 < nk) load(kc + PF - 1, wb[(u + PF - 1) % PF], sb[(u + PF - 1) % PF]);
                        const int s = it % kStages;
                        if (!mbar_wait(empty + s, ((it / kStages) & 1) ^ 1, abort_flag)) {
                            ok = false;
                        } else {
                            uint32_t out[16];
                            const float r0 = sb[u][0] * inv, r1 = sb[u][1] * inv;
                            const int pos0 = (kc * kBK + 32 * h) % F::kCW;
                            if constexpr (LEVELS == 8) {
                                switch (pos0) {
                                    case 0: decode32<LEVELS, 0, XT>(wb[u], r0, r1, lut, out); break;
                                    case 2: decode32<LEVELS, 2, XT>(wb[u], r0, r1, lut, out); break;
                                    case 4: decode32<LEVELS, 4, XT>(wb[u], r0, r1, lut, out); break;
                                    case 6: decode32<LEVELS, 6, XT>(wb[u], r0, r1, lut, out); break;
                                    default: decode32<LEVELS, 8, XT>(wb[u], r0, r1, lut, out); break;
                                }
                            } else {
                                decode32<LEVELS, 0, XT>(wb[u], r0, r1, lut, out);
                            }
                            uint8_t* arow = sA + s * kABytes + r * 128;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const int chunk = 4 * h + c;
                                *reinterpret_cast<uint4*>(arow + ((chunk ^ (r & 7)) << 4)) =
                                    make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]);
                            }
                            fence_async_smem();
                            mbar_arrive(full + s);
                            ++it;
                        }
                    }
                }
            }
            if (!ok) break;
            // epilogue: TMEM -> registers -> y (rows of the sorted pairs)
            if (!mbar_wait(tile_full, tile_it & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            if (!dec_sync()) { ok = false; break; }  // rowscale visible
            const int m = quarter * 32 + lane;
            const float rs = rowscale[m];
            for (int c0 = chalf * 128; c0 < chalf * 128 + 128; c0 += 32) {
                if (c0 < nvalid) {
                    uint32_t v[32];
                    tc_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < nvalid)
                            store_from_float(p.y, (int64_t)(i0 + c0 + j) * p.rows + m0 + m, p.ydt,
                                             __uint_as_float(v[j]) * rs);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tile_empty);
        }
    }

    __syncthreads();
    if (tid == 0 && *abort_flag && p.err) atomicOr(p.err, TQ_DEVERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kNT) : "memory");
    }
}

// ---------------------------------------------------------------- staged variant
//
// Same contraction and tile walk as gather_qmm_kernel, with the data movement
// reorganised so that neither the copies nor the decode starve the tensor core:
//   warp 0      issues the MMAs (one thread);
//   warps 1-2   gather the pairs' input rows: each thread keeps the source row
//               indices of its 32 rows in registers for the whole tile and
//               issues one 16-byte cp.async per row and stage, 8 lanes per
//               128-byte row segment (3-stage ring of 256 x 64 operand tiles);
//   warp 3      stages the m-tile's scale block and its packed codes, 32 words
//               (128 bytes) per row and chunk, in a 2-slot ring; word w of row r
//               is stored at word w ^ (r & 31) of the row so that the decoders'
//               reads (one word of 32 consecutive rows) are free of bank conflicts;
//   warps 4-19  decode in two groups of 8 warps taking alternate stages: pairs
//               of codes index a per-lane copy of a table of packed operand
//               pairs and one half2 multiply applies s_group / s_rowmax; then
//               all 16 drain the accumulator (epilogue).
constexpr int kStagesA = 4, kStagesB = 3, kChunkSlots = 2;
constexpr int kChunkBytes = kBM * 128;   // 32 code words of each of the 128 rows
constexpr int kScaleBlock = kBM * 128;   // up to 64 fp16 scales of each row
constexpr int kDec2 = 16;                // decoder warps
constexpr int kFirstDec2 = 4;
constexpr int kThreads2 = 32 * (kFirstDec2 + kDec2);
constexpr int kDecThreads2 = 32 * kDec2;

template <int LEVELS>
struct Q2Fmt {
    using F = BitFmt<LEVELS>;
    static constexpr int kSPC = F::kCW / 2;                    // stages (64 codes) per 32-word chunk
    static constexpr int kLutCopies = LEVELS == 16 ? 1 : 32;  // per-lane copies when small enough
};

template <int XT>
TQ_DEVFN uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    if constexpr (XT == 0) {
        __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    } else {
        __nv_bfloat162 r =
            __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
        return *reinterpret_cast<uint32_t*>(&r);
    }
}

TQ_DEVFN uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
TQ_DEVFN uint32_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
TQ_DEVFN void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
TQ_DEVFN void cp_async4(uint32_t dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

template <int LEVELS, int G, int XT>
__global__ void __launch_bounds__(kThreads2, 1) gather_qmm2_kernel(const QmmParams p) {
    using F = BitFmt<LEVELS>;
    using Q = Q2Fmt<LEVELS>;
    constexpr int SPC = Q::kSPC, NL = LEVELS * LEVELS, COPIES = Q::kLutCopies;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;                                      // [4][128 x 64]
    uint8_t* sB = sA + kStagesA * kABytes;                   // [3][256 x 64]
    uint8_t* sC = sB + kStagesB * kBBytes;                   // [2][128 rows x 128 B] code chunks
    uint8_t* sS = sC + kChunkSlots * kChunkBytes;            // [128 rows x 128 B] scale block
    uint32_t* lut = reinterpret_cast<uint32_t*>(sS + kScaleBlock);       // [NL][COPIES] operand pairs
    float* rowscale = reinterpret_cast<float*>(lut + NL * COPIES);       // [128]
    float* rowmax_part = rowscale + kBM;                                 // [4][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(rowmax_part + 4 * kBM);
    uint64_t* fullA = bars;
    uint64_t* emptyA = fullA + kStagesA;
    uint64_t* fullB = emptyA + kStagesA;
    uint64_t* emptyB = fullB + kStagesB;
    uint64_t* cfull = emptyB + kStagesB;
    uint64_t* cempty = cfull + kChunkSlots;
    uint64_t* sfull = cempty + kChunkSlots;
    uint64_t* sempty = sfull + 1;
    uint64_t* tile_full = sempty + 1;
    uint64_t* tile_empty = tile_full + 1;
    uint64_t* drain = tile_empty + 1;
    uint64_t* decbar = drain + 1;
    int* ctl = reinterpret_cast<int*>(decbar + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl);
    volatile int* abort_flag = ctl + 1;
    int* total_items = ctl + 2;
    int* cum = ctl + 8;  // [experts + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.experts;
    const int mtiles = p.rows / kBM;
    const int nk = p.cols / kBK;
    const int ngroups = p.cols / G;
    const int nchunks = (nk + SPC - 1) / SPC;

    for (int i = tid; i <= E; i += kThreads2) cum[i] = p.offsets[i];
    for (int i = tid; i < NL * COPIES; i += kThreads2) {
        const int idx = i / COPIES;
        lut[i] = pack2<XT>(p.centroids[idx & (LEVELS - 1)], p.centroids[idx / LEVELS]);
    }
    __syncthreads();
    if (tid == 0) {
        bool ok = cum[0] == 0 && cum[E] == p.P;
        int prev = 0, acc = 0;
        for (int e = 0; e <= E; ++e) {
            const int off = cum[e];
            if (e > 0) {
                const int n = off - prev;
                ok = ok && n >= 0;
                const int nt = n > 0 ? (n + kNT - 1) / kNT : 0;
                cum[e - 1] = acc;
                acc += nt * mtiles;
            }
            prev = off;
        }
        cum[E] = acc;
        *total_items = ok ? acc : -1;
        *abort_flag = 0;
        for (int s = 0; s < kStagesA; ++s) {
            mbar_init(fullA + s, 32 * kDec2 / 2);
            mbar_init(emptyA + s, 1);
        }
        for (int s = 0; s < kStagesB; ++s) {
            mbar_init(fullB + s, 64);
            mbar_init(emptyB + s, 1);
        }
        for (int s = 0; s < kChunkSlots; ++s) {
            mbar_init(cfull + s, 32);
            mbar_init(cempty + s, kDecThreads2);
        }
        mbar_init(sfull, 32);
        mbar_init(sempty, kDecThreads2);
        mbar_init(tile_full, 1);
        mbar_init(tile_empty, kDecThreads2);
        mbar_init(drain, 1);
        mbar_init(decbar, kDecThreads2);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int total = *total_items;
    if (total < 0) {
        if (tid == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        return;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kNT)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto item_coords = [&](int item, int& e, int& mt, int& nt, int& i0, int& nvalid) {
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum[mid] <= item) lo = mid; else hi = mid - 1;
        }
        e = lo;
        const int off0 = p.offsets[e], n = p.offsets[e + 1] - off0;
        const int ntiles = (n + kNT - 1) / kNT;
        const int local = item - cum[e];
        mt = local / ntiles;
        nt = local - mt * ntiles;
        i0 = off0 + nt * kNT;
        nvalid = min(kNT, n - nt * kNT);
    };

    if (warp == 0) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            uint32_t it = 0, tile_it = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++tile_it) {
                int e, mt, nt, i0, nvalid;
                item_coords(item, e, mt, nt, i0, nvalid);
                const uint32_t idesc = f16_idesc(XT, (nvalid + 15) & ~15);
                if (!mbar_wait(tile_empty, (tile_it & 1) ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int sa = it % kStagesA, sb = it % kStagesB;
                    if (!mbar_wait(fullA + sa, (it / kStagesA) & 1, abort_flag) ||
                        !mbar_wait(fullB + sb, (it / kStagesB) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(a0 + sa * kABytes), bd = sw128_desc(b0 + sb * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) tc_mma(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kc | kk) != 0);
                    tc_commit(emptyA + sa);
                    tc_commit(emptyB + sb);
                }
                if (!ok) break;
                tc_commit(tile_full);
            }
            tc_commit(drain);
            if (!mbar_wait_drain(drain, 0)) *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp < 3) {
        // ------------------------------------------------ B producers: rows rb + 8 i of every stage
        const int t = tid - 32;            // 0..63
        const int q = t & 7, rb = t >> 3;  // 16-byte piece; first row (rows rb + 8 i share r & 7 == rb)
        const uint8_t* xq = reinterpret_cast<const uint8_t*>(p.x) + q * 16;
        const uint32_t pitch = (uint32_t)p.cols * 2u;
        uint32_t it = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
            int e, mt, nt, i0, nvalid;
            item_coords(item, e, mt, nt, i0, nvalid);
            const int ninst = (nvalid + 15) & ~15;
            const int cnt = (ninst - rb + 7) >> 3;  // my rows below ninst (ninst >= 16 > rb)
            // Source rows; padding rows past nvalid read row 0 (their outputs are not stored),
            // rows with an invalid pair id are zero-filled.
            uint32_t rowv[32];
            uint32_t bad = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int r = rb + 8 * i;
                uint32_t row = 0;
                if (r < nvalid) {
                    if (p.per_pair) {
                        row = (uint32_t)(i0 + r);
                    } else {
                        const int f = __ldg(p.perm + i0 + r);
                        if (f < 0 || f >= p.P) {
                            bad |= 1u << i;
                            if (p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
                        } else {
                            row = (uint32_t)(f / p.k);
                        }
                    }
                }
                rowv[i] = row;
            }
            int prev_s = -1;
            for (int kc = 0; kc < nk; ++kc, ++it) {
                const int s = it % kStagesB;
                if (!mbar_wait(emptyB + s, ((it / kStagesB) & 1) ^ 1, abort_flag)) { ok = false; break; }
                const uint32_t dst = smem_u32(sB + s * kBBytes) + rb * 128 + ((q ^ rb) << 4);
                const uint8_t* g = xq + (size_t)kc * (kBK * 2);
                if (bad == 0) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < cnt) cp_async16(dst + i * 1024, g + (size_t)rowv[i] * pitch, 16u);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < cnt) cp_async16(dst + i * 1024, g + (size_t)rowv[i] * pitch, (bad >> i) & 1 ? 0u : 16u);
                }
                cp_async_commit();
                if (prev_s >= 0) {
                    cp_async_wait<1>();
                    fence_async_smem();
                    mbar_arrive(fullB + prev_s);
                }
                prev_s = s;
            }
            cp_async_wait<0>();
            fence_async_smem();
            if (ok && prev_s >= 0) mbar_arrive(fullB + prev_s);
        }
        cp_async_wait<0>();
    } else if (warp < kFirstDec2) {
        // ------------------------------------------------ scale block and code chunks
        const int nsw = ngroups >> 1;  // scale words per row (ngroups even, at most 64)
        const uint32_t sS0 = smem_u32(sS), sC0 = smem_u32(sC);
        uint32_t cc = 0, tile_it = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++tile_it) {
            int e, mt, nt, i0, nvalid;
            item_coords(item, e, mt, nt, i0, nvalid);
            const int m0 = mt * kBM;
            if (!mbar_wait(sempty, (tile_it & 1) ^ 1, abort_flag)) { ok = false; break; }
            const uint32_t* sbase =
                reinterpret_cast<const uint32_t*>(p.scales + (int64_t)e * p.ess + (int64_t)m0 * ngroups);
            if (lane < nsw) {
                for (int r = 0; r < kBM; ++r)
                    cp_async4(sS0 + r * 128 + ((lane ^ (r & 31)) << 2), sbase + (int64_t)r * nsw + lane, 4u);
            }
            cp_async_commit();
            cp_async_wait<0>();
            mbar_arrive(sfull);
            const uint32_t* cbase = p.codes + (int64_t)e * p.esw + (int64_t)m0 * p.row_stride;
            for (int c = 0; c < nchunks; ++c, ++cc) {
                const int slot = cc % kChunkSlots;
                if (!mbar_wait(cempty + slot, ((cc / kChunkSlots) & 1) ^ 1, abort_flag)) { ok = false; break; }
                const uint32_t dst = sC0 + slot * kChunkBytes;
                const int64_t gw = (int64_t)c * 32 + lane;
                const bool in = gw < p.row_stride;  // words past the padded row read as zero
                const uint32_t* src = cbase + (in ? gw : 0);
                for (int r = 0; r < kBM; ++r)
                    cp_async4(dst + r * 128 + ((lane ^ (r & 31)) << 2), src + (int64_t)r * p.row_stride,
                              in ? 4u : 0u);
                cp_async_commit();
                cp_async_wait<0>();
                mbar_arrive(cfull + slot);
            }
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------ decoders, then epilogue
        const int dw = warp - kFirstDec2;  // 0..15
        const int grp = dw >> 3;           // takes the stages with it & 1 == grp
        const int h = (dw >> 2) & 1;       // which 32 codes of the 64-wide stage
        const int part = dw >> 2;          // row-max quarter; epilogue column quarter
        const int r = (dw & 3) * 32 + lane;
        const int quarter = warp & 3;      // TMEM lanes this warp may access (== dw & 3)
        const uint32_t lutl = smem_u32(lut) + (COPIES == 32 ? lane * 4 : 0);
        const uint32_t srow = smem_u32(sS) + r * 128 + ((r & 31) << 2);  // word w of the row: srow ^ (w << 2)
        const uint32_t crow0 = smem_u32(sC) + r * 128 + ((r & 31) << 2);
        const uint32_t arow0 = smem_u32(sA) + r * 128 + ((r & 7) << 4);  // 16-byte piece c: arow ^ (c << 4)
        uint32_t it = 0, tile_it = 0, dec_phase = 0, cc = 0;
        bool ok = true;
        auto dec_sync = [&]() -> bool {
            mbar_arrive(decbar);
            const bool rr = mbar_wait(decbar, dec_phase, abort_flag);
            dec_phase ^= 1;
            return rr;
        };
        auto scale_at = [&](int g) -> float {
            return half_bits_to_float((uint16_t)lds16((srow ^ ((g >> 1) << 2)) + (g & 1) * 2));
        };
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++tile_it) {
            int e, mt, nt, i0, nvalid;
            item_coords(item, e, mt, nt, i0, nvalid);
            const int m0 = mt * kBM;
            if (!mbar_wait(sfull, tile_it & 1, abort_flag)) { ok = false; break; }
            float mx = 0.f;
            for (int g = part; g < ngroups; g += 4) mx = fmaxf(mx, scale_at(g));
            rowmax_part[part * kBM + r] = mx;
            if (!dec_sync()) { ok = false; break; }
            float smax = fmaxf(fmaxf(rowmax_part[r], rowmax_part[kBM + r]),
                               fmaxf(rowmax_part[2 * kBM + r], rowmax_part[3 * kBM + r]));
            if (!(smax > 0.f)) smax = 1.f;
            const float inv = 1.0f / smax;
            if (part == 0) rowscale[r] = smax;
            uint32_t crow = crow0;
            int sub = 0;
            for (int kc = 0; kc < nk && ok; ++kc, ++it) {
                if (sub == 0) {
                    const int slot = cc % kChunkSlots;
                    if (!mbar_wait(cfull + slot, (cc / kChunkSlots) & 1, abort_flag)) { ok = false; break; }
                    crow = crow0 + slot * kChunkBytes;
                }
                if ((int)(it & 1) == grp) {
                    const int s = it % kStagesA;
                    if (!mbar_wait(emptyA + s, ((it / kStagesA) & 1) ^ 1, abort_flag)) { ok = false; break; }
                    const int lq = 64 * sub + 32 * h;  // first code of this thread within the chunk
                    const int w0 = lq / F::kCW, pos0 = lq - w0 * F::kCW;
                    uint32_t W[F::kWords];
#pragma unroll
                    for (int j = 0; j < F::kWords; ++j) W[j] = lds32(crow ^ ((w0 + j) << 2));
                    const int g0 = (kc * kBK + 32 * h) / G;
                    const float r0 = scale_at(g0) * inv;
                    const float r1 = G == 16 ? scale_at(g0 + 1) * inv : r0;
                    const uint32_t rr0 = pack2<XT>(r0, r0), rr1 = pack2<XT>(r1, r1);
                    uint32_t out[16];
                    auto dec = [&](auto pos_c) {
                        constexpr int POS0 = decltype(pos_c)::value;
                        constexpr uint32_t kMask = (1u << (2 * F::kBits)) - 1u;
                        constexpr int kStride = COPIES * 4;  // bytes between table entries
                        constexpr int kLog = COPIES == 32 ? 7 : 2;
#pragma unroll
                        for (int pp = 0; pp < 16; ++pp) {
                            const int tt = POS0 + 2 * pp;
                            const int sh = F::kBits * (tt % F::kCW);
                            const uint32_t w = W[tt / F::kCW];
                            const uint32_t off =
                                (sh >= kLog ? (w >> (sh - kLog)) : (w << (kLog - sh))) & (kMask * kStride);
                            out[pp] = hmul2_bits<XT>(lds32(lutl + off), pp < 8 ? rr0 : rr1);
                        }
                    };
                    if constexpr (LEVELS == 8) {
                        switch (pos0) {
                            case 0: dec(std::integral_constant<int, 0>{}); break;
                            case 2: dec(std::integral_constant<int, 2>{}); break;
                            case 4: dec(std::integral_constant<int, 4>{}); break;
                            case 6: dec(std::integral_constant<int, 6>{}); break;
                            default: dec(std::integral_constant<int, 8>{}); break;
                        }
                    } else {
                        dec(std::integral_constant<int, 0>{});
                    }
                    const uint32_t arow = arow0 + s * kABytes;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        sts128(arow ^ ((4 * h + c4) << 4), out[4 * c4], out[4 * c4 + 1], out[4 * c4 + 2],
                               out[4 * c4 + 3]);
                    fence_async_smem();
                    mbar_arrive(fullA + s);
                }
                if (++sub == SPC || kc == nk - 1) {
                    mbar_arrive(cempty + cc % kChunkSlots);
                    ++cc;
                    sub = 0;
                }
            }
            if (!ok) break;
            mbar_arrive(sempty);  // scale block no longer read (row scales kept in rowscale)
            if (!mbar_wait(tile_full, tile_it & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            if (!dec_sync()) { ok = false; break; }
            const int m = quarter * 32 + lane;
            const float rs = rowscale[m];
            for (int c0 = part * 64; c0 < part * 64 + 64; c0 += 32) {
                if (c0 < nvalid) {
                    uint32_t v[32];
                    tc_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < nvalid)
                            store_from_float(p.y, (int64_t)(i0 + c0 + j) * p.rows + m0 + m, p.ydt,
                                             __uint_as_float(v[j]) * rs);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(tile_empty);
        }
    }

    __syncthreads();
    if (tid == 0 && *abort_flag && p.err) atomicOr(p.err, TQ_DEVERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kNT) : "memory");
    }
}

size_t qmm2_smem_bytes(int levels, int experts) {
    const int copies = levels == 16 ? 1 : 32;
    return 1024 + (size_t)kStagesA * kABytes + (size_t)kStagesB * kBBytes + (size_t)kChunkSlots * kChunkBytes +
           kScaleBlock + (size_t)levels * levels * copies * 4 + 5 * kBM * 4 + 32 * 8 + 32 +
           (size_t)(experts + 1) * 4;
}

size_t qmm_smem_bytes(int levels, int experts) {
    return 1024 + (size_t)kStages * (kABytes + kBBytes) + (2 * kStages + 4) * 8 + 32 + (size_t)levels * levels * 8 +
           3 * kBM * 4 + (size_t)(experts + 1) * 4;
}

template <int LEVELS, int G, int XT>
tq_status launch_qmm(const QmmParams& p, cudaStream_t st) {
    const size_t smem = qmm_smem_bytes(LEVELS, p.experts);
    if (smem > 227 * 1024) return TQ_ERR_UNSUPPORTED;
    if (ensure_smem((const void*)gather_qmm_kernel<LEVELS, G, XT>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    gather_qmm_kernel<LEVELS, G, XT><<<sms > 0 ? sms : 148, kThreads, smem, st>>>(p);
    return launch_status();
}

// The staged kernel holds a tile's scale block in 128 bytes per row: it takes
// an even group count of at most 64 per row; other shapes use the first kernel.
bool staged_fits(const QmmParams& p, int G, int levels) {
    const int ngroups = p.cols / G;
    return ngroups <= 64 && ngroups % 2 == 0 && p.ess % 2 == 0 && aligned(p.scales, 4) &&
           qmm2_smem_bytes(levels, p.experts) <= 227 * 1024;
}

template <int LEVELS, int G, int XT>
tq_status launch_qmm2(const QmmParams& p, cudaStream_t st) {
    const size_t smem = qmm2_smem_bytes(LEVELS, p.experts);
    if (ensure_smem((const void*)gather_qmm2_kernel<LEVELS, G, XT>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    gather_qmm2_kernel<LEVELS, G, XT><<<sms > 0 ? sms : 148, kThreads2, smem, st>>>(p);
    return launch_status();
}

template <int LEVELS, int G, int XT>
tq_status launch_any(const QmmParams& p, cudaStream_t st) {
    return staged_fits(p, G, LEVELS) ? launch_qmm2<LEVELS, G, XT>(p, st) : launch_qmm<LEVELS, G, XT>(p, st);
}

template <int LEVELS, int G>
tq_status dispatch_xt(const QmmParams& p, int xt, cudaStream_t st) {
    return xt == 0 ? launch_any<LEVELS, G, 0>(p, st) : launch_any<LEVELS, G, 1>(p, st);
}

template <int LEVELS>
tq_status dispatch_g(const QmmParams& p, int group, int xt, cudaStream_t st) {
    switch (group) {
        case 16: return dispatch_xt<LEVELS, 16>(p, xt, st);
        case 32: return dispatch_xt<LEVELS, 32>(p, xt, st);
        case 64: return dispatch_xt<LEVELS, 64>(p, xt, st);
        case 128: return dispatch_xt<LEVELS, 128>(p, xt, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace

extern "C" size_t tq_gather_qmm_workspace_bytes(int32_t experts) { return 0; }

extern "C" tq_status tq_gather_qmm(const tq_qweight_t* w, const void* x, tq_dtype xdt, const int32_t* perm,
                                   const int32_t* offsets, int32_t P, int32_t k, int32_t per_pair_input, void* y,
                                   tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream) {
    (void)ws;
    (void)ws_bytes;
    if (!w || !w->codes || !w->scales || !w->cb.centroids) return TQ_ERR_INVALID;
    if (w->experts <= 0 || w->experts > kMaxExperts || w->rows <= 0 || w->cols <= 0) return TQ_ERR_INVALID;
    if (!(w->group == 16 || w->group == 32 || w->group == 64 || w->group == 128) || w->cols % w->group)
        return TQ_ERR_INVALID;
    if (w->row_stride_words < tq_row_words(w->cb.levels, w->cols)) return TQ_ERR_INVALID;
    if (w->experts > 1 && (w->expert_stride_words < (int64_t)w->rows * w->row_stride_words ||
                           w->expert_stride_scales < (int64_t)w->rows * (w->cols / w->group)))
        return TQ_ERR_INVALID;
    if (P < 0 || k <= 0 || !(xdt == TQ_F16 || xdt == TQ_BF16) || !(ydt == TQ_F32 || ydt == TQ_BF16))
        return TQ_ERR_INVALID;
    if (!(w->cb.levels == 4 || w->cb.levels == 8 || w->cb.levels == 16)) return TQ_ERR_UNSUPPORTED;
    if (w->rows % kBM || w->cols % kBK) return TQ_ERR_UNSUPPORTED;
    if (!offsets || (P > 0 && (!x || !y || (!per_pair_input && !perm)))) return TQ_ERR_INVALID;
    if (!aligned(x, 16)) return TQ_ERR_INVALID;
    if (P == 0) return TQ_OK;
    QmmParams p{};
    p.codes = w->codes;
    p.scales = w->scales;
    p.row_stride = w->row_stride_words;
    p.esw = w->experts > 1 ? w->expert_stride_words : 0;
    p.ess = w->experts > 1 ? w->expert_stride_scales : 0;
    p.rows = w->rows;
    p.cols = w->cols;
    p.experts = w->experts;
    p.centroids = w->cb.centroids;
    p.x = x;
    p.perm = perm;
    p.offsets = offsets;
    p.P = P;
    p.k = k;
    p.per_pair = per_pair_input ? 1 : 0;
    p.y = y;
    p.ydt = ydt;
    p.err = err;
    const int xt = xdt == TQ_F16 ? 0 : 1;
    cudaStream_t st = as_stream(stream);
    switch (w->cb.levels) {
        case 4: return dispatch_g<4>(p, w->group, xt, st);
        case 8: return dispatch_g<8>(p, w->group, xt, st);
        case 16: return dispatch_g<16>(p, w->group, xt, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}
