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

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "tma.cuh"

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
TQ_DEVFN void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : TQ_R8(0), TQ_R8(8)
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
    const float* colscale;  // split-K form: per input row, the factor applied to its outputs
    long long wait_cycles;  // budget of each bounded wait (wait_budget() at launch)
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
                if (!mbar_wait(tile_empty, (tile_it & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                tc_fence_after();
                for (int kc = 0; kc < nk; ++kc, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(full + s, (it / kStages) & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
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
                if (!mbar_wait(empty + s, ((it / kStages) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
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
            const bool r = mbar_wait(decbar, dec_phase, abort_flag, p.wait_cycles);
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
                        if (!mbar_wait(empty + s, ((it / kStages) & 1) ^ 1, abort_flag, p.wait_cycles)) {
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
            if (!mbar_wait(tile_full, tile_it & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
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
// Same contraction and tile walk as gather_qmm_kernel, organised so that the
// tensor core is fed continuously across tiles:
//   warps 0-1   issue the MMAs (one thread each, sharing each tile) into one of
//               two TMEM accumulators (2 x 256 columns), so that the next tile's
//               MMAs run while the previous accumulator is drained;
//   warps 2-3   load B stages, alternately, each with one 2-D tensor copy
//               (128-byte swizzle) of the pairs' input rows, which are
//               contiguous in sorted order (token rows are gathered into that
//               order by a first pass).  A thread is blocked for a few hundred
//               cycles by each copy it issues, hence one copy per stage and two
//               issuing warps;
//   warp 4      loads the m-tile's packed codes, 32 words of 128 rows per
//               chunk, with one 3-D tensor copy (128-byte swizzle) into a
//               2-slot ring;
//   warp 5      copies the scales those codes need into the same slot
//               (cp.async, SW words per row, SW a power of two; word j of row
//               r stored at j ^ ((r / (32 / SW)) % SW) so that one group read
//               across 32 rows hits 32 banks);
//   warps 6-21  decode in two groups of 8 warps taking alternate stages: pairs
//               of codes index a per-lane copy of a table of packed operand
//               pairs and one half2 multiply applies the group scale, so the
//               operand is c[code] * s_group in the operand type;
//   warps 22-25 drain the accumulators (epilogue).
constexpr int kChunkSlots = 2;
constexpr int kChunkCodeBytes = kBM * 128;            // 32 code words of each of the 128 rows
constexpr int kDec2 = 16;                             // decoder warps
constexpr int kMmaWarps = 2;                          // MMA issuers (warps 0, 1)
constexpr int kBWarps = 2;                            // B producers (warps 2, 3)
constexpr int kCodeWarp = kMmaWarps + kBWarps, kScaleWarp = kCodeWarp + 1;
constexpr int kFirstDec2 = kScaleWarp + 1;
constexpr int kEpiWarps = 4;
constexpr int kFirstEpi = kFirstDec2 + kDec2;
constexpr int kThreads2 = 32 * (kFirstEpi + kEpiWarps);
constexpr int kDecThreads2 = 32 * kDec2;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBoxRows[5] = {256, 128, 64, 32, 16};  // host side; the kernel uses 256 >> i

struct QmmMaps {
    CUtensorMap b[5];  // pair rows, boxes of 64 columns x kBoxRows[i] rows
    CUtensorMap c;     // codes [experts][rows][row_stride] words, box 32 x 128 x 1
};

// Most scale words (pairs of fp16 group scales) one row of a code chunk needs.
constexpr int chunk_scale_words(int cpc, int g) {
    int most = 0;
    for (int c = 0; c <= 2 * g; ++c) {
        const int w = (((c + 1) * cpc - 1) / g >> 1) - ((c * cpc / g) >> 1) + 1;
        most = w > most ? w : most;
    }
    return most;
}
constexpr int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

template <int LEVELS, int G, int NT, int ST>
struct Q2Fmt {
    using F = BitFmt<LEVELS>;
    static_assert(NT == 256 || (NT >= 16 && NT <= 128 && NT % 16 == 0), "pair tile");
    static constexpr int kBBytes = NT * kBK * 2;                // one B stage
    static constexpr int kHalf = NT <= 128 ? NT : 128;          // columns of one MMA thread's accumulator
    static constexpr int kBuf = 2 * kHalf;                      // columns of one accumulator buffer
    static constexpr int kTmemCols = 2 * kBuf;                  // two buffers
    static constexpr int kSPC = F::kCW / 2;                    // stages (64 codes) per 32-word chunk
    static constexpr int kCPC = 32 * F::kCW;                   // codes per chunk
    static constexpr int kLutCopies = LEVELS == 16 ? 1 : 32;  // per-lane copies when small enough
    static constexpr int kLutBytes = LEVELS * LEVELS * kLutCopies * 4;
    static constexpr int kSW = pow2_at_least(chunk_scale_words(kCPC, G));  // scale words per row in a slot
    static constexpr int kChunkBytes = kChunkCodeBytes + kBM * kSW * 4;
    // A and B stages share one ring (one full and one empty barrier per stage, so the MMA
    // thread waits once and commits once per stage).
    static constexpr int kStages = ST;
    static_assert(2 * ST + 2 * kChunkSlots + 5 <= 64, "barrier area");
    static constexpr int kSmem = 8192 + kStages * (kABytes + kBBytes) + kChunkSlots * kChunkBytes + kLutBytes + 64 * 8 +
                                 32;  // plus 8 * (experts + 1)
    static_assert(kSW <= 16, "scale words per chunk row");
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

// fp16 scale bits -> the operand type, in both halves of a word.
template <int XT>
TQ_DEVFN uint32_t scale_pair(uint32_t hbits) {
    if constexpr (XT == 0) {
        return hbits | (hbits << 16);
    } else {
        const float f = half_bits_to_float((uint16_t)hbits);
        return pack2<1>(f, f);
    }
}

TQ_DEVFN uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
TQ_DEVFN uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
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
// SK (split K, one expert, all pairs in one tile of at most NT): the work is the
// (row tile, code chunk) units, and CTA b takes a contiguous range of them, so
// every SM has work even when the row tiles are fewer than the SMs; each run of
// a row tile's chunks is one item, whose partial sums are added to y (zeroed
// beforehand) with atomics.
template <int LEVELS, int G, int XT, int NT, int ST, bool SK>
__global__ void __launch_bounds__(kThreads2, 1)
    gather_qmm2_kernel(const QmmParams p, const __grid_constant__ QmmMaps tm) {
    using F = BitFmt<LEVELS>;
    using Q = Q2Fmt<LEVELS, G, NT, ST>;
    constexpr int SPC = Q::kSPC, CPC = Q::kCPC, NL = LEVELS * LEVELS, COPIES = Q::kLutCopies;
    constexpr int kStages = Q::kStages, kChunkBytes = Q::kChunkBytes, SW = Q::kSW, kBBytes = Q::kBBytes;
    constexpr int kHalf = Q::kHalf, kBuf = Q::kBuf;
    extern __shared__ uint8_t smem_raw[];
    // The table sits at an 8 KB boundary, so its per-lane entry addresses are ORs of disjoint bit
    // fields (lane * 4 in bits 2..6, the code pair above); the tiles follow at 1 KB multiples.
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 8191) & ~uintptr_t(8191));
    uint32_t* lut = reinterpret_cast<uint32_t*>(base);                    // [NL][COPIES] operand pairs
    uint8_t* sA = base + Q::kLutBytes;                                    // [kStages][128 x 64]
    uint8_t* sB = sA + kStages * kABytes;                                 // [kStages][NT x 64]
    uint8_t* sC = sB + kStages * kBBytes;  // [2] x (codes 128 x 128 B, scales 128 x SW words)
    static_assert(Q::kLutBytes % 1024 == 0, "table size");
    uint64_t* bars = reinterpret_cast<uint64_t*>(sC + kChunkSlots * kChunkBytes);
    // full[s]: stage s's A (its decoder group) and B (the copy's bytes) are in place;
    // empty[s]: the MMAs that read stage s have completed.
    uint64_t* full = bars;
    uint64_t* empty = full + kStages;
    uint64_t* cfull = empty + kStages;
    uint64_t* cempty = cfull + kChunkSlots;
    uint64_t* tile_full = cempty + kChunkSlots;  // [2]
    uint64_t* tile_empty = tile_full + 2;        // [2]
    uint64_t* drain = tile_empty + 2;
    int* ctl = reinterpret_cast<int*>(drain + 1);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl);
    volatile int* abort_flag = ctl + 1;
    int* total_items = ctl + 2;
    int* cum = ctl + 8;              // [experts + 1]
    int* offs = cum + (p.experts + 1);  // [experts + 1] pair offsets

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.experts;
    const int mtiles = p.rows / kBM;
    const int nk = p.cols / kBK;
    const int ngroups = p.cols / G;
    const int nchunks = (nk + SPC - 1) / SPC;

    if constexpr (!SK) {
        for (int i = tid; i <= E; i += kThreads2) cum[i] = offs[i] = p.offsets[i];
        __syncthreads();
    }
    if (tid == 0) {
        if constexpr (SK) {
            *total_items = mtiles * nchunks;  // units
        } else {
            bool ok = cum[0] == 0 && cum[E] == p.P;
            int prev = 0, acc = 0;
            for (int e = 0; e <= E; ++e) {
                const int off = cum[e];
                if (e > 0) {
                    const int n = off - prev;
                    ok = ok && n >= 0;
                    const int nt = n > 0 ? (n + NT - 1) / NT : 0;
                    cum[e - 1] = acc;
                    acc += nt * mtiles;
                }
                prev = off;
            }
            cum[E] = acc;
            *total_items = ok ? acc : -1;
        }
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full + s, 32 * kDec2 / 2 + 1);  // a decoder group + the B copy
            mbar_init(empty + s, kMmaWarps);          // a commit from each MMA thread
        }
        for (int s = 0; s < kChunkSlots; ++s) {
            mbar_init(cfull + s, 1 + 32);  // the code copy's arrival and the 32 scale lanes
            mbar_init(cempty + s, kDecThreads2);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tile_full + b, kMmaWarps);
            mbar_init(tile_empty + b, 32 * kEpiWarps);
        }
        mbar_init(drain, kMmaWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int total = *total_items;
    if (total < 0) {
        if (tid == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        return;
    }
    // The code and scale warps start their copies at once; the others fill the table and
    // allocate TMEM, then meet at a named barrier (the copying warps use neither).
    uint32_t tmem = 0;
    if (warp != kCodeWarp && warp != kScaleWarp) {
        const int ftid = warp < kCodeWarp ? tid : tid - 64;
        for (int i = ftid; i < NL * COPIES; i += kThreads2 - 64) {
            const int idx = i / COPIES;
            lut[i] = pack2<XT>(p.centroids[idx & (LEVELS - 1)], p.centroids[idx / LEVELS]);
        }
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(Q::kTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"r"(kThreads2 - 64) : "memory");
        tc_fence_after();
        tmem = *tmem_slot;
    }

    // One item: chunks [c0, c1) (stages [kb, ke)) of row tile mt of expert e against pair
    // tile nt (pairs i0 .. i0 + nvalid - 1).  Every role walks the same item sequence.
    struct Item {
        int e, mt, nt, i0, nvalid, c0, c1, kb, ke, state;
    };
    const int ub = SK ? (int)((int64_t)blockIdx.x * total / gridDim.x) : 0;  // this CTA's units (SK)
    const int ue = SK ? (int)((int64_t)(blockIdx.x + 1) * total / gridDim.x) : 0;
    auto load_item = [&](Item& I) -> bool {
        if constexpr (SK) {
            const int u = I.state;
            if (u >= ue) return false;
            I.e = 0;
            I.nt = 0;
            I.i0 = 0;
            I.nvalid = p.P;
            I.mt = u / nchunks;
            I.c0 = u - I.mt * nchunks;
            I.c1 = min(nchunks, I.c0 + (ue - u));
        } else {
            const int item = I.state;
            if (item >= total) return false;
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cum[mid] <= item) lo = mid; else hi = mid - 1;
            }
            I.e = lo;
            const int off0 = offs[lo], n = offs[lo + 1] - off0;
            const int ntiles = (n + NT - 1) / NT;
            const int local = item - cum[lo];
            I.mt = local / ntiles;
            I.nt = local - I.mt * ntiles;
            I.i0 = off0 + I.nt * NT;
            I.nvalid = min(NT, n - I.nt * NT);
            I.c0 = 0;
            I.c1 = nchunks;
        }
        I.kb = I.c0 * SPC;
        I.ke = min(I.c1 * SPC, nk);
        return true;
    };
    auto first_item = [&](Item& I) -> bool {
        I.state = SK ? ub : (int)blockIdx.x;
        return load_item(I);
    };
    auto next_item = [&](Item& I) -> bool {
        I.state += SK ? I.c1 - I.c0 : (int)gridDim.x;
        return load_item(I);
    };

    if (warp < kMmaWarps) {
        // ------------------------------------------------ MMA issuers (one thread each)
        // Each MMA instruction blocks its thread for tens of cycles and each commit for about a
        // hundred, so two threads share a tile of at most 128 pairs: they take alternate K
        // stages into their own 128 accumulator columns (the epilogue adds the two).  A wider
        // tile is one N = 256 MMA per K step from thread 0 (the tensor pipe runs at full rate
        // only at N = 256), thread 1 only committing.  Both wait for every stage and commit
        // every stage, so a slot is released only after both.
        if (lane == 0) {
            const int me = warp;
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
            uint32_t it = 0, tile_it = 0;
            bool ok = true;
            Item I;
            for (bool have = first_item(I); have && ok; have = next_item(I), ++tile_it) {
                const int kb = I.kb, ke = I.ke;
                const int ninst = (I.nvalid + 15) & ~15;
                const bool ksplit = ninst <= 128 && ke - kb >= 2;
                const int ncols = ksplit ? ninst : (me == 0 ? ninst : 0);
                const uint32_t idesc = f16_idesc(XT, ncols > 0 ? ncols : 16);
                const int buf = tile_it & 1;
                if (!mbar_wait(tile_empty + buf, ((tile_it >> 1) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * kBuf + me * kHalf);
                const uint32_t boff = 0u;
                for (int kc = kb; kc < ke; ++kc, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(full + s, (it / kStages) & 1, abort_flag, p.wait_cycles)) {
                        ok = false;
                        break;
                    }
                    const bool mine = ksplit ? ((kc - kb) & 1) == me : ncols > 0;
                    if (mine) {
                        const bool first = ksplit ? kc - kb == me : kc == kb;
                        const uint64_t ad = sw128_desc(a0 + s * kABytes), bd = sw128_desc(b0 + s * kBBytes + boff);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc_mma(d, ad + 2 * kk, bd + 2 * kk, idesc, !(first && kk == 0));
                    }
                    tc_commit(empty + s);
                }
                if (!ok) break;
                tc_commit(tile_full + buf);
            }
            tc_commit(drain);
            if (!mbar_wait_drain(drain, 0)) *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp < kMmaWarps + kBWarps) {
        // ------------------------------------------------ B: one tensor copy per stage, warps alternate stages
        if (lane == 0) {
            if constexpr (SK) asm volatile("griddepcontrol.wait;" ::: "memory");  // x16 written
            const int bw = warp - kMmaWarps;
            const uint32_t b0 = smem_u32(sB);
            uint32_t it = 0;
            bool ok = true;
            Item I;
            for (bool have = first_item(I); have && ok; have = next_item(I)) {
                int bi = 0;
                while (bi < 4 && (128 >> bi) >= I.nvalid) ++bi;  // smallest box of 256 >> bi rows >= nvalid
                const int box_rows = 256 >> bi;                   // at most NT (the host checks)
                const int i0 = I.i0;
                for (int kc = I.kb; kc < I.ke; ++kc, ++it) {
                    if ((int)(it % kBWarps) != bw) continue;
                    const int s = it % kStages;
                    if (!mbar_wait(empty + s, ((it / kStages) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                    uint64_t* fb = full + s;
                    mbar_expect_tx(fb, (uint32_t)box_rows * 128u);
                    tma_load_2d(b0 + s * kBBytes, &tm.b[bi], kc * kBK, i0, fb);
                }
            }
            // copies this thread issued that may still be in flight complete before the CTA may exit
            // (the full barrier also waits for the decoders' arrivals, which come unless they aborted)
            for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
                if ((int)(j % kBWarps) == bw && !mbar_wait_drain(full + j % kStages, (j / kStages) & 1))
                    *abort_flag = 1;
        }
        __syncwarp();
    } else if (warp == kCodeWarp) {
        // ------------------------------------------------ code chunks: one tensor copy each
        if (lane == 0) {
            const uint32_t c0 = smem_u32(sC);
            uint32_t cc = 0;
            bool ok = true;
            Item I;
            for (bool have = first_item(I); have && ok; have = next_item(I)) {
                const int e = I.e, mt = I.mt;
                for (int c = I.c0; c < I.c1; ++c, ++cc) {
                    const int slot = cc % kChunkSlots;
                    if (!mbar_wait(cempty + slot, ((cc / kChunkSlots) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                    mbar_expect_tx(cfull + slot, (uint32_t)kChunkCodeBytes);
                    tma_load_3d(c0 + slot * kChunkBytes, &tm.c, c * 32, mt * kBM, e, cfull + slot);
                }
            }
            for (uint32_t j = cc > (uint32_t)kChunkSlots ? cc - kChunkSlots : 0; j < cc; ++j) {
                // the slot's phase also waits for the scale lanes: wait on the copy's bytes alone is not
                // possible, so wait for the phase (the scale lanes arrive unless they aborted)
                if (!mbar_wait_drain(cfull + j % kChunkSlots, (j / kChunkSlots) & 1)) *abort_flag = 1;
            }
        }
        __syncwarp();
    } else if (warp == kScaleWarp) {
        // ------------------------------------------------ the scales of each code chunk
        const uint32_t* sc32 = reinterpret_cast<const uint32_t*>(p.scales);  // ngroups and ess are even
        const int nsw_row = ngroups >> 1;
        uint32_t cc = 0;
        Item I;
        for (bool have = first_item(I); have; have = next_item(I)) {
            const uint32_t* rows0 = sc32 + ((int64_t)I.e * p.ess + (int64_t)I.mt * kBM * ngroups) / 2;
            bool ok = true;
            for (int c = I.c0; c < I.c1; ++c, ++cc) {
                const int slot = cc % kChunkSlots;
                if (!mbar_wait(cempty + slot, ((cc / kChunkSlots) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                const int wlo = (c * CPC / G) >> 1;
                const int ghi = min(ngroups - 1, ((c + 1) * CPC - 1) / G);
                const int nw = (ghi >> 1) - wlo + 1;  // 1..SW words per row
                const int rpi = 32 / nw;              // rows per instruction
                const int rr = lane / nw, j = lane - rr * nw;
                const uint32_t dst0 = smem_u32(sC) + slot * kChunkBytes + kChunkCodeBytes;
                if (rr < rpi) {
                    for (int r = rr; r < kBM; r += rpi)
                        cp_async4(dst0 + r * (SW * 4) + ((j ^ ((r / (32 / SW)) & (SW - 1))) << 2),
                                  rows0 + (int64_t)r * nsw_row + wlo + j, 4u);
                }
                cp_async_commit();
                cp_async_wait<0>();
                mbar_arrive(cfull + slot);
            }
            if (!ok) break;
        }
        cp_async_wait<0>();
    } else if (warp < kFirstEpi) {
        // ------------------------------------------------ decoders
        const int dw = warp - kFirstDec2;  // 0..15
        const int grp = dw >> 3;           // takes the stages with it & 1 == grp
        const int h = (dw >> 2) & 1;       // which 32 codes of the 64-wide stage
        const int r = (dw & 3) * 32 + lane;
        const int rx = r & 7;
        const uint32_t lutl = smem_u32(lut) + (COPIES == 32 ? lane * 4 : 0);
        const uint32_t crow0 = smem_u32(sC) + r * 128;  // 16-byte piece q of the row: crow + ((q ^ rx) << 4)
        const uint32_t srow0 = smem_u32(sC) + kChunkCodeBytes + r * (SW * 4);  // word j: srow + ((j ^ sx) << 2)
        const int sx = (r / (32 / SW)) & (SW - 1);
        const uint32_t arow0 = smem_u32(sA) + r * 128 + (rx << 4);  // piece q of the A row: arow ^ (q << 4)
        // The stage counter it runs over every stage of the CTA; this group decodes those with
        // (it & 1) == grp.  Each code chunk is waited for once and released once by every
        // decoder thread; the empty barrier of the group's next stage is tested before the
        // current stage is decoded, so that its latency overlaps the decode.
        uint32_t it = 0, cc = 0;
        bool ok = true, pre = false;  // pre: the empty test of the next stage succeeded
        Item I;
        for (bool have = first_item(I); have && ok; have = next_item(I)) {
            for (int c = I.c0; c < I.c1 && ok; ++c, ++cc) {
                const int k0 = c * SPC, nsub = min(SPC, I.ke - k0);
                const int slot = cc % kChunkSlots;
                if (!mbar_wait(cfull + slot, (cc / kChunkSlots) & 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                const uint32_t crow = crow0 + slot * kChunkBytes, srow = srow0 + slot * kChunkBytes;
                const int gbase = (c * CPC / G) & ~1;  // group at word 0 of the chunk's scale rows
                for (int sub = (int)((it ^ (uint32_t)grp) & 1u); sub < nsub; sub += 2) {
                    const uint32_t sit = it + (uint32_t)sub;
                    const int kc = k0 + sub;
                    const int s = sit % kStages;
                    if (!pre && !mbar_wait(empty + s, ((sit / kStages) & 1) ^ 1, abort_flag, p.wait_cycles)) { ok = false; break; }
                    {
                        const uint32_t nit = sit + 2;  // this group's next stage
                        pre = mbar_peek(empty + nit % kStages, ((nit / kStages) & 1) ^ 1);
                    }
                    const int lq = 64 * sub + 32 * h;  // first code of this thread within the chunk
                    const int w0 = lq / F::kCW, pos0 = lq - w0 * F::kCW;
                    const int o = w0 & 3, q0 = w0 >> 2;
                    // words w0 .. w0 + kWords - 1 lie in pieces q0 and, for 3-bit codes with o != 0, q0 + 1
                    const uint4 P0 = lds128(crow + ((q0 ^ rx) << 4));
                    uint4 P1 = P0;
                    if (F::kBits == 3 && o != 0) P1 = lds128(crow + (((q0 + 1) ^ rx) << 4));
                    const uint32_t WW[8] = {P0.x, P0.y, P0.z, P0.w, P1.x, P1.y, P1.z, P1.w};
                    const int g0 = (kc * kBK + 32 * h) / G - gbase;
                    const uint32_t rr0 = scale_pair<XT>(lds16(srow + (((g0 >> 1) ^ sx) << 2) + (g0 & 1) * 2));
                    uint32_t rr1 = rr0;
                    if (G == 16) {
                        const int g1 = g0 + 1;
                        rr1 = scale_pair<XT>(lds16(srow + (((g1 >> 1) ^ sx) << 2) + (g1 & 1) * 2));
                    }
                    uint32_t out[16];
                    auto dec = [&](auto pos_c, auto o_c) {
                        constexpr int POS0 = decltype(pos_c)::value, O = decltype(o_c)::value;
                        constexpr uint32_t kMask = (1u << (2 * F::kBits)) - 1u;
                        constexpr int kStride = COPIES * 4;  // bytes between table entries
                        constexpr int kLog = COPIES == 32 ? 7 : 2;
#pragma unroll
                        for (int pp = 0; pp < 16; ++pp) {
                            const int tt = POS0 + 2 * pp;
                            const int sh = F::kBits * (tt % F::kCW);
                            const uint32_t w = WW[O + tt / F::kCW];
                            const uint32_t off =
                                (sh >= kLog ? (w >> (sh - kLog)) : (w << (kLog - sh))) & (kMask * kStride);
                            out[pp] = hmul2_bits<XT>(lds32(lutl | off), pp < 8 ? rr0 : rr1);
                        }
                    };
                    using I0 = std::integral_constant<int, 0>;
                    if constexpr (LEVELS == 8) {
                        switch (pos0) {  // pos0 fixes o: (0,0) (2,3) (4,2) (6,1) (8,0)
                            case 0: dec(I0{}, I0{}); break;
                            case 2: dec(std::integral_constant<int, 2>{}, std::integral_constant<int, 3>{}); break;
                            case 4: dec(std::integral_constant<int, 4>{}, std::integral_constant<int, 2>{}); break;
                            case 6: dec(std::integral_constant<int, 6>{}, std::integral_constant<int, 1>{}); break;
                            default: dec(std::integral_constant<int, 8>{}, I0{}); break;
                        }
                    } else if constexpr (LEVELS == 4) {
                        if (o == 0) dec(I0{}, I0{});
                        else dec(I0{}, std::integral_constant<int, 2>{});
                    } else {
                        dec(I0{}, I0{});
                    }
                    const uint32_t arow = arow0 + s * kABytes;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        sts128(arow ^ ((4 * h + c4) << 4), out[4 * c4], out[4 * c4 + 1], out[4 * c4 + 2],
                               out[4 * c4 + 3]);
                    fence_async_smem();
                    mbar_arrive(full + s);
                }
                if (!ok) break;
                it += (uint32_t)nsub;
                mbar_arrive(cempty + slot);
            }
        }
    } else {
        // ------------------------------------------------ epilogue: accumulator -> y rows of the sorted pairs
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int m = quarter * 32 + lane;
        uint32_t tile_it = 0;
        if constexpr (SK) asm volatile("griddepcontrol.wait;" ::: "memory");  // y zeroed, scales written
        Item I;
        for (bool have = first_item(I); have; have = next_item(I), ++tile_it) {
            const int mt = I.mt, i0 = I.i0, nvalid = I.nvalid;
            const int buf = tile_it & 1;
            if (!mbar_wait(tile_full + buf, (tile_it >> 1) & 1, abort_flag, p.wait_cycles)) break;
            tc_fence_after();
            const int64_t ybase = (int64_t)i0 * p.rows + mt * kBM + m;
            const bool ksplit = ((nvalid + 15) & ~15) <= 128 && I.ke - I.kb >= 2;  // as the MMA threads decided
            const uint32_t t0 = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * kBuf);
            // SK: partial sums of a run of chunks, added (y is f32 and zeroed beforehand)
            auto put = [&](int c, float v) {
                if constexpr (SK) {  // the per-row input scale of the prep kernel, then a partial sum
                    atomicAdd(static_cast<float*>(p.y) + ybase + (int64_t)c * p.rows, v * __ldg(p.colscale + i0 + c));
                } else {
                    store_from_float(p.y, ybase + (int64_t)c * p.rows, p.ydt, v);
                }
            };
            if (ksplit) {
                for (int c0 = 0; c0 < nvalid; c0 += 16) {  // the two K halves' partial sums
                    uint32_t v[16], w[16];
                    tc_ld16(t0 + (uint32_t)c0, v);
                    tc_ld16(t0 + (uint32_t)kHalf + (uint32_t)c0, w);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < nvalid) put(c0 + j, __uint_as_float(v[j]) + __uint_as_float(w[j]));
                }
            } else {
                for (int c0 = 0; c0 < nvalid; c0 += 32) {
                    uint32_t v[32];
                    tc_ld32(t0 + (uint32_t)c0, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < nvalid) put(c0 + j, __uint_as_float(v[j]));
                }
            }
            tc_fence_before();
            mbar_arrive(tile_empty + buf);
        }
    }

    __syncthreads();
    if (tid == 0 && *abort_flag && p.err) atomicOr(p.err, TQ_DEVERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Q::kTmemCols) : "memory");
    }
}

// Token rows into sorted pair order: xs[i] = x[perm[i] / k] (zero and BAD_ID for
// an out-of-range perm entry).  One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ perm,
                                                          int P, int k, int vecs, uint4* __restrict__ xs,
                                                          uint32_t* err) {
    const int wpb = blockDim.x >> 5, lane = threadIdx.x & 31;
    for (int i = blockIdx.x * wpb + (threadIdx.x >> 5); i < P; i += gridDim.x * wpb) {
        const int f = __ldg(perm + i);
        const bool ok = f >= 0 && f < P;
        if (!ok && lane == 0 && err) atomicOr(err, TQ_DEVERR_BAD_ID);
        const uint4* src = x + (size_t)(ok ? f / k : 0) * vecs;
        uint4* dst = xs + (size_t)i * vecs;
#pragma unroll 4
        for (int v = lane; v < vecs; v += 32) dst[v] = ok ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Pair tiles and ring depths of the staged kernel: 256-pair tiles with 3 stages for
// expert-sorted batches; for the dense split-K form, tiles of 16 or 64 pairs,
// whose small B stages leave room for a deeper ring (the decode and MMA latencies
// of a stage are about a thousand cycles each).
constexpr int kSkSmallNT = 16, kSkSmallST = 8, kSkNT = 64, kSkST = 6;

template <int LEVELS, int G, int NT = kNT, int ST = 3>
size_t qmm2_smem_bytes(int experts) {
    return (size_t)Q2Fmt<LEVELS, G, NT, ST>::kSmem + (size_t)(experts + 1) * 8;
}

template <int LEVELS>
size_t qmm2_smem_bytes_g(int G, int experts) {
    switch (G) {
        case 16: return qmm2_smem_bytes<LEVELS, 16>(experts);
        case 32: return qmm2_smem_bytes<LEVELS, 32>(experts);
        case 64: return qmm2_smem_bytes<LEVELS, 64>(experts);
        default: return qmm2_smem_bytes<LEVELS, 128>(experts);
    }
}

size_t qmm2_smem_for(int levels, int G, int experts) {
    return levels == 4 ? qmm2_smem_bytes_g<4>(G, experts)
                       : levels == 8 ? qmm2_smem_bytes_g<8>(G, experts) : qmm2_smem_bytes_g<16>(G, experts);
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

// The staged kernel holds a tile's scale block in 128 bytes per row (an even
// group count of at most 64) and reads codes by tensor copies (rows and experts
// a multiple of 16 bytes apart); other shapes use the first kernel.
bool staged_fits(const QmmParams& p, int G, int levels) {
    const int ngroups = p.cols / G;
    return ngroups <= 64 && ngroups % 2 == 0 && p.ess % 2 == 0 && aligned(p.scales, 4) && aligned(p.codes, 16) &&
           p.row_stride % 4 == 0 && p.esw % 4 == 0 && p.row_stride <= (int64_t)1 << 31 &&
           qmm2_smem_for(levels, G, p.experts) <= (size_t)kSmemLimit && tensor_map_encoder() != nullptr;
}

// Tensor maps of the pair rows (P x cols, 2-byte elements) and of the codes.
bool encode_maps(const QmmParams& p, const void* rows_base, QmmMaps& m) {
    const EncodeFn enc = tensor_map_encoder();
    for (int i = 0; i < 5; ++i) {
        const cuuint64_t dims[2] = {(cuuint64_t)p.cols, (cuuint64_t)p.P};
        const cuuint64_t strides[1] = {(cuuint64_t)p.cols * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBoxRows[i]};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&m.b[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(rows_base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    const int64_t esw = p.experts > 1 ? p.esw : (int64_t)p.rows * p.row_stride;
    const cuuint64_t dims[3] = {(cuuint64_t)p.row_stride, (cuuint64_t)p.rows, (cuuint64_t)p.experts};
    const cuuint64_t strides[2] = {(cuuint64_t)p.row_stride * 4, (cuuint64_t)esw * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)kBM, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(&m.c, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(p.codes), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

template <int LEVELS, int G, int XT>
tq_status launch_qmm2(const QmmParams& p, const QmmMaps& maps, cudaStream_t st) {
    const size_t smem = qmm2_smem_bytes<LEVELS, G>(p.experts);
    if (ensure_smem((const void*)gather_qmm2_kernel<LEVELS, G, XT, kNT, 3, false>, smem) != cudaSuccess)
        return TQ_ERR_CUDA;
    gather_qmm2_kernel<LEVELS, G, XT, kNT, 3, false><<<sm_count(), kThreads2, smem, st>>>(p, maps);
    return launch_status();
}

// Dense split-K form (fp16 operands): one CTA per SM at most, each over a
// contiguous range of the (row tile, code chunk) units.
template <int LEVELS, int G, int NT, int ST>
tq_status launch_sk(const QmmParams& p, const QmmMaps& maps, cudaStream_t st) {
    using Q = Q2Fmt<LEVELS, G, NT, ST>;
    const size_t smem = qmm2_smem_bytes<LEVELS, G, NT, ST>(1);
    if (smem > (size_t)kSmemLimit) return TQ_ERR_UNSUPPORTED;
    const int units = (p.rows / kBM) * ((p.cols / kBK + Q::kSPC - 1) / Q::kSPC);
    const int grid = units < sm_count() ? units : sm_count();
    if (ensure_smem((const void*)gather_qmm2_kernel<LEVELS, G, 0, NT, ST, true>, smem) != cudaSuccess)
        return TQ_ERR_CUDA;
    // Programmatic dependent launch: the prologue and the first code chunks overlap the prep
    // kernel; only the input-row copies and the epilogue wait for it (griddepcontrol.wait).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads2);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, gather_qmm2_kernel<LEVELS, G, 0, NT, ST, true>, p, maps);
    return launch_status();
}

template <int LEVELS, int G>
tq_status launch_sk_nt(const QmmParams& p, const QmmMaps& maps, cudaStream_t st) {
    return p.P <= kSkSmallNT ? launch_sk<LEVELS, G, kSkSmallNT, kSkSmallST>(p, maps, st)
                             : launch_sk<LEVELS, G, kSkNT, kSkST>(p, maps, st);
}

template <int LEVELS>
tq_status launch_sk_g(const QmmParams& p, int group, const QmmMaps& maps, cudaStream_t st) {
    switch (group) {
        case 16: return launch_sk_nt<LEVELS, 16>(p, maps, st);
        case 32: return launch_sk_nt<LEVELS, 32>(p, maps, st);
        case 64: return launch_sk_nt<LEVELS, 64>(p, maps, st);
        case 128: return launch_sk_nt<LEVELS, 128>(p, maps, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

// x (f32 [T, cols], cols a multiple of 64) -> x16 = fp16(x / 2^e_t) with 2^e_t the power of
// two just above max |x[t, :]| (colscale[t] = 2^e_t, so the outputs of row t are scaled back
// exactly), one block per input row, four 16-byte loads in flight per thread; the remaining
// blocks zero y (f32, ny values) for the split-K sums.  The dependent matvec may launch at once.
TQ_DEVFN float4 ld_row4(const float* r, int i, bool v4) {
    if (v4) return __ldg(reinterpret_cast<const float4*>(r) + i);
    return make_float4(__ldg(r + 4 * i), __ldg(r + 4 * i + 1), __ldg(r + 4 * i + 2), __ldg(r + 4 * i + 3));
}

__global__ void __launch_bounds__(256) qmv_tc_prep_kernel(const float* __restrict__ x, int T, int cols,
                                                          __half* __restrict__ x16, float* __restrict__ colscale,
                                                          float* __restrict__ y, int64_t ny) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float red[8];
    const int tid = threadIdx.x;
    if ((int)blockIdx.x >= T) {
        const int64_t n0 = (int64_t)(blockIdx.x - T) * blockDim.x + tid, step = (int64_t)(gridDim.x - T) * blockDim.x;
        for (int64_t i = n0; i < ny; i += step) y[i] = 0.f;
        return;
    }
    const float* xr = x + (int64_t)blockIdx.x * cols;
    const bool v4 = (reinterpret_cast<uintptr_t>(xr) & 15) == 0;
    const int n4 = cols / 4, nt = blockDim.x;
    float m = 0.f;
    for (int i0 = tid; i0 < n4; i0 += 4 * nt) {
        float4 v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = i0 + t * nt < n4 ? ld_row4(xr, i0 + t * nt, v4) : make_float4(0, 0, 0, 0);
#pragma unroll
        for (int t = 0; t < 4; ++t)
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v[t].x), fabsf(v[t].y)), fmaxf(fabsf(v[t].z), fabsf(v[t].w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    m = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    int e = 0;
    if (m > 0.f && m <= 3.4e38f) frexpf(m, &e);  // m = f * 2^e, f in [0.5, 1): |x| / 2^e < 1
    const float inv = ldexpf(1.f, -e);
    if (tid == 0) colscale[blockIdx.x] = ldexpf(1.f, e);
    uint2* dr = reinterpret_cast<uint2*>(x16 + (int64_t)blockIdx.x * cols);  // 4 halves per 8 bytes
    for (int i0 = tid; i0 < n4; i0 += 4 * nt) {
        float4 v[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) v[t] = i0 + t * nt < n4 ? ld_row4(xr, i0 + t * nt, v4) : make_float4(0, 0, 0, 0);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (i0 + t * nt < n4) {
                __half2 a = __floats2half2_rn(v[t].x * inv, v[t].y * inv), b = __floats2half2_rn(v[t].z * inv, v[t].w * inv);
                dr[i0 + t * nt] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
            }
        }
    }
}

template <int LEVELS, int G, int XT>
tq_status launch_any(const QmmParams& p, const QmmMaps* maps, cudaStream_t st) {
    return maps ? launch_qmm2<LEVELS, G, XT>(p, *maps, st) : launch_qmm<LEVELS, G, XT>(p, st);
}

template <int LEVELS, int G>
tq_status dispatch_xt(const QmmParams& p, int xt, const QmmMaps* maps, cudaStream_t st) {
    return xt == 0 ? launch_any<LEVELS, G, 0>(p, maps, st) : launch_any<LEVELS, G, 1>(p, maps, st);
}

template <int LEVELS>
tq_status dispatch_g(const QmmParams& p, int group, int xt, const QmmMaps* maps, cudaStream_t st) {
    switch (group) {
        case 16: return dispatch_xt<LEVELS, 16>(p, xt, maps, st);
        case 32: return dispatch_xt<LEVELS, 32>(p, xt, maps, st);
        case 64: return dispatch_xt<LEVELS, 64>(p, xt, maps, st);
        case 128: return dispatch_xt<LEVELS, 128>(p, xt, maps, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace

extern "C" size_t tq_gather_qmm_workspace_bytes(int32_t P, int32_t cols, int32_t per_pair_input) {
    return per_pair_input || P <= 0 || cols <= 0 ? 0 : (size_t)P * (size_t)cols * 2;
}

extern "C" tq_status tq_gather_qmm(const tq_qweight_t* w, const void* x, tq_dtype xdt, const int32_t* perm,
                                   const int32_t* offsets, int32_t P, int32_t k, int32_t per_pair_input, void* y,
                                   tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream) {
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
    const size_t need = tq_gather_qmm_workspace_bytes(P, w->cols, per_pair_input);
    if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16))) return TQ_ERR_INVALID;
    if (P == 0) return TQ_OK;
    QmmParams p{};
    p.wait_cycles = wait_budget();
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
    QmmMaps maps;
    const QmmMaps* mp = nullptr;
    if (staged_fits(p, w->group, w->cb.levels)) {
        const void* rows = x;
        if (!per_pair_input) {  // token rows into sorted pair order first
            const int vecs = w->cols / 8;
            gather_rows_kernel<<<sm_count() * 8, 256, 0, st>>>(reinterpret_cast<const uint4*>(x), perm, P, k, vecs,
                                                               reinterpret_cast<uint4*>(ws), err);
            const tq_status s = launch_status();
            if (s != TQ_OK) return s;
            rows = ws;
        }
        if (!encode_maps(p, rows, maps)) return TQ_ERR_CUDA;
        mp = &maps;
    }
    switch (w->cb.levels) {
        case 4: return dispatch_g<4>(p, w->group, xt, mp, st);
        case 8: return dispatch_g<8>(p, w->group, xt, mp, st);
        case 16: return dispatch_g<16>(p, w->group, xt, mp, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

extern "C" size_t tq_qmv_tc_workspace_bytes(int32_t T, int32_t cols) {
    if (T <= 0 || cols <= 0) return 0;
    return ((size_t)T * (size_t)cols * 2 + 15) / 16 * 16 + ((size_t)T * 4 + 15) / 16 * 16;
}

extern "C" tq_status tq_qmv_tc(const tq_qweight_t* w, const float* x_rot, int32_t T, float* y, void* ws,
                               size_t ws_bytes, uint32_t* err, void* stream) {
    if (!w || !w->codes || !w->scales || !w->cb.centroids) return TQ_ERR_INVALID;
    if (w->experts <= 0 || w->rows <= 0 || w->cols <= 0) return TQ_ERR_INVALID;
    if (!(w->group == 16 || w->group == 32 || w->group == 64 || w->group == 128) || w->cols % w->group)
        return TQ_ERR_INVALID;
    if (w->row_stride_words < tq_row_words(w->cb.levels, w->cols)) return TQ_ERR_INVALID;
    if (T < 0) return TQ_ERR_INVALID;
    if (T == 0) return TQ_OK;
    if (!x_rot || !y) return TQ_ERR_INVALID;
    if (!(w->cb.levels == 4 || w->cb.levels == 8 || w->cb.levels == 16)) return TQ_ERR_UNSUPPORTED;
    if (w->rows % kBM || w->cols % kBK || T > kSkNT) return TQ_ERR_UNSUPPORTED;
    const size_t need = tq_qmv_tc_workspace_bytes(T, w->cols);
    if (!ws || ws_bytes < need || !aligned(ws, 16)) return TQ_ERR_INVALID;
    QmmParams p{};
    p.wait_cycles = wait_budget();
    p.codes = w->codes;
    p.scales = w->scales;
    p.row_stride = w->row_stride_words;
    p.esw = 0;
    p.ess = 0;
    p.rows = w->rows;
    p.cols = w->cols;
    p.experts = 1;  // the dense matrix is expert 0
    p.centroids = w->cb.centroids;
    __half* x16 = static_cast<__half*>(ws);
    float* cs = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ((size_t)T * w->cols * 2 + 15) / 16 * 16);
    p.x = x16;
    p.P = T;
    p.k = 1;
    p.per_pair = 1;
    p.y = y;
    p.ydt = TQ_F32;
    p.colscale = cs;
    p.err = err;
    if (!staged_fits(p, w->group, w->cb.levels)) return TQ_ERR_UNSUPPORTED;
    QmmMaps maps;
    if (!encode_maps(p, x16, maps)) return TQ_ERR_CUDA;
    cudaStream_t st = as_stream(stream);
    const int64_t ny = (int64_t)T * w->rows;
    const int zb = (int)std::min<int64_t>((ny + 255) / 256, 4 * (int64_t)sm_count());
    qmv_tc_prep_kernel<<<T + zb, 256, 0, st>>>(x_rot, T, w->cols, x16, cs, y, ny);
    const tq_status s = launch_status();
    if (s != TQ_OK) return s;
    switch (w->cb.levels) {
        case 4: return launch_sk_g<4>(p, w->group, maps, st);
        case 8: return launch_sk_g<8>(p, w->group, maps, st);
        default: return launch_sk_g<16>(p, w->group, maps, st);
    }
}
