// Ternary inline-decode matvec (one input vector per item): the kernel behind
// tq_qmv / tq_gather_qmv / tq_multi_gather_qmv for three-level books.
//
// "How it works", "The ternary tier (1.58 bits)": 20 trits per 32-bit word in
// base 3; "Running a quantized layer": decode inline, no per-weight integer
// division.
//
// Decode.  A word w = sum_j d_j 3^j is split into two ten-digit halves
// (w / 3^10 is a multiply by a constant).  Each half h becomes the 32-bit
// fixed-point fraction F = h*72736 + 8860 (in [h, h+1) 2^32/3^10 for every h),
// and mul.hi(F, 81) yields the next four digits as one number v in [0, 81)
// (mul.hi(F, 9) the last two).  v indexes a per-lane copy of an 81-entry table
// in shared memory whose entry packs the four digits into four bytes; two
// dp2a instructions multiply them by the input, which is held as 16-bit
// integers (per group: x = xs_g * xq, |xq| <= 32767).  The three-level book is
// affine (c0 + d*delta), so per group
//     sum_k c[d_k] x_k = delta * xs_g * (sum_k d_k xq_k) + c0 * sum_k x_k,
// an exact integer dot product plus two precomputed per-group terms.
//
// Work layout.  A warp takes RPW rows of one item and walks their columns in
// steps of UPW consecutive units (RPW * UPW = 32 lanes): lane (r, c) decodes
// unit s*UPW + c of row r.  A load instruction thus covers RPW contiguous
// segments of UPW units (coalesced), and the UPW units in flight read their
// quantized input from shared-memory blocks that start on distinct 4-bank
// groups, shared by the RPW lanes of each unit (broadcast).  CTAs are
// persistent: each takes a contiguous range of (item, row block) tasks,
// prepares the quantized input once per distinct input vector, and its warps
// share the tasks round-robin.
#include <algorithm>
#include <cstdlib>
#include <numeric>

#include "qmv_impl.cuh"
#include "tma.cuh"

namespace tq {
namespace {

template <int G>
struct TritFmt {
    static constexpr int kUT = 20 / Gcd<20, G>::v * G;  // trits per unit: lcm(20, G)
    static constexpr int kUW = kUT / 20;                // words per unit
    static constexpr int kGPU = kUT / G;                // groups per unit
    static constexpr int kXW = 12;                      // shared words of 16-bit x pairs per code word (10 used)
    static constexpr int kAB = kUW * kXW;               // offset of the (a_g, b_g) floats in a unit block
    static constexpr int kRaw = kAB + 2 * kGPU;
    // unit block stride: whole 16-byte chunks, = 4 (mod 8) words so that 8
    // consecutive units start on distinct 4-bank groups
    static constexpr int kUS = ((kRaw + 3) / 4 * 4) % 8 == 4 ? (kRaw + 3) / 4 * 4 : (kRaw + 3) / 4 * 4 + 4;
};

TQ_DEVFN uint32_t dp2a_lo(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
TQ_DEVFN uint32_t dp2a_hi(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

struct TritParams {
    QmvParams q;
    int units;      // units per row
    int nsteps;     // steps of UPW units per row
    int tasks_per_item;
    int n_items;
    int total_tasks;
    // input stage of the tensor-copy kernel: 0 = q.x is the rotated input; 1 = xin rows are
    // rotated here; 2 = xin rows are [gate | up] pairs, SwiGLU'd then rotated here
    int xmode;
    const void* xin;
    int xdt;
    const int8_t* xsigns;
    int xblock;
};

template <int G, int RPW>
__global__ void __launch_bounds__(256, 2) qmv_trit_kernel(const TritParams tp) {
    using F = TritFmt<G>;
    constexpr int UPW = 32 / RPW;
    constexpr int UW = F::kUW, GPU = F::kGPU, US = F::kUS;
    const QmvParams& p = tp.q;
    extern __shared__ __align__(16) uint32_t sm[];
    uint32_t* lut = sm;            // [81][32]: per-lane copies, entry v of lane l at v*32 + l
    uint32_t* xb = lut + 81 * 32;  // [nsteps*UPW units][US]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    for (int i = tid; i < 81 * 32; i += blockDim.x) {
        const int v = i >> 5;
        lut[i] = (uint32_t)(v / 27) | ((uint32_t)((v / 9) % 3) << 8) | ((uint32_t)((v / 3) % 3) << 16) |
                 ((uint32_t)(v % 3) << 24);
    }
    // centroid c[d] = c0 + d * delta (three-level affine book)
    const float c0 = __ldg(p.centroids), delta = __ldg(p.centroids + 1) - c0;
    if (tid == 0 && p.err && fabsf((__ldg(p.centroids + 2) - __ldg(p.centroids + 1)) - delta) > 1e-6f * fabsf(delta))
        atomicOr(p.err, TQ_DEVERR_BAD_BOOK);

    const int t_begin = (int)((int64_t)blockIdx.x * tp.total_tasks / gridDim.x);
    const int t_end = (int)((int64_t)(blockIdx.x + 1) * tp.total_tasks / gridDim.x);
    const int r = lane / UPW, c = lane % UPW;
    const uint32_t* lut_lane = lut + lane;
    const int ngroups = p.ngroups;
    const int nunits_pad = tp.nsteps * UPW;
    int cur_vec = -1;

    for (int t0 = t_begin; t0 < t_end;) {
        const int item = t0 / tp.tasks_per_item;
        const int t1 = min(t_end, (item + 1) * tp.tasks_per_item);
        int e, vec;
        if (p.mode == kModeDense) {
            e = 0;
            vec = item;
        } else {
            e = __ldg(p.ids + item);
            vec = p.mode == kModeGather ? item / p.k : item;
        }
        const int64_t out0 = (int64_t)item * p.rows;
        if (vec != cur_vec) {
            // Quantize this vector per group: xs = max|x| / 32767, xq = rint(x / xs),
            // a_g = delta * xs, b_g = c0 * sum(x); zero beyond the last column.
            __syncthreads();
            const float* xv = p.x + (int64_t)vec * p.cols;
            for (int g = tid; g < nunits_pad * GPU; g += blockDim.x) {
                const int u = g / GPU, gl = g - u * GPU;  // unit, group within the unit
                float mx = 0.f, sum = 0.f;
                if (g < ngroups) {
#pragma unroll 8
                    for (int k = 0; k < G; ++k) {
                        const float v = xv[g * G + k];
                        mx = fmaxf(mx, fabsf(v));
                        sum += v;
                    }
                }
                uint32_t* blk = xb + u * US;
                reinterpret_cast<float*>(blk + F::kAB)[2 * gl] = delta * (mx / 32767.0f);
                reinterpret_cast<float*>(blk + F::kAB)[2 * gl + 1] = c0 * sum;
                const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
                // pair pp of word w holds the 16-bit inputs of unit trits (20w + 19 - 2pp, 20w + 18 - 2pp)
#pragma unroll 4
                for (int k = 0; k < G; k += 2) {
                    const int tl = gl * G + k;  // even unit-local trit
                    const int w = tl / 20, pp = (18 - (tl - 20 * w)) / 2;
                    const int tg = g * G + k;   // global trit
                    const float xlo = g < ngroups ? xv[tg] : 0.f;
                    const float xhi = g < ngroups ? xv[tg + 1] : 0.f;
                    const int qlo = __float2int_rn(xlo * inv), qhi = __float2int_rn(xhi * inv);
                    blk[w * F::kXW + pp] = ((uint32_t)qhi & 0xffffu) | ((uint32_t)qlo << 16);
                }
            }
            __syncthreads();
            cur_vec = vec;
        }
        const bool bad = e < 0 || e >= p.experts;
        if (bad && tid == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);

        for (int t = t0 + warp; t < t1; t += nwarps) {
            const int row = (t - item * tp.tasks_per_item) * RPW + r;
            const int rowc = row < p.rows ? row : p.rows - 1;
            float tot = 0.f;
            if (!bad) {
                const uint32_t* wrow = p.codes + (int64_t)e * p.expert_stride_w + (int64_t)rowc * p.row_stride;
                const uint16_t* srow = p.scales + (int64_t)e * p.expert_stride_s + (int64_t)rowc * ngroups;
                // prefetch depth in steps: about 64 bytes of codes in flight per lane
                constexpr int PF = UW >= 16 ? 1 : (UW == 8 ? 2 : 4);
                uint32_t wb[PF][UW];
                float sb[PF][GPU];
                auto load = [&](int s, uint32_t (&W)[UW], float (&S)[GPU]) {
                    const int u = s * UPW + c;
#pragma unroll
                    for (int m = 0; m < UW; m += 4) {
                        const int64_t wi = (int64_t)u * UW + m;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (wi < p.row_stride) v = ldg_u4(wrow + wi);
                        W[m] = v.x;
                        W[m + 1] = v.y;
                        W[m + 2] = v.z;
                        W[m + 3] = v.w;
                    }
#pragma unroll
                    for (int g = 0; g < GPU; ++g) {
                        const int gg = u * GPU + g;
                        S[g] = gg < ngroups ? half_bits_to_float(__ldg(srow + gg)) : 0.f;
                    }
                };
#pragma unroll
                for (int i = 0; i < PF - 1; ++i)
                    if (i < tp.nsteps) load(i, wb[i], sb[i]);
                for (int s0 = 0; s0 < tp.nsteps; s0 += PF) {
#pragma unroll
                    for (int uu = 0; uu < PF; ++uu) {
                        const int s = s0 + uu;
                        if (s < tp.nsteps) {
                            if (s + PF - 1 < tp.nsteps) load(s + PF - 1, wb[(uu + PF - 1) % PF], sb[(uu + PF - 1) % PF]);
                            uint32_t acc[GPU];
#pragma unroll
                            for (int g = 0; g < GPU; ++g) acc[g] = 0u;
                            const uint32_t* blk = xb + (s * UPW + c) * US;
#pragma unroll
                            for (int w = 0; w < UW; ++w) {
                                const uint4 xa = *reinterpret_cast<const uint4*>(blk + w * F::kXW);
                                const uint4 xc = *reinterpret_cast<const uint4*>(blk + w * F::kXW + 4);
                                const uint2 xd = *reinterpret_cast<const uint2*>(blk + w * F::kXW + 8);
                                const uint32_t xp[10] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w, xd.x, xd.y};
                                const uint32_t word = wb[uu][w];
                                const uint32_t hh = word / 59049u;
                                const uint32_t ll = word - hh * 59049u;
#pragma unroll
                                for (int half = 0; half < 2; ++half) {
                                    uint32_t Fx = (half == 0 ? hh : ll) * 72736u + 8860u;
                                    const int pb = half * 5;  // first pair of this half
                                    // digits 4 at a time (v in [0, 81)), then the last 2 (v in [0, 9))
                                    const uint32_t v1 = __umulhi(Fx, 81u);
                                    Fx *= 81u;
                                    const uint32_t v2 = __umulhi(Fx, 81u);
                                    Fx *= 81u;
                                    const uint32_t v3 = __umulhi(Fx, 9u);
                                    const uint32_t e1 = lut_lane[v1 << 5], e2 = lut_lane[v2 << 5], e3 = lut_lane[v3 << 5];
                                    // group of pair pp of word w: unit-local trit (20w + 18 - 2pp) / G
#define TQ_GRP(pp) ((20 * w + 18 - 2 * (pp)) / G)
                                    acc[TQ_GRP(pb + 0)] = dp2a_lo(xp[pb + 0], e1, acc[TQ_GRP(pb + 0)]);
                                    acc[TQ_GRP(pb + 1)] = dp2a_hi(xp[pb + 1], e1, acc[TQ_GRP(pb + 1)]);
                                    acc[TQ_GRP(pb + 2)] = dp2a_lo(xp[pb + 2], e2, acc[TQ_GRP(pb + 2)]);
                                    acc[TQ_GRP(pb + 3)] = dp2a_hi(xp[pb + 3], e2, acc[TQ_GRP(pb + 3)]);
                                    acc[TQ_GRP(pb + 4)] = dp2a_hi(xp[pb + 4], e3, acc[TQ_GRP(pb + 4)]);
#undef TQ_GRP
                                }
                            }
                            const float* abu = reinterpret_cast<const float*>(blk + F::kAB);
#pragma unroll
                            for (int g = 0; g < GPU; ++g)
                                tot = fmaf(sb[uu][g], fmaf(abu[2 * g], (float)(int)acc[g], abu[2 * g + 1]), tot);
                        }
                    }
                }
            }
#pragma unroll
            for (int m = 1; m < UPW; m <<= 1) tot += __shfl_xor_sync(kFull, tot, m);
            if (c == 0 && row < p.rows) store_from_float(p.y, out0 + row, p.ydt, tot);
        }
        t0 = t1;
    }
}

template <int G, int RPW>
tq_status launch_trit(const QmvParams& qp, int n_items, cudaStream_t st) {
    using F = TritFmt<G>;
    constexpr int UPW = 32 / RPW;
    TritParams tp{};
    tp.q = qp;
    tp.units = (qp.cols + F::kUT - 1) / F::kUT;
    tp.nsteps = (tp.units + UPW - 1) / UPW;
    tp.tasks_per_item = (qp.rows + RPW - 1) / RPW;
    tp.n_items = n_items;
    const int64_t total = (int64_t)n_items * tp.tasks_per_item;
    if (total > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    tp.total_tasks = (int)total;
    const size_t smem = 4 * ((size_t)81 * 32 + (size_t)tp.nsteps * UPW * F::kUS);
    if (smem > 200 * 1024) return TQ_ERR_UNSUPPORTED;
    const void* kfn = (const void*)qmv_trit_kernel<G, RPW>;
    if (ensure_smem(kfn, smem) != cudaSuccess) return TQ_ERR_CUDA;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmv_trit_kernel<G, RPW>, 256, smem) != cudaSuccess ||
        per_sm <= 0)
        per_sm = 1;
    int64_t grid = (int64_t)sms * per_sm;
    const int64_t max_grid = (total + 7) / 8;  // at least one task per warp
    if (grid > max_grid) grid = max_grid;
    if (grid < 1) grid = 1;
    qmv_trit_kernel<G, RPW><<<(unsigned)grid, 256, smem, st>>>(tp);
    return launch_status();
}

// ---------------------------------------------------------------- pipelined variant
//
// Same decode, but codes and scales are staged in a per-warp ring of NS
// shared-memory stages with cp.async (16 bytes per lane, one commit group per
// stage and lane), so NS-1 stages are in flight while the warp decodes the
// oldest one and no registers hold data in flight.  A stage holds 8
// consecutive units of each of the warp's 4 rows: their code words
// (8 * UW * 4 bytes per row) followed by their 40 fp16 scales (80 bytes per
// row).  Each cp.async instruction covers 4 contiguous 128-byte row segments.
// (1-D bulk copies were measured at about one request per 38 cycles per SM,
// too slow for 128-byte pieces.)

TQ_DEVFN uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
TQ_DEVFN uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

TQ_DEVFN void cp16(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
TQ_DEVFN void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
TQ_DEVFN void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kPipeRPW = 4, kPipeUPW = 8;
constexpr int kPipeUPL = 4;  // units per lane and stage: lane c takes units c, c + 8, c + 16, c + 24
constexpr int kPipeNS = 2;   // stages per warp ring (a stage is long enough to hide the load latency)

template <int G>
struct PipeFmt {
    using F = TritFmt<G>;
    static constexpr int kS = kPipeUPW * kPipeUPL;               // units per row and stage
    static constexpr int kCodeRow = kS * F::kUW * 4;              // code bytes per row and stage
    static constexpr int kScaleRow = kS * F::kGPU * 2;            // scale bytes per row and stage
    static constexpr int kStage = kPipeRPW * (kCodeRow + kScaleRow);
    static constexpr int kScaleCopies = (kScaleRow / 16 + kPipeUPW - 1) / kPipeUPW;  // 16-byte copies per lane
    static_assert(kScaleRow % 16 == 0, "scale row copy");
};

template <int G>
__global__ void __launch_bounds__(256, 3) qmv_trit_pipe_kernel(const TritParams tp) {
    using F = TritFmt<G>;
    using B = PipeFmt<G>;
    constexpr int RPW = kPipeRPW, UPW = kPipeUPW, UPL = kPipeUPL, NS = kPipeNS, S = B::kS;
    constexpr int UW = F::kUW, GPU = F::kGPU, US = F::kUS;
    constexpr int nwarps = 8;
    const QmvParams& p = tp.q;
    extern __shared__ __align__(16) uint32_t sm[];
    uint32_t* lut = sm;                                           // [81][32]
    uint32_t* xb = lut + 81 * 32;                                 // [nsteps * S units][US]
    const int nunits_pad = tp.nsteps * S;
    uint8_t* ring0 = reinterpret_cast<uint8_t*>(xb + nunits_pad * US);  // [8 warps][NS][stage]
    float* rowsum = reinterpret_cast<float*>(ring0 + nwarps * NS * B::kStage);  // [max tasks per CTA][RPW]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 81 * 32; i += blockDim.x) {
        const int v = i >> 5;
        lut[i] = (uint32_t)(v / 27) | ((uint32_t)((v / 9) % 3) << 8) | ((uint32_t)((v / 3) % 3) << 16) |
                 ((uint32_t)(v % 3) << 24);
    }
    const float c0 = __ldg(p.centroids), delta = __ldg(p.centroids + 1) - c0;
    if (tid == 0 && p.err && fabsf((__ldg(p.centroids + 2) - __ldg(p.centroids + 1)) - delta) > 1e-6f * fabsf(delta))
        atomicOr(p.err, TQ_DEVERR_BAD_BOOK);

    const int t_begin = (int)((int64_t)blockIdx.x * tp.total_tasks / gridDim.x);
    const int t_end = (int)((int64_t)(blockIdx.x + 1) * tp.total_tasks / gridDim.x);
    const int r = lane / UPW, c = lane % UPW;
    // shared address of table entry v of this lane is lut_bias + ((0x4B400000 + v) << 7), mod 2^32
    const uint32_t lut_bias = smem_addr(lut + lane) - (0x4B400000u << 7);
    const int ngroups = p.ngroups;
    const int nst = tp.nsteps;  // stages (of S units) per task
    const int tpi = tp.tasks_per_item;
    const int64_t row_stride = p.row_stride;
    uint8_t* ring = ring0 + warp * NS * B::kStage;
    int cur_vec = -1;

    auto item_info = [&](int item, int& e, int& vec) {
        if (p.mode == kModeDense) {
            e = 0;
            vec = item;
        } else {
            e = __ldg(p.ids + item);
            vec = p.mode == kModeGather ? item / p.k : item;
        }
    };

    // Segments: maximal runs of this CTA's tasks whose items share one input vector.
    for (int s0 = t_begin; s0 < t_end;) {
        int e0, vec;
        item_info(s0 / tpi, e0, vec);
        int s1 = min(t_end, (s0 / tpi + 1) * tpi);
        while (s1 < t_end) {  // extend over following items with the same vector
            int e1, v1;
            item_info(s1 / tpi, e1, v1);
            if (v1 != vec) break;
            s1 = min(t_end, (s1 / tpi + 1) * tpi);
        }
        __syncthreads();  // previous segment's row sums written out, x no longer read

        // This warp's share of the segment's (task, stage) units: a contiguous range.
        const int nunits_seg = (s1 - s0) * nst;
        const int f_begin = (int)((int64_t)warp * nunits_seg / nwarps);
        const int f_end = (int)((int64_t)(warp + 1) * nunits_seg / nwarps);
        const int L = f_end - f_begin;

        // Producer: task pt, stage ps; pcode/pscale point at this lane's first unit of the stage.
        int pt = s0 + f_begin / nst, ps = f_begin % nst, pslot = 0;
        const uint32_t* pcode = nullptr;
        const uint16_t* pscale = nullptr;
        int pword = 0;  // word index of this lane's first unit in the row
        int pgrp = 0;   // first scale group of this lane's first scale chunk
        const int rs32 = (int)row_stride;
        auto set_prod_task = [&]() {
            int e, v;
            item_info(pt / tpi, e, v);
            if (e < 0 || e >= p.experts) e = 0;  // rows of a bad id are summed as zero below
            const int row = min((pt % tpi) * RPW + r, p.rows - 1);
            pcode = p.codes + (int64_t)e * p.expert_stride_w + (int64_t)row * row_stride;
            pscale = p.scales + (int64_t)e * p.expert_stride_s + (int64_t)row * ngroups;
            pword = (ps * S + c) * UW;
            pgrp = ps * S * GPU + c * 8;
        };
        if (L > 0) set_prod_task();
        auto issue = [&]() {
            uint8_t* dst = ring + pslot * B::kStage;
#pragma unroll
            for (int j = 0; j < UPL; ++j) {
#pragma unroll
                for (int m = 0; m < UW; m += 4) {
                    const int wi = pword + j * UPW * UW + m;
                    const bool in = wi < rs32;  // past the padded row: zero
                    cp16(dst + r * B::kCodeRow + ((c + j * UPW) * UW + m) * 4, pcode + (in ? wi : 0), in ? 16u : 0u);
                }
            }
#pragma unroll
            for (int q = 0; q < B::kScaleCopies; ++q) {  // the row's scale bytes, 16 per lane and copy
                const int chunk = c + q * UPW;
                if (chunk * 16 < B::kScaleRow) {
                    const int g0 = pgrp + q * UPW * 8;
                    const bool in = g0 < ngroups;  // scale rows are whole 16-byte chunks
                    cp16(dst + RPW * B::kCodeRow + r * B::kScaleRow + chunk * 16, pscale + (in ? g0 : 0),
                         in ? 16u : 0u);
                }
            }
            cp_commit();
            pslot = pslot + 1 == NS ? 0 : pslot + 1;
            pword += S * UW;
            pgrp += S * GPU;
            if (++ps == nst) {
                ps = 0;
                ++pt;
                if (pt < s1) set_prod_task();
            }
        };
        // weights start streaming before the input is prepared
        for (int j = 0; j < NS - 1; ++j) {
            if (j < L) issue(); else cp_commit();
        }

        for (int i = tid; i < (s1 - s0) * RPW; i += blockDim.x) rowsum[i] = 0.f;
        if (vec != cur_vec) {
            // Quantize this vector per group: xs = max|x| / 32767, xq = rint(x / xs),
            // a_g = delta * xs, b_g = c0 * sum(x); zero beyond the last column.
            // One thread per group, the group's values read once into registers.
            const float* xv = p.x + (int64_t)vec * p.cols;
            const bool x16 = (reinterpret_cast<uintptr_t>(xv) & 15) == 0;
            for (int g = tid; g < nunits_pad * GPU; g += blockDim.x) {
                const int u = g / GPU, gl = g - u * GPU;
                float xr[G];
                if (g < ngroups) {
                    if (x16) {
#pragma unroll
                        for (int k = 0; k < G; k += 4) {
                            const float4 v4 = __ldg(reinterpret_cast<const float4*>(xv + g * G + k));
                            xr[k] = v4.x;
                            xr[k + 1] = v4.y;
                            xr[k + 2] = v4.z;
                            xr[k + 3] = v4.w;
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < G; ++k) xr[k] = __ldg(xv + g * G + k);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < G; ++k) xr[k] = 0.f;
                }
                float mx = 0.f, sum = 0.f;
#pragma unroll
                for (int k = 0; k < G; ++k) {
                    mx = fmaxf(mx, fabsf(xr[k]));
                    sum += xr[k];
                }
                uint32_t* blk = xb + u * US;
                reinterpret_cast<float*>(blk + F::kAB)[2 * gl] = delta * (mx / 32767.0f);
                reinterpret_cast<float*>(blk + F::kAB)[2 * gl + 1] = c0 * sum;
                const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
#pragma unroll
                for (int k = 0; k < G; k += 2) {
                    // pair of unit-local trits (tl, tl + 1), tl even, lives at pair pp of word w
                    const int tl = gl * G + k;
                    const int w = tl / 20, pp = (18 - (tl - 20 * w)) / 2;
                    const int qlo = __float2int_rn(xr[k] * inv), qhi = __float2int_rn(xr[k + 1] * inv);
                    blk[w * F::kXW + pp] = ((uint32_t)qhi & 0xffffu) | ((uint32_t)qlo << 16);
                }
            }
            cur_vec = vec;
        }
        __syncthreads();

        // consumer position
        int ct = s0 + f_begin / nst, cs = f_begin % nst, cslot = 0;
        bool cbad;
        {
            int e, v;
            item_info(ct / tpi, e, v);
            cbad = e < 0 || e >= p.experts;
            if (cbad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        }
        float tot = 0.f;
        for (int j = 0; j < L; ++j) {
            cp_wait<NS - 2>();  // stage j has landed
            __syncwarp();       // and every lane is done with the slot of stage j - 1
            if (j + NS - 1 < L) issue(); else cp_commit();  // stage j + NS - 1 into that slot
            const uint8_t* stg = ring + cslot * B::kStage;
            // Units past the row's last one read zero words and zero input blocks.
#pragma unroll
            for (int ju = 0; ju < UPL; ++ju) {
                const int uloc = c + ju * UPW;
                const uint32_t* blk = xb + (cs * S + uloc) * US;
                const uint32_t* wsrc = reinterpret_cast<const uint32_t*>(stg + r * B::kCodeRow + uloc * UW * 4);
                uint32_t acc[GPU];
#pragma unroll
                for (int g = 0; g < GPU; ++g) acc[g] = 0u;
#pragma unroll
                for (int w4 = 0; w4 < UW; w4 += 4) {
                    const uint4 wq = *reinterpret_cast<const uint4*>(wsrc + w4);
                    const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        const int w = w4 + wi;
                        const uint4 xa = *reinterpret_cast<const uint4*>(blk + w * F::kXW);
                        const uint4 xc = *reinterpret_cast<const uint4*>(blk + w * F::kXW + 4);
                        const uint2 xd = *reinterpret_cast<const uint2*>(blk + w * F::kXW + 8);
                        const uint32_t xp[10] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w, xd.x, xd.y};
                        const uint32_t word = wv[wi];
                        const uint32_t hh = word / 59049u;
                        const uint32_t ll = word - hh * 59049u;
                        // Digits of each half h < 3^10 in fp32, every value an integer below 2^24.
                        // With M = 1.5 * 2^23 (unit spacing), adding M rounds to an integer, and
                        // round((h - 364) / 729) = floor(h / 729) for every h (the remainder offset
                        // stays within 0.4993 of zero); the same with 4 and 9 for the remainder.
                        // t1, t2 hold M + the table index of digits 9..6 and 5..2 of a half, t3 the
                        // index 9 (h0 % 9) + (h1 % 9) of both halves' last two digits; their bits
                        // (0x4B400000 + v) << 7 address the per-lane table of 128-byte-spaced entries.
                        float t1[2], t2[2], b2[2];
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const float hb = __uint_as_float((half == 0 ? hh : ll) | 0x4B000000u) - 8388972.0f;
                            t1[half] = fmaf(hb, 1.0f / 729.0f, 12582912.0f);              // M + h / 729
                            const float b1 = fmaf(t1[half] - 12582912.0f, -729.0f, hb);   // h % 729 - 364
                            t2[half] = fmaf(b1, 1.0f / 9.0f, 12582952.0f);                // M + h % 729 / 9
                            b2[half] = fmaf(t2[half] - 12582912.0f, -9.0f, b1);           // h % 9 - 364
                        }
                        const float t3 = fmaf(b2[0], 9.0f, b2[1] + 12586552.0f);  // M + 9 (h0 % 9) + h1 % 9
                        const uint32_t e3 = lds_u32(lut_bias + (__float_as_uint(t3) << 7));
#define TQ_GRP(pp) ((20 * w + 18 - 2 * (pp)) / G)
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int pb = half * 5;
                            const uint32_t e1 = lds_u32(lut_bias + (__float_as_uint(t1[half]) << 7));
                            const uint32_t e2 = lds_u32(lut_bias + (__float_as_uint(t2[half]) << 7));
                            acc[TQ_GRP(pb + 0)] = dp2a_lo(xp[pb + 0], e1, acc[TQ_GRP(pb + 0)]);
                            acc[TQ_GRP(pb + 1)] = dp2a_hi(xp[pb + 1], e1, acc[TQ_GRP(pb + 1)]);
                            acc[TQ_GRP(pb + 2)] = dp2a_lo(xp[pb + 2], e2, acc[TQ_GRP(pb + 2)]);
                            acc[TQ_GRP(pb + 3)] = dp2a_hi(xp[pb + 3], e2, acc[TQ_GRP(pb + 3)]);
                        }
                        acc[TQ_GRP(4)] = dp2a_lo(xp[4], e3, acc[TQ_GRP(4)]);  // half 0's last digits: bytes 0, 1
                        acc[TQ_GRP(9)] = dp2a_hi(xp[9], e3, acc[TQ_GRP(9)]);  // half 1's: bytes 2, 3
#undef TQ_GRP
                    }
                }
                const uint16_t* ssrc =
                    reinterpret_cast<const uint16_t*>(stg + RPW * B::kCodeRow + r * B::kScaleRow) + uloc * GPU;
                const float* abu = reinterpret_cast<const float*>(blk + F::kAB);
                // Groups past the last column have a_g = b_g = 0 and zero-filled scales.  The
                // group sum |acc| <= 2 G 32767 < 2^22 becomes a float exactly by adding it to 1.5 * 2^23.
#pragma unroll
                for (int g = 0; g < GPU; ++g) {
                    const float accf = __int_as_float((int)acc[g] + 0x4B400000) - 12582912.0f;
                    tot = fmaf(half_bits_to_float(ssrc[g]), fmaf(abu[2 * g], accf, abu[2 * g + 1]), tot);
                }
            }
            cslot = cslot + 1 == NS ? 0 : cslot + 1;
            if (++cs == nst || j == L - 1) {  // task finished or this warp's share ends: add the row sums
                float v = cbad ? 0.f : tot;
#pragma unroll
                for (int m = 1; m < UPW; m <<= 1) v += __shfl_xor_sync(kFull, v, m);
                if (c == 0) atomicAdd(rowsum + (ct - s0) * RPW + r, v);
                tot = 0.f;
                if (cs == nst) {
                    cs = 0;
                    ++ct;
                    if (ct < s1) {
                        int e, vv;
                        item_info(ct / tpi, e, vv);
                        cbad = e < 0 || e >= p.experts;
                        if (cbad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
                    }
                }
            }
        }
        cp_wait<0>();
        __syncthreads();  // all row sums of the segment complete
        for (int i = tid; i < (s1 - s0) * RPW; i += blockDim.x) {
            const int t = s0 + i / RPW, row = (t % tpi) * RPW + i % RPW;
            if (row < p.rows) store_from_float(p.y, (int64_t)(t / tpi) * p.rows + row, p.ydt, rowsum[i]);
        }
        s0 = s1;
    }
}

template <int G>
tq_status launch_trit_pipe(const QmvParams& qp, int n_items, cudaStream_t st) {
    using F = TritFmt<G>;
    using B = PipeFmt<G>;
    TritParams tp{};
    tp.q = qp;
    tp.units = (qp.cols + F::kUT - 1) / F::kUT;
    tp.nsteps = (tp.units + B::kS - 1) / B::kS;
    tp.tasks_per_item = (qp.rows + kPipeRPW - 1) / kPipeRPW;
    tp.n_items = n_items;
    const int64_t total = (int64_t)n_items * tp.tasks_per_item;
    if (total > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    tp.total_tasks = (int)total;
    int max_grid_tasks = 0;  // tasks of the largest CTA range, for the row-sum buffer
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const size_t smem_fixed = 4 * ((size_t)81 * 32 + (size_t)tp.nsteps * B::kS * F::kUS) +
                              (size_t)8 * kPipeNS * B::kStage;
    const void* kfn = (const void*)qmv_trit_pipe_kernel<G>;
    // The most resident CTAs per SM (3, 2 or 1) whose shared memory, including the row-sum
    // buffer of the tasks each then takes, fits; one wave of them, at most 128 tasks per CTA.
    int64_t grid = 0;
    size_t smem = 0;
    for (int per_sm = 3; per_sm >= 1 && grid == 0; --per_sm) {
        int64_t g = (int64_t)sms * per_sm;
        const int64_t max_grid = (total + 7) / 8;
        if (g > max_grid) g = max_grid;
        if (g < (total + 127) / 128) g = (total + 127) / 128;
        if (g < 1) g = 1;
        if (g > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
        max_grid_tasks = (int)((total + g - 1) / g) + 1;
        const size_t need = smem_fixed + (size_t)max_grid_tasks * kPipeRPW * 4;
        if (need > 200 * 1024) continue;
        if (ensure_smem(kfn, need) != cudaSuccess) return TQ_ERR_CUDA;
        int fit = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, qmv_trit_pipe_kernel<G>, 256, need) != cudaSuccess)
            return TQ_ERR_CUDA;
        if (fit >= per_sm || per_sm == 1) {
            grid = g;
            smem = need;
        }
    }
    if (grid == 0) return TQ_ERR_UNSUPPORTED;
    qmv_trit_pipe_kernel<G><<<(unsigned)grid, 256, smem, st>>>(tp);
    return launch_status();
}

// ---------------------------------------------------------------- tensor-copy pipeline (group 16)
//
// Warp-specialised version of the staged pipeline, built to cut the
// instructions per code word and to keep more bytes in flight:
//  * one producer warp streams the codes and scales with tensor copies (two per
//    stage: a 16-row x 128-byte code box, 128-byte swizzled, and a 16-row x
//    80-byte scale box) into per-consumer rings of three slots; rows, words,
//    groups and expert ids past the tensor read as zeros, so no bounds checks
//    remain on the data path;
//  * each consumer lane decodes the same unit of two rows, so one load of the
//    quantized input serves two code words; a consumer warp covers 16 rows
//    (rows r and r + 8 for lane row r) and 4 unit columns, and a unit pass that
//    lies wholly past the row is skipped;
//  * the table holds signed digits t = d - 1: for an affine three-level book
//    c[d] = c1 + t * delta,
//        sum_k c[d_k] x_k = delta * sum_k t_k x_k + c1 * sum_k x_k,
//    and with one input scale per vector (x = xs * xq, |xq| <= 32767) a group's
//    integer sum only needs its weight scale: y = delta * xs * sum_g s_g acc_g
//    (+ c1 * sum_g s_g X_g when the middle level is not zero);
//  * the dp2a accumulators start at the bits of 1.5 * 2^23, so their final bits
//    are the float 1.5 * 2^23 + acc exactly (|acc| <= 16 * 32767 < 2^22).
// Every wait is bounded; on expiry the CTA raises TQ_DEVERR_TIMEOUT, stops, and
// waits (bounded) for its copies in flight before it exits.

TQ_DEVFN uint32_t dp2a_lo_ss(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
TQ_DEVFN uint32_t dp2a_hi_ss(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
template <int D>
TQ_DEVFN uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a), "n"(D));
    return v;
}
template <int D>
TQ_DEVFN uint2 lds_v2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(D));
    return v;
}
template <int D>
TQ_DEVFN uint32_t lds_w(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(D));
    return v;
}
#ifndef TQ_TC_WARPS
#define TQ_TC_WARPS 15
#endif
// Consumer warps (warp 0 produces): 15 + 1 puts four warps on each scheduler, which
// leaves each thread up to 128 registers.
constexpr int kTcWarps = TQ_TC_WARPS;
constexpr int kTcDepth = 3;                  // slots per consumer warp
constexpr int kTcSlots = kTcWarps * kTcDepth;
constexpr int kTcRows = 16;                  // rows per task
constexpr int kTcS = 8;                      // units per row and stage
constexpr int kTcCode = kTcRows * kTcS * 16;  // 2048 code bytes per slot: one 128-byte line per row
constexpr int kTcScale = kTcRows * kTcS * 10;  // 1280 scale bytes per slot: 80 per row
constexpr int kTcUS = 52;                    // input block words per unit: 4 x 12, = 4 (mod 8)
constexpr int kTcThreads = 32 * (1 + kTcWarps);

// Barrier `id` over the first `count` threads' warps (count a multiple of 32).
TQ_DEVFN void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Signal barrier `id` without waiting on it.
TQ_DEVFN void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// M-point Hadamard transforms down the 32 columns of every block of M rows of a padded
// [rows][33] float array (rows = a multiple of M; M a power of two up to 256).  A warp takes
// 32 / L columns at a time, L = min(M, 32) lanes per column, each lane E = M / L elements
// (rows i0 + L j): in-register butterflies over j, then shuffles over the lane bits.
template <int M>
TQ_DEVFN void hadamard_columns_m(float* xf, int nrows, int warp, int nwarps, int lane) {
    constexpr int L = M < 32 ? M : 32, E = M / L, CPW = 32 / L;
    constexpr int P = E >= 8 ? 1 : 8 / E;  // independent column groups per pass (ILP)
    const int ncols = (nrows / M) * 32;     // (block, column) pairs
    const int i0 = lane % L;
    for (int cb = warp * CPW; cb < ncols; cb += P * nwarps * CPW) {
        float e[P][E];
        float* base[P];
        bool on[P];
#pragma unroll
        for (int g = 0; g < P; ++g) {
            const int col = cb + g * nwarps * CPW + lane / L;
            on[g] = col < ncols;
            const int blk = on[g] ? col >> 5 : 0, c = col & 31;
            base[g] = xf + (blk * M + i0) * 33 + c;
#pragma unroll
            for (int j = 0; j < E; ++j) e[g][j] = on[g] ? base[g][L * j * 33] : 0.f;
        }
#pragma unroll
        for (int g = 0; g < P; ++g)
#pragma unroll
            for (int st = 1; st < E; st <<= 1)
#pragma unroll
                for (int j = 0; j < E; ++j)
                    if (!(j & st)) {
                        const float x0 = e[g][j], x1 = e[g][j + st];
                        e[g][j] = x0 + x1;
                        e[g][j + st] = x0 - x1;
                    }
#pragma unroll
        for (int m = 1; m < L; m <<= 1) {
            const float sgn = (i0 & m) ? -1.0f : 1.0f;
#pragma unroll
            for (int g = 0; g < P; ++g)
#pragma unroll
                for (int j = 0; j < E; ++j) e[g][j] = fmaf(sgn, e[g][j], __shfl_xor_sync(kFull, e[g][j], m));
        }
#pragma unroll
        for (int g = 0; g < P; ++g)
            if (on[g]) {
#pragma unroll
                for (int j = 0; j < E; ++j) base[g][L * j * 33] = e[g][j];
            }
    }
}

TQ_DEVFN void hadamard_columns(float* xf, int nrows, int M, int warp, int nwarps, int lane) {
    switch (M) {
        case 1: break;
        case 2: hadamard_columns_m<2>(xf, nrows, warp, nwarps, lane); break;
        case 4: hadamard_columns_m<4>(xf, nrows, warp, nwarps, lane); break;
        case 8: hadamard_columns_m<8>(xf, nrows, warp, nwarps, lane); break;
        case 16: hadamard_columns_m<16>(xf, nrows, warp, nwarps, lane); break;
        case 32: hadamard_columns_m<32>(xf, nrows, warp, nwarps, lane); break;
        case 64: hadamard_columns_m<64>(xf, nrows, warp, nwarps, lane); break;
        case 128: hadamard_columns_m<128>(xf, nrows, warp, nwarps, lane); break;
        default: hadamard_columns_m<256>(xf, nrows, warp, nwarps, lane); break;
    }
}

struct TritMaps {
    CUtensorMap codes;   // [experts][rows][row_stride] words, box 32 x 16 x 1, 128-byte swizzle
    CUtensorMap scales;  // [experts][rows][ngroups] fp16, box 40 x 16 x 1
};

// The 64-bit pair (v, v) of fp32 lanes.
TQ_DEVFN uint64_t f32x2_splat(float v) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
    return r;
}

// One 20-trit word against its 20 quantized inputs (pair words xp), added into the
// unit's five group accumulators.  W is the word's index in the unit.
template <int W>
TQ_DEVFN void trit_word_signed(uint32_t word, const uint32_t (&xp)[10], uint32_t (&acc)[5], uint32_t lut_bias) {
    constexpr int G = 16;
    const uint32_t hh = word / 59049u;
    const uint32_t ll = word - hh * 59049u;
    // Both halves' digit steps at once, as pairs of fp32 lanes (same arithmetic, lane by lane).
    float t1[2], t2[2], b2[2];
    {
        uint64_t H, hb, T1, D1, B1, T2, D2, B2;
        asm("mov.b64 %0, {%1, %2};" : "=l"(H) : "r"(hh | 0x4B000000u), "r"(ll | 0x4B000000u));
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(hb) : "l"(H), "l"(f32x2_splat(-8388972.0f)));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(T1) : "l"(hb), "l"(f32x2_splat(1.0f / 729.0f)), "l"(f32x2_splat(12582912.0f)));
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(D1) : "l"(T1), "l"(f32x2_splat(-12582912.0f)));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(B1) : "l"(D1), "l"(f32x2_splat(-729.0f)), "l"(hb));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(T2) : "l"(B1), "l"(f32x2_splat(1.0f / 9.0f)), "l"(f32x2_splat(12582952.0f)));
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(D2) : "l"(T2), "l"(f32x2_splat(-12582912.0f)));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(B2) : "l"(D2), "l"(f32x2_splat(-9.0f)), "l"(B1));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(t1[0]), "=f"(t1[1]) : "l"(T1));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(t2[0]), "=f"(t2[1]) : "l"(T2));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(b2[0]), "=f"(b2[1]) : "l"(B2));
    }
    const float t3 = fmaf(b2[0], 9.0f, b2[1] + 12586552.0f);
    const uint32_t e3 = lds_u32(lut_bias + (__float_as_uint(t3) << 7));
    constexpr int g0 = (20 * W + 18) / G, g1 = (20 * W + 16) / G, g2 = (20 * W + 14) / G, g3 = (20 * W + 12) / G,
                  g4 = (20 * W + 10) / G, g5 = (20 * W + 8) / G, g6 = (20 * W + 6) / G, g7 = (20 * W + 4) / G,
                  g8 = (20 * W + 2) / G, g9 = (20 * W) / G;
    {
        const uint32_t e1 = lds_u32(lut_bias + (__float_as_uint(t1[0]) << 7));
        const uint32_t e2 = lds_u32(lut_bias + (__float_as_uint(t2[0]) << 7));
        acc[g0] = dp2a_lo_ss(xp[0], e1, acc[g0]);
        acc[g1] = dp2a_hi_ss(xp[1], e1, acc[g1]);
        acc[g2] = dp2a_lo_ss(xp[2], e2, acc[g2]);
        acc[g3] = dp2a_hi_ss(xp[3], e2, acc[g3]);
    }
    {
        const uint32_t e1 = lds_u32(lut_bias + (__float_as_uint(t1[1]) << 7));
        const uint32_t e2 = lds_u32(lut_bias + (__float_as_uint(t2[1]) << 7));
        acc[g5] = dp2a_lo_ss(xp[5], e1, acc[g5]);
        acc[g6] = dp2a_hi_ss(xp[6], e1, acc[g6]);
        acc[g7] = dp2a_lo_ss(xp[7], e2, acc[g7]);
        acc[g8] = dp2a_hi_ss(xp[8], e2, acc[g8]);
    }
    acc[g4] = dp2a_lo_ss(xp[4], e3, acc[g4]);
    acc[g9] = dp2a_hi_ss(xp[9], e3, acc[g9]);
}

// The five fp16 scales of a unit as floats: three words from the 4-byte aligned address
// a + D, shifted right by sh bits (0, or 16 when the unit starts mid-word).
template <int D>
TQ_DEVFN void unit_scales(uint32_t a, uint32_t sh, float (&s)[5]) {
    const uint32_t w0 = lds_w<D>(a), w1 = lds_w<D + 4>(a), w2 = lds_w<D + 8>(a);
    const uint32_t v0 = __funnelshift_r(w0, w1, sh), v1 = __funnelshift_r(w1, w2, sh), v2 = w2 >> sh;
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v0));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v1));
    s[0] = f0.x;
    s[1] = f0.y;
    s[2] = f1.x;
    s[3] = f1.y;
    s[4] = __low2float(*reinterpret_cast<const __half2*>(&v2));
}

// XS: the kernel carries the input stage (xmode 1 or 2); without it (xmode 0) none of that code
// or its registers is in the plain matvec.
template <bool XS>
__global__ void __launch_bounds__(kTcThreads, 1) qmv_trit_tc_kernel(const TritParams tp, const __grid_constant__ TritMaps maps) {
    const int xmode = XS ? tp.xmode : 0;
    constexpr int G = 16;
    using F = TritFmt<G>;
    constexpr int GPU = 5, S = kTcS, US = kTcUS, D = kTcDepth, NC = kTcWarps, RT = kTcRows;
    constexpr int NCT = NC * 32;  // consumer threads
    static_assert(F::kUW == 4 && F::kGPU == GPU, "group 16 units");
    const QmvParams& p = tp.q;
    const int nst = tp.nsteps;
    const int nunits_pad = nst * S;
    extern __shared__ __align__(16) uint8_t smraw[];
    const uint32_t raw_addr = smem_u32(smraw);
    uint8_t* sm = smraw + (((raw_addr + 1023u) & ~1023u) - raw_addr);  // swizzled boxes want 1024-byte alignment
    uint8_t* ring_c = sm;                                               // [slots][2048]
    uint8_t* ring_s = ring_c + kTcSlots * kTcCode;                      // [slots][1280]
    uint32_t* lut = reinterpret_cast<uint32_t*>(ring_s + kTcSlots * kTcScale);  // [81][32] signed digits
    float* red = reinterpret_cast<float*>(lut + 81 * 32);               // [32]
    uint32_t* xb = reinterpret_cast<uint32_t*>(red + 32);               // [nunits_pad][US]
    float* xsum = reinterpret_cast<float*>(xb + nunits_pad * US);       // [nunits_pad * 5, padded to 4]
    uint64_t* full = reinterpret_cast<uint64_t*>(xsum + (nunits_pad * GPU + 3) / 4 * 4);
    uint64_t* empty = full + kTcSlots;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kTcSlots);
    int* tag = reinterpret_cast<int*>(empty + kTcSlots + 1);            // [slots]: (task << 8) | stage, or -1
    float* xf = reinterpret_cast<float*>(tag + (kTcSlots + 3) / 4 * 4);  // [cols / 32][33] input stage (xmode != 0)
    float* rowsum = xf + (xmode ? (p.cols / 32) * 33 : 0);             // [tasks of this CTA][RT]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t_begin = (int)((int64_t)blockIdx.x * tp.total_tasks / gridDim.x);
    const int t_end = (int)((int64_t)(blockIdx.x + 1) * tp.total_tasks / gridDim.x);
    const int tpi = tp.tasks_per_item;
    const uint32_t ring_c_addr = smem_u32(ring_c), ring_s_addr = smem_u32(ring_s);
    uint32_t uses = 0;  // stages this warp (consumer) or this lane's consumer (producer) has passed through its ring

    auto vec_of = [&](int item) { return p.mode == kModeGather ? item / p.k : item; };
    // Segments: maximal runs of this CTA's tasks whose items share one input vector.
    auto seg_end = [&](int s0) {
        const int vec = vec_of(s0 / tpi);
        int s1 = min(t_end, (s0 / tpi + 1) * tpi);
        while (s1 < t_end && vec_of(s1 / tpi) == vec) s1 = min(t_end, (s1 / tpi + 1) * tpi);
        return s1;
    };

    if (warp == 0) {
        // ---------------- producer: lane w fills consumer warp w's ring.  Stages are handed out
        // in order to whichever consumers have a free slot, and each slot's tag says which
        // stage it holds (-1: the segment is over).  No block-wide barrier is taken after this
        // point: the rings order producer and consumers.
        int cur_item = -1, e = 0;  // the expert id of the item last handed out by this lane
        if (t_begin < t_end && p.mode != kModeDense) {  // in flight while the barriers are set up
            cur_item = t_begin / tpi;
            e = __ldg(p.ids + cur_item);
            if ((e < 0 || e >= p.experts) && p.err && lane == 0) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        }
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.codes)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.scales)) : "memory");
        for (int i = lane; i < kTcSlots; i += 32) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        if (lane == 0) *abort_flag = 0;
        fence_mbar_init();
        __syncwarp();
        named_bar_arrive(2, kTcThreads);  // barriers ready
        for (int s0 = t_begin; s0 < t_end && !*abort_flag;) {
            const int s1 = seg_end(s0);
            const int nunits_seg = (s1 - s0) * nst;
            int next = 0;            // next stage of the segment to hand out (same in every lane)
            bool done = lane >= NC;  // this lane's consumer has its end mark
            long long t0 = clock64();
            for (;;) {
                if (__all_sync(kFull, done)) break;
                const int slot = lane * D + (int)(uses % D);
                const bool ready = !done && mbar_peek(empty + slot, ((uses / D) & 1) ^ 1);
                const unsigned rmask = __ballot_sync(kFull, ready);
                if (ready) {
                    const int j = next + __popc(rmask & ((1u << lane) - 1));
                    if (j < nunits_seg) {
                        const int tl = j / nst, stage = j - tl * nst, task = s0 + tl;
                        const int item = task / tpi;
                        if (item != cur_item) {  // an id past the bank reads zeros (and is reported)
                            e = p.mode == kModeDense ? 0 : __ldg(p.ids + item);
                            cur_item = item;
                            if ((e < 0 || e >= p.experts) && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
                        }
                        const int row0 = (task % tpi) * RT;
                        tag[slot] = (tl << 8) | stage;
                        mbar_expect_tx(full + slot, kTcCode + kTcScale);
                        tma_load_3d(ring_c_addr + slot * kTcCode, &maps.codes, stage * S * 4, row0, e, full + slot);
                        tma_load_3d(ring_s_addr + slot * kTcScale, &maps.scales, stage * S * GPU, row0, e, full + slot);
                    } else {
                        tag[slot] = -1;
                        mbar_arrive(full + slot);
                        done = true;
                    }
                    ++uses;
                }
                next += __popc(rmask);
                if (rmask) {
                    t0 = clock64();
                } else {
                    if (*abort_flag) break;
                    if (clock64() - t0 > p.wait_cycles) {
                        *abort_flag = 1;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            s0 = s1;
        }
        __syncthreads();  // every consumer is done
        if (*abort_flag && lane < NC) {
            // Stopped early: let the copies this lane issued land before the CTA exits.
            if (lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_TIMEOUT);
            for (uint32_t k = 0; k < (uses < D ? uses : (uint32_t)D); ++k) {
                const uint32_t u = uses - 1 - k;  // the last D uses of this lane's slots
                mbar_wait_drain(full + lane * D + (int)(u % D), (u / D) & 1);
            }
        }
        return;
    }

    // ---------------- consumers
    const int cw = warp - 1, ctid = tid - 32;
    // input stage: quads of 4 columns of vector vec, 4 per thread in flight (r = 0..3 -> quad ctid + r NCT)
    const int nq = p.cols / 4;
    auto load_quads = [&](int64_t vec, int q0, float4 (&xv4)[4], uint32_t (&sg)[4]) {
        const uint32_t* sg4 = reinterpret_cast<const uint32_t*>(tp.xsigns);  // 4 signs per word
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int q = q0 + ctid + r * NCT;
            if (q < nq) {
                sg[r] = __ldg(sg4 + q);
                if (xmode == 1) {
                    if (tp.xdt == TQ_F32) {
                        xv4[r] = __ldg(reinterpret_cast<const float4*>(tp.xin) + vec * nq + q);
                    } else {
                        const uint2 b = __ldg(reinterpret_cast<const uint2*>(tp.xin) + vec * nq + q);
                        xv4[r] = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u),
                                             __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u));
                    }
                } else {
                    const float4* gu = reinterpret_cast<const float4*>(tp.xin) + vec * 2 * nq;
                    const float4 g = __ldg(gu + q), u = __ldg(gu + nq + q);
                    xv4[r] = make_float4(g.x / (1.0f + expf(-g.x)) * u.x, g.y / (1.0f + expf(-g.y)) * u.y,
                                         g.z / (1.0f + expf(-g.z)) * u.z, g.w / (1.0f + expf(-g.w)) * u.w);
                }
            }
        }
    };
    float4 pre_x[4];
    uint32_t pre_sg[4];
    const int64_t pre_vec = xmode != 0 && t_begin < t_end && nq <= 4 * NCT ? vec_of(t_begin / tpi) : -1;
    if (pre_vec >= 0) load_quads(pre_vec, 0, pre_x, pre_sg);  // in flight while the table is built
    if (t_begin < t_end) {  // start fetching the first input vector while the table is built
        const int64_t v0 = vec_of(t_begin / tpi);
        const int64_t bytes = xmode == 0 ? (int64_t)p.cols * 4
                              : xmode == 1 ? (int64_t)p.cols * (tp.xdt == TQ_F32 ? 4 : 2)
                                              : (int64_t)p.cols * 8;  // [gate | up] in f32
        const char* x0 = xmode == 0 ? reinterpret_cast<const char*>(p.x) : reinterpret_cast<const char*>(tp.xin);
        x0 += v0 * bytes;
        for (int64_t off = ctid * 128; off < bytes; off += NCT * 128)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(x0 + off));
    }
    for (int i = ctid; i < 81 * 32; i += NCT) {
        const int v = i >> 5;
        lut[i] = (((uint32_t)(v / 27 - 1)) & 0xffu) | ((((uint32_t)((v / 9) % 3 - 1)) & 0xffu) << 8) |
                 ((((uint32_t)((v / 3) % 3 - 1)) & 0xffu) << 16) | (((uint32_t)(v % 3 - 1)) << 24);
    }
    const float cmid = __ldg(p.centroids + 1), delta = __ldg(p.centroids + 2) - cmid;
    if (ctid == 0 && p.err && fabsf((cmid - __ldg(p.centroids)) - delta) > 1e-6f * fabsf(delta))
        atomicOr(p.err, TQ_DEVERR_BAD_BOOK);
    const bool has_off = cmid != 0.f;  // uniform
    // lane row lr takes rows rA = (lr >> 1) + 4 (lr & 1) and rA + 8, so the two rows a quarter
    // warp reads differ in bit 2 and their swizzled 16-byte pieces fall in different bank halves
    const int lr = lane >> 2, c = lane & 3;
    const int rA = (lr >> 1) + 4 * (lr & 1);
    const uint32_t coff0 = (uint32_t)(rA * 128 + ((c ^ rA) * 16));  // piece of unit c (unit c + 4: ^ 64)
    const uint32_t soff = (uint32_t)(rA * 80 + ((10 * c) & ~3));    // row B: + 640
    const uint32_t ssh = (uint32_t)(c & 1) * 16u;
    const uint32_t xoff = smem_u32(xb) + (uint32_t)(c * US * 4);
    const uint32_t lut_bias = smem_u32(lut + lane) - (0x4B400000u << 7);
    int cur_vec = -1;
    float yscale = 0.f;  // delta * xs of the current vector
    named_bar_sync(2, kTcThreads);  // the producer has initialised the barriers

    for (int s0 = t_begin; s0 < t_end && !*abort_flag;) {
        const int s1 = seg_end(s0);
        const int vec = vec_of(s0 / tpi);
        for (int i = ctid; i < (s1 - s0) * RT; i += NCT) rowsum[i] = 0.f;
        if (vec != cur_vec) {
            // One scale for the vector: xs = max|x| / 32767, xq = rint(x / xs); pair word pp of
            // word w of a unit holds the inputs of unit trits 20w + 19 - 2pp (low half) and
            // 20w + 18 - 2pp (high half), zero past the last column.
            const float* xv = p.x + (int64_t)vec * p.cols;
            // the pair of columns (k, k + 1), k even, sits at pair word pp of word w of unit u
            auto pair_at = [&](int k) {
                const int u = k / F::kUT, tl = k - u * F::kUT, w = tl / 20;
                return u * US + w * F::kXW + (18 - (tl - 20 * w)) / 2;
            };
            auto pack = [](int qlo, int qhi) { return ((uint32_t)qhi & 0xffffu) | ((uint32_t)qlo << 16); };
            constexpr int kV4 = 4;  // 16-byte input loads per thread when the vector fits
            const int nv4 = p.cols >> 2;
            if (xmode != 0) {
                // The input stage: x (or silu(gate) * up) times the signs, into rows of 32 floats
                // padded to 33, then the block Hadamard transform of the rotation as 32-point
                // transforms along the rows and M-point transforms down the columns of every
                // block (H_{32M} = H_M (x) H_32), scaled by 1 / sqrt(block) through yscale.
                const int K = p.cols, nrows = K / 32;
                // quads of 4 columns, 4 quads per thread in flight at a time
                for (int q0 = 0; q0 < nq; q0 += 4 * NCT) {
                    float4 xv4[4];
                    uint32_t sg[4];
                    if (q0 == 0 && vec == pre_vec) {  // loaded at the start
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            xv4[r] = pre_x[r];
                            sg[r] = pre_sg[r];
                        }
                    } else {
                        load_quads(vec, q0, xv4, sg);
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int q = q0 + ctid + r * NCT;
                        if (q < nq) {
                            const int k = 4 * q;  // 4 columns inside one row of 32
                            float* dst = xf + (k >> 5) * 33 + (k & 31);
                            dst[0] = xv4[r].x * (float)(int8_t)(sg[r]);
                            dst[1] = xv4[r].y * (float)(int8_t)(sg[r] >> 8);
                            dst[2] = xv4[r].z * (float)(int8_t)(sg[r] >> 16);
                            dst[3] = xv4[r].w * (float)(int8_t)(sg[r] >> 24);
                        }
                    }
                }
                named_bar_sync(1, NCT);
                for (int r0 = cw; r0 < nrows; r0 += 4 * NC) {  // four independent rows per pass
                    float v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] = r0 + i * NC < nrows ? xf[(r0 + i * NC) * 33 + lane] : 0.f;
#pragma unroll
                    for (int m = 1; m < 32; m <<= 1) {
                        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) v[i] = fmaf(sgn, v[i], __shfl_xor_sync(kFull, v[i], m));
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (r0 + i * NC < nrows) xf[(r0 + i * NC) * 33 + lane] = v[i];
                }
                named_bar_sync(1, NCT);
                hadamard_columns(xf, nrows, tp.xblock / 32, cw, NC, lane);
                named_bar_sync(1, NCT);
                float mx = 0.f;
                for (int k = ctid; k < K; k += NCT) mx = fmaxf(mx, fabsf(xf[(k >> 5) * 33 + (k & 31)]));
#pragma unroll
                for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
                if (lane == 0) red[cw] = mx;
                named_bar_sync(1, NCT);
                mx = 0.f;
#pragma unroll
                for (int i = 0; i < NC; ++i) mx = fmaxf(mx, red[i]);
                const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
                const float rs = rsqrtf((float)tp.xblock);
                yscale = delta * (rs * mx / 32767.0f);
                for (int k = 2 * ctid; k < nunits_pad * F::kUT; k += 2 * NCT) {
                    const float lo = k < K ? xf[(k >> 5) * 33 + (k & 31)] : 0.f;
                    const float hi = k + 1 < K ? xf[((k + 1) >> 5) * 33 + ((k + 1) & 31)] : 0.f;
                    xb[pair_at(k)] = pack(__float2int_rn(lo * inv), __float2int_rn(hi * inv));
                }
                if (has_off) {
                    for (int g = ctid; g < nunits_pad * GPU; g += NCT) {
                        float sum = 0.f;
                        for (int k = g * G; k < min((g + 1) * G, K); ++k) sum += xf[(k >> 5) * 33 + (k & 31)];
                        xsum[g] = rs * sum;
                    }
                }
            } else if ((p.cols & 3) == 0 && (reinterpret_cast<uintptr_t>(xv) & 15) == 0 && nv4 <= kV4 * NCT) {
                float4 xr[kV4];
                float mx = 0.f;
#pragma unroll
                for (int r = 0; r < kV4; ++r) {
                    const int f = ctid + r * NCT;
                    xr[r] = f < nv4 ? __ldg(reinterpret_cast<const float4*>(xv) + f) : make_float4(0.f, 0.f, 0.f, 0.f);
                    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(xr[r].x), fabsf(xr[r].y)), fmaxf(fabsf(xr[r].z), fabsf(xr[r].w))));
                }
#pragma unroll
                for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
                if (lane == 0) red[cw] = mx;
                named_bar_sync(1, NCT);
                mx = 0.f;
#pragma unroll
                for (int i = 0; i < NC; ++i) mx = fmaxf(mx, red[i]);
                const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
                yscale = delta * (mx / 32767.0f);
#pragma unroll
                for (int r = 0; r < kV4; ++r) {
                    const int f = ctid + r * NCT;
                    if (f < nv4) {
                        xb[pair_at(4 * f)] = pack(__float2int_rn(xr[r].x * inv), __float2int_rn(xr[r].y * inv));
                        xb[pair_at(4 * f + 2)] = pack(__float2int_rn(xr[r].z * inv), __float2int_rn(xr[r].w * inv));
                    }
                }
                for (int k = p.cols + 2 * ctid; k < nunits_pad * F::kUT; k += 2 * NCT) xb[pair_at(k)] = 0u;  // past the row
            } else {
                float mx = 0.f;
                for (int k = ctid; k < p.cols; k += NCT) mx = fmaxf(mx, fabsf(__ldg(xv + k)));
#pragma unroll
                for (int m = 16; m; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
                if (lane == 0) red[cw] = mx;
                named_bar_sync(1, NCT);
                mx = 0.f;
#pragma unroll
                for (int i = 0; i < NC; ++i) mx = fmaxf(mx, red[i]);
                const float inv = mx > 0.f ? 32767.0f / mx : 0.f;
                yscale = delta * (mx / 32767.0f);
                for (int k = 2 * ctid; k < nunits_pad * F::kUT; k += 2 * NCT) {
                    const float lo = k < p.cols ? __ldg(xv + k) : 0.f, hi = k + 1 < p.cols ? __ldg(xv + k + 1) : 0.f;
                    xb[pair_at(k)] = pack(__float2int_rn(lo * inv), __float2int_rn(hi * inv));
                }
            }
            if (has_off && xmode == 0) {
                for (int g = ctid; g < nunits_pad * GPU; g += NCT) {
                    float sum = 0.f;
                    for (int k = g * G; k < min((g + 1) * G, p.cols); ++k) sum += __ldg(xv + k);
                    xsum[g] = sum;
                }
            }
            cur_vec = vec;
        }
        named_bar_sync(1, NCT);  // table, input blocks and row sums ready

        auto consume = [&](auto off_c) {
            constexpr bool OFF = decltype(off_c)::value;
            uint32_t slot = cw * D + uses % D, par = (uses / D) & 1;
            for (;;) {
                if (!mbar_wait_short(full + slot, par, abort_flag, p.wait_cycles)) break;
                const int tg = tag[slot];
                if (tg < 0) {  // end of the segment
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty + slot);
                    ++uses;
                    break;
                }
                const int cs = tg & 255;                        // stage within the task
                float* rs = rowsum + (tg >> 8) * RT + rA;       // row sums of the task, row A
                const uint32_t cbase = ring_c_addr + slot * kTcCode;
                const uint32_t sbase = ring_s_addr + slot * kTcScale + soff;
                const uint32_t xs = xoff + (uint32_t)(cs * S * US * 4);
                float totA = 0.f, totB = 0.f, offA = 0.f, offB = 0.f;
                // unit pass JU: unit c + 4 JU of the stage, rows A and B (a pass past the row
                // decodes zero words against zero inputs and scales)
                auto pass = [&](auto ju_c) {
                    constexpr int JU = decltype(ju_c)::value;
                    const uint32_t ca = cbase + (JU == 0 ? coff0 : (coff0 ^ 64u));
                    uint32_t accA[GPU], accB[GPU];
#pragma unroll
                    for (int g = 0; g < GPU; ++g) accA[g] = accB[g] = 0x4B400000u;
                    const uint4 qa = lds_v4<0>(ca), qb = lds_v4<1024>(ca);
                    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
                    static_for<0, 4>([&](auto wi_c) {
                        constexpr int wi = decltype(wi_c)::value;
                        constexpr int xd = (JU * 4 * US + wi * F::kXW) * 4;
                        const uint4 xa = lds_v4<xd>(xs), xc = lds_v4<xd + 16>(xs);
                        const uint2 xe = lds_v2<xd + 32>(xs);
                        const uint32_t xp[10] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w, xe.x, xe.y};
                        trit_word_signed<wi>(wa[wi], xp, accA, lut_bias);
                        trit_word_signed<wi>(wb[wi], xp, accB, lut_bias);
                    });
                    float sA[5], sB[5];
                    unit_scales<JU * 40>(sbase, ssh, sA);
                    unit_scales<JU * 40 + 640>(sbase, ssh, sB);
#pragma unroll
                    for (int g = 0; g < GPU; ++g) {
                        totA = fmaf(sA[g], __uint_as_float(accA[g]) - 12582912.0f, totA);
                        totB = fmaf(sB[g], __uint_as_float(accB[g]) - 12582912.0f, totB);
                    }
                    if (OFF) {
                        const float* xg = xsum + (cs * S + c + 4 * JU) * GPU;
#pragma unroll
                        for (int g = 0; g < GPU; ++g) {
                            offA = fmaf(sA[g], xg[g], offA);
                            offB = fmaf(sB[g], xg[g], offB);
                        }
                    }
                };
                pass(std::integral_constant<int, 0>{});
                pass(std::integral_constant<int, 1>{});
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + slot);  // slot free for the producer
                // this stage's partial row sums
                float vA = OFF ? fmaf(yscale, totA, cmid * offA) : yscale * totA;
                float vB = OFF ? fmaf(yscale, totB, cmid * offB) : yscale * totB;
                vA += __shfl_xor_sync(kFull, vA, 1);
                vB += __shfl_xor_sync(kFull, vB, 1);
                vA += __shfl_xor_sync(kFull, vA, 2);
                vB += __shfl_xor_sync(kFull, vB, 2);
                if (c == 0) {
                    atomicAdd(rs, vA);
                    atomicAdd(rs + 8, vB);
                }
                ++uses;
                if (++slot == (uint32_t)(cw * D + D)) {
                    slot = cw * D;
                    par ^= 1u;
                }
            }
        };
        if (has_off) consume(std::true_type{}); else consume(std::false_type{});
        named_bar_sync(1, NCT);  // all row sums of the segment complete
        for (int i = ctid; i < (s1 - s0) * RT; i += NCT) {
            const int t = s0 + i / RT, row = (t % tpi) * RT + i % RT;
            if (row < p.rows) store_from_float(p.y, (int64_t)(t / tpi) * p.rows + row, p.ydt, rowsum[i]);
        }
        named_bar_sync(1, NCT);  // row sums read out before the next segment clears them
        s0 = s1;
    }
    __syncthreads();  // the producer drains its copies on an abort before the CTA exits
}

size_t trit_tc_smem(int nsteps, int max_tasks, int xf_floats) {
    const size_t nunits_pad = (size_t)nsteps * kTcS;
    return 1024 + (size_t)kTcSlots * (kTcCode + kTcScale) + 4 * ((size_t)81 * 32 + 32) + 4 * nunits_pad * kTcUS +
           4 * ((nunits_pad * 5 + 3) / 4 * 4) + 8 * (size_t)(2 * kTcSlots + 1) + 4 * (size_t)((kTcSlots + 3) / 4 * 4) +
           4 * (size_t)xf_floats + 4 * (size_t)max_tasks * kTcRows;
}

// Tensor maps of the code and scale banks (3-D: experts x rows x row).
bool encode_trit_maps(const QmvParams& qp, TritMaps& m) {
    const EncodeFn enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t ne = qp.mode == kModeDense ? 1 : qp.experts;
    const int64_t esw = ne > 1 ? qp.expert_stride_w : (int64_t)qp.rows * qp.row_stride;
    const int64_t ess = ne > 1 ? qp.expert_stride_s : (int64_t)qp.rows * qp.ngroups;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)qp.row_stride, (cuuint64_t)qp.rows, (cuuint64_t)ne};
        const cuuint64_t strides[2] = {(cuuint64_t)qp.row_stride * 4, (cuuint64_t)esw * 4};
        const cuuint32_t box[3] = {32, (cuuint32_t)kTcRows, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&m.codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(qp.codes), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)qp.ngroups, (cuuint64_t)qp.rows, (cuuint64_t)ne};
        const cuuint64_t strides[2] = {(cuuint64_t)qp.ngroups * 2, (cuuint64_t)ess * 2};
        const cuuint32_t box[3] = {(cuuint32_t)(kTcS * 5), (cuuint32_t)kTcRows, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&m.scales, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(qp.scales), dims, strides, box,
                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

// Group 16 with tensor-copyable banks: 16-byte aligned bases, rows and experts a
// multiple of 16 bytes apart.
bool trit_tc_ok(const QmvParams& qp, int group) {
    const bool dense = qp.mode == kModeDense || qp.experts <= 1;
    return group == 16 && qp.rows > 0 && qp.cols > 0 && qp.row_stride % 4 == 0 && qp.ngroups % 8 == 0 &&
           (dense || (qp.expert_stride_w % 4 == 0 && qp.expert_stride_s % 8 == 0)) &&
           (reinterpret_cast<uintptr_t>(qp.codes) & 15) == 0 && (reinterpret_cast<uintptr_t>(qp.scales) & 15) == 0 &&
           tensor_map_encoder() != nullptr;
}

tq_status launch_trit_tc(const QmvParams& qp, int n_items, cudaStream_t st, const TritParams* xstage) {
    using F = TritFmt<16>;
    TritParams tp{};
    if (xstage) tp = *xstage;
    tp.q = qp;
    tp.units = (qp.cols + F::kUT - 1) / F::kUT;
    tp.nsteps = (tp.units + kTcS - 1) / kTcS;
    tp.tasks_per_item = (qp.rows + kTcRows - 1) / kTcRows;
    tp.n_items = n_items;
    const int64_t total = (int64_t)n_items * tp.tasks_per_item;
    if (total > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    tp.total_tasks = (int)total;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    // one CTA per SM, fewer when there are fewer (task, stage) units than consumer warps
    const int64_t work = total * tp.nsteps;
    int64_t grid = std::min<int64_t>(sms, (work + kTcWarps - 1) / kTcWarps);
    if (grid < (total + 255) / 256) grid = (total + 255) / 256;  // row-sum buffer: at most 256 tasks per CTA
    if (grid < 1) grid = 1;
    if (grid > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    const int max_tasks = (int)((total + grid - 1) / grid) + 1;
    const size_t smem = trit_tc_smem(tp.nsteps, max_tasks, tp.xmode ? (qp.cols / 32) * 33 : 0);
    if (smem > 227 * 1024) return TQ_ERR_UNSUPPORTED;
    TritMaps maps;
    if (!encode_trit_maps(qp, maps)) return TQ_ERR_UNSUPPORTED;
    if (tp.xmode) {
        if (ensure_smem((const void*)qmv_trit_tc_kernel<true>, smem) != cudaSuccess) return TQ_ERR_CUDA;
        qmv_trit_tc_kernel<true><<<(unsigned)grid, kTcThreads, smem, st>>>(tp, maps);
    } else {
        if (ensure_smem((const void*)qmv_trit_tc_kernel<false>, smem) != cudaSuccess) return TQ_ERR_CUDA;
        qmv_trit_tc_kernel<false><<<(unsigned)grid, kTcThreads, smem, st>>>(tp, maps);
    }
    return launch_status();
}

}  // namespace

// The tensor-copy kernel with its input stage (xmode 1: rotate xin rows; 2: SwiGLU then rotate).
tq_status qmv_trit_xstage_run(const QmvParams& p, int group, int n_items, int xmode, const void* xin, int xdt,
                              const int8_t* signs, int block, cudaStream_t st) {
    // 16-byte input loads (8-byte for bf16) and one 32-bit word per 4 signs
    const uintptr_t xa = xmode == 1 && xdt == TQ_BF16 ? 7 : 15;
    if (!trit_tc_ok(p, group) || p.cols % 32 || block < 32 || block > 8192 || (block & (block - 1)) ||
        p.cols % block || (reinterpret_cast<uintptr_t>(xin) & xa) || (reinterpret_cast<uintptr_t>(signs) & 3))
        return TQ_ERR_UNSUPPORTED;
    TritParams xs{};
    xs.xmode = xmode;
    xs.xin = xin;
    xs.xdt = xdt;
    xs.xsigns = signs;
    xs.xblock = block;
    return launch_trit_tc(p, n_items, st, &xs);
}

// Rows per warp step: 4 rows x 8 units when a row holds many units, else 8 rows
// x 4 units (keeps the last, partial step of short rows cheap).
tq_status qmv_trit_run(const QmvParams& p, int group, int n_items, cudaStream_t st) {
    // Staged pipeline when every copy is 16-byte aligned: 16-byte code rows
    // (always), scale rows and expert scale strides in whole 16-byte chunks.
    const bool pipe_ok = (group == 16 || group == 32) && ((int64_t)p.ngroups * 2) % 16 == 0 && p.row_stride < (1 << 30) &&
                         (p.expert_stride_s * 2) % 16 == 0 && (reinterpret_cast<uintptr_t>(p.scales) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.codes) & 15) == 0;
    if (pipe_ok) {
        // group 16: the tensor-copy pipeline when the banks can be described by tensor maps
        if (trit_tc_ok(p, group)) {
            const tq_status s = launch_trit_tc(p, n_items, st, nullptr);
            if (s != TQ_ERR_UNSUPPORTED) return s;
        }
        return group == 16 ? launch_trit_pipe<16>(p, n_items, st) : launch_trit_pipe<32>(p, n_items, st);
    }
    const int ut = 20 / std::gcd(20, group) * group;
    const bool wide = (p.cols + ut - 1) / ut >= 48;
    switch (group) {
        case 16: return wide ? launch_trit<16, 4>(p, n_items, st) : launch_trit<16, 8>(p, n_items, st);
        case 32: return wide ? launch_trit<32, 4>(p, n_items, st) : launch_trit<32, 8>(p, n_items, st);
        case 64: return wide ? launch_trit<64, 4>(p, n_items, st) : launch_trit<64, 8>(p, n_items, st);
        case 128: return wide ? launch_trit<128, 4>(p, n_items, st) : launch_trit<128, 8>(p, n_items, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
