// Quantized matvec with inline decode: tq_qmv, tq_gather_qmv, tq_multi_gather_qmv.
//
// "How it works", "Running a quantized layer": the input is rotated once and
// multiplied by the packed codes, which are decoded inline, so full-precision
// weights never exist.  The three MoE situations of that section map to the
// item modes below (dense matrix, gather with a shared input, per-pair input).
//
// Work layout (GB300): a CTA owns 32 consecutive output rows of one item and
// splits the input dimension over its warps; inside a warp each lane owns one
// row, so all lanes walk the same columns at the same time: the rotated input
// in shared memory is read with broadcast loads, and each lane streams its own
// row with 16-byte loads.  Columns are walked in "units" of lcm(codes per
// word, group) codes, so group boundaries sit at compile-time positions and no
// per-code division or branch is needed.  The partial sums of the warps are
// added in shared memory at the end.  The kernel is bound by HBM bytes and by
// the integer/FP issue rate of the decode.
#pragma once

#include "common.cuh"

namespace tq {

template <int A, int B>
struct Gcd {
    static constexpr int v = Gcd<B, A % B>::v;
};
template <int A>
struct Gcd<A, 0> {
    static constexpr int v = A;
};

template <int LEVELS, int G>
struct QFmt {
    static constexpr bool kTrit = LEVELS == 3;
    static constexpr int kBits = LEVELS == 3 ? 0 : (LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4));
    static constexpr int kCW = LEVELS == 3 ? 20 : (LEVELS == 8 ? 10 : 32 / kBits);  // codes per word
    static constexpr int kUC = kCW / Gcd<kCW, G>::v * G;                          // codes per unit
    static constexpr int kUW = kUC / kCW;                                           // words per unit
    static constexpr int kS = kUW >= 16 ? 1 : 16 / kUW;                            // units per step
    static constexpr int kSW = kS * kUW;                                            // words per step
    static constexpr int kSC = kSW * kCW;                                           // codes per step
    static constexpr int kSG = kSC / G;                                             // groups per step
    static constexpr int kCB = kCW == 10 ? 20 : kCW;                                // codes per x block
    static constexpr int kCBW = kCB / kCW;                                          // words per x block
    static_assert(kSW % 4 == 0, "steps are whole 16-byte loads");
    static_assert(kSC % G == 0, "steps hold whole groups");
    static_assert(kCB % 4 == 0, "x blocks are whole float4");
};

// kModeGroups: multi-gather with the pairs grouped by expert; item g is record g of `groups`
// (groups[0] = number of records; record g at groups + 2 + g * (1 + NV) = expert, then up to NV
// pair indices, -1 where empty), so each expert's weights are decoded once for all its pairs.
enum QmvMode { kModeDense = 0, kModeGather = 1, kModeMulti = 2, kModeGroups = 3 };

struct QmvParams {
    const uint32_t* codes;
    const uint16_t* scales;
    int64_t row_stride, expert_stride_w, expert_stride_s;
    int rows, cols, ngroups, experts;
    const float* centroids;
    int levels;
    const float* x;  // [*, cols] rotated input, fp32
    int T;           // dense: number of vectors
    int mode;
    const int32_t* ids;
    int k;           // gather: experts per token
    int item0;       // first item of this launch
    void* y;
    int ydt;
    uint32_t* err;
    int kpad;        // padded x length in shared memory (multiple of the step)
    int gpad;        // padded group count
    int nsteps;      // steps per row
    const int32_t* groups;  // kModeGroups: the expert records
    long long wait_cycles = 1ll << 31;  // budget of each bounded wait of the tensor-copy kernel
};

TQ_DEVFN uint4 ldg_u4(const uint32_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

template <int LEVELS, int G, int NV>
__global__ void __launch_bounds__(256) qmv_kernel(const QmvParams p) {
    using F = QFmt<LEVELS, G>;
    constexpr int SW = F::kSW, SC = F::kSC, SG = F::kSG, CW = F::kCW, CB = F::kCB, CBW = F::kCBW;
    constexpr int NQ = SW / 4;
    constexpr bool kDouble = SW <= 16;

    extern __shared__ __align__(16) float smem[];
    float* xs = smem;                       // [NV][kpad]
    float* xsum = xs + NV * p.kpad;         // [NV][gpad], ternary only
    float* lut = xsum + NV * p.gpad;        // [16]
    float* red = lut + 16;                  // [nwarps][NV][32]

    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = p.item0 + blockIdx.y;
    const int row = blockIdx.x * 32 + lane;
    const int rowc = row < p.rows ? row : p.rows - 1;

    int e, vec0, nv;
    int64_t out0, out_stride;
    const int32_t* glist = nullptr;  // kModeGroups: this item's pair indices
    if (p.mode == kModeGroups) {
        if (item >= __ldg(p.groups)) return;  // uniform: fewer records than the launch's bound
        const int32_t* rec = p.groups + 2 + (int64_t)item * (1 + NV);
        e = __ldg(rec);
        glist = rec + 1;
        vec0 = 0;
        nv = NV;
        out0 = 0;
        out_stride = 0;
    } else if (p.mode == kModeDense) {
        e = 0;
        vec0 = item * NV;
        nv = min(NV, p.T - vec0);
        out0 = (int64_t)vec0 * p.rows;
        out_stride = p.rows;
    } else if (p.mode == kModeGather) {
        e = p.ids[item];
        vec0 = item / p.k;
        nv = 1;
        out0 = (int64_t)item * p.rows;
        out_stride = 0;
    } else {
        e = p.ids[item];
        vec0 = item;
        nv = 1;
        out0 = (int64_t)item * p.rows;
        out_stride = 0;
    }
    if (e < 0 || e >= p.experts) {  // uniform over the CTA
        if (threadIdx.x == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        if (glist) return;  // records hold valid experts only; nothing to write here
        for (int i = threadIdx.x; i < 32 * nv; i += blockDim.x) {
            const int r = blockIdx.x * 32 + (i & 31);
            if (r < p.rows) store_from_float(p.y, out0 + (i >> 5) * out_stride + r, p.ydt, 0.f);
        }
        return;
    }

    const uint32_t* wrow = p.codes + (int64_t)e * p.expert_stride_w + (int64_t)rowc * p.row_stride;
    const uint16_t* srow = p.scales + (int64_t)e * p.expert_stride_s + (int64_t)rowc * p.ngroups;
    const int s0 = (int)((int64_t)warp * p.nsteps / nwarps);
    const int s1 = (int)((int64_t)(warp + 1) * p.nsteps / nwarps);

    uint4 cur[NQ];
    auto load_step = [&](uint4 (&buf)[NQ], int s) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int64_t widx = (int64_t)s * SW + 4 * q;
            buf[q] = widx < p.row_stride ? ldg_u4(wrow + widx) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    if (s0 < s1) load_step(cur, s0);  // first weight bytes in flight before the x fill

    // Rotated input (zero padded), per-group input sums (ternary) and the codebook.
    int vidx[NV];  // input / output row of each vector (-1: none)
#pragma unroll
    for (int v = 0; v < NV; ++v) vidx[v] = glist ? __ldg(glist + v) : (v < nv ? vec0 + v : -1);
    for (int v = 0; v < NV; ++v) {
        const bool has = vidx[v] >= 0;
        const float* xv = p.x + (int64_t)(has ? vidx[v] : 0) * p.cols;
        for (int i = threadIdx.x; i < p.kpad; i += blockDim.x) xs[v * p.kpad + i] = (has && i < p.cols) ? xv[i] : 0.f;
    }
    if (threadIdx.x < 16) lut[threadIdx.x] = threadIdx.x < LEVELS ? p.centroids[threadIdx.x] : 0.f;
    __syncthreads();
    float c0 = 0.f, dc = 0.f;
    if (F::kTrit) {
        for (int i = threadIdx.x; i < NV * p.gpad; i += blockDim.x) {
            const int v = i / p.gpad, g = i - v * p.gpad;
            const float* a = xs + v * p.kpad + g * G;
            float s = 0.f;
#pragma unroll 16
            for (int j = 0; j < G; ++j) s += a[j];
            xsum[i] = s;
        }
        c0 = lut[0];
        dc = lut[1] - lut[0];
        if (threadIdx.x == 0 && p.err && fabsf((lut[2] - lut[1]) - dc) > 1e-6f * fabsf(dc))
            atomicOr(p.err, TQ_DEVERR_BAD_BOOK);
        __syncthreads();
    }

    float tot[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) tot[v] = 0.f;

    for (int s = s0; s < s1; ++s) {
        uint4 nxt[kDouble ? NQ : 1];
        if constexpr (kDouble) {
            if (s + 1 < s1) load_step(nxt, s + 1);
        }
        float sc[SG];
#pragma unroll
        for (int g = 0; g < SG; ++g) {
            const int gi = s * SG + g;
            sc[g] = gi < p.ngroups ? half_bits_to_float(__ldg(srow + gi)) : 0.f;
        }
        const int kbase = s * SC;
        float acc[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[v] = 0.f;
        const uint32_t* wv = reinterpret_cast<const uint32_t*>(cur);

#pragma unroll
        for (int j = 0; j < SW; j += CBW) {
            // x values of this block of CB codes, for each vector
            float4 xf[NV][CB / 4];
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int q = 0; q < CB / 4; ++q)
                    xf[v][q] = reinterpret_cast<const float4*>(xs + v * p.kpad + kbase + j * CW)[q];
            float cv[CB];
            if constexpr (F::kTrit) {
                const TritHalves th = trit_split(wv[j]);
                uint32_t Fh = th.hi, Fl = th.lo;
#pragma unroll
                for (int t = 0; t < 10; ++t) cv[19 - t] = trit_next(Fh);
#pragma unroll
                for (int t = 0; t < 10; ++t) cv[9 - t] = trit_next(Fl);
            } else {
#pragma unroll
                for (int i = 0; i < CB; ++i) {
                    const uint32_t w = wv[j + i / CW];
                    const int pos = i % CW;
                    const uint32_t off = (pos == 0 ? (w << 2) : (w >> (F::kBits * pos - 2))) & ((LEVELS - 1) << 2);
                    cv[i] = *reinterpret_cast<const float*>(reinterpret_cast<const char*>(lut) + off);
                }
            }
#pragma unroll
            for (int i = 0; i < CB; ++i) {
                const int kk = j * CW + i;  // code index within the step
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const float4 f = xf[v][i / 4];
                    const float xk = (i & 3) == 0 ? f.x : ((i & 3) == 1 ? f.y : ((i & 3) == 2 ? f.z : f.w));
                    acc[v] = fmaf(cv[i], xk, acc[v]);
                }
                if ((kk + 1) % G == 0) {
                    const int g = kk / G;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        if constexpr (F::kTrit) {
                            const float xg = xsum[v * p.gpad + s * SG + g];
                            tot[v] = fmaf(sc[g], fmaf(dc, acc[v], c0 * xg), tot[v]);
                        } else {
                            tot[v] = fmaf(sc[g], acc[v], tot[v]);
                        }
                        acc[v] = 0.f;
                    }
                }
            }
        }
        if constexpr (kDouble) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) cur[q] = nxt[q];
        } else {
            if (s + 1 < s1) load_step(cur, s + 1);
        }
    }

#pragma unroll
    for (int v = 0; v < NV; ++v) red[(warp * NV + v) * 32 + lane] = tot[v];
    __syncthreads();
    for (int i = threadIdx.x; i < NV * 32; i += blockDim.x) {
        const int v = i >> 5, l = i & 31;
        float sum = 0.f;
        for (int w = 0; w < nwarps; ++w) sum += red[(w * NV + v) * 32 + l];
        const int r = blockIdx.x * 32 + l;
        if (glist) {
            const int pv = __ldg(glist + v);
            if (r < p.rows && pv >= 0) store_from_float(p.y, (int64_t)pv * p.rows + r, p.ydt, sum);
        } else if (r < p.rows && v < nv) {
            store_from_float(p.y, out0 + (int64_t)v * out_stride + r, p.ydt, sum);
        }
    }
}

// Host-side launch of one (levels, group, NV) instantiation.
template <int LEVELS, int G, int NV>
tq_status launch_qmv(QmvParams p, int n_items, cudaStream_t st) {
    using F = QFmt<LEVELS, G>;
    const int units = (p.cols + F::kUC - 1) / F::kUC;
    p.nsteps = (units + F::kS - 1) / F::kS;
    p.kpad = p.nsteps * F::kSC;
    p.gpad = F::kTrit ? p.kpad / G : 0;
    const int nwarps = p.nsteps < 8 ? p.nsteps : 8;
    const size_t smem = sizeof(float) * ((size_t)NV * p.kpad + (size_t)NV * p.gpad + 16 + (size_t)nwarps * NV * 32);
    if (smem > 200 * 1024) return TQ_ERR_UNSUPPORTED;
    if (ensure_smem((const void*)qmv_kernel<LEVELS, G, NV>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    const int tiles = (p.rows + 31) / 32;
    if (tiles > 65535) return TQ_ERR_UNSUPPORTED;
    for (int i0 = 0; i0 < n_items; i0 += 65535) {
        const int n = n_items - i0 < 65535 ? n_items - i0 : 65535;
        p.item0 = i0;
        qmv_kernel<LEVELS, G, NV><<<dim3(tiles, n), nwarps * 32, smem, st>>>(p);
        const tq_status s = launch_status();
        if (s != TQ_OK) return s;
    }
    return TQ_OK;
}

// Shared-memory floats per input vector, for choosing NV on the host.
template <int LEVELS, int G>
int qmv_kpad(int cols) {
    using F = QFmt<LEVELS, G>;
    const int units = (cols + F::kUC - 1) / F::kUC;
    const int nsteps = (units + F::kS - 1) / F::kS;
    return nsteps * F::kSC;
}

template <int LEVELS, int G>
tq_status dispatch_qmv_nv(QmvParams p, int nv, int n_items, cudaStream_t st) {
    switch (nv) {
        case 1: return launch_qmv<LEVELS, G, 1>(p, n_items, st);
        case 2: return launch_qmv<LEVELS, G, 2>(p, n_items, st);
        case 4: return launch_qmv<LEVELS, G, 4>(p, n_items, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

// Ternary books with one input vector per item (qmv_trit.cu).
tq_status qmv_trit_run(const QmvParams& p, int group, int n_items, cudaStream_t st);
// The ternary tensor-copy kernel with an input stage: xmode 1 rotates rows of xin (dtype xdt),
// xmode 2 takes rows [gate | up] of f32 xin, applies SwiGLU, then rotates.  TQ_ERR_UNSUPPORTED
// where that kernel does not apply.
tq_status qmv_trit_xstage_run(const QmvParams& p, int group, int n_items, int xmode, const void* xin, int xdt,
                              const int8_t* signs, int block, cudaStream_t st);
// Ternary books by table lookup (qmv_lut.cu): gather and multi modes.  Rows wider than one
// column slice need qmv_lut_workspace_bytes of scratch for the slices' partial sums.
bool qmv_lut_ok(const QmvParams& p, int group);
size_t qmv_lut_workspace_bytes(int cols, int64_t n_items, int rows);
tq_status qmv_lut_run(const QmvParams& p, int n_items, void* ws, size_t ws_bytes, cudaStream_t st);
bool qmv_bits_ok(const QmvParams& p, int group);
tq_status qmv_bits_run(const QmvParams& p, int group, int n_items, cudaStream_t st);
// Bit-packed books, one matrix row per lane (qmv_rows.cu): every mode but kModeGroups (dense
// vectors go four, two or one to a task; gather and multi items one pair to a task).  Rows
// longer than one column chunk need qmv_rows_workspace_bytes of scratch for the chunks'
// partial sums; without it an f32 output is zeroed and the chunks add into it.
bool qmv_rows_ok(const QmvParams& p, int group);
size_t qmv_rows_workspace_bytes(int levels, int group, int cols, int64_t n_items, int rows);
tq_status qmv_rows_run(const QmvParams& p, int group, int n_items, void* ws, size_t ws_bytes, cudaStream_t st);
// The same kernel over pairs grouped by expert: lists[i] holds the grouping's records of 4, 2
// and 1 pairs (count, pad, then expert and pair indices per record), written on the device;
// each expert's words are decoded once per record.  Scratch as for P items.
tq_status qmv_rows_run_groups(const QmvParams& p, int group, const int32_t* const lists[3], int P, void* ws,
                              size_t ws_bytes, cudaStream_t st);

// One entry point per (levels, group), each compiled in its own translation unit.
#define TQ_QMV_DECL(L, G) tq_status qmv_run_l##L##_g##G(QmvParams p, int nv, int n_items, cudaStream_t st);
#define TQ_QMV_DECL_L(L) TQ_QMV_DECL(L, 16) TQ_QMV_DECL(L, 32) TQ_QMV_DECL(L, 64) TQ_QMV_DECL(L, 128)
TQ_QMV_DECL_L(3)
TQ_QMV_DECL_L(4)
TQ_QMV_DECL_L(8)
TQ_QMV_DECL_L(16)
#undef TQ_QMV_DECL_L
#undef TQ_QMV_DECL

}  // namespace tq
