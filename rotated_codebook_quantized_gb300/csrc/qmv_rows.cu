// Bit-packed matvec with one matrix row per lane (2-, 3- and 4-bit books): the kernel behind
// tq_gather_qmv, tq_multi_gather_qmv and tq_qmv for bit-packed books.
//
// "How it works", "Quantizing a weight" (codes packed into 32-bit words: 16 / 10 / 8 codes of
// 2 / 3 / 4 bits) and "Running a quantized layer" (the rotated input times the codes, decoded
// inline, one fp16 scale per group).
//
// Work layout.  A task is (item, block of 32 rows, chunk of columns); lane l of the warp that
// takes it owns row 32·block + l, so all 32 lanes walk the same columns: the input values are
// one broadcast load per four codes (from L1), and the group boundaries fall at the same,
// compile-time positions for every lane.  A chunk is a whole number of units of lcm(80, 64, ...)
// codes: lcm(8 words of codes, group), so each unit holds whole groups at fixed offsets.
// Decode: a pair of codes (2·bits) indexes a per-lane table of (c[a], c[b]) pairs, so a pair
// costs one shift, one masked OR into the lane's table column, one 8-byte shared load and two
// FMAs; a group's sum is scaled once.
//
// Pipeline.  One persistent CTA per SM, 16 warps; each warp takes a contiguous run of the CTA's
// tasks and streams their stages (8 code words of each of its 32 rows, 1 KB) with 16-byte
// cp.async into a private ring of 4 stages, 3 in flight while it decodes one.  Words beyond a
// row, rows beyond the matrix and experts outside the bank read as zeros.  Rows longer than one
// chunk write one partial sum per chunk: into scratch (added in chunk order by a second kernel,
// launched as a programmatic dependent) or, for a call without scratch, added into a zeroed f32
// output with atomics.
#include <algorithm>

#include "qmv_impl.cuh"

namespace tq {
namespace {

constexpr int kRWarps = 16;
constexpr int kRThreads = 32 * kRWarps;
constexpr int kRDepth = 4;              // ring stages per warp (3 in flight)
constexpr int kRCodeBytes = 32 * 32;    // a stage's codes: 8 words of each of 32 rows
constexpr int kRMaxChunkGroups = 8;     // scale registers per task

template <int LEVELS>
struct RFmt {
    static constexpr int kBits = LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4);
    static constexpr int kCW = LEVELS == 8 ? 10 : 32 / kBits;  // codes per word
    static constexpr int kPW = kCW / 2;                        // code pairs per word
    static constexpr int kTab = 1 << (2 * kBits);              // pair-table entries
    static constexpr uint32_t kTabBytes = kTab * 32 * 8;       // one float2 per entry and lane
    static constexpr int kSC = 8 * kCW;                        // codes per stage
    static constexpr int kStageBytes = kRCodeBytes + kSC * 4;  // codes, then the stage's input values
};

template <int LEVELS, int G>
struct RUnit {
    using F = RFmt<LEVELS>;
    static constexpr int kCodes = F::kSC / Gcd<F::kSC, G>::v * G;  // lcm(stage codes, group)
    static constexpr int kStages = kCodes / F::kSC;
    static constexpr int kGroups = kCodes / G;
    static constexpr int kChunkUnits = kRMaxChunkGroups / kGroups > 0 ? kRMaxChunkGroups / kGroups : 1;
    static_assert(kGroups <= kRMaxChunkGroups, "unit groups");
};

struct RowsParams {
    QmvParams q;
    int units;        // units per row
    int chunk_units;  // units per task (<= the instance's kChunkUnits)
    int nchunks;      // chunks per row
    int row_blocks;   // ceil(rows / 32)
    int n_items;
    int ntasks;
    float* part;      // [nchunks][n_items][rows]: partial sums (nchunks > 1, with scratch)
    int atomic_out;   // nchunks > 1 without scratch: add into y (f32, zeroed beforehand)
};

TQ_DEVFN uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
TQ_DEVFN void cp16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
TQ_DEVFN void commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
TQ_DEVFN void wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
TQ_DEVFN uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
TQ_DEVFN float2 lds64f(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}

// What one task reads: row `row` of expert `e` (bad: outside the bank), input vector `vec`.
struct RTask {
    int item, rb, ch, row, vec, e;
    bool bad;
    const uint32_t* w;  // the lane's row, first word of the chunk
};

TQ_DEVFN RTask task_of(const RowsParams& rp, int t, int lane, int nst) {
    const QmvParams& p = rp.q;
    RTask k;
    const int per_item = rp.row_blocks * rp.nchunks;
    k.item = t / per_item;
    const int rem = t - k.item * per_item;
    k.rb = rem / rp.nchunks;
    k.ch = rem - k.rb * rp.nchunks;
    k.row = k.rb * 32 + lane;
    int e = 0;
    if (p.mode == kModeDense) {
        k.vec = k.item;
    } else {
        e = __ldg(p.ids + k.item);
        k.vec = p.mode == kModeGather ? k.item / p.k : k.item;
    }
    k.bad = e < 0 || e >= p.experts;
    k.e = k.bad ? 0 : e;
    const int64_t ee = k.e;
    const int rowc = k.row < p.rows ? k.row : 0;
    k.w = p.codes + ee * p.expert_stride_w + (int64_t)rowc * p.row_stride + (int64_t)k.ch * nst * 8;
    return k;
}

// The task after k (t + 1), without divisions.
TQ_DEVFN void task_next(const RowsParams& rp, RTask& k, int lane, int nst) {
    const QmvParams& p = rp.q;
    if (++k.ch == rp.nchunks) {
        k.ch = 0;
        if (++k.rb == rp.row_blocks) {
            k.rb = 0;
            ++k.item;
            int e = 0;
            if (p.mode == kModeDense) {
                k.vec = k.item;
            } else {
                e = __ldg(p.ids + k.item);
                k.vec = p.mode == kModeGather ? k.item / p.k : k.item;
            }
            k.bad = e < 0 || e >= p.experts;
            k.e = k.bad ? 0 : e;
        }
        k.row = k.rb * 32 + lane;
    }
    const int rowc = k.row < p.rows ? k.row : 0;
    k.w = p.codes + (int64_t)k.e * p.expert_stride_w + (int64_t)rowc * p.row_stride + (int64_t)k.ch * nst * 8;
}

// The lane's scales of task k's groups (zero past the row's groups, for a bad expert or a row
// past the matrix).
template <int NG, int UG>
TQ_DEVFN void task_scales(const RowsParams& rp, const RTask& k, float (&sc)[NG]) {
    const QmvParams& p = rp.q;
    const uint16_t* s0 = p.scales + (int64_t)k.e * p.expert_stride_s + (int64_t)(k.row < p.rows ? k.row : 0) * p.ngroups;
    const int g0 = k.ch * rp.chunk_units * UG;
    const bool live = !k.bad && k.row < p.rows;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const int gi = g0 + g;
        sc[g] = (live && g < rp.chunk_units * UG && gi < p.ngroups) ? half_bits_to_float(__ldg(s0 + gi)) : 0.f;
    }
}

template <int LEVELS, int G>
__global__ void __launch_bounds__(kRThreads, 1) qmv_rows_kernel(const RowsParams rp) {
    using F = RFmt<LEVELS>;
    using U = RUnit<LEVELS, G>;
    constexpr int CW = F::kCW, PW = F::kPW, BITS = F::kBits, SC = F::kSC;
    constexpr int NG = U::kChunkUnits * U::kGroups;  // scale registers
    const QmvParams& p = rp.q;
    extern __shared__ __align__(16) uint8_t smraw[];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // The pair table sits on a multiple of its own size, so an entry's address is the OR of
    // disjoint bit fields (lane * 8 in bits 3..7, the code pair above).
    const uint32_t raw = smem_addr(smraw);
    const uint32_t tab = (raw + F::kTabBytes - 1) & ~(F::kTabBytes - 1);
    uint8_t* tabp = smraw + (tab - raw);
    const uint32_t ring = tab + F::kTabBytes + (uint32_t)(warp * kRDepth * F::kStageBytes);
    for (int i = tid; i < F::kTab * 32; i += kRThreads) {
        const int v = i >> 5;
        reinterpret_cast<float2*>(tabp)[i] =
            make_float2(__ldg(p.centroids + (v & (LEVELS - 1))), __ldg(p.centroids + (v >> BITS)));
    }
    __syncthreads();

    const int nst = rp.chunk_units * U::kStages;  // stages per task
    const int tb = (int)((int64_t)blockIdx.x * rp.ntasks / gridDim.x);
    const int te = (int)((int64_t)(blockIdx.x + 1) * rp.ntasks / gridDim.x);
    const int ta = tb + (int)((int64_t)(te - tb) * warp / kRWarps);
    const int tz = tb + (int)((int64_t)(te - tb) * (warp + 1) / kRWarps);
    if (ta >= tz) return;
    const int64_t nstages = (int64_t)(tz - ta) * nst;
    const uint32_t lanetab = tab + (uint32_t)lane * 8u;
    const uint32_t swz = (uint32_t)((lane >> 2) & 1);
    const uint32_t my0 = (uint32_t)lane * 32u + (swz << 4), my1 = (uint32_t)lane * 32u + ((swz ^ 1u) << 4);

    // stream of stages: task ts, stage ss within it
    int ts = ta, ss = 0;
    RTask sk = task_of(rp, ts, lane, nst);
    auto issue = [&](int64_t j) {
        const uint32_t dst = ring + (uint32_t)((j % kRDepth) * F::kStageBytes);
        const int64_t word0 = (int64_t)sk.ch * nst * 8 + (int64_t)ss * 8;
        const bool rok = !sk.bad && sk.row < p.rows;
        const uint32_t* src = sk.w + ss * 8;
        cp16(dst + my0, src, rok && word0 + 4 <= p.row_stride ? 16u : 0u);
        cp16(dst + my1, src + 4, rok && word0 + 8 <= p.row_stride ? 16u : 0u);
        // the stage's input values (columns past the row read as zeros; cols is a multiple of 16)
        const int xcol = sk.ch * rp.chunk_units * U::kCodes + ss * SC + 4 * lane;
        if (lane < SC / 4)
            cp16(dst + kRCodeBytes + 16u * (uint32_t)lane, p.x + (int64_t)sk.vec * p.cols + (xcol < p.cols ? xcol : 0),
                 xcol < p.cols ? 16u : 0u);
        if (++ss == nst) {
            ss = 0;
            if (++ts < tz) task_next(rp, sk, lane, nst);
        }
    };
#pragma unroll
    for (int j = 0; j < kRDepth - 1; ++j) {
        if (j < nstages) issue(j);
        commit();
    }

    // scales one task ahead: the loads of task t + 1 are in flight while task t decodes
    float sc[NG], scn[NG];
    RTask k = task_of(rp, ta, lane, nst);
    task_scales<NG, U::kGroups>(rp, k, scn);
    int64_t j = 0;  // stage being decoded
    for (int t = ta; t < tz; ++t) {
        if (t > ta) task_next(rp, k, lane, nst);
        if (k.bad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
#pragma unroll
        for (int g = 0; g < NG; ++g) sc[g] = scn[g];
        if (t + 1 < tz) {
            RTask kn = k;
            task_next(rp, kn, lane, nst);
            task_scales<NG, U::kGroups>(rp, kn, scn);
        }
        float tot = 0.f;
        for (int u = 0; u < rp.chunk_units; ++u) {
            float acc0 = 0.f, acc1 = 0.f;
            static_for<0, U::kStages>([&](auto s_c) {
                constexpr int S = decltype(s_c)::value;
                if (j + kRDepth - 1 < nstages) issue(j + kRDepth - 1);
                commit();
                wait_group<kRDepth - 1>();
                __syncwarp();
                const uint32_t sb = ring + (uint32_t)((j % kRDepth) * F::kStageBytes);
                const uint32_t sbx = sb + kRCodeBytes;  // the stage's input values (broadcast reads)
                const uint4 P0 = lds128(sb + my0), P1 = lds128(sb + my1);
                const uint32_t W[8] = {P0.x, P0.y, P0.z, P0.w, P1.x, P1.y, P1.z, P1.w};
                static_for<0, 8>([&](auto w_c) {
                    constexpr int WI = decltype(w_c)::value;
                    const uint32_t w = W[WI];
                    // the word's input values, broadcast (every lane reads the same address)
                    // the word's input values from the stage (every lane reads the same address):
                    // four per load where the column is a multiple of 4, else two
                    float xw[CW];
                    static_for<0, CW / 2>([&](auto q_c) {
                        constexpr int Q = 2 * decltype(q_c)::value;
                        constexpr int kOff = WI * CW + Q;  // column within the stage
                        constexpr bool kQuad = kOff % 4 == 0 && Q + 4 <= CW;
                        if constexpr (kOff % 4 == 2 && Q >= 2) return;  // loaded with the pair before it
                        if constexpr (kQuad) {
                            const uint4 xx = lds128(sbx + 4u * kOff);
                            xw[Q] = __uint_as_float(xx.x);
                            xw[Q + 1] = __uint_as_float(xx.y);
                            xw[Q + 2] = __uint_as_float(xx.z);
                            xw[Q + 3] = __uint_as_float(xx.w);
                        } else {
                            const float2 xx = lds64f(sbx + 4u * kOff);
                            xw[Q] = xx.x;
                            xw[Q + 1] = xx.y;
                        }
                    });
                    static_for<0, PW>([&](auto p_c) {
                        constexpr int PI = decltype(p_c)::value;
                        constexpr int SH = 2 * BITS * PI;  // bit offset of the pair
                        constexpr uint32_t kMask = ((1u << (2 * BITS)) - 1u) << 8;
                        const uint32_t off = (SH >= 8 ? (w >> (SH - 8)) : (w << (8 - SH))) & kMask;
                        const float2 c = lds64f(lanetab | off);
                        float& acc = (PI & 1) ? acc1 : acc0;
                        acc = fmaf(c.x, xw[2 * PI], acc);
                        acc = fmaf(c.y, xw[2 * PI + 1], acc);
                        constexpr int kEnd = S * SC + WI * CW + 2 * PI + 2;  // codes of the unit done
                        if constexpr (kEnd % G == 0) {
                            tot = fmaf(sc[kEnd / G - 1], acc0 + acc1, tot);
                            acc0 = 0.f;
                            acc1 = 0.f;
                        }
                    });
                });
                __syncwarp();  // the slot (codes and input values) is read before a later stage refills it
                ++j;
            });
#pragma unroll
            for (int g = 0; g + U::kGroups < NG; ++g) sc[g] = sc[g + U::kGroups];  // the next unit's scales first
        }
        if (k.row < p.rows) {
            const int64_t o = (int64_t)k.item * p.rows + k.row;
            if (rp.nchunks == 1) store_from_float(p.y, o, p.ydt, tot);
            else if (rp.atomic_out) atomicAdd(static_cast<float*>(p.y) + o, tot);
            else rp.part[(int64_t)k.ch * rp.n_items * p.rows + o] = tot;
        }
    }
    wait_group<0>();
}

// y[i] = sum over chunks of part[c][i], in chunk order.
__global__ void __launch_bounds__(256) rows_chunk_sum_kernel(const float* __restrict__ part, int nchunks, int64_t n,
                                                             void* y, int ydt) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        for (int c = 0; c < nchunks; ++c) v += part[c * n + i];
        store_from_float(y, i, ydt, v);
    }
}

int sm_count_rows() {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    return sms;
}

// Units per chunk: the fewest decoded units per row (least padding), then the fewest chunks
// while the tasks still give every warp of the GPU two or more.
template <int LEVELS, int G>
void plan_chunks(RowsParams& rp, int cols) {
    using U = RUnit<LEVELS, G>;
    rp.units = (cols + U::kCodes - 1) / U::kCodes;
    const int64_t want = 2ll * sm_count_rows() * kRWarps;
    int best = 1;
    int64_t best_dec = -1;
    for (int cu = 1; cu <= U::kChunkUnits; ++cu) {
        const int nch = (rp.units + cu - 1) / cu;
        const int64_t dec = (int64_t)nch * cu;
        const int64_t tasks = (int64_t)rp.n_items * rp.row_blocks * nch;
        if (tasks < want && cu > 1) break;
        if (best_dec < 0 || dec < best_dec || (dec == best_dec)) {
            best = cu;
            best_dec = dec;
        }
    }
    rp.chunk_units = best;
    rp.nchunks = (rp.units + best - 1) / best;
}

template <int LEVELS, int G>
size_t rows_smem() {
    return (size_t)RFmt<LEVELS>::kTabBytes * 2 + (size_t)kRWarps * kRDepth * RFmt<LEVELS>::kStageBytes;
}

template <int LEVELS, int G>
tq_status rows_launch(const QmvParams& qp, int n_items, void* ws, size_t ws_bytes, cudaStream_t st) {
    RowsParams rp{};
    rp.q = qp;
    rp.n_items = n_items;
    rp.row_blocks = (qp.rows + 31) / 32;
    plan_chunks<LEVELS, G>(rp, qp.cols);
    const int64_t ntasks = (int64_t)n_items * rp.row_blocks * rp.nchunks;
    if (ntasks > 0x7fffffffll || ntasks == 0) return TQ_ERR_UNSUPPORTED;
    rp.ntasks = (int)ntasks;
    const int64_t n = (int64_t)n_items * qp.rows;
    const size_t need = rp.nchunks > 1 ? (size_t)rp.nchunks * (size_t)n * 4 : 0;
    if (need > 0) {
        if (ws && ws_bytes >= need && (reinterpret_cast<uintptr_t>(ws) & 15) == 0) {
            rp.part = static_cast<float*>(ws);
        } else {
            if (qp.ydt != TQ_F32) return TQ_ERR_UNSUPPORTED;
            rp.atomic_out = 1;
            if (cudaMemsetAsync(qp.y, 0, (size_t)n * 4, st) != cudaSuccess) return TQ_ERR_CUDA;
        }
    }
    const size_t smem = rows_smem<LEVELS, G>();
    if (ensure_smem((const void*)qmv_rows_kernel<LEVELS, G>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    const int sms = sm_count_rows();
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, (ntasks + kRWarps - 1) / kRWarps));
    tq_status s;
    if (rp.atomic_out) {
        qmv_rows_kernel<LEVELS, G><<<grid, kRThreads, smem, st>>>(rp);
        s = launch_status();
    } else {
        s = launch_pdl(qmv_rows_kernel<LEVELS, G>, dim3(grid), dim3(kRThreads), smem, st, rp);
    }
    if (s != TQ_OK || rp.nchunks == 1 || rp.atomic_out) return s;
    return launch_pdl(rows_chunk_sum_kernel, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4 * (int64_t)sms)),
                      dim3(256), 0, st, (const float*)rp.part, rp.nchunks, n, qp.y, qp.ydt);
}

template <int LEVELS>
tq_status rows_g(const QmvParams& p, int group, int n_items, void* ws, size_t ws_bytes, cudaStream_t st) {
    switch (group) {
        case 16: return rows_launch<LEVELS, 16>(p, n_items, ws, ws_bytes, st);
        case 32: return rows_launch<LEVELS, 32>(p, n_items, ws, ws_bytes, st);
        case 64: return rows_launch<LEVELS, 64>(p, n_items, ws, ws_bytes, st);
        case 128: return rows_launch<LEVELS, 128>(p, n_items, ws, ws_bytes, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

template <int LEVELS, int G>
size_t rows_ws(int cols, int64_t n_items, int rows) {
    RowsParams rp{};
    rp.n_items = (int)std::min<int64_t>(n_items, 0x7fffffff);
    rp.row_blocks = (rows + 31) / 32;
    plan_chunks<LEVELS, G>(rp, cols);
    return rp.nchunks > 1 ? (size_t)rp.nchunks * (size_t)n_items * (size_t)rows * 4 : 0;
}

template <int LEVELS>
size_t rows_ws_g(int group, int cols, int64_t n_items, int rows) {
    switch (group) {
        case 16: return rows_ws<LEVELS, 16>(cols, n_items, rows);
        case 32: return rows_ws<LEVELS, 32>(cols, n_items, rows);
        case 64: return rows_ws<LEVELS, 64>(cols, n_items, rows);
        case 128: return rows_ws<LEVELS, 128>(cols, n_items, rows);
        default: return 0;
    }
}

}  // namespace

// Whether the row-per-lane kernel takes this matvec: a 2-, 3- or 4-bit book, code rows and
// expert strides whole 16-byte pieces from a 16-byte aligned base, an input whose rows can be
// read as float pairs, and items that fit the task count.
bool qmv_rows_ok(const QmvParams& p, int group) {
    const bool dense = p.mode == kModeDense || p.experts <= 1;
    return (p.levels == 4 || p.levels == 8 || p.levels == 16) &&
           (group == 16 || group == 32 || group == 64 || group == 128) && p.rows > 0 && p.cols > 0 &&
           p.cols % 16 == 0 && p.row_stride % 4 == 0 && (dense || p.expert_stride_w % 4 == 0) &&
           (reinterpret_cast<uintptr_t>(p.codes) & 15) == 0 && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0 &&
           (p.mode != kModeGroups);
}

size_t qmv_rows_workspace_bytes(int levels, int group, int cols, int64_t n_items, int rows) {
    if (n_items <= 0 || rows <= 0 || cols <= 0) return 0;
    switch (levels) {
        case 4: return rows_ws_g<4>(group, cols, n_items, rows);
        case 8: return rows_ws_g<8>(group, cols, n_items, rows);
        case 16: return rows_ws_g<16>(group, cols, n_items, rows);
        default: return 0;
    }
}

tq_status qmv_rows_run(const QmvParams& p, int group, int n_items, void* ws, size_t ws_bytes, cudaStream_t st) {
    switch (p.levels) {
        case 4: return rows_g<4>(p, group, n_items, ws, ws_bytes, st);
        case 8: return rows_g<8>(p, group, n_items, ws, ws_bytes, st);
        case 16: return rows_g<16>(p, group, n_items, ws, ws_bytes, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
