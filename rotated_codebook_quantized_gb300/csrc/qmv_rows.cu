// Bit-packed matvec with one matrix row per lane (2-, 3- and 4-bit books): the kernel behind
// tq_gather_qmv, tq_multi_gather_qmv and tq_qmv for bit-packed books.
//
// "How it works", "Quantizing a weight" (codes packed into 32-bit words: 16 / 10 / 8 codes of
// 2 / 3 / 4 bits) and "Running a quantized layer" (the rotated input times the codes, decoded
// inline, one fp16 scale per group; with a different input per expert, each expert's weights
// read once for all the inputs routed to it).
//
// Work layout.  A record is one matrix (an expert, or the dense matrix) with up to four input
// vectors; records come in three segments of 4, 2 and 1 vectors.  A task is (record, block of
// 32 rows, chunk of columns); lane l of the warp that takes it owns row 32·block + l, so all 32
// lanes walk the same columns: the input values are one broadcast load per four codes, and the
// group boundaries fall at the same, compile-time positions for every lane.  A chunk is a whole
// number of units of lcm(8 words of codes, group) codes, so each unit holds whole groups at
// fixed offsets.  Decode: a pair of codes (2·bits) indexes a per-lane table of (c[a], c[b])
// pairs, so a pair costs one shift, one masked OR into the lane's table column and one 8-byte
// shared load, then two FMAs per input vector; a group's sum is scaled once per vector.  Every
// vector's sums are formed in the same order as with one vector per record, so grouping the
// inputs changes no bit of the results.
//
// Pipeline.  One persistent CTA per SM, 16 warps; the tasks are split between the warps of the
// grid by weight (a task of v vectors weighs 5 + v), each warp taking a contiguous run, and
// each warp streams its stages (8 code words of each of its 32 rows, 1 KB, and the record's
// input values for those columns) with 16-byte cp.async into a private ring, the later stages
// in flight while it decodes one.  Words beyond a row, rows beyond the matrix and experts
// outside the bank read as zeros.  Rows longer than one chunk write one partial sum per chunk:
// into scratch (added in chunk order by a second kernel, launched as a programmatic dependent)
// or, for a call without scratch, added into a zeroed f32 output with atomics.
#include <algorithm>
#include <type_traits>

#include "qmv_impl.cuh"

// The build compiles this file once per book (TQ_ROWS_LEVELS 4, 8, 16: that book's kernel
// instances) and once for the entry points (TQ_ROWS_LEVELS 0); undefined, it holds everything.
#if !defined(TQ_ROWS_LEVELS)
#define TQ_ROWS_ALL 1
#define TQ_ROWS_LEVELS 0
#endif

namespace tq {

struct RowsParams {
    QmvParams q;
    int units;        // units per row
    int chunk_units;  // units per task (<= the instance's kChunkUnits)
    int nchunks;      // chunks per row
    int row_blocks;   // ceil(rows / 32)
    // Records of segment i: count[i] of them (-1: the count is list[i][0], written on the device).
    // list[i]: explicit records (count, pad, then per record the expert and seg_nv(i) pair
    // indices, -1 where empty); null: implicit, record r of segment i holding the pairs
    // base_i + r·seg_nv(i) + s (base_i: the pairs of the segments before it), of expert ids[pair]
    // (one-vector records) or of the dense matrix.
    int count[3];
    const int32_t* list[3];
    int n_out;        // output rows: y is [n_out][rows]
    float* part;      // [nchunks][n_out][rows]: partial sums (nchunks > 1, with scratch)
    int atomic_out;   // nchunks > 1 without scratch: add into y (f32, zeroed beforehand)
};

// The kernel and its chunk sum for one book (any group size).
tq_status qmv_rows_launch_l4(const RowsParams& rp, int group, int64_t n_rec, void* ws, size_t ws_bytes,
                             cudaStream_t st);
tq_status qmv_rows_launch_l8(const RowsParams& rp, int group, int64_t n_rec, void* ws, size_t ws_bytes,
                             cudaStream_t st);
tq_status qmv_rows_launch_l16(const RowsParams& rp, int group, int64_t n_rec, void* ws, size_t ws_bytes,
                              cudaStream_t st);

namespace {

constexpr int kRWarps = 16;
constexpr int kRThreads = 32 * kRWarps;
constexpr int kRCodeBytes = 32 * 32;    // a stage's codes: 8 words of each of 32 rows
constexpr int kRMaxChunkGroups = 8;     // scale registers per task
constexpr int kRMaxNV = 4;              // input vectors per record

// Vectors of a record of segment i, and a task's weight in the split between warps.
__host__ __device__ constexpr int seg_nv(int i) { return i == 0 ? 4 : (i == 1 ? 2 : 1); }
__host__ __device__ constexpr int seg_weight(int i) { return 5 + seg_nv(i); }

template <int LEVELS, int MAXNV>
struct RFmt {
    static constexpr int kBits = LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4);
    static constexpr int kCW = LEVELS == 8 ? 10 : 32 / kBits;  // codes per word
    static constexpr int kPW = kCW / 2;                        // code pairs per word
    static constexpr int kTab = 1 << (2 * kBits);              // pair-table entries
    static constexpr uint32_t kTabBytes = kTab * 32 * 8;       // one float2 per entry and lane
    static constexpr int kSC = 8 * kCW;                        // codes per stage
    static constexpr int kXBytes = kSC * 4;                    // one vector's input values of a stage
    static constexpr int kStageBytes = kRCodeBytes + MAXNV * kXBytes;
    // ring stages per warp: 4 (3 in flight); 3 for the 4-bit book with four vectors, whose 64 KB
    // table takes the room
    static constexpr int kDepth = LEVELS == 16 && MAXNV > 1 ? 3 : 4;
};

template <int LEVELS, int G>
struct RUnit {
    using F = RFmt<LEVELS, 1>;
    static constexpr int kCodes = F::kSC / Gcd<F::kSC, G>::v * G;  // lcm(stage codes, group)
    static constexpr int kStages = kCodes / F::kSC;
    static constexpr int kGroups = kCodes / G;
    static constexpr int kChunkUnits = kRMaxChunkGroups / kGroups > 0 ? kRMaxChunkGroups / kGroups : 1;
    static_assert(kGroups <= kRMaxChunkGroups, "unit groups");
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
TQ_DEVFN int pick3(const int (&a)[3], int i) { return i == 0 ? a[0] : (i == 1 ? a[1] : a[2]); }

// The segments as one warp sees them: record counts and first implicit pairs.
struct RSegs {
    int cnt[3];
    int base[3];
};

// What one task reads: rows 32·rb .. of expert `e` (bad: outside the bank), the pairs pr[] of
// its record.
struct RTask {
    int seg, rec, rb, ch, row, e, nv;
    bool bad;
    int pr[kRMaxNV];    // pair (output row) of each vector slot, -1 where empty
    int vec0;           // input row of slot 0
    const uint32_t* w;  // the lane's row, first word of the chunk
};

TQ_DEVFN void load_record(const RowsParams& rp, const RSegs& sg, RTask& k) {
    const QmvParams& p = rp.q;
    k.nv = seg_nv(k.seg);
    const int32_t* L = k.seg == 0 ? rp.list[0] : (k.seg == 1 ? rp.list[1] : rp.list[2]);
    int e = 0;
    if (L) {
        const int32_t* r = L + 2 + (int64_t)k.rec * (1 + k.nv);
        e = __ldcg(r);
#pragma unroll
        for (int s = 0; s < kRMaxNV; ++s) k.pr[s] = s < k.nv ? __ldcg(r + 1 + s) : -1;
    } else {
        const int b = pick3(sg.base, k.seg) + k.rec * k.nv;
#pragma unroll
        for (int s = 0; s < kRMaxNV; ++s) k.pr[s] = s < k.nv ? b + s : -1;
        if (p.mode != kModeDense) e = __ldg(p.ids + b);
    }
    k.bad = e < 0 || e >= p.experts;
    k.e = k.bad ? 0 : e;
    k.vec0 = k.pr[0] < 0 ? 0 : (p.mode == kModeGather ? k.pr[0] / p.k : k.pr[0]);
}

TQ_DEVFN void set_row(const RowsParams& rp, RTask& k, int lane, int nst) {
    const QmvParams& p = rp.q;
    k.row = k.rb * 32 + lane;
    const int rowc = k.row < p.rows ? k.row : 0;
    k.w = p.codes + (int64_t)k.e * p.expert_stride_w + (int64_t)rowc * p.row_stride + (int64_t)k.ch * nst * 8;
}

// Task t of the launch (segments in order, records, row blocks, chunks; the host keeps the
// task count below 2^31).
TQ_DEVFN void task_of(const RowsParams& rp, const RSegs& sg, int t, int lane, int nst, RTask& k) {
    const int per_rec = rp.row_blocks * rp.nchunks;
    int seg = 0;
    while (seg < 2 && t >= pick3(sg.cnt, seg) * per_rec) {
        t -= pick3(sg.cnt, seg) * per_rec;
        ++seg;
    }
    k.seg = seg;
    k.rec = t / per_rec;
    const int rem = t - k.rec * per_rec;
    k.rb = rem / rp.nchunks;
    k.ch = rem - k.rb * rp.nchunks;
    load_record(rp, sg, k);
    set_row(rp, k, lane, nst);
}

// The task after k, without divisions (called only while one follows).
TQ_DEVFN void task_next(const RowsParams& rp, const RSegs& sg, RTask& k, int lane, int nst) {
    if (++k.ch == rp.nchunks) {
        k.ch = 0;
        if (++k.rb == rp.row_blocks) {
            k.rb = 0;
            if (++k.rec == pick3(sg.cnt, k.seg)) {
                k.rec = 0;
                do ++k.seg;
                while (k.seg < 2 && pick3(sg.cnt, k.seg) == 0);
            }
            load_record(rp, sg, k);
        }
    }
    set_row(rp, k, lane, nst);
}

// Tasks whose start, in the running sum of the task weights, lies below x.
TQ_DEVFN int64_t tasks_below(const RSegs& sg, int64_t per_rec, int64_t x) {
    int64_t n = 0, c = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int64_t ni = (int64_t)sg.cnt[i] * per_rec, wi = seg_weight(i);
        if (x > c) n += min(ni, (x - c + wi - 1) / wi);
        c += ni * wi;
    }
    return n;
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

// MAXNV: the most vectors of a record the instance takes (1: every record has one, and the
// instance holds the one-vector body alone; 4: records of 4, 2 and 1).
template <int LEVELS, int G, int MAXNV>
__global__ void __launch_bounds__(kRThreads, 1) qmv_rows_kernel(const RowsParams rp) {
    using F = RFmt<LEVELS, MAXNV>;
    using U = RUnit<LEVELS, G>;
    constexpr int CW = F::kCW, PW = F::kPW, BITS = F::kBits, SC = F::kSC, D = F::kDepth;
    constexpr int NG = U::kChunkUnits * U::kGroups;  // scale registers
    constexpr int kPieces = SC / 4;                    // 16-byte pieces of one vector's stage values
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
    const uint32_t ring = tab + F::kTabBytes + (uint32_t)(warp * D * F::kStageBytes);
    for (int i = tid; i < F::kTab * 32; i += kRThreads) {
        const int v = i >> 5;
        reinterpret_cast<float2*>(tabp)[i] =
            make_float2(__ldg(p.centroids + (v & (LEVELS - 1))), __ldg(p.centroids + (v >> BITS)));
    }
    __syncthreads();

    // the segments' record counts (from the grouping kernel's lists where they come from there)
    RSegs sg;
#pragma unroll
    for (int i = 0; i < 3; ++i) sg.cnt[i] = rp.count[i] >= 0 ? rp.count[i] : __ldcg(rp.list[i]);
    sg.base[0] = 0;
    sg.base[1] = 4 * sg.cnt[0];
    sg.base[2] = sg.base[1] + 2 * sg.cnt[1];
    const int nst = rp.chunk_units * U::kStages;  // stages per task
    const int64_t per_rec = (int64_t)rp.row_blocks * rp.nchunks;
    int64_t wsum = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) wsum += (int64_t)sg.cnt[i] * per_rec * seg_weight(i);
    const int64_t nw = (int64_t)gridDim.x * kRWarps, gw = (int64_t)blockIdx.x * kRWarps + warp;
    const int ta = (int)tasks_below(sg, per_rec, wsum * gw / nw);
    const int tz = (int)tasks_below(sg, per_rec, wsum * (gw + 1) / nw);
    if (ta >= tz) return;
    const int64_t nstages = (tz - ta) * nst;
    const uint32_t lanetab = tab + (uint32_t)lane * 8u;
    const uint32_t swz = (uint32_t)((lane >> 2) & 1);
    const uint32_t my0 = (uint32_t)lane * 32u + (swz << 4), my1 = (uint32_t)lane * 32u + ((swz ^ 1u) << 4);

    // stream of stages: task ts, stage ss within it
    int ts = ta;
    int ss = 0;
    RTask sk;
    task_of(rp, sg, ta, lane, nst, sk);
    auto issue = [&](int64_t j) {
        const uint32_t dst = ring + (uint32_t)((j % D) * F::kStageBytes);
        const int64_t word0 = (int64_t)sk.ch * nst * 8 + (int64_t)ss * 8;
        const bool rok = !sk.bad && sk.row < p.rows;
        const uint32_t* src = sk.w + ss * 8;
        cp16(dst + my0, src, rok && word0 + 4 <= p.row_stride ? 16u : 0u);
        cp16(dst + my1, src + 4, rok && word0 + 8 <= p.row_stride ? 16u : 0u);
        // the stage's input values of each vector of the record (columns past the row read as
        // zeros; cols is a multiple of 16); an empty slot is left as it is, its sums unused
        const int xcol0 = sk.ch * rp.chunk_units * U::kCodes + ss * SC;
        if constexpr (MAXNV == 1) {
            const int xcol = xcol0 + 4 * lane;
            if (lane < kPieces)
                cp16(dst + kRCodeBytes + 16u * (uint32_t)lane,
                     p.x + (int64_t)sk.vec0 * p.cols + (xcol < p.cols ? xcol : 0), xcol < p.cols ? 16u : 0u);
        } else {
            for (int q = lane; q < sk.nv * kPieces; q += 32) {
                const int v = q / kPieces, c = q - v * kPieces;
                const int pv = v == 0 ? sk.pr[0] : (v == 1 ? sk.pr[1] : (v == 2 ? sk.pr[2] : sk.pr[3]));
                if (pv < 0) continue;
                const int vec = v == 0 ? sk.vec0 : (p.mode == kModeGather ? pv / p.k : pv);
                const int xcol = xcol0 + 4 * c;
                cp16(dst + kRCodeBytes + (uint32_t)(v * F::kXBytes + 16 * c),
                     p.x + (int64_t)vec * p.cols + (xcol < p.cols ? xcol : 0), xcol < p.cols ? 16u : 0u);
            }
        }
        if (++ss == nst) {
            ss = 0;
            if (++ts < tz) task_next(rp, sg, sk, lane, nst);
        }
    };
#pragma unroll
    for (int j = 0; j < D - 1; ++j) {
        if (j < nstages) issue(j);
        commit();
    }

    // scales one task ahead: the loads of task t + 1 are in flight while task t decodes
    float sc[NG], scn[NG];
    RTask k;
    task_of(rp, sg, ta, lane, nst, k);
    task_scales<NG, U::kGroups>(rp, k, scn);
    int64_t j = 0;  // stage being decoded

    // One task of NV vectors: every stage's words decoded once, each pair's table entry
    // multiplied into every vector of the record.
    auto run_task = [&](auto nv_c) {
        constexpr int NV = decltype(nv_c)::value;
        float tot[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) tot[v] = 0.f;
        for (int u = 0; u < rp.chunk_units; ++u) {
            float acc0[NV], acc1[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) acc0[v] = acc1[v] = 0.f;
            static_for<0, U::kStages>([&](auto s_c) {
                constexpr int S = decltype(s_c)::value;
                if (j + D - 1 < nstages) issue(j + D - 1);
                commit();
                wait_group<D - 1>();
                __syncwarp();
                const uint32_t sb = ring + (uint32_t)((j % D) * F::kStageBytes);
                const uint32_t sbx = sb + kRCodeBytes;  // the stage's input values (broadcast reads)
                const uint4 P0 = lds128(sb + my0), P1 = lds128(sb + my1);
                const uint32_t W[8] = {P0.x, P0.y, P0.z, P0.w, P1.x, P1.y, P1.z, P1.w};
                static_for<0, 8>([&](auto w_c) {
                    constexpr int WI = decltype(w_c)::value;
                    const uint32_t w = W[WI];
                    // the word's table entries, one per pair of codes
                    float2 c[PW];
                    static_for<0, PW>([&](auto p_c) {
                        constexpr int PI = decltype(p_c)::value;
                        constexpr int SH = 2 * BITS * PI;  // bit offset of the pair
                        constexpr uint32_t kMask = ((1u << (2 * BITS)) - 1u) << 8;
                        const uint32_t off = (SH >= 8 ? (w >> (SH - 8)) : (w << (8 - SH))) & kMask;
                        c[PI] = lds64f(lanetab | off);
                    });
                    static_for<0, NV>([&](auto v_c) {
                        constexpr int V = decltype(v_c)::value;
                        const uint32_t sxv = sbx + (uint32_t)(V * F::kXBytes);
                        // the word's input values of vector V (every lane reads the same address):
                        // four per load where the column is a multiple of 4, else two
                        float xw[CW];
                        static_for<0, CW / 2>([&](auto q_c) {
                            constexpr int Q = 2 * decltype(q_c)::value;
                            constexpr int kOff = WI * CW + Q;  // column within the stage
                            constexpr bool kQuad = kOff % 4 == 0 && Q + 4 <= CW;
                            if constexpr (kOff % 4 == 2 && Q >= 2) return;  // loaded with the pair before it
                            if constexpr (kQuad) {
                                const uint4 xx = lds128(sxv + 4u * kOff);
                                xw[Q] = __uint_as_float(xx.x);
                                xw[Q + 1] = __uint_as_float(xx.y);
                                xw[Q + 2] = __uint_as_float(xx.z);
                                xw[Q + 3] = __uint_as_float(xx.w);
                            } else {
                                const float2 xx = lds64f(sxv + 4u * kOff);
                                xw[Q] = xx.x;
                                xw[Q + 1] = xx.y;
                            }
                        });
                        static_for<0, PW>([&](auto p_c) {
                            constexpr int PI = decltype(p_c)::value;
                            float& acc = (PI & 1) ? acc1[V] : acc0[V];
                            acc = fmaf(c[PI].x, xw[2 * PI], acc);
                            acc = fmaf(c[PI].y, xw[2 * PI + 1], acc);
                            constexpr int kEnd = S * SC + WI * CW + 2 * PI + 2;  // codes of the unit done
                            if constexpr (kEnd % G == 0) {
                                tot[V] = fmaf(sc[kEnd / G - 1], acc0[V] + acc1[V], tot[V]);
                                acc0[V] = 0.f;
                                acc1[V] = 0.f;
                            }
                        });
                    });
                });
                __syncwarp();  // the slot (codes and input values) is read before a later stage refills it
                ++j;
            });
#pragma unroll
            for (int g = 0; g + U::kGroups < NG; ++g) sc[g] = sc[g + U::kGroups];  // the next unit's scales first
        }
        if (k.row < p.rows) {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                if (k.pr[v] < 0) continue;
                const int64_t o = (int64_t)k.pr[v] * p.rows + k.row;
                if (rp.nchunks == 1) store_from_float(p.y, o, p.ydt, tot[v]);
                else if (rp.atomic_out) atomicAdd(static_cast<float*>(p.y) + o, tot[v]);
                else rp.part[(int64_t)k.ch * rp.n_out * p.rows + o] = tot[v];
            }
        }
    };

    for (int t = ta; t < tz; ++t) {
        if (t > ta) task_next(rp, sg, k, lane, nst);
        if (k.bad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
#pragma unroll
        for (int g = 0; g < NG; ++g) sc[g] = scn[g];
        if (t + 1 < tz) {
            RTask kn = k;
            task_next(rp, sg, kn, lane, nst);
            task_scales<NG, U::kGroups>(rp, kn, scn);
        }
        if constexpr (MAXNV == 1) {
            run_task(std::integral_constant<int, 1>{});
        } else {
            if (k.nv == 4) run_task(std::integral_constant<int, 4>{});
            else if (k.nv == 2) run_task(std::integral_constant<int, 2>{});
            else run_task(std::integral_constant<int, 1>{});
        }
    }
    wait_group<0>();
}

// y[i] = sum over chunks of part[c][i], in chunk order; zero for a pair whose expert id is
// outside the bank (ids non-null; the grouped records never hold such a pair).
__global__ void __launch_bounds__(256) rows_chunk_sum_kernel(const float* __restrict__ part, int nchunks, int64_t n,
                                                             void* y, int ydt, const int32_t* __restrict__ ids,
                                                             int rows, int experts) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        bool bad = false;
        if (ids) {
            const int e = __ldg(ids + i / rows);
            bad = e < 0 || e >= experts;
        }
        if (!bad)
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
// while the tasks (n_rec records) still give every warp of the GPU two or more.
template <int LEVELS, int G>
void plan_chunks(RowsParams& rp, int cols, int64_t n_rec) {
    using U = RUnit<LEVELS, G>;
    rp.units = (cols + U::kCodes - 1) / U::kCodes;
    const int64_t want = 2ll * sm_count_rows() * kRWarps;
    int best = 1;
    int64_t best_dec = -1;
    for (int cu = 1; cu <= U::kChunkUnits; ++cu) {
        const int nch = (rp.units + cu - 1) / cu;
        const int64_t dec = (int64_t)nch * cu;
        const int64_t tasks = n_rec * rp.row_blocks * nch;
        if (tasks < want && cu > 1) break;
        if (best_dec < 0 || dec < best_dec || (dec == best_dec)) {
            best = cu;
            best_dec = dec;
        }
    }
    rp.chunk_units = best;
    rp.nchunks = (rp.units + best - 1) / best;
}

template <int LEVELS, int MAXNV>
size_t rows_smem() {
    using F = RFmt<LEVELS, MAXNV>;
    return (size_t)F::kTabBytes * 2 + (size_t)kRWarps * F::kDepth * F::kStageBytes;
}

template <int LEVELS, int G, int MAXNV>
tq_status rows_kernel_launch(const RowsParams& rp, int grid, cudaStream_t st) {
    const size_t smem = rows_smem<LEVELS, MAXNV>();
    if (ensure_smem((const void*)qmv_rows_kernel<LEVELS, G, MAXNV>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    if (rp.atomic_out) {  // after the output's memset: no programmatic overlap
        qmv_rows_kernel<LEVELS, G, MAXNV><<<grid, kRThreads, smem, st>>>(rp);
        return launch_status();
    }
    return launch_pdl(qmv_rows_kernel<LEVELS, G, MAXNV>, dim3(grid), dim3(kRThreads), smem, st, rp);
}

// Launches the kernel over rp's records (count / list set by the caller), n_rec an upper bound
// of their number, then the chunk sum where the rows take more than one chunk.
template <int LEVELS, int G>
tq_status rows_launch(RowsParams rp, int64_t n_rec, void* ws, size_t ws_bytes, cudaStream_t st) {
    const QmvParams& qp = rp.q;
    rp.row_blocks = (qp.rows + 31) / 32;
    plan_chunks<LEVELS, G>(rp, qp.cols, n_rec);
    const int64_t ntasks = n_rec * rp.row_blocks * rp.nchunks;
    if (ntasks > 0x7fffffffll || ntasks == 0) return TQ_ERR_UNSUPPORTED;
    const int64_t n = (int64_t)rp.n_out * qp.rows;
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
    const int sms = sm_count_rows();
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, (ntasks + kRWarps - 1) / kRWarps));
    // records of one vector only (counts known here, no record lists): the one-vector instance
    const bool single = rp.count[0] == 0 && rp.count[1] == 0;
    const tq_status s = single ? rows_kernel_launch<LEVELS, G, 1>(rp, grid, st)
                               : rows_kernel_launch<LEVELS, G, kRMaxNV>(rp, grid, st);
    if (s != TQ_OK || rp.nchunks == 1 || rp.atomic_out) return s;
    const int32_t* ids = qp.mode == kModeDense ? nullptr : qp.ids;
    return launch_pdl(rows_chunk_sum_kernel, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4 * (int64_t)sms)),
                      dim3(256), 0, st, (const float*)rp.part, rp.nchunks, n, qp.y, qp.ydt, ids, qp.rows,
                      qp.experts);
}

template <int LEVELS>
tq_status rows_g(const RowsParams& rp, int group, int64_t n_rec, void* ws, size_t ws_bytes, cudaStream_t st) {
    switch (group) {
        case 16: return rows_launch<LEVELS, 16>(rp, n_rec, ws, ws_bytes, st);
        case 32: return rows_launch<LEVELS, 32>(rp, n_rec, ws, ws_bytes, st);
        case 64: return rows_launch<LEVELS, 64>(rp, n_rec, ws, ws_bytes, st);
        case 128: return rows_launch<LEVELS, 128>(rp, n_rec, ws, ws_bytes, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

tq_status rows_dispatch(const RowsParams& rp, int group, int64_t n_rec, void* ws, size_t ws_bytes, cudaStream_t st) {
    switch (rp.q.levels) {
        case 4: return qmv_rows_launch_l4(rp, group, n_rec, ws, ws_bytes, st);
        case 8: return qmv_rows_launch_l8(rp, group, n_rec, ws, ws_bytes, st);
        case 16: return qmv_rows_launch_l16(rp, group, n_rec, ws, ws_bytes, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

template <int LEVELS, int G>
size_t rows_ws(int cols, int64_t n_items, int rows) {
    RowsParams rp{};
    rp.row_blocks = (rows + 31) / 32;
    plan_chunks<LEVELS, G>(rp, cols, n_items);
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

#define TQ_ROWS_LAUNCHER(L)                                                                             \
    tq_status qmv_rows_launch_l##L(const RowsParams& rp, int group, int64_t n_rec, void* ws, size_t ws_bytes, \
                                   cudaStream_t st) {                                                   \
        return rows_g<L>(rp, group, n_rec, ws, ws_bytes, st);                                           \
    }
#if defined(TQ_ROWS_ALL) || TQ_ROWS_LEVELS == 4
TQ_ROWS_LAUNCHER(4)
#endif
#if defined(TQ_ROWS_ALL) || TQ_ROWS_LEVELS == 8
TQ_ROWS_LAUNCHER(8)
#endif
#if defined(TQ_ROWS_ALL) || TQ_ROWS_LEVELS == 16
TQ_ROWS_LAUNCHER(16)
#endif
#undef TQ_ROWS_LAUNCHER

#if defined(TQ_ROWS_ALL) || TQ_ROWS_LEVELS == 0
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
    if (n_items <= 0) return TQ_ERR_UNSUPPORTED;
    RowsParams rp{};
    rp.q = p;
    rp.n_out = n_items;
    if (p.mode == kModeDense) {  // the vectors of one matrix, four at a time, then two, then one
        rp.count[0] = n_items / 4;
        rp.count[1] = (n_items % 4) / 2;
        rp.count[2] = n_items % 2;
    } else {  // one pair per record, each of its own expert
        rp.count[2] = n_items;
    }
    const int64_t n_rec = (int64_t)rp.count[0] + rp.count[1] + rp.count[2];
    return rows_dispatch(rp, group, n_rec, ws, ws_bytes, st);
}

tq_status qmv_rows_run_groups(const QmvParams& p, int group, const int32_t* const lists[3], int P, void* ws,
                              size_t ws_bytes, cudaStream_t st) {
    if (P <= 0 || p.mode == kModeDense) return TQ_ERR_UNSUPPORTED;
    RowsParams rp{};
    rp.q = p;
    rp.n_out = P;
    for (int i = 0; i < 3; ++i) {
        rp.count[i] = -1;
        rp.list[i] = lists[i];
    }
    return rows_dispatch(rp, group, P, ws, ws_bytes, st);
}
#endif

}  // namespace tq
