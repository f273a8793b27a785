// Bit-packed inline-decode matvec (2-, 3- and 4-bit books, one input vector
// per item): the kernel behind tq_qmv / tq_gather_qmv / tq_multi_gather_qmv
// when the scale rows are whole 16-byte chunks.
//
// "How it works", "Quantizing a weight" (codes packed into 32-bit words) and
// "Running a quantized layer" (the rotated input times the codes, decoded
// inline).
//
// Work layout (the same as the ternary kernel).  A warp takes 4 rows of one
// item and walks their columns in stages of 8 chunks; a chunk is a whole
// number of lcm(codes per word, group) units and at least 4 words, so group
// boundaries sit at compile-time positions.  Lane (r, c) decodes chunk c of
// the stage for row r; the copies interleave 16-byte pieces over the lanes so
// that one instruction covers 128 contiguous bytes of each of 4 rows.  Codes and scales stream through a 2-slot per-warp
// cp.async ring (the next stage is issued before the current one is decoded);
// the input is copied once per CTA and distinct vector into shared blocks, one
// per chunk, whose starts fall on distinct 4-bank groups, so the 8 chunks in
// flight are read without conflicts (the 4 rows of a chunk share a broadcast).
// Decode: with 2- and 3-bit codes a pair of codes indexes a per-lane table of
// float2 (c[lo], c[hi]), with 4-bit codes each code a per-lane float table; the
// products accumulate per group and are scaled once per group.
#include <type_traits>

#include "qmv_impl.cuh"

namespace tq {
namespace {

template <int LEVELS, int G>
struct BitsFmt {
    static constexpr int kBits = LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4);
    static constexpr int kCW = LEVELS == 8 ? 10 : 32 / kBits;  // codes per word
    static constexpr int kUC = kCW / Gcd<kCW, G>::v * G;       // codes per unit: lcm(codes per word, G)
    static constexpr int kUW = kUC / kCW;                       // words per unit
    static constexpr int kChW = kUW >= 4 ? kUW : 4;             // words per chunk
    static constexpr int kChC = kChW * kCW;                     // codes per chunk
    static constexpr int kGPC = kChC / G;                       // groups per chunk
    static constexpr bool kPair = kBits <= 3;                   // two codes per table entry
    static constexpr int kTab = kPair ? (1 << (2 * kBits)) : LEVELS;  // table entries
    static constexpr int kXS = (kChC + 31) / 32 * 32 + 4;       // floats per input block (= 4 mod 32 words)
    static constexpr int kXQ = kCW == 10 ? 2 : 1;               // words per 16-byte-aligned input step
    static constexpr int kSUB = kChW > 16 ? kChW / 16 : 1;      // stages (parts) per chunk
    static constexpr int kPW = kChW / kSUB;                     // words per part
    static constexpr int kPPC = kPW / 4;                        // 16-byte pieces per part
    static_assert(kChW % 4 == 0 && kChC % G == 0 && kGPC <= 8 && kPW % 4 == 0, "chunk shape");
};

constexpr int kRPW = 4, kUPW = 8, kNS = 3;

// Position of 16-byte piece P of a row's stage span in shared memory.  A chunk holds PPC
// pieces; XOR-ing the low bits of P with a function of its chunk puts piece i of the 8
// chunks on 8 different 16-byte bank groups, so the lanes reading piece i of their own
// chunks (the 4 rows of a chunk excepted) are conflict-free.
template <int PPC>
TQ_DEVFN int swz_piece(int P) {
    const int ch = P / PPC;
    if constexpr (PPC >= 8) return P ^ (ch & 7);
    else return P ^ (ch / (8 / PPC) & (PPC - 1));
}

template <int LEVELS, int G>
struct BitsStage {
    using F = BitsFmt<LEVELS, G>;
    static constexpr int kCodeRow = kUPW * F::kPW * 4;    // code bytes per row and stage (one part of 8 chunks)
    static constexpr int kScaleRow = kUPW * F::kGPC * 2;  // scale bytes per row and stage (16 * groups per chunk)
    static constexpr int kStage = kRPW * (kCodeRow + kScaleRow);
};

TQ_DEVFN uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
TQ_DEVFN void cp16(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr(dst)), "l"(src), "r"(bytes) : "memory");
}
TQ_DEVFN void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
TQ_DEVFN void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct BitsParams {
    QmvParams q;
    int nchunks;  // chunks per row
    int nsteps;   // stages of 8 chunks per row
    int tasks_per_item;
    int n_items;
    int total_tasks;
};

template <int LEVELS, int G>
__global__ void __launch_bounds__(256, 2) qmv_bits_kernel(const BitsParams bp) {
    using F = BitsFmt<LEVELS, G>;
    using B = BitsStage<LEVELS, G>;
    constexpr int RPW = kRPW, UPW = kUPW, NS = kNS;
    constexpr int ChW = F::kChW, ChC = F::kChC, GPC = F::kGPC, CW = F::kCW, XS = F::kXS, BITS = F::kBits;
    constexpr int nwarps = 8;
    const QmvParams& p = bp.q;
    extern __shared__ __align__(16) uint32_t sm[];
    // per-lane table: entry v of lane l at [v][l] (float2 pairs, or floats for 4-bit codes)
    uint32_t* lut = sm;
    constexpr int kLutWords = F::kTab * 32 * (F::kPair ? 2 : 1);
    float* xb = reinterpret_cast<float*>(lut + kLutWords);  // [nsteps * 8 chunks][XS]
    const int nchunk_pad = bp.nsteps * UPW;
    uint8_t* ring0 = reinterpret_cast<uint8_t*>(xb + nchunk_pad * XS);        // [8 warps][NS][stage]
    float* rowsum = reinterpret_cast<float*>(ring0 + nwarps * NS * B::kStage);  // [max tasks per CTA][RPW]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ float cbk[LEVELS];  // the codebook, read from global memory once
    if (tid < LEVELS) cbk[tid] = __ldg(p.centroids + tid);
    __syncthreads();
    for (int i = tid; i < F::kTab * 32; i += blockDim.x) {
        const int v = i >> 5;
        if constexpr (F::kPair) {
            reinterpret_cast<float2*>(lut)[i] = make_float2(cbk[v & (LEVELS - 1)], cbk[v >> BITS]);
        } else {
            reinterpret_cast<float*>(lut)[i] = cbk[v];
        }
    }
    constexpr int SUB = F::kSUB, PW = F::kPW, PPC = F::kPPC;
    const int t_begin = (int)((int64_t)blockIdx.x * bp.total_tasks / gridDim.x);
    const int t_end = (int)((int64_t)(blockIdx.x + 1) * bp.total_tasks / gridDim.x);
    const int r = lane / UPW, c = lane % UPW;
    const uint32_t lut_lane = saddr(lut) + lane * (F::kPair ? 8 : 4);
    const int ngroups = p.ngroups;
    const int nsc = bp.nsteps;  // chunk stages (of 8 chunks) per task; each is SUB part stages
    const int tpi = bp.tasks_per_item;
    const int rs32 = (int)p.row_stride;
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

        // This warp's share: a contiguous range of part stages (SUB per chunk stage, nsc chunk
        // stages per task); a share may start or end inside a chunk stage.
        const int nps = nsc * SUB;  // part stages per task
        const int nparts_seg = (s1 - s0) * nps;
        const int f_begin = (int)((int64_t)warp * nparts_seg / nwarps);
        const int f_end = (int)((int64_t)(warp + 1) * nparts_seg / nwarps);
        const int L = f_end - f_begin;  // part stages

        // producer: task pt, chunk stage pcs, part pp
        int pt = s0 + f_begin / nps, pcs = (f_begin % nps) / SUB, pp = f_begin % SUB, pslot = 0;
        const uint32_t* pcode = nullptr;
        const uint16_t* pscale = nullptr;
        auto set_prod_task = [&]() {
            int e, v;
            item_info(pt / tpi, e, v);
            if (e < 0 || e >= p.experts) e = 0;  // rows of a bad id are summed as zero below
            const int row = min((pt % tpi) * RPW + r, p.rows - 1);
            pcode = p.codes + (int64_t)e * p.expert_stride_w + (int64_t)row * p.row_stride;
            pscale = p.scales + (int64_t)e * p.expert_stride_s + (int64_t)row * ngroups;
        };
        if (L > 0) set_prod_task();
        auto issue = [&]() {
            uint8_t* dst = ring + pslot * B::kStage;
            // part pp of the stage's 8 chunks of the row, 8 * PPC pieces of 16 bytes, lane c taking
            // pieces c, c + 8, ...: one instruction covers 8 consecutive pieces (whole parts of
            // consecutive chunks) of each of the 4 rows; a lane's own part arrives through the
            // other lanes' copies (the warp syncs before decoding)
#pragma unroll
            for (int i = 0; i < PPC; ++i) {
                const int P = c + 8 * i, ch = P / PPC, ip = P - ch * PPC;
                const int wi = (pcs * UPW + ch) * ChW + pp * PW + 4 * ip;
                const bool in = wi < rs32;  // past the padded row: zero
                cp16(dst + r * B::kCodeRow + swz_piece<PPC>(P) * 16, pcode + (in ? wi : 0), in ? 16u : 0u);
            }
            if (c < GPC) {  // the stage's scales of the row: GPC pieces of 8 groups
                const int g0 = pcs * UPW * GPC + c * 8;
                const bool in = g0 < ngroups;  // scale rows are whole 16-byte chunks
                cp16(dst + RPW * B::kCodeRow + r * B::kScaleRow + c * 16, pscale + (in ? g0 : 0), in ? 16u : 0u);
            }
            cp_commit();
            pslot = pslot + 1 == NS ? 0 : pslot + 1;
            if (++pp == SUB) {
                pp = 0;
                if (++pcs == nsc) {
                    pcs = 0;
                    ++pt;
                    if (pt < s1) set_prod_task();
                }
            }
        };
        for (int j = 0; j < NS - 1; ++j) {
            if (j < L) issue(); else cp_commit();
        }

        for (int i = tid; i < (s1 - s0) * RPW; i += blockDim.x) rowsum[i] = 0.f;
        if (vec != cur_vec) {
            // The input vector, chunk by chunk, zero past the last column: four floats per thread
            // and step (chunks hold a multiple of 4 codes), the loads of a few steps in flight
            // before their stores.
            const float* xv = p.x + (int64_t)vec * p.cols;
            const bool x16 = (reinterpret_cast<uintptr_t>(xv) & 15) == 0;
            const int n4 = nchunk_pad * ChC / 4;
            for (int i0 = tid; i0 < n4; i0 += 4 * blockDim.x) {
                float4 v[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int i = 4 * (i0 + t * blockDim.x);
                    if (x16 && i + 3 < p.cols) {
                        v[t] = __ldg(reinterpret_cast<const float4*>(xv + i));
                    } else {
                        v[t].x = i < p.cols ? __ldg(xv + i) : 0.f;
                        v[t].y = i + 1 < p.cols ? __ldg(xv + i + 1) : 0.f;
                        v[t].z = i + 2 < p.cols ? __ldg(xv + i + 2) : 0.f;
                        v[t].w = i + 3 < p.cols ? __ldg(xv + i + 3) : 0.f;
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int i4 = i0 + t * blockDim.x;
                    if (i4 < n4) {
                        const int u = 4 * i4 / ChC, jj = 4 * i4 - u * ChC;
                        *reinterpret_cast<float4*>(xb + u * XS + jj) = v[t];
                    }
                }
            }
            cur_vec = vec;
        }
        __syncthreads();

        int ct = s0 + f_begin / nps, ccs = (f_begin % nps) / SUB, cpart = f_begin % SUB, cslot = 0;
        bool cbad;
        {
            int e, v;
            item_info(ct / tpi, e, v);
            cbad = e < 0 || e >= p.experts;
            if (cbad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
        }
        float tot = 0.f;
        float acc[GPC];
#pragma unroll
        for (int g = 0; g < GPC; ++g) acc[g] = 0.f;  // a share may start inside a chunk stage
        for (int j = 0; j < L; ++j) {
            cp_wait<NS - 2>();  // stage j has landed
            __syncwarp();       // and every lane is done with the slot of stage j - 1
            if (j + NS - 1 < L) issue(); else cp_commit();
            const uint8_t* stg = ring + cslot * B::kStage;
            const uint8_t* wrow = stg + r * B::kCodeRow;  // this lane's part: pieces c * PPC + i, swizzled
            const float* xc = xb + (ccs * UPW + c) * XS;   // zero past the row's last chunk
            if (cpart == 0) {
#pragma unroll
                for (int g = 0; g < GPC; ++g) acc[g] = 0.f;
            }
            // Part PART of this lane's chunk: words PART * PW .. + PW - 1, groups at compile-time
            // positions (the part index is the same for the whole warp).
            auto decode_part = [&](auto part_c) {
                constexpr int PART = decltype(part_c)::value;
                static_for<0, PPC>([&](auto qc) {
                    constexpr int q = decltype(qc)::value * 4;  // word in the part
                    const uint4 wq = *reinterpret_cast<const uint4*>(wrow + swz_piece<PPC>(c * PPC + q / 4) * 16);
                    const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int w2 = 0; w2 < 4; w2 += F::kXQ) {
                        constexpr int NX = F::kXQ * CW;
                        float xv[NX];
                        const int wc = PART * PW + q + w2;  // word in the chunk
#pragma unroll
                        for (int t = 0; t < NX; t += 4) {
                            const float4 x4 = *reinterpret_cast<const float4*>(xc + wc * CW + t);
                            xv[t] = x4.x;
                            xv[t + 1] = x4.y;
                            xv[t + 2] = x4.z;
                            xv[t + 3] = x4.w;
                        }
#pragma unroll
                        for (int wi = 0; wi < F::kXQ; ++wi) {
                            // one word's products on their own (independent chains across words),
                            // split where a group boundary falls inside the word (3-bit codes only)
                            const uint32_t word = wv[w2 + wi];
                            const int j0 = (wc + wi) * CW;  // first code of the word in the chunk
                            const int g0 = j0 / G;
                            float ws[2] = {0.f, 0.f};
                            if constexpr (F::kPair) {
#pragma unroll
                                for (int pr = 0; pr < CW / 2; ++pr) {
                                    const int jc = j0 + 2 * pr;
                                    const uint32_t idx = (word >> (2 * BITS * pr)) & ((1u << (2 * BITS)) - 1u);
                                    float2 cc;
                                    asm("ld.shared.v2.f32 {%0, %1}, [%2];"
                                        : "=f"(cc.x), "=f"(cc.y)
                                        : "r"(lut_lane + idx * 256u));
                                    ws[jc / G - g0] = fmaf(cc.x, xv[wi * CW + 2 * pr], ws[jc / G - g0]);
                                    ws[jc / G - g0] = fmaf(cc.y, xv[wi * CW + 2 * pr + 1], ws[jc / G - g0]);
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < CW; ++k) {
                                    const int jc = j0 + k;
                                    const uint32_t idx = (word >> (BITS * k)) & ((1u << BITS) - 1u);
                                    float cv;
                                    asm("ld.shared.f32 %0, [%1];" : "=f"(cv) : "r"(lut_lane + idx * 128u));
                                    ws[jc / G - g0] = fmaf(cv, xv[wi * CW + k], ws[jc / G - g0]);
                                }
                            }
                            acc[g0] += ws[0];
                            if ((j0 + CW - 1) / G != g0) acc[g0 + 1] += ws[1];
                        }
                    }
                });
            };
            if constexpr (SUB == 1) {
                decode_part(std::integral_constant<int, 0>{});
            } else {
                static_for<0, SUB>([&](auto pc) {
                    if (cpart == decltype(pc)::value) decode_part(pc);
                });
            }
            const bool last = j == L - 1;
            if (cpart == SUB - 1 || last) {  // the chunk stage's (or this share's) group sums, scaled
                const uint16_t* ssrc =
                    reinterpret_cast<const uint16_t*>(stg + RPW * B::kCodeRow + r * B::kScaleRow) + c * GPC;
#pragma unroll
                for (int g = 0; g < GPC; ++g) tot = fmaf(half_bits_to_float(ssrc[g]), acc[g], tot);
            }
            cslot = cslot + 1 == NS ? 0 : cslot + 1;
            const bool stage_end = ++cpart == SUB;
            if (stage_end) {
                cpart = 0;
                ++ccs;
            }
            const bool task_end = stage_end && ccs == nsc;
            if (task_end || last) {  // task finished or this warp's share ends: add the row sums
                float v = cbad ? 0.f : tot;
#pragma unroll
                for (int m = 1; m < UPW; m <<= 1) v += __shfl_xor_sync(kFull, v, m);
                if (c == 0) atomicAdd(rowsum + (ct - s0) * RPW + r, v);
                tot = 0.f;
            }
            if (task_end) {
                ccs = 0;
                ++ct;
                if (ct < s1) {
                    int e, vv;
                    item_info(ct / tpi, e, vv);
                    cbad = e < 0 || e >= p.experts;
                    if (cbad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
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

template <int LEVELS, int G>
tq_status launch_bits(const QmvParams& qp, int n_items, cudaStream_t st) {
    using F = BitsFmt<LEVELS, G>;
    using B = BitsStage<LEVELS, G>;
    BitsParams bp{};
    bp.q = qp;
    bp.nchunks = (qp.cols + F::kChC - 1) / F::kChC;
    bp.nsteps = (bp.nchunks + kUPW - 1) / kUPW;
    bp.tasks_per_item = (qp.rows + kRPW - 1) / kRPW;
    bp.n_items = n_items;
    const int64_t total = (int64_t)n_items * bp.tasks_per_item;
    if (total > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    bp.total_tasks = (int)total;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const size_t lut_bytes = (size_t)F::kTab * 32 * (F::kPair ? 8 : 4);
    const size_t smem_fixed = lut_bytes + (size_t)bp.nsteps * kUPW * F::kXS * 4 + (size_t)8 * kNS * B::kStage;
    const void* kfn = (const void*)qmv_bits_kernel<LEVELS, G>;
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
        const int max_tasks = (int)((total + g - 1) / g) + 1;
        const size_t need = smem_fixed + (size_t)max_tasks * kRPW * 4;
        if (need > 220 * 1024) continue;
        if (ensure_smem(kfn, need) != cudaSuccess) return TQ_ERR_CUDA;
        int fit = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, qmv_bits_kernel<LEVELS, G>, 256, need) != cudaSuccess)
            return TQ_ERR_CUDA;
        if (fit >= per_sm || per_sm == 1) {
            grid = g;
            smem = need;
        }
    }
    if (grid == 0) return TQ_ERR_UNSUPPORTED;
    qmv_bits_kernel<LEVELS, G><<<(unsigned)grid, 256, smem, st>>>(bp);
    return launch_status();
}

template <int LEVELS>
tq_status bits_g(const QmvParams& p, int group, int n_items, cudaStream_t st) {
    switch (group) {
        case 16: return launch_bits<LEVELS, 16>(p, n_items, st);
        case 32: return launch_bits<LEVELS, 32>(p, n_items, st);
        case 64: return launch_bits<LEVELS, 64>(p, n_items, st);
        case 128: return launch_bits<LEVELS, 128>(p, n_items, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace

// Staged bit-packed pipeline when every copy is 16-byte aligned: code rows
// (always, row strides are whole 16-byte chunks), scale rows and expert scale
// strides in whole 16-byte chunks (group counts a multiple of 8).
bool qmv_bits_ok(const QmvParams& p, int group) {
    return (p.levels == 4 || p.levels == 8 || p.levels == 16) &&
           (group == 16 || group == 32 || group == 64 || group == 128) && p.ngroups % 8 == 0 &&
           p.expert_stride_s % 8 == 0 && (reinterpret_cast<uintptr_t>(p.scales) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(p.codes) & 15) == 0 && p.row_stride < (1 << 30);
}

tq_status qmv_bits_run(const QmvParams& p, int group, int n_items, cudaStream_t st) {
    switch (p.levels) {
        case 4: return bits_g<4>(p, group, n_items, st);
        case 8: return bits_g<8>(p, group, n_items, st);
        case 16: return bits_g<16>(p, group, n_items, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}

}  // namespace tq
