// Ternary matvec by table lookup: the decode kernel behind tq_gather_qmv and
// tq_multi_gather_qmv for symmetric three-level books {-c, 0, +c}, group 16.
//
// "How it works", "The ternary tier (1.58 bits)": 20 trits per 32-bit word in
// base 3 (digit j of weight 3^j); "Running a quantized layer": the rotated
// input times the packed codes, decoded inline (no per-weight division).
//
// Arithmetic.  A word is read as five chunks of four consecutive trits (base-81
// digits: trits 0-3, 4-7, 8-11, 12-15, 16-19).  For the input vector x the CTA
// builds, for every chunk position p of its slice of columns and every chunk
// value d in [0, 81), the partial dot product
//     e(p, d) = sum_{j<4} (digit_j(d) - 1) * xq[4p + j],
// where xq is x quantized to integers per group of 16 columns (x ~= xs_g * xq,
// xs_g = max|x| / 8191 over the group, so |e| <= 4 * 8191 fits 16 bits).  A
// weight group (16 trits = 4 chunks) then costs four table reads and two
// integer adds:  sum_k t_k x_k = xs_g * sum_{chunks} e(p, d_p)  exactly in
// integers, and the row result is  c * sum_g s_g * xs_g * (that sum).
//
// Table layout (GB300 shared memory, 32 banks).  Lane l of every warp owns unit l
// (80 columns = 4 words = 5 groups) of the slice, so the 32 lanes of one lookup
// read 32 different chunk positions: entry (unit u, position i, value d) lives in
// bank u, and a warp's lookup is one conflict-free wavefront whatever the digits.
// Word ((i mod 10) * 81 + d) * 32 + u holds position i (< 10) in its low half and
// position i + 10 in its high half, biased by 2^15.  One slice is 32 units =
// 2560 columns (101 KB of table); wider rows are split into slices handled by
// different CTAs, whose partial sums a second kernel adds.
//
// Digits.  w = u * 3^12 + v: u = mulhi(w, ceil(2^51 / 3^12)) >> 19, exact for every
// w < 3^20 (the multiplier's excess over 2^51 / 3^12 times 3^20 stays below 2^51 / 3^12);
// v < 3^12 holds chunks 0-2 and u < 3^8 chunks 3-4, split by multiply-highs with
// ceil(2^32 / 6561) and ceil(2^32 / 81) (exact for these ranges, checked for every
// value) and multiply-subtracts.  A chunk's table address is the lane's base + 128 d.
//
// Pipeline.  One persistent CTA per SM, 16 warps, all decoding.  Each warp streams
// its own stages (2 rows x one slice: 1 KB of code words, 640 B of scales) with
// 16-byte cp.async copies into a private ring of 4 stages, 3 in flight while it
// decodes one; words, groups, rows and expert ids outside the bank are filled
// with zeros.  (A single producer warp issuing tensor copies of such small boxes
// could not keep up: measured with the decode removed, the copies alone ran at
// 2.8 TB/s.)  The first stages are requested before the table is built, so the
// build overlaps their latency.
#include <algorithm>

#include "qmv_impl.cuh"
#include "route.cuh"

namespace tq {
namespace {

constexpr int kLWarps = 16;                          // warps, every one decoding
constexpr int kLThreads = 32 * kLWarps;
constexpr int kLDepth = 4;                           // ring stages per warp (3 in flight)
constexpr int kLRows = 2;                            // rows per stage
constexpr int kLUnits = 32;                          // units per slice, one per lane
constexpr int kLSliceCols = kLUnits * 80;            // 2560
constexpr int kLSliceWords = kLUnits * 4;            // 128
constexpr int kLSliceGroups = kLUnits * 5;           // 160
constexpr int kLCodeRow = kLSliceWords * 4;          // 512 bytes of codes per row
constexpr int kLScaleRow = kLSliceGroups * 2;        // 320 bytes of scales per row
constexpr int kLStage = kLRows * (kLCodeRow + kLScaleRow);  // 1664
constexpr int kLTableWords = 10 * 81 * 32;
constexpr int kLQ = 8191;                            // |xq| <= 8191 per group
constexpr uint32_t kMBits = 0x4B400000u;             // bits of 1.5 * 2^23

// Shared-memory carve-up (byte offsets from a 128-byte aligned base).
constexpr size_t kOffTable = 0;
constexpr size_t kOffRing = kOffTable + (size_t)kLTableWords * 4;
constexpr size_t kOffXq = kOffRing + (size_t)kLWarps * kLDepth * kLStage;
constexpr size_t kOffXs = kOffXq + (size_t)kLSliceCols * 2;
constexpr size_t kLSmem = kOffXs + (size_t)kLSliceGroups * 8 + 128;  // xs_g and group sums; + alignment slack

struct LutParams {
    QmvParams q;
    int nslices;        // column slices of 32 units
    int row_tasks;      // ceil(rows / 4)
    int n_items;
    int cta_per_slice;
    float* part;        // [nslices][n_items * rows] when nslices > 1, else unused (y written directly)
};

// 16-bit shared load zero-extended into a 32-bit register.
template <int D>
TQ_DEVFN uint32_t lds_u16(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1+%2];" : "=r"(v) : "r"(a), "n"(D));
    return v;
}
TQ_DEVFN uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
TQ_DEVFN uint4 lds_u4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
TQ_DEVFN uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
TQ_DEVFN uint32_t iadd3(uint32_t a, uint32_t b, uint32_t c) { return a + b + c; }

// 16-byte global -> shared copy; src_bytes 0 writes zeros (src is then not read).
TQ_DEVFN void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
TQ_DEVFN void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
TQ_DEVFN void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Table entry of chunk position P (0..19 within the lane's unit) at address a = lane base + 128 d.
template <int P>
TQ_DEVFN uint32_t lut_lookup(uint32_t a) {
    constexpr int kImm = (P % 10) * 81 * 128 + (P >= 10 ? 2 : 0);
    return lds_u16<kImm>(a);
}

// Table addresses of the five chunks of a word: a[i] = tb + 128 * (trits 4i..4i+3 as a base-81 digit).
TQ_DEVFN void chunk_addrs(uint32_t w, uint32_t tb, uint32_t (&a)[5]) {
    const uint32_t u = __umulhi(w, 4237158620u) >> 19;  // w / 3^12, exact for every w < 3^20
    const uint32_t v = w - u * 531441u;            // trits 0..11
    const uint32_t c4 = __umulhi(u, 53024288u);    // u / 81
    const uint32_t c3 = u - 81u * c4;
    const uint32_t c2 = __umulhi(v, 654621u);      // v / 6561
    const uint32_t r = v - 6561u * c2;
    const uint32_t c1 = __umulhi(r, 53024288u);    // r / 81
    const uint32_t c0 = r - 81u * c1;
    a[0] = tb + (c0 << 7);
    a[1] = tb + (c1 << 7);
    a[2] = tb + (c2 << 7);
    a[3] = tb + (c3 << 7);
    a[4] = tb + (c4 << 7);
}

// One unit-row: four words against the lane's table column.  Returns sum_g s_g xs_g S_g, S_g the
// group's integer dot product.
TQ_DEVFN float unit_row(const uint4 q, uint32_t tb, const float (&s)[5], const float (&xs)[5]) {
    uint32_t a[4][5];
    chunk_addrs(q.x, tb, a[0]);
    chunk_addrs(q.y, tb, a[1]);
    chunk_addrs(q.z, tb, a[2]);
    chunk_addrs(q.w, tb, a[3]);
    // chunk position P = 5 W + i belongs to group P / 4; pairs of chunks of one group are added
    // together; each group sum starts at the bits of 1.5 * 2^23
    uint32_t acc[5];
    static_for<0, 10>([&](auto k_c) {
        constexpr int k = decltype(k_c)::value;
        constexpr int P0 = 2 * k, P1 = 2 * k + 1;
        const uint32_t e0 = lut_lookup<P0>(a[P0 / 5][P0 % 5]);
        const uint32_t e1 = lut_lookup<P1>(a[P1 / 5][P1 % 5]);
        acc[P0 / 4] = iadd3(k % 2 == 0 ? kMBits : acc[P0 / 4], e0, e1);
    });
    float tot = 0.f;
#pragma unroll
    for (int g = 0; g < 5; ++g) {
        // acc = bits of 1.5 * 2^23 + sum(e + 2^15) over the group's four chunks (< 2^22)
        const float v = __uint_as_float(acc[g]) - (12582912.0f + 131072.0f);
        tot = fmaf(s[g] * xs[g], v, tot);
    }
    return tot;
}

// The five fp16 scales of the lane's unit in one row: 10 bytes at byte offset 10 * lane.
TQ_DEVFN void lane_scales(uint32_t a, uint32_t sh, float (&s)[5]) {
    const uint32_t w0 = lds_u32(a), w1 = lds_u32(a + 4), w2 = lds_u32(a + 8);
    const uint32_t v0 = __funnelshift_r(w0, w1, sh), v1 = __funnelshift_r(w1, w2, sh), v2 = w2 >> sh;
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v0));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v1));
    s[0] = f0.x;
    s[1] = f0.y;
    s[2] = f1.x;
    s[3] = f1.y;
    s[4] = __low2float(*reinterpret_cast<const __half2*>(&v2));
}

// Stream state of one warp: the next stage to request.
struct LutStream {
    const uint32_t* c;  // code words of row `row` of the item's expert (this lane's piece)
    const uint16_t* s;  // scales of that row (this lane's piece)
    int item, row;
    bool bad;           // expert id outside the bank: the stage reads as zeros
};

// Point the stream at `row` of `item` (reads the item's expert id; COH: through L2, for ids
// written earlier by the same launch).
template <bool COH>
TQ_DEVFN void lut_seek(LutStream& st, const QmvParams& p, int item, int row, int64_t wofs, int64_t gofs, int lane) {
    st.item = item;
    st.row = row;
    const int e = p.mode == kModeDense ? 0 : (COH ? __ldcg(p.ids + item) : __ldg(p.ids + item));
    st.bad = e < 0 || e >= p.experts;
    if (st.bad && lane == 0 && p.err) atomicOr(p.err, TQ_DEVERR_BAD_ID);
    const int64_t ee = st.bad ? 0 : e;
    st.c = p.codes + ee * p.expert_stride_w + (int64_t)row * p.row_stride + wofs;
    st.s = p.scales + ee * p.expert_stride_s + (int64_t)row * p.ngroups + gofs;
}

// Request the stream's next stage (2 rows) into the ring slot at shared address dst, then advance.
template <bool COH>
TQ_DEVFN void lut_issue(LutStream& st, const QmvParams& p, int n_items, int rt_n, uint32_t dst, bool wok, bool gok,
                        int64_t wofs, int64_t gofs, int lane) {
#pragma unroll
    for (int r = 0; r < kLRows; ++r) {
        const bool rok = !st.bad && st.row + r < p.rows;
        cp_async16(dst + r * kLCodeRow + lane * 16, st.c + r * p.row_stride, rok && wok ? 16u : 0u);
        if (lane < kLScaleRow / 16)
            cp_async16(dst + kLRows * kLCodeRow + r * kLScaleRow + lane * 16, st.s + r * p.ngroups,
                       rok && gok ? 16u : 0u);
    }
    st.row += kLRows;
    if (st.row >= rt_n * kLRows) {
        if (st.item + 1 < n_items) lut_seek<COH>(st, p, st.item + 1, 0, wofs, gofs, lane);
    } else {
        st.c += kLRows * p.row_stride;
        st.s += kLRows * p.ngroups;
    }
}

// The matvec of CTA `cta` of the launch (the table-lookup kernel, or a phase of the fused decode
// layer).  sm: the 128-byte aligned shared memory of the layout above.  COH: the ids and the
// input were written earlier by the same launch, so they are read through L2.
template <bool COH>
TQ_DEVFN void lut_body(const LutParams& lp, uint8_t* sm, int cta) {
    const QmvParams& p = lp.q;
    uint32_t* table = reinterpret_cast<uint32_t*>(sm + kOffTable);
    int16_t* xq = reinterpret_cast<int16_t*>(sm + kOffXq);
    float* xsg = reinterpret_cast<float*>(sm + kOffXs);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = cta / lp.cta_per_slice, cb = cta - slice * lp.cta_per_slice;
    const int rt_n = lp.row_tasks, n_items = lp.n_items;
    const int64_t ntasks = (int64_t)n_items * rt_n;
    const int t_begin = (int)(cb * ntasks / lp.cta_per_slice);
    const int t_end = (int)((cb + 1) * ntasks / lp.cta_per_slice);
    const int kper = p.mode == kModeGather ? p.k : 1;  // items per input vector

    // three-level book c[d] = c1 + (d - 1) delta: sum_k c[d_k] x_k = delta sum_k t_k x_k + c1 sum_k x_k
    const float c1 = __ldg(p.centroids + 1), delta = __ldg(p.centroids + 2) - c1;
    if (tid == 0 && cb == 0 && p.err && fabsf((c1 - __ldg(p.centroids)) - delta) > 1e-6f * fabsf(delta))
        atomicOr(p.err, TQ_DEVERR_BAD_BOOK);
    const bool has_off = c1 != 0.f;  // uniform
    const int col0 = slice * kLSliceCols;
    const uint32_t tb = smem_u32(table) + (uint32_t)lane * 4u;
    const uint32_t ring = smem_u32(sm + kOffRing) + (uint32_t)(warp * kLDepth * kLStage);
    const uint32_t soff = (uint32_t)((10 * lane) & ~3), ssh = (uint32_t)(lane & 1) * 16u;
    // this lane's 16-byte pieces: code words 4 lane.. of the slice, scale piece `lane` (lanes < 20)
    const int64_t wofs_raw = (int64_t)slice * kLSliceWords + 4 * lane;
    const int64_t gofs_raw = (int64_t)slice * kLSliceGroups + 8 * lane;
    const bool wok = wofs_raw < p.row_stride, gok = lane < kLScaleRow / 16 && gofs_raw < p.ngroups;
    const int64_t wofs = wok ? wofs_raw : 0, gofs = gok ? gofs_raw : 0;
    float xs[5] = {0.f, 0.f, 0.f, 0.f, 0.f}, xsum[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
    int cur_vec = -1;
    LutStream st{p.codes, p.scales, 0, 0, false};

    for (int s0 = t_begin; s0 < t_end;) {
        // the segment: the maximal run of this CTA's tasks whose items share one input vector
        const int vec = (s0 / rt_n) / kper;
        const int s1 = min(t_end, (vec + 1) * kper * rt_n);
        // this warp's tasks of the segment: a contiguous run [ta, ta + nmine)
        const int ta = s0 + (int)((int64_t)(s1 - s0) * warp / kLWarps);
        const int nmine = s0 + (int)((int64_t)(s1 - s0) * (warp + 1) / kLWarps) - ta;
        // The slice of the input vector is loaded first: requested after the weight stages below,
        // it would wait behind them in the memory pipeline.
        const bool new_vec = vec != cur_vec;  // uniform
        constexpr int kXPer = (kLSliceCols / 4 + kLThreads - 1) / kLThreads;  // float4s per thread
        float4 xv4[kXPer];
        if (new_vec) {
            const float* xv = p.x + (int64_t)vec * p.cols;
#pragma unroll
            for (int r = 0; r < kXPer; ++r) {
                const int f = tid + r * kLThreads, c = col0 + 4 * f;
                const float4* src = reinterpret_cast<const float4*>(xv + c);
                xv4[r] = f < kLSliceCols / 4 && c < p.cols ? (COH ? __ldcg(src) : __ldg(src))
                                                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (nmine > 0) lut_seek<COH>(st, p, ta / rt_n, (ta % rt_n) * kLRows, wofs, gofs, lane);
        // the first stages go out before the table is (re)built
#pragma unroll
        for (int j = 0; j < kLDepth - 1; ++j) {
            if (j < nmine) lut_issue<COH>(st, p, n_items, rt_n, ring + j * kLStage, wok, gok, wofs, gofs, lane);
            cp_commit();
        }
        if (new_vec) {
            __syncthreads();  // no warp still reads the previous table
            // Quantize the slice of x per group of 16 (four lanes hold one group as float4s):
            // xq = rint(x * 8191 / max|x|), and keep xs_g = max|x| / 8191 and the group sum.
#pragma unroll
            for (int r = 0; r < kXPer; ++r) {
                const int f = tid + r * kLThreads;
                static_assert((kLSliceCols / 4) % 32 == 0, "whole warps quantize or skip");
                if (f >= kLSliceCols / 4) continue;  // uniform over the warp
                const float4 v = xv4[r];
                float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
                float sm4 = (v.x + v.y) + (v.z + v.w);
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                sm4 += __shfl_xor_sync(kFull, sm4, 1);
                sm4 += __shfl_xor_sync(kFull, sm4, 2);
                const float inv = mx > 0.f ? (float)kLQ / mx : 0.f;
                const int q0 = __float2int_rn(v.x * inv), q1 = __float2int_rn(v.y * inv);
                const int q2 = __float2int_rn(v.z * inv), q3 = __float2int_rn(v.w * inv);
                uint2 pk;
                pk.x = ((uint32_t)q0 & 0xffffu) | ((uint32_t)q1 << 16);
                pk.y = ((uint32_t)q2 & 0xffffu) | ((uint32_t)q3 << 16);
                *reinterpret_cast<uint2*>(xq + 4 * f) = pk;
                if ((f & 3) == 0) {
                    xsg[f >> 2] = mx / (float)kLQ;
                    xsg[kLSliceGroups + (f >> 2)] = sm4;
                }
            }
            __syncthreads();
            // Table words: thread task (unit u, position pair i, upper digit pair dh) writes the
            // nine words of lower digit pairs dl, d = dl + 9 dh.
            for (int tsk = tid; tsk < 32 * 90; tsk += kLThreads) {
                const int u = tsk & 31, ih = tsk >> 5, i = ih / 9, dh = ih - 9 * i;
                const uint2 lo = *reinterpret_cast<const uint2*>(xq + 80 * u + 4 * i);
                const uint2 hi = *reinterpret_cast<const uint2*>(xq + 80 * u + 4 * i + 40);
                const int a0 = (int16_t)(lo.x & 0xffffu), a1 = (int16_t)(lo.x >> 16);
                const int a2 = (int16_t)(lo.y & 0xffffu), a3 = (int16_t)(lo.y >> 16);
                const int b0 = (int16_t)(hi.x & 0xffffu), b1 = (int16_t)(hi.x >> 16);
                const int b2 = (int16_t)(hi.y & 0xffffu), b3 = (int16_t)(hi.y >> 16);
                const int d2 = dh % 3 - 1, d3 = dh / 3 - 1;
                const int base_a = d2 * a2 + d3 * a3 + 32768, base_b = d2 * b2 + d3 * b3 + 32768;
                uint32_t* dst = table + (i * 81 + 9 * dh) * 32 + u;
#pragma unroll
                for (int dl = 0; dl < 9; ++dl) {
                    const int d0 = dl % 3 - 1, d1 = dl / 3 - 1;
                    const uint32_t ea = (uint32_t)(base_a + d0 * a0 + d1 * a1);
                    const uint32_t eb = (uint32_t)(base_b + d0 * b0 + d1 * b1);
                    dst[dl * 32] = ea | (eb << 16);
                }
            }
#pragma unroll
            for (int g = 0; g < 5; ++g) {
                xs[g] = xsg[5 * lane + g];
                xsum[g] = xsg[kLSliceGroups + 5 * lane + g];
            }
            __syncthreads();
            cur_vec = vec;
        }

        // output position of the stage being decoded
        int o_item = ta / rt_n, o_row = (ta % rt_n) * kLRows;
        for (int j = 0; j < nmine; ++j) {
            if (j + kLDepth - 1 < nmine)
                lut_issue<COH>(st, p, n_items, rt_n, ring + ((j + kLDepth - 1) % kLDepth) * kLStage, wok, gok, wofs,
                               gofs, lane);
            cp_commit();
            cp_wait<kLDepth - 1>();  // this lane's pieces of stage j have landed
            __syncwarp();            // ... and every lane's
            const uint32_t sb = ring + (uint32_t)((j % kLDepth) * kLStage);
            float tot[kLRows];
#pragma unroll
            for (int r = 0; r < kLRows; ++r) {
                const uint4 q = lds_u4(sb + r * kLCodeRow + lane * 16);
                float sc[5];
                lane_scales(sb + kLRows * kLCodeRow + r * kLScaleRow + soff, ssh, sc);
                float off = 0.f;
                tot[r] = delta * unit_row(q, tb, sc, xs);
                if (has_off) {
#pragma unroll
                    for (int g = 0; g < 5; ++g) off = fmaf(sc[g], xsum[g], off);
                    tot[r] = fmaf(c1, off, tot[r]);
                }
            }
            __syncwarp();  // the slot is read out before a later stage refills it
            // reduce-scatter of the two row sums over the warp: lane l ends with row (l >> 4)
            const bool h16 = lane & 16;
            float k = h16 ? tot[1] : tot[0];
            k += __shfl_xor_sync(kFull, h16 ? tot[0] : tot[1], 16);
            k += __shfl_xor_sync(kFull, k, 8);
            k += __shfl_xor_sync(kFull, k, 4);
            k += __shfl_xor_sync(kFull, k, 2);
            k += __shfl_xor_sync(kFull, k, 1);
            const int row = o_row + (lane >> 4);
            if ((lane & 15) == 0 && row < p.rows) {
                const int64_t o = (int64_t)o_item * p.rows + row;
                if (lp.nslices > 1) lp.part[(int64_t)slice * n_items * p.rows + o] = k;
                else store_from_float(p.y, o, p.ydt, k);
            }
            o_row += kLRows;
            if (o_row >= rt_n * kLRows) {
                o_row = 0;
                ++o_item;
            }
        }
        cp_wait<0>();
        s0 = s1;
    }
}

__global__ void __launch_bounds__(kLThreads, 1) qmv_lut_kernel(const LutParams lp) {
    extern __shared__ __align__(16) uint8_t smraw[];
    const uint32_t raw_addr = smem_u32(smraw);
    uint8_t* sm = smraw + (((raw_addr + 127u) & ~127u) - raw_addr);
    pdl_trigger();  // the slice sum (or the next call) may launch; it waits for this grid
    pdl_wait();     // ids, x, y and the scratch may belong to the kernel before
    lut_body<false>(lp, sm, blockIdx.x);
}

// y[i] = sum over slices of part[s][i], in slice order.
__global__ void __launch_bounds__(256) lut_slice_sum_kernel(const float* __restrict__ part, int nslices, int64_t n,
                                                            void* y, int ydt) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        for (int s = 0; s < nslices; ++s) v += part[s * n + i];
        store_from_float(y, i, ydt, v);
    }
}

int lut_nslices(int cols) { return (cols + kLSliceCols - 1) / kLSliceCols; }

}  // namespace

// Whether the table-lookup kernel takes this matvec: a three-level book, group 16, code rows and
// scale rows whole 16-byte pieces (16-byte aligned bases, row and expert strides a multiple of 16
// bytes) and a 16-byte aligned input with cols a multiple of 4.
bool qmv_lut_ok(const QmvParams& p, int group) {
    const bool dense = p.mode == kModeDense || p.experts <= 1;
    return p.levels == 3 && group == 16 && p.rows > 0 && p.cols > 0 && p.cols % 4 == 0 && p.row_stride % 4 == 0 &&
           p.ngroups % 8 == 0 && (dense || (p.expert_stride_w % 4 == 0 && p.expert_stride_s % 8 == 0)) &&
           (reinterpret_cast<uintptr_t>(p.codes) & 15) == 0 && (reinterpret_cast<uintptr_t>(p.scales) & 15) == 0 &&
           (reinterpret_cast<uintptr_t>(p.x) & 15) == 0;
}

size_t qmv_lut_workspace_bytes(int cols, int64_t n_items, int rows) {
    const int ns = lut_nslices(cols);
    return ns > 1 ? (size_t)ns * (size_t)n_items * (size_t)rows * 4 : 0;
}

// Launch on n_items items (gather / multi modes).  ws: qmv_lut_workspace_bytes bytes (partial
// sums of the column slices), may be null when the row fits one slice.
tq_status qmv_lut_run(const QmvParams& qp, int n_items, void* ws, size_t ws_bytes, cudaStream_t st) {
    LutParams lp{};
    lp.q = qp;
    lp.nslices = lut_nslices(qp.cols);
    lp.row_tasks = (qp.rows + kLRows - 1) / kLRows;
    lp.n_items = n_items;
    const size_t need = qmv_lut_workspace_bytes(qp.cols, n_items, qp.rows);
    if (need > 0 && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15))) return TQ_ERR_INVALID;
    lp.part = static_cast<float*>(ws);
    const int64_t ntasks = (int64_t)n_items * lp.row_tasks;
    if (ntasks > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    // one CTA per SM, the SMs shared evenly by the slices; no more CTAs than stages per slice
    lp.cta_per_slice = (int)std::max<int64_t>(1, std::min<int64_t>(sms / lp.nslices, (ntasks + 1) / 2));
    const int grid = lp.cta_per_slice * lp.nslices;
    if (ensure_smem((const void*)qmv_lut_kernel, kLSmem) != cudaSuccess) return TQ_ERR_CUDA;
    tq_status s = launch_pdl(qmv_lut_kernel, dim3(grid), dim3(kLThreads), kLSmem, st, lp);
    if (s != TQ_OK || lp.nslices == 1) return s;
    // the slices' partial sums: a programmatic dependent of the matvec, so its launch overlaps
    const int64_t n = (int64_t)n_items * qp.rows;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4 * (int64_t)sms));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, lut_slice_sum_kernel, (const float*)lp.part, lp.nslices, n, qp.y, qp.ydt) !=
        cudaSuccess)
        return TQ_ERR_CUDA;
    return TQ_OK;
}


// ---------------------------------------------------------------- the fused decode layer

namespace {

// One token through a Mixture-of-Experts layer in one cooperative launch: route + input rotation,
// the gate||up gather, SwiGLU + the intermediate rotation of each routed pair, the down
// gather, the router-weighted combine.  Phases are separated by grid barriers (a counter the
// host zeroes before the launch; each wait bounded by the wait budget, after which the CTA
// raises TQ_DEVERR_TIMEOUT and stops).  Every phase does what the separate kernels do, in the
// same order of operations, so the result has their bits.
struct DecodeParams {
    LutParams gu, dn;  // the two matvec phases
    const float* logits;
    int E, k;
    const void* x;
    int xdt;
    const int8_t* sig_h;
    int H, block_h, span_h;
    float scale_h;
    const int8_t* sig_i;
    int I, block_i;
    float scale_i;
    float* x_rot;   // [H]
    int32_t* ids;   // [k]
    float* probs;   // [k]
    float* h_rot;   // [k][I]
    float* y_dn;    // [k][H]
    void* out;      // [H]
    int odt;
    unsigned* bar;  // grid barrier counter, zero at launch
    uint32_t* err;
    long long wait_cycles;
};

// All CTAs of the launch meet; false (and TQ_DEVERR_TIMEOUT) if the others did not arrive in time.
TQ_DEVFN bool grid_meet(const DecodeParams& dp, unsigned target, int* flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(dp.bar, 1u);
        const long long t0 = clock64();
        int ok = 1;
        while (*reinterpret_cast<volatile unsigned*>(dp.bar) < target) {
            if (clock64() - t0 > dp.wait_cycles) {
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        if (!ok && dp.err) atomicOr(dp.err, TQ_DEVERR_TIMEOUT);
        *flag = ok;
    }
    __syncthreads();
    return *flag != 0;
}

template <int EH, int EI>
__global__ void __launch_bounds__(kLThreads, 1) moe_decode_kernel(const DecodeParams dp) {
    extern __shared__ __align__(16) uint8_t smraw[];
    const uint32_t raw_addr = smem_u32(smraw);
    uint8_t* sm = smraw + (((raw_addr + 127u) & ~127u) - raw_addr);
    float* fw = reinterpret_cast<float*>(sm);  // transform scratch of the rotation phases
    __shared__ int flag;
    const int cta = blockIdx.x, tid = threadIdx.x, G = gridDim.x;
    pdl_trigger();
    pdl_wait();
    // phase 1: the input rotation (one CTA per span of whole Hadamard blocks) and the router
    const int nrot = dp.H / dp.span_h;
    if (cta < nrot) {
        const int base = cta * dp.span_h + tid * EH;
        float v[EH];
#pragma unroll
        for (int i = 0; i < EH; ++i) v[i] = load_as_float(dp.x, base + i, dp.xdt) * (float)dp.sig_h[base + i];
        fwht_cta<EH>(v, fw, dp.block_h);
#pragma unroll
        for (int i = 0; i < EH; ++i) dp.x_rot[base + i] = v[i] * dp.scale_h;
    } else if (cta == nrot && tid < 32) {
        route_token<16>(dp.logits, dp.E, dp.k, dp.ids, dp.probs, nullptr);
    }
    if (!grid_meet(dp, 1u * G, &flag)) return;
    // phase 2: gate||up of the k routed experts (column slices: partial sums)
    if (cta < dp.gu.cta_per_slice * dp.gu.nslices) lut_body<true>(dp.gu, sm, cta);
    if (!grid_meet(dp, 2u * G, &flag)) return;
    // phase 3: per pair, the slices' sum (in slice order), silu(gate) * up, the rotation
    if (cta < dp.k) {
        const int64_t n = (int64_t)dp.k * 2 * dp.I;
        const float* a = dp.gu.part + (int64_t)cta * 2 * dp.I;
        const int base = tid * EI;
        float v[EI];
#pragma unroll
        for (int i = 0; i < EI; ++i) {
            float g = 0.f, u = 0.f;
            for (int sl = 0; sl < dp.gu.nslices; ++sl) {
                g += __ldcg(a + sl * n + base + i);
                u += __ldcg(a + sl * n + dp.I + base + i);
            }
            v[i] = g / (1.0f + expf(-g)) * u * (float)dp.sig_i[base + i];
        }
        fwht_cta<EI>(v, fw, dp.block_i);
#pragma unroll
        for (int i = 0; i < EI; ++i) dp.h_rot[(int64_t)cta * dp.I + base + i] = v[i] * dp.scale_i;
    }
    if (!grid_meet(dp, 3u * G, &flag)) return;
    // phase 4: down projection of each pair (one column slice: y directly)
    if (cta < dp.dn.cta_per_slice * dp.dn.nslices) lut_body<true>(dp.dn, sm, cta);
    if (!grid_meet(dp, 4u * G, &flag)) return;
    // phase 5: out = sum_j probs[j] y_j
    for (int c = cta * kLThreads + tid; c < dp.H; c += G * kLThreads) {
        float acc = 0.f;
        for (int j = 0; j < dp.k; ++j) acc = fmaf(__ldcg(dp.probs + j), __ldcg(dp.y_dn + (int64_t)j * dp.H + c), acc);
        store_from_float(dp.out, c, dp.odt, acc);
    }
}

// The span of whole Hadamard blocks one rotation CTA takes (as the rotation kernel chooses it).
int decode_span(int dim, int block) {
    int span = block;
    while (span * 2 <= 2048 && dim % (span * 2) == 0) span *= 2;
    return span;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

struct DecodeLayout {
    size_t bar, ids, probs, xrot, part, hrot, ydn, total;
};

DecodeLayout decode_layout(int H, int I, int k) {
    DecodeLayout L{};
    size_t o = 0;
    L.bar = o;
    o += 256;
    L.ids = o;
    o += align256((size_t)k * 4);
    L.probs = o;
    o += align256((size_t)k * 4);
    L.xrot = o;
    o += align256((size_t)H * 4);
    L.part = o;
    o += align256((size_t)lut_nslices(H) * k * 2 * I * 4);
    L.hrot = o;
    o += align256((size_t)k * I * 4);
    L.ydn = o;
    o += align256((size_t)k * H * 4);
    L.total = o;
    return L;
}

bool decode_ok(const tq_qweight_t* gu, const tq_qweight_t* dn, const tq_rotation_t* rh, const tq_rotation_t* ri,
               int k) {
    if (!gu || !dn || !rh || !ri || !rh->signs || !ri->signs) return false;
    const int H = gu->cols, I = dn->cols;
    if (gu->cb.levels != 3 || dn->cb.levels != 3 || gu->group != 16 || dn->group != 16) return false;
    if (gu->rows != 2 * I || dn->rows != H || gu->experts != dn->experts || gu->experts > 512) return false;
    if (k < 1 || k > 32 || k > gu->experts || rh->dim != H || ri->dim != I) return false;
    if (lut_nslices(I) != 1 || lut_nslices(H) > 8) return false;
    const int sh = decode_span(H, rh->block), si = decode_span(I, ri->block);
    return sh == 2 * kLThreads && si == 4 * kLThreads && H % sh == 0 && I % si == 0 && I == si &&
           H / sh < 152;
}

}  // namespace

}  // namespace tq

using namespace tq;

extern "C" size_t tq_moe_decode_layer_workspace_bytes(const tq_qweight_t* gate_up, const tq_qweight_t* down,
                                                      int32_t k) {
    if (!gate_up || !down || k < 1) return 0;
    return decode_layout(gate_up->cols, down->cols, k).total;
}

extern "C" tq_status tq_moe_decode_layer(const tq_qweight_t* gate_up, const tq_qweight_t* down,
                                         const tq_rotation_t* rot_h, const tq_rotation_t* rot_i,
                                         const float* logits, const void* x, tq_dtype xdt, int32_t k, void* out,
                                         tq_dtype odt, void* ws, size_t ws_bytes, uint32_t* err, void* stream) {
    if (!gate_up || !down || !logits || !x || !out || !ws) return TQ_ERR_INVALID;
    if (!(xdt == TQ_F32 || xdt == TQ_BF16 || xdt == TQ_F16) || !(odt == TQ_F32 || odt == TQ_BF16))
        return TQ_ERR_INVALID;
    if (!gate_up->codes || !gate_up->scales || !down->codes || !down->scales || !gate_up->cb.centroids ||
        !down->cb.centroids)
        return TQ_ERR_INVALID;
    if (!decode_ok(gate_up, down, rot_h, rot_i, k)) return TQ_ERR_UNSUPPORTED;
    const int H = gate_up->cols, I = down->cols;
    const DecodeLayout L = decode_layout(H, I, k);
    if (ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return TQ_ERR_INVALID;
    uint8_t* b = static_cast<uint8_t*>(ws);
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    DecodeParams dp{};
    dp.logits = logits;
    dp.E = gate_up->experts;
    dp.k = k;
    dp.x = x;
    dp.xdt = xdt;
    dp.sig_h = rot_h->signs;
    dp.H = H;
    dp.block_h = rot_h->block;
    dp.span_h = decode_span(H, rot_h->block);
    dp.scale_h = (float)(1.0 / sqrt((double)rot_h->block));
    dp.sig_i = rot_i->signs;
    dp.I = I;
    dp.block_i = rot_i->block;
    dp.scale_i = (float)(1.0 / sqrt((double)rot_i->block));
    dp.bar = reinterpret_cast<unsigned*>(b + L.bar);
    dp.ids = reinterpret_cast<int32_t*>(b + L.ids);
    dp.probs = reinterpret_cast<float*>(b + L.probs);
    dp.x_rot = reinterpret_cast<float*>(b + L.xrot);
    dp.h_rot = reinterpret_cast<float*>(b + L.hrot);
    dp.y_dn = reinterpret_cast<float*>(b + L.ydn);
    dp.out = out;
    dp.odt = odt;
    dp.err = err;
    dp.wait_cycles = wait_budget();
    // the two matvec phases, as the table-lookup kernel would be launched for them
    auto qparams = [&](const tq_qweight_t* w, const float* xin, int mode, void* y) {
        QmvParams q{};
        q.codes = w->codes;
        q.scales = w->scales;
        q.row_stride = w->row_stride_words;
        q.expert_stride_w = w->experts > 1 ? w->expert_stride_words : 0;
        q.expert_stride_s = w->experts > 1 ? w->expert_stride_scales : 0;
        q.rows = w->rows;
        q.cols = w->cols;
        q.ngroups = w->cols / w->group;
        q.experts = w->experts;
        q.centroids = w->cb.centroids;
        q.levels = 3;
        q.x = xin;
        q.T = 1;
        q.mode = mode;
        q.ids = dp.ids;
        q.k = mode == kModeGather ? k : 1;
        q.y = y;
        q.ydt = TQ_F32;
        q.err = err;
        q.wait_cycles = dp.wait_cycles;
        return q;
    };
    auto lparams = [&](const QmvParams& q, float* part) {
        LutParams lp{};
        lp.q = q;
        lp.nslices = lut_nslices(q.cols);
        lp.row_tasks = (q.rows + kLRows - 1) / kLRows;
        lp.n_items = k;
        const int64_t ntasks = (int64_t)k * lp.row_tasks;
        lp.cta_per_slice = (int)std::max<int64_t>(1, std::min<int64_t>(sms / lp.nslices, (ntasks + 1) / 2));
        lp.part = part;
        return lp;
    };
    dp.gu = lparams(qparams(gate_up, dp.x_rot, kModeGather, nullptr), reinterpret_cast<float*>(b + L.part));
    dp.dn = lparams(qparams(down, dp.h_rot, kModeMulti, dp.y_dn), nullptr);
    if (!qmv_lut_ok(dp.gu.q, 16) || !qmv_lut_ok(dp.dn.q, 16)) return TQ_ERR_UNSUPPORTED;
    if (dp.gu.nslices < 2 || dp.dn.nslices != 1) return TQ_ERR_UNSUPPORTED;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(dp.bar, 0, sizeof(unsigned), st) != cudaSuccess) return TQ_ERR_CUDA;
    if (ensure_smem((const void*)moe_decode_kernel<2, 4>, kLSmem) != cudaSuccess) return TQ_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)sms);
    cfg.blockDim = dim3(kLThreads);
    cfg.dynamicSmemBytes = kLSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_decode_kernel<2, 4>, dp) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

namespace tq {
}  // namespace tq
