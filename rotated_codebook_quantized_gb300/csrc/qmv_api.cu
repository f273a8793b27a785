// C ABI of the inline-decode matvec family and of the expert dequantizer.
//
// "How it works", "Running a quantized layer": polar_gather_qmv (one token,
// every routed expert reads the shared input), polar_multi_gather_qmv (a
// different input per expert), the dense quantized layer, and
// polar_dequant_experts ("anything else": decode, then a regular matmul).
#include <algorithm>

#include "qmv_impl.cuh"

using namespace tq;

namespace {

int gcd_i(int a, int b) { return b ? gcd_i(b, a % b) : a; }

// Padded x length per vector in the kernel's shared memory (mirrors QFmt).
int host_kpad(int levels, int group, int cols) {
    const int cw = host_codes_per_word(levels);
    const int uc = cw / gcd_i(cw, group) * group;
    const int uw = uc / cw;
    const int s = uw >= 16 ? 1 : 16 / uw;
    const int units = (cols + uc - 1) / uc;
    const int nsteps = (units + s - 1) / s;
    return nsteps * s * uc;
}

tq_status check_qweight(const tq_qweight_t* w) {
    if (!w || !w->codes || !w->scales || !w->cb.centroids) return TQ_ERR_INVALID;
    const int L = w->cb.levels;
    if (host_codes_per_word(L) == 0) return TQ_ERR_INVALID;
    if (w->experts <= 0 || w->rows <= 0 || w->cols <= 0) return TQ_ERR_INVALID;
    if (!(w->group == 16 || w->group == 32 || w->group == 64 || w->group == 128) || w->cols % w->group)
        return TQ_ERR_INVALID;
    if (w->row_stride_words < tq_row_words(L, w->cols) || w->row_stride_words % 4) return TQ_ERR_INVALID;
    if (w->experts > 1 && (w->expert_stride_words < (int64_t)w->rows * w->row_stride_words ||
                           w->expert_stride_words % 4 ||
                           w->expert_stride_scales < (int64_t)w->rows * (w->cols / w->group)))
        return TQ_ERR_INVALID;
    if (!aligned(w->codes, 16)) return TQ_ERR_INVALID;
    return TQ_OK;
}

bool ydt_ok(int d) { return d == TQ_F32 || d == TQ_BF16; }

QmvParams make_params(const tq_qweight_t* w, const float* x, void* y, tq_dtype ydt, uint32_t* err) {
    QmvParams p{};
    p.codes = w->codes;
    p.scales = w->scales;
    p.row_stride = w->row_stride_words;
    p.expert_stride_w = w->experts > 1 ? w->expert_stride_words : 0;
    p.expert_stride_s = w->experts > 1 ? w->expert_stride_scales : 0;
    p.rows = w->rows;
    p.cols = w->cols;
    p.ngroups = w->cols / w->group;
    p.experts = w->experts;
    p.centroids = w->cb.centroids;
    p.levels = w->cb.levels;
    p.x = x;
    p.y = y;
    p.ydt = ydt;
    p.err = err;
    p.wait_cycles = wait_budget();
    return p;
}

tq_status run(const QmvParams& p, int group, int nv, int n_items, cudaStream_t st) {
    if (p.levels == 3 && nv == 1) return qmv_trit_run(p, group, n_items, st);
#define TQ_QMV_G(L)                                                     \
    switch (group) {                                                    \
        case 16: return qmv_run_l##L##_g16(p, nv, n_items, st);         \
        case 32: return qmv_run_l##L##_g32(p, nv, n_items, st);         \
        case 64: return qmv_run_l##L##_g64(p, nv, n_items, st);         \
        case 128: return qmv_run_l##L##_g128(p, nv, n_items, st);       \
        default: return TQ_ERR_UNSUPPORTED;                             \
    }
    switch (p.levels) {
        case 3: TQ_QMV_G(3)
        case 4: TQ_QMV_G(4)
        case 8: TQ_QMV_G(8)
        case 16: TQ_QMV_G(16)
        default: return TQ_ERR_UNSUPPORTED;
    }
#undef TQ_QMV_G
}

// Largest vector batch (1, 2 or 4, at most `want`) whose inputs fit the shared-memory budget.
int pick_nv(int want, int kpad) {
    int nv = 1;
    while (nv * 2 <= want && nv * 2 <= 4 && (size_t)(nv * 2) * kpad * 4 <= 160 * 1024) nv *= 2;
    return nv;
}

}  // namespace

extern "C" tq_status tq_qmv(const tq_qweight_t* w, const float* x_rot, int32_t T, void* y, tq_dtype ydt, void* stream) {
    tq_status s = check_qweight(w);
    if (s != TQ_OK) return s;
    if (T < 0 || !ydt_ok(ydt)) return TQ_ERR_INVALID;
    if (T == 0) return TQ_OK;
    if (!x_rot || !y) return TQ_ERR_INVALID;
    if (w->cb.levels == 2 || w->cb.levels == 256) return TQ_ERR_UNSUPPORTED;
    QmvParams p = make_params(w, x_rot, y, ydt, nullptr);
    p.mode = kModeDense;
    p.T = T;
    // Bit-packed books up to T = 8 take the row-per-lane kernel, which decodes each weight word
    // once for up to four vectors (a second group of four re-reads the weights, mostly from L2;
    // 11008 x 4096 3-bit: 17.4 us at T = 1, 27.1 at 4, 45.8 at 8, 84.4 at 16); beyond, the
    // batched kernel below.
    if (T <= 8 && qmv_rows_ok(p, w->group)) {
        const tq_status rs = qmv_rows_run(p, w->group, T, nullptr, 0, as_stream(stream));
        if (rs != TQ_ERR_UNSUPPORTED) return rs;
    }
    if (T <= 8 && qmv_bits_ok(p, w->group)) return qmv_bits_run(p, w->group, T, as_stream(stream));
    const int nv = pick_nv(T, host_kpad(w->cb.levels, w->group, w->cols));
    return run(p, w->group, nv, (T + nv - 1) / nv, as_stream(stream));
}

namespace {

// The table-lookup kernel (three-level books) or the row-per-lane kernel (bit-packed books) when
// it applies and its scratch is there; else the single-pass kernels.
tq_status run_items(const QmvParams& p, int group, int n_items, void* ws, size_t ws_bytes, cudaStream_t st) {
    if (qmv_lut_ok(p, group)) {
        const size_t need = qmv_lut_workspace_bytes(p.cols, n_items, p.rows);
        if (need == 0 || (ws && ws_bytes >= need && aligned(ws, 16))) {
            const tq_status s = qmv_lut_run(p, n_items, ws, ws_bytes, st);
            if (s != TQ_ERR_UNSUPPORTED) return s;
        }
    }
    if (qmv_rows_ok(p, group)) {
        const size_t need = qmv_rows_workspace_bytes(p.levels, group, p.cols, n_items, p.rows);
        if (need == 0 || (ws && ws_bytes >= need && aligned(ws, 16))) {
            const tq_status s = qmv_rows_run(p, group, n_items, ws, ws_bytes, st);
            if (s != TQ_ERR_UNSUPPORTED) return s;
        }
    }
    return run(p, group, 1, n_items, st);
}

size_t items_workspace(const tq_qweight_t* w, int64_t n_items) {
    if (!w || w->rows <= 0 || w->cols <= 0 || n_items <= 0) return 0;
    if (w->cb.levels == 3) return w->group == 16 ? qmv_lut_workspace_bytes(w->cols, n_items, w->rows) : 0;
    return qmv_rows_workspace_bytes(w->cb.levels, w->group, w->cols, n_items, w->rows);
}

}  // namespace

namespace {

// Multi-gather of bit-packed books, pairs grouped by expert.  An expert with c pairs gets
// c / 4 records of four pairs and its remainder as one record of 3, 2 or 1 pairs; records of
// three or four pairs, of two and of one go to three lists, each run by the matvec instance
// with as many input vectors (4, 2, 1), so each expert's weights are decoded once per record
// and no instance multiplies empty vector slots beyond a record of three.
constexpr int kListNV[3] = {4, 2, 1};

bool groups_apply(const tq_qweight_t* w, int64_t P) {
    return w && (w->cb.levels == 4 || w->cb.levels == 8 || w->cb.levels == 16) && P >= 2 && w->experts >= 1 &&
           w->experts <= (1 << 20) && P <= (1 << 26);
}

// Most records list i can hold, and its size in ints (a count, a pad, then the records).
int64_t list_cap(int i, int64_t P) { return i == 0 ? (P + 2) / 3 : (i == 1 ? P / 2 : P); }
int64_t list_ints(int i, int64_t P) { return 2 + list_cap(i, P) * (1 + kListNV[i]); }

// Workspace of the grouping: the three record lists, then per expert its pair count, fill
// counter and first record in each list (5 * experts ints).
size_t groups_workspace(const tq_qweight_t* w, int64_t P) {
    if (!groups_apply(w, P)) return 0;
    int64_t ints = 5 * (int64_t)w->experts;
    for (int i = 0; i < 3; ++i) ints += list_ints(i, P);
    return (size_t)ints * 4 + 16;
}

struct GroupLists {
    int32_t* list[3];
};

// One CTA: count each expert's pairs, lay out its records (experts in ascending order in each
// list), then place every pair in a slot of a record of its expert.  The slot order within an
// expert follows atomics, which changes nothing in the results (each pair's sums are its own).
// A pair whose id is outside the bank gets a zero output row and raises BAD_ID.
__global__ void __launch_bounds__(1024) group_pairs_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                           GroupLists L, int32_t* __restrict__ cnt, void* y,
                                                           int rows, int ydt, uint32_t* err) {
    __shared__ int wsum[3][32];
    __shared__ int any_bad;
    int32_t* fill = cnt + E;
    int32_t* first = fill + E;  // [3][E]
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid == 0) any_bad = 0;
    for (int e = tid; e < E; e += nt) cnt[e] = fill[e] = 0;
    __syncthreads();
    for (int i = tid; i < P; i += nt) {
        const int e = __ldg(ids + i);
        if (e >= 0 && e < E) atomicAdd(cnt + e, 1);
        else any_bad = 1;
    }
    __syncthreads();
    // records of each expert in each list: four-slot list c/4 + (c%4 == 3), two-slot c%4 == 2,
    // one-slot c%4 == 1; exclusive prefixes over the experts (a contiguous range per thread)
    auto nrec = [](int c, int i) { return i == 0 ? c / 4 + (c % 4 == 3) : (i == 1 ? (c % 4 == 2) : (c % 4 == 1)); };
    const int per = (E + nt - 1) / nt, e0 = min(E, tid * per), e1 = min(E, e0 + per);
    const int lane = tid & 31, wid = tid >> 5, nwarp = nt >> 5;
    int loc[3], inc[3];
    for (int i = 0; i < 3; ++i) {
        int local = 0;
        for (int e = e0; e < e1; ++e) local += nrec(cnt[e], i);
        loc[i] = inc[i] = local;
        for (int d = 1; d < 32; d <<= 1) {  // inclusive scan within the warp
            const int v = __shfl_up_sync(0xffffffffu, inc[i], d);
            if (lane >= d) inc[i] += v;
        }
        if (lane == 31) wsum[i][wid] = inc[i];
    }
    __syncthreads();
    if (wid == 0) {  // inclusive scan of the warps' totals
        for (int i = 0; i < 3; ++i) {
            int v = lane < nwarp ? wsum[i][lane] : 0;
            for (int d = 1; d < 32; d <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, d);
                if (lane >= d) v += u;
            }
            if (lane < nwarp) wsum[i][lane] = v;
        }
    }
    __syncthreads();
    if (tid < 3) {
        L.list[tid][0] = wsum[tid][nwarp - 1];
        L.list[tid][1] = 0;
    }
    for (int i = 0; i < 3; ++i) {
        int run = inc[i] - loc[i] + (wid > 0 ? wsum[i][wid - 1] : 0);  // records of the experts before e0
        for (int e = e0; e < e1; ++e) {
            first[i * E + e] = run;
            run += nrec(cnt[e], i);
        }
    }
    for (int i = 0; i < 3; ++i) {  // the records' slots empty (-1) until their pairs are placed
        const int nv = i == 0 ? 4 : (i == 1 ? 2 : 1), nr = wsum[i][nwarp - 1];
        for (int j = tid; j < nr * nv; j += nt) L.list[i][2 + (j / nv) * (1 + nv) + 1 + j % nv] = -1;
    }
    __syncthreads();
    for (int i = tid; i < P; i += nt) {
        const int e = __ldg(ids + i);
        if (e < 0 || e >= E) continue;
        const int c = cnt[e], q = c / 4, slot = atomicAdd(fill + e, 1);
        int li, rec, pos;
        if (slot < 4 * q || c % 4 == 3) {
            li = 0;
            rec = first[e] + slot / 4;
            pos = slot % 4;
        } else {
            li = c % 4 == 2 ? 1 : 2;
            rec = first[li * E + e];
            pos = slot - 4 * q;
        }
        const int nv = li == 0 ? 4 : (li == 1 ? 2 : 1);
        int32_t* r = L.list[li] + 2 + (int64_t)rec * (1 + nv);
        r[0] = e;
        r[1 + pos] = i;
    }
    if (!any_bad) return;  // uniform
    if (tid == 0 && err) atomicOr(err, TQ_DEVERR_BAD_ID);
    for (int i = 0; i < P; ++i) {
        const int e = __ldg(ids + i);
        if (e >= 0 && e < E) continue;
        for (int r = tid; r < rows; r += nt) store_from_float(y, (int64_t)i * rows + r, ydt, 0.f);
    }
}

// Builds the record lists in ws (groups_workspace bytes) on the stream.
tq_status group_pairs(const QmvParams& p, const tq_qweight_t* w, int P, void* ws, GroupLists& L, cudaStream_t st) {
    int32_t* base = static_cast<int32_t*>(ws);
    int64_t off = 0;
    for (int i = 0; i < 3; ++i) {
        L.list[i] = base + off;
        off += list_ints(i, P);
    }
    int32_t* cnt = base + off;
    group_pairs_kernel<<<1, 1024, 0, st>>>(p.ids, P, w->experts, L, cnt, p.y, p.rows, p.ydt, p.err);
    return launch_status();
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// Scratch of the row-per-lane kernel over grouped pairs: the lists, then the chunks' partial sums.
size_t rows_groups_workspace(const tq_qweight_t* w, int64_t P) {
    const size_t g = groups_workspace(w, P);
    return g ? round256(g) + items_workspace(w, P) : 0;
}

// Gather (p.mode kModeGather, P = T * k pairs) or multi-gather of bit-packed books through the
// row-per-lane kernel with the pairs grouped by expert: the lists are built first, then each
// expert's words are decoded once for up to four of its pairs.
tq_status run_groups_rows(const QmvParams& p, const tq_qweight_t* w, int P, void* ws, size_t ws_bytes,
                          cudaStream_t st) {
    GroupLists L;
    tq_status s = group_pairs(p, w, P, ws, L, st);
    if (s != TQ_OK) return s;
    const size_t off = round256(groups_workspace(w, P));
    const int32_t* lists[3] = {L.list[0], L.list[1], L.list[2]};
    return qmv_rows_run_groups(p, w->group, lists, P, static_cast<char*>(ws) + off, ws_bytes - off, st);
}

// Whether the grouped row-per-lane path takes these pairs with this scratch.
bool groups_rows_apply(const QmvParams& p, const tq_qweight_t* w, int64_t P, const void* ws, size_t ws_bytes) {
    const size_t need = rows_groups_workspace(w, P);
    return need > 0 && qmv_rows_ok(p, w->group) && ws && aligned(ws, 16) && ws_bytes >= need;
}

tq_status run_groups(QmvParams p, const tq_qweight_t* w, int P, void* ws, cudaStream_t st) {
    GroupLists L;
    tq_status s = group_pairs(p, w, P, ws, L, st);
    if (s != TQ_OK) return s;
    p.mode = kModeGroups;
    for (int i = 0; i < 3; ++i) {  // each launch has room for the list's most records; the rest return at once
        p.groups = L.list[i];
        s = run(p, w->group, kListNV[i], (int)std::max<int64_t>(1, list_cap(i, P)), st);
        if (s != TQ_OK) return s;
    }
    return TQ_OK;
}

}  // namespace

extern "C" size_t tq_gather_qmv_workspace_bytes(const tq_qweight_t* w, int32_t T, int32_t k) {
    if (T <= 0 || k <= 0) return 0;
    const int64_t P = (int64_t)T * k;
    // more than one token: room to group the pairs by expert (bit-packed books)
    return std::max(items_workspace(w, P), T > 1 ? rows_groups_workspace(w, P) : (size_t)0);
}

extern "C" size_t tq_multi_gather_qmv_workspace_bytes(const tq_qweight_t* w, int32_t P) {
    return std::max(std::max(items_workspace(w, P), groups_workspace(w, P)), rows_groups_workspace(w, P));
}

extern "C" tq_status tq_gather_qmv(const tq_qweight_t* w, const float* x_rot, const int32_t* ids, int32_t T, int32_t k,
                                   void* y, tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err, void* stream) {
    tq_status s = check_qweight(w);
    if (s != TQ_OK) return s;
    if (T < 0 || k <= 0 || !ydt_ok(ydt)) return TQ_ERR_INVALID;
    if (T == 0) return TQ_OK;
    if (!x_rot || !ids || !y) return TQ_ERR_INVALID;
    if (w->cb.levels == 2 || w->cb.levels == 256) return TQ_ERR_UNSUPPORTED;
    if ((int64_t)T * k > 0x7fffffffll) return TQ_ERR_INVALID;
    QmvParams p = make_params(w, x_rot, y, ydt, err);
    p.mode = kModeGather;
    p.ids = ids;
    p.k = k;
    if (T > 1 && groups_rows_apply(p, w, (int64_t)T * k, ws, ws_bytes))
        return run_groups_rows(p, w, T * k, ws, ws_bytes, as_stream(stream));
    return run_items(p, w->group, T * k, ws, ws_bytes, as_stream(stream));
}

extern "C" tq_status tq_multi_gather_qmv(const tq_qweight_t* w, const float* x_rot, const int32_t* ids, int32_t P,
                                         void* y, tq_dtype ydt, void* ws, size_t ws_bytes, uint32_t* err,
                                         void* stream) {
    tq_status s = check_qweight(w);
    if (s != TQ_OK) return s;
    if (P < 0 || !ydt_ok(ydt)) return TQ_ERR_INVALID;
    if (P == 0) return TQ_OK;
    if (!x_rot || !ids || !y) return TQ_ERR_INVALID;
    if (w->cb.levels == 2 || w->cb.levels == 256) return TQ_ERR_UNSUPPORTED;
    QmvParams p = make_params(w, x_rot, y, ydt, err);
    p.mode = kModeMulti;
    p.ids = ids;
    p.k = 1;
    if (groups_rows_apply(p, w, P, ws, ws_bytes)) return run_groups_rows(p, w, P, ws, ws_bytes, as_stream(stream));
    const size_t gneed = groups_workspace(w, P);
    if (!qmv_rows_ok(p, w->group) && gneed > 0 && ws && ws_bytes >= gneed && aligned(ws, 16))
        return run_groups(p, w, P, ws, as_stream(stream));
    return run_items(p, w->group, P, ws, ws_bytes, as_stream(stream));
}

extern "C" tq_status tq_gather_qmv_rotate(const tq_qweight_t* w, const void* x, tq_dtype xdt,
                                          const tq_rotation_t* rot, const int32_t* ids, int32_t T, int32_t k,
                                          void* y, tq_dtype ydt, uint32_t* err, void* stream) {
    tq_status s = check_qweight(w);
    if (s != TQ_OK) return s;
    if (T < 0 || k <= 0 || !ydt_ok(ydt) || (xdt != TQ_F32 && xdt != TQ_BF16)) return TQ_ERR_INVALID;
    if (!rot || !rot->signs || rot->dim != w->cols) return TQ_ERR_INVALID;
    if (T == 0) return TQ_OK;
    if (!x || !ids || !y) return TQ_ERR_INVALID;
    if (w->cb.levels != 3 || (int64_t)T * k > 0x7fffffffll) return TQ_ERR_UNSUPPORTED;
    QmvParams p = make_params(w, nullptr, y, ydt, err);
    p.mode = kModeGather;
    p.ids = ids;
    p.k = k;
    return qmv_trit_xstage_run(p, w->group, T * k, 1, x, xdt, rot->signs, rot->block, as_stream(stream));
}

extern "C" tq_status tq_multi_gather_qmv_swiglu(const tq_qweight_t* w, const float* gate_up,
                                               const tq_rotation_t* rot, const int32_t* ids, int32_t P, void* y,
                                               tq_dtype ydt, uint32_t* err, void* stream) {
    tq_status s = check_qweight(w);
    if (s != TQ_OK) return s;
    if (P < 0 || !ydt_ok(ydt)) return TQ_ERR_INVALID;
    if (!rot || !rot->signs || rot->dim != w->cols) return TQ_ERR_INVALID;
    if (P == 0) return TQ_OK;
    if (!gate_up || !ids || !y) return TQ_ERR_INVALID;
    if (w->cb.levels != 3) return TQ_ERR_UNSUPPORTED;
    QmvParams p = make_params(w, nullptr, y, ydt, err);
    p.mode = kModeMulti;
    p.ids = ids;
    p.k = 1;
    return qmv_trit_xstage_run(p, w->group, P, 2, gate_up, TQ_F32, rot->signs, rot->block, as_stream(stream));
}

// ---------------------------------------------------------------- dequant_experts

namespace {

// 1-bit, ternary and 8-bit books.  One CTA per (selected expert, run of up to kDqRows rows), in
// two passes over shared memory: each thread decodes whole words into one code byte per column;
// then each thread writes 8 consecutive columns (one group, as 8 divides the
// group) as a single 16-byte store for 16-bit outputs (two for f32), so a warp
// writes 512 contiguous bytes per instruction.
constexpr int kDqRows = 4;

template <int LEVELS>
__global__ void __launch_bounds__(256) dequant_kernel(const uint32_t* __restrict__ codes,
                                                      const uint16_t* __restrict__ scales, int64_t row_stride,
                                                      int64_t esw, int64_t ess, int rows, int cols, int gshift,
                                                      int experts, const float* __restrict__ centroids,
                                                      const int32_t* __restrict__ ids, void* out, int odt, int rpc,
                                                      int cpad, uint32_t* err) {
    constexpr int BITS = LEVELS == 3 ? 0 : (LEVELS == 2 ? 1 : (LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : (LEVELS == 16 ? 4 : 8))));
    constexpr int CW = LEVELS == 3 ? 20 : (LEVELS == 8 ? 10 : 32 / BITS);
    extern __shared__ __align__(16) uint8_t dq[];  // [rpc][cpad] code bytes
    __shared__ float lut[LEVELS];
    for (int i = threadIdx.x; i < LEVELS; i += blockDim.x) lut[i] = centroids[i];
    const int n0 = blockIdx.x * rpc;
    const int nr = min(rpc, rows - n0);
    const int64_t i_sel = blockIdx.y;
    const int e = ids[i_sel];
    const bool bad = e < 0 || e >= experts;
    if (bad && threadIdx.x == 0 && err) atomicOr(err, TQ_DEVERR_BAD_ID);
    const int nw = (cols + CW - 1) / CW;
    const uint32_t* w0 = codes + (bad ? 0 : (int64_t)e * esw + (int64_t)n0 * row_stride);
    for (int r = 0; r < nr; ++r) {
        for (int j = threadIdx.x; j < nw; j += blockDim.x) {
            const uint32_t w = bad ? 0u : __ldg(w0 + (int64_t)r * row_stride + j);
            uint8_t* d = dq + r * cpad + j * CW;  // cpad >= nw * CW: the last word's tail lands in padding
            if constexpr (LEVELS == 3) {
                const TritHalves th = trit_split(w);
                uint32_t Fh = th.hi, Fl = th.lo;
#pragma unroll
                for (int q = 0; q < 10; ++q) d[19 - q] = (uint8_t)trit_next_int(Fh);
#pragma unroll
                for (int q = 0; q < 10; ++q) d[9 - q] = (uint8_t)trit_next_int(Fl);
            } else {
#pragma unroll
                for (int q = 0; q < CW; ++q) d[q] = (uint8_t)((w >> (BITS * q)) & ((1u << BITS) - 1u));
            }
        }
    }
    __syncthreads();
    const int nv = cols / 8;
    const int ngroups = cols >> gshift;
    const uint16_t* s0 = scales + (bad ? 0 : (int64_t)e * ess + (int64_t)n0 * ngroups);
    for (int r = 0; r < nr; ++r) {
        for (int v = threadIdx.x; v < nv; v += blockDim.x) {
            const int kk = v * 8;
            const float sc = bad ? 0.f : half_bits_to_float(__ldg(s0 + (int64_t)r * ngroups + (kk >> gshift)));
            const uint2 cb = *reinterpret_cast<const uint2*>(dq + r * cpad + kk);
            float f[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = sc * lut[((q < 4 ? cb.x : cb.y) >> (8 * (q & 3))) & 0xffu];
            const int64_t o = (i_sel * rows + n0 + r) * (int64_t)cols + kk;  // a multiple of 8 elements
            if (odt == TQ_F32) {
                float4* y = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
                y[0] = make_float4(f[0], f[1], f[2], f[3]);
                y[1] = make_float4(f[4], f[5], f[6], f[7]);
            } else {
                uint32_t h[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (odt == TQ_BF16) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);
                        h[q] = *reinterpret_cast<const uint32_t*>(&b2);
                    } else {
                        const __half2 b2 = __floats2half2_rn(f[2 * q], f[2 * q + 1]);
                        h[q] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                }
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + o) = make_uint4(h[0], h[1], h[2], h[3]);
            }
        }
    }
}

// Bit-packed books (2, 3, 4 bits) in one pass: each thread writes 8 consecutive columns of one
// row (one 16-byte store for 16-bit outputs), so a warp's stores cover 512 contiguous bytes.
// The 8 codes come from one word, or for 3-bit books from two (a word holds 10 codes in its low
// 30 bits, so the pair read as one 64-bit value is a contiguous run of codes); they go through a
// per-lane table (pairs of centroids for 2- and 3-bit books, one centroid for 4-bit ones; entry
// e of lane l at (32 e + l) entries, so a warp's lookups are conflict-free whatever the codes)
// and are multiplied by the group's scale in fp32, as in the two-pass kernel above.
template <int LEVELS>
struct DqFmt {
    static constexpr int kBits = LEVELS == 4 ? 2 : (LEVELS == 8 ? 3 : 4);
    static constexpr int kCW = LEVELS == 8 ? 10 : 32 / kBits;  // codes per word
    static constexpr bool kPair = LEVELS != 16;
    static constexpr int kEntries = 1 << ((kPair ? 2 : 1) * kBits);
    static constexpr int kEntryBytes = kPair ? 8 : 4;
    static constexpr int kTabBytes = kEntries * 32 * kEntryBytes;
};

TQ_DEVFN float2 dq_lds64(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}
TQ_DEVFN float dq_lds32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

// Eight consecutive outputs from element o on (a multiple of 8): one 16-byte store for 16-bit
// outputs, two for f32.
TQ_DEVFN void dq_store8(void* out, int odt, int64_t o, const float (&f)[8]) {
    if (odt == TQ_F32) {
        float4* y = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
        y[0] = make_float4(f[0], f[1], f[2], f[3]);
        y[1] = make_float4(f[4], f[5], f[6], f[7]);
        return;
    }
    uint32_t h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (odt == TQ_BF16) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);
            h[q] = *reinterpret_cast<const uint32_t*>(&b2);
        } else {
            const __half2 b2 = __floats2half2_rn(f[2 * q], f[2 * q + 1]);
            h[q] = *reinterpret_cast<const uint32_t*>(&b2);
        }
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + o) = make_uint4(h[0], h[1], h[2], h[3]);
}

template <int LEVELS>
__global__ void __launch_bounds__(256) dequant_bits_kernel(const uint32_t* __restrict__ codes,
                                                           const uint16_t* __restrict__ scales, int64_t row_stride,
                                                           int64_t esw, int64_t ess, int rows, int cols, int gshift,
                                                           int experts, const float* __restrict__ centroids,
                                                           const int32_t* __restrict__ ids, void* out, int odt,
                                                           uint32_t* err) {
    using D = DqFmt<LEVELS>;
    constexpr int CW = D::kCW, BITS = D::kBits;
    extern __shared__ __align__(16) uint8_t dtab[];
    for (int i = threadIdx.x; i < D::kEntries * 32; i += blockDim.x) {
        const int v = i >> 5;
        if constexpr (D::kPair)
            reinterpret_cast<float2*>(dtab)[i] =
                make_float2(__ldg(centroids + (v & (LEVELS - 1))), __ldg(centroids + (v >> BITS)));
        else
            reinterpret_cast<float*>(dtab)[i] = __ldg(centroids + v);
    }
    __syncthreads();
    const int vpr = cols >> 3;  // 8-column vectors per row
    const int nvec = rows * vpr;
    const int64_t i_sel = blockIdx.y;
    const int e = __ldg(ids + i_sel);
    const bool bad = e < 0 || e >= experts;
    if (bad && err && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, TQ_DEVERR_BAD_ID);
    const int64_t ee = bad ? 0 : e;
    const uint32_t lbase = (uint32_t)__cvta_generic_to_shared(dtab) + (threadIdx.x & 31) * D::kEntryBytes;
    // vectors of the selected expert's rows, strided over the CTAs of this id (the table is built
    // once per CTA)
    for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < nvec; f += gridDim.x * blockDim.x) {
        const int n = f / vpr, k0 = (f - n * vpr) * 8;  // row, first column
        const uint32_t* wrow = codes + ee * esw + (int64_t)n * row_stride;
        const int a = k0 / CW, ob = (k0 - a * CW) * BITS;  // the first code's word and bit
        uint32_t lo;  // the 8 codes from bit 0 on
        if constexpr (LEVELS == 8) {
            const uint32_t wa = __ldg(wrow + a);
            const uint32_t wb = (ob > 6 && a + 1 < row_stride) ? __ldg(wrow + a + 1) : 0u;  // codes past word a
            lo = (uint32_t)((((uint64_t)wb << 30) | wa) >> ob);
        } else {
            lo = __ldg(wrow + a) >> ob;  // 2-bit: 8 codes from bit 0 or 16; 4-bit: a whole word
        }
        const float sc =
            bad ? 0.f : half_bits_to_float(__ldg(scales + ee * ess + (int64_t)n * (cols >> gshift) + (k0 >> gshift)));
        float v8[8];
        if constexpr (D::kPair) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t pv = (lo >> (2 * BITS * j)) & ((1u << (2 * BITS)) - 1u);
                const float2 c = dq_lds64(lbase + (pv << 8));
                v8[2 * j] = c.x * sc;
                v8[2 * j + 1] = c.y * sc;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v8[q] = dq_lds32(lbase + (((lo >> (4 * q)) & 15u) << 7)) * sc;
        }
        dq_store8(out, odt, (i_sel * rows + n) * (int64_t)cols + k0, v8);
    }
}

template <int LEVELS>
tq_status launch_dequant_bits(const tq_qweight_t* w, const int32_t* ids, int32_t n_ids, void* out, tq_dtype odt,
                              uint32_t* err, cudaStream_t st) {
    const int64_t nvec = (int64_t)w->rows * (w->cols / 8);
    if (nvec > 0x7fffffffll / 2) return TQ_ERR_UNSUPPORTED;
    // about eight CTAs per SM over all ids, each looping over its id's vectors
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t per_id = std::max<int64_t>(1, (int64_t)(sms > 0 ? sms : 152) * 8 / n_ids);
    const unsigned blocks = (unsigned)std::min<int64_t>((nvec + 255) / 256, per_id);
    dequant_bits_kernel<LEVELS><<<dim3(blocks, (unsigned)n_ids), 256, DqFmt<LEVELS>::kTabBytes, st>>>(
        w->codes, w->scales, w->row_stride_words, w->experts > 1 ? w->expert_stride_words : 0,
        w->experts > 1 ? w->expert_stride_scales : 0, w->rows, w->cols, __builtin_ctz((unsigned)w->group),
        w->experts, w->cb.centroids, ids, out, (int)odt, err);
    return launch_status();
}

template <int LEVELS>
tq_status launch_dequant(const tq_qweight_t* w, const int32_t* ids, int32_t n_ids, void* out, tq_dtype odt,
                         uint32_t* err, int rpc, int cpad, cudaStream_t st) {
    const size_t smem = (size_t)rpc * cpad;
    if (ensure_smem((const void*)dequant_kernel<LEVELS>, smem) != cudaSuccess) return TQ_ERR_CUDA;
    const int gshift = __builtin_ctz((unsigned)w->group);
    dequant_kernel<LEVELS><<<dim3((w->rows + rpc - 1) / rpc, n_ids), 256, smem, st>>>(
        w->codes, w->scales, w->row_stride_words, w->experts > 1 ? w->expert_stride_words : 0,
        w->experts > 1 ? w->expert_stride_scales : 0, w->rows, w->cols, gshift, w->experts, w->cb.centroids, ids, out,
        (int)odt, rpc, cpad, err);
    return launch_status();
}

}  // namespace

extern "C" tq_status tq_dequant_experts(const tq_qweight_t* w, const int32_t* ids, int32_t n_ids, void* out,
                                        tq_dtype odt, uint32_t* err, void* stream) {
    tq_status s = check_qweight(w);
    if (s != TQ_OK) return s;
    if (n_ids < 0 || !(odt == TQ_F32 || odt == TQ_BF16 || odt == TQ_F16)) return TQ_ERR_INVALID;
    if (n_ids == 0) return TQ_OK;
    if (!ids || !out || n_ids > 65535 || !aligned(out, 16)) return TQ_ERR_INVALID;
    cudaStream_t st = as_stream(stream);
    // 2-, 3- and 4-bit books: one pass, one 8-column store per thread
    switch (w->cb.levels) {
        case 4: return launch_dequant_bits<4>(w, ids, n_ids, out, odt, err, st);
        case 8: return launch_dequant_bits<8>(w, ids, n_ids, out, odt, err, st);
        case 16: return launch_dequant_bits<16>(w, ids, n_ids, out, odt, err, st);
        default: break;
    }
    // the others (1-bit, ternary, 8-bit books): the two-pass kernel
    const int cw = host_codes_per_word(w->cb.levels);
    const int cpad = (int)((tq_row_words(w->cb.levels, w->cols) * cw + 15) / 16 * 16);
    if (cpad > 160 * 1024) return TQ_ERR_UNSUPPORTED;
    const int rpc = std::max(1, std::min(kDqRows, 40960 / cpad));
    switch (w->cb.levels) {
        case 2: return launch_dequant<2>(w, ids, n_ids, out, odt, err, rpc, cpad, st);
        case 3: return launch_dequant<3>(w, ids, n_ids, out, odt, err, rpc, cpad, st);
        case 256: return launch_dequant<256>(w, ids, n_ids, out, odt, err, rpc, cpad, st);
        default: return TQ_ERR_UNSUPPORTED;
    }
}
