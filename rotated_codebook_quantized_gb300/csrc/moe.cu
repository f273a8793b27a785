// Mixture-of-Experts glue: tq_moe_route (top-k, softmax, expert-sorted pair
// order) and tq_moe_combine (router-weighted sum of expert outputs).
//
// "Running a 1T-Parameter Model on a Laptop": a router picks 8 of 384 experts
// per token and their outputs are combined; "How it works", row "A large batch
// sorted by expert" (the order polar_gather_qmm consumes).
#include <math.h>

#include "common.cuh"
#include "route.cuh"

using namespace tq;

namespace {

constexpr int kMaxK = 32;

// One warp per token: route_token (the routing body shared with the fused decode layer).
template <int kPer>  // experts per lane: E <= 32 * kPer
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ ids, float* __restrict__ probs,
                                                         int32_t* __restrict__ counts) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;
    route_token<kPer>(logits + (int64_t)t * E, E, k, ids + (int64_t)t * k, probs + (int64_t)t * k, counts);
}

// offsets[e] = sum of counts below e (one CTA, E <= 1024).
__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* __restrict__ counts, int E,
                                                          int32_t* __restrict__ offsets) {
    __shared__ int32_t s[1024];
    const int i = threadIdx.x;
    s[i] = i < E ? counts[i] : 0;
    __syncthreads();
    for (int d = 1; d < 1024; d <<= 1) {  // inclusive Hillis-Steele scan
        const int v = i >= d ? s[i - d] : 0;
        __syncthreads();
        s[i] += v;
        __syncthreads();
    }
    if (i < E) offsets[i + 1] = s[i];
    if (i == 0) offsets[0] = 0;
}

// One CTA per expert: walk all pairs in order and compact those routed to it
// (a stable counting sort: pairs keep their flat order within an expert).
__global__ void __launch_bounds__(256) route_compact_kernel(const int32_t* __restrict__ ids, int P,
                                                            const int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ perm, int32_t* __restrict__ pair_pos) {
    __shared__ int warp_tot[8];
    __shared__ int base_s;
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    if (threadIdx.x == 0) base_s = offsets[e];
    __syncthreads();
    for (int f0 = 0; f0 < P; f0 += blockDim.x) {
        const int f = f0 + threadIdx.x;
        const bool hit = f < P && ids[f] == e;
        const unsigned bal = __ballot_sync(kFull, hit);
        if (lane == 0) warp_tot[warp] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < nwarps; ++w) {
            before += w < warp ? warp_tot[w] : 0;
            total += warp_tot[w];
        }
        if (hit) {
            const int pos = base_s + before + __popc(bal & ((1u << lane) - 1u));
            perm[pos] = f;
            if (pair_pos) pair_pos[f] = pos;
        }
        __syncthreads();
        if (threadIdx.x == 0) base_s += total;
        __syncthreads();
    }
}

__global__ void combine_kernel(const float* __restrict__ y, const float* __restrict__ probs,
                               const int32_t* __restrict__ pair_pos, int k, int H, void* out, int odt) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= H) return;
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
        const int64_t f = (int64_t)t * k + j;
        const int64_t r = pair_pos ? pair_pos[f] : f;
        acc = fmaf(probs[f], y[r * H + n], acc);
    }
    store_from_float(out, (int64_t)t * H + n, odt, acc);
}

}  // namespace

extern "C" size_t tq_route_workspace_bytes(int32_t E) { return E > 0 ? ((size_t)E * 4 + 255) / 256 * 256 : 0; }

extern "C" tq_status tq_moe_route(const float* logits, int32_t T, int32_t E, int32_t k, int32_t* ids, float* probs,
                                  int32_t* perm, int32_t* pair_pos, int32_t* offsets, void* ws, size_t ws_bytes,
                                  void* stream) {
    if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > kMaxK || k > E) return TQ_ERR_INVALID;
    if ((int64_t)T * k > 0x7fffffffll) return TQ_ERR_INVALID;
    const bool sort = perm || pair_pos || offsets;
    if (sort && (!perm || !offsets || !ws || ws_bytes < tq_route_workspace_bytes(E))) return TQ_ERR_INVALID;
    if (T > 0 && (!logits || !ids || !probs)) return TQ_ERR_INVALID;
    cudaStream_t st = as_stream(stream);
    int32_t* counts = sort ? reinterpret_cast<int32_t*>(ws) : nullptr;
    if (sort && cudaMemsetAsync(counts, 0, (size_t)E * 4, st) != cudaSuccess) return TQ_ERR_CUDA;
    if (T > 0) {
        const int warps = 8;
        const dim3 grid((T + warps - 1) / warps), block(warps * 32);
        // without sorting the top-k kernel is the call's only launch: a programmatic dependent of
        // the previous kernel (with sorting it follows the counts' memset)
        auto go = [&](auto kern) -> tq_status {
            if (!sort) return launch_pdl(kern, grid, block, 0, st, logits, T, E, k, ids, probs, counts);
            kern<<<grid, block, 0, st>>>(logits, T, E, k, ids, probs, counts);
            return launch_status();
        };
        tq_status s = E <= 128 ? go(route_topk_kernel<4>)
                      : E <= 256 ? go(route_topk_kernel<8>)
                      : E <= 512 ? go(route_topk_kernel<16>)
                                 : go(route_topk_kernel<32>);
        if (s != TQ_OK) return s;
    }
    if (!sort) return TQ_OK;
    route_scan_kernel<<<1, 1024, 0, st>>>(counts, E, offsets);
    tq_status s = launch_status();
    if (s != TQ_OK || T == 0) return s;
    route_compact_kernel<<<E, 256, 0, st>>>(ids, T * k, offsets, perm, pair_pos);
    return launch_status();
}

extern "C" tq_status tq_moe_combine(const float* y, const float* probs, const int32_t* pair_pos, int32_t T, int32_t k,
                                    int32_t H, void* out, tq_dtype odt, void* stream) {
    if (T < 0 || k <= 0 || H <= 0 || !(odt == TQ_F32 || odt == TQ_BF16)) return TQ_ERR_INVALID;
    if (T == 0) return TQ_OK;
    if (!y || !probs || !out || T > 65535) return TQ_ERR_INVALID;
    return launch_pdl(combine_kernel, dim3((H + 255) / 256, T), dim3(256), 0, as_stream(stream), y, probs, pair_pos, k,
                      H, out, (int)odt);
}
