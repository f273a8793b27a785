// Router top-k of one token: the body shared by the routing kernel and the fused decode layer.
//
// "Running a 1T-Parameter Model on a Laptop": the router picks k of E experts per token (ties
// to the lower id) and their weights are a softmax over the k chosen logits.  One warp: the
// row's logits in registers (lane l holds experts l, l + 32, ...), each lane keeps its best
// untaken expert, and each of the k rounds is two warp-wide reductions (the largest value as an
// order-preserving 32-bit key, -0 folded into +0, then the lowest id among the lanes holding
// it), after which only the winning lane rescans.  ids[0..k) and probs[0..k) of the token are
// written; counts (if not NULL) receives each chosen expert's pair count.
#pragma once

#include "common.cuh"

namespace tq {

template <int kPer, bool kCoherent = false>  // experts per lane: E <= 32 * kPer
TQ_DEVFN void route_token(const float* __restrict__ row, int E, int k, int32_t* __restrict__ ids,
                          float* __restrict__ probs, int32_t* __restrict__ counts) {
    const int lane = threadIdx.x & 31;
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = lane + 32 * j;
        v[j] = i < E ? (kCoherent ? __ldcg(row + i) : __ldg(row + i)) : -INFINITY;
    }
    unsigned taken = 0;  // bit j: expert lane + 32 j already chosen
    float chosen_v = 0.f;  // lane r keeps the r-th chosen logit
    // The lane's best untaken expert (ascending ids within the lane: strict > keeps the lower id);
    // only the lane that wins a round looks again.
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    auto lane_best = [&]() {
        bv = -INFINITY;
        bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = lane + 32 * j;
            if (i < E && !(taken >> j & 1u) && (v[j] > bv || bi == 0x7fffffff)) {
                bv = v[j];
                bi = i;
            }
        }
    };
    lane_best();
    for (int r = 0; r < k; ++r) {
        // round winner: the largest value (an order-preserving 32-bit key, 0 for a lane with no
        // candidate), then the lowest id among the lanes holding it -- two warp reductions
        const uint32_t u0 = __float_as_uint(bv);
        const uint32_t u = (u0 << 1) == 0u ? 0u : u0;  // -0 and +0 are one value
        const uint32_t key = bi == 0x7fffffff ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
        const uint32_t mk = __reduce_max_sync(kFull, key);
        const uint32_t wi = __reduce_min_sync(kFull, key == mk && bi != 0x7fffffff ? (uint32_t)bi : 0xffffffffu);
        if ((int)(wi & 31u) == lane) {
            taken |= 1u << (wi >> 5);
            lane_best();
        }
        if (lane == 0) {
            ids[r] = (int32_t)wi;
            if (counts) atomicAdd(counts + wi, 1);
        }
        if (lane == r) chosen_v = __uint_as_float((mk & 0x80000000u) ? (mk ^ 0x80000000u) : ~mk);
    }
    // softmax over the k chosen logits; the first is the largest
    const float mx = __shfl_sync(kFull, chosen_v, 0);
    const float ex = lane < k ? expf(chosen_v - mx) : 0.f;
    float sum = ex;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) sum += __shfl_xor_sync(kFull, sum, m);
    if (lane < k) probs[lane] = ex / sum;
}

}  // namespace tq
