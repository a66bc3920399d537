// topk.cuh -- top-k softmax routing of one token by one warp.
//
// "Warp decode", section on the conventional MoE path: every token selects
// k of E experts.  Selection is by logit, which orders experts exactly as the
// softmax probabilities do; ties go to the lower expert id and slots come out
// in descending order.  The k weights are the softmax probabilities
// renormalised over the chosen experts, exp(l_j - l_max) / sum over the
// chosen of exp(l_i - l_max), in FP32.
//
// Each round takes the warp-wide maximum of order-preserving integer keys of
// the remaining logits (redux.sync), then the lowest expert id holding it.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving key of a float (larger float -> larger key; -0 as +0);
// 0 is never produced for a non-NaN input and marks an absent entry.
__device__ __forceinline__ uint32_t topk_key(float v)
{
    const uint32_t u = __float_as_uint(v + 0.0f);
    return u ^ ((u >> 31) ? 0xFFFFFFFFu : 0x80000000u);
}

__device__ __forceinline__ float topk_unkey(uint32_t key)
{
    return __uint_as_float(key ^ ((key >> 31) ? 0x80000000u : 0xFFFFFFFFu));
}

// Lane j < k receives slot j: its expert id and renormalised weight.  All 32
// lanes call it; l holds E logits; PER_LANE * 32 >= E.  `hook` runs after the
// logit loads are issued and before their values are used (set-up work that
// can overlap the memory latency).
template <int PER_LANE, typename Hook>
__device__ __forceinline__ void topk_warp(const float *__restrict__ l, int E, int k, int lane, int &slot_e,
                                          float &slot_w, Hook hook)
{
    float lg[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = i * 32 + lane;
        lg[i] = e < E ? __ldcg(l + e) : 0.f;
    }
    hook();
    uint32_t key[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = i * 32 + lane;
        key[i] = e < E ? topk_key(lg[i]) : 0u;
    }
    float my_l = -INFINITY;
    int my_e = -1;
    constexpr int NW = (PER_LANE + 31) / 32;
    uint32_t taken[NW];                      // bit i: this lane's entry i already chosen
#pragma unroll
    for (int w = 0; w < NW; ++w)
        taken[w] = 0;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0;
        int bi = 0;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
            if (!((taken[i >> 5] >> (i & 31)) & 1u) && key[i] > bk) {   // strictly greater: lower id wins in a lane
                bk = key[i];
                bi = i;
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        // a unique maximum (the usual case) names its lane directly; equal
        // maxima in several lanes take the lowest expert id among them
        const bool have = bk == mk && bk != 0u;
        const unsigned holders = __ballot_sync(0xffffffffu, have);
        uint32_t win;
        if ((holders & (holders - 1u)) == 0u) {
            const int wl = holders ? __ffs(holders) - 1 : 0;
            win = static_cast<uint32_t>(__shfl_sync(0xffffffffu, bi, wl) * 32 + wl);
        } else {
            win = __reduce_min_sync(0xffffffffu, have ? static_cast<uint32_t>(bi * 32 + lane) : 0xFFFFFFFFu);
        }
        if (static_cast<int>(win & 31u) == lane) {
            const int wi = static_cast<int>(win >> 5);
            if constexpr (NW == 1) {
                taken[0] |= 1u << wi;
            } else {
#pragma unroll
                for (int w = 0; w < NW; ++w)
                    if (w == (wi >> 5))
                        taken[w] |= 1u << (wi & 31);
            }
        }
        if (lane == j) {
            my_l = topk_unkey(mk);
            my_e = static_cast<int>(win);
        }
    }
    const float mx = __shfl_sync(0xffffffffu, my_l, 0);
    const float p = lane < k ? expf(my_l - mx) : 0.f;
    const float z = warp_sum(p);
    slot_e = my_e;
    slot_w = lane < k ? p / z : 0.f;
}

template <int PER_LANE>
__device__ __forceinline__ void topk_warp(const float *__restrict__ l, int E, int k, int lane, int &slot_e,
                                          float &slot_w)
{
    topk_warp<PER_LANE>(l, E, k, lane, slot_e, slot_w, [] {});
}

}  // namespace moe
