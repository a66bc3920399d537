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

// Selection only: lane j < k receives slot j's expert id and logit.  All 32
// lanes call it; l holds E logits; PER_LANE * 32 >= E.  `hook` runs after the
// logit loads are issued and before their values are used (set-up work that
// can overlap the memory latency).
template <int PER_LANE, typename Hook>
__device__ __forceinline__ void topk_select(const float *__restrict__ l, int E, int k, int lane, int &slot_e,
                                            float &slot_l, Hook hook)
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
    if constexpr (PER_LANE <= 8) {
        // tournament: each lane sorts its keys once (descending; equal keys
        // keep the lower index, i.e. the lower expert id, first), then every
        // round takes the warp maximum of the lanes' heads and the winning
        // lane pops its head
        int idx[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i)
            idx[i] = i;
#pragma unroll
        for (int i = 1; i < PER_LANE; ++i)
#pragma unroll
            for (int j = i; j > 0; --j) {
                // insertion step: move entry j up while strictly larger
                const bool sw = key[j] > key[j - 1];
                const uint32_t ka = key[j - 1], kb = key[j];
                const int ia = idx[j - 1], ib = idx[j];
                key[j - 1] = sw ? kb : ka;
                key[j] = sw ? ka : kb;
                idx[j - 1] = sw ? ib : ia;
                idx[j] = sw ? ia : ib;
            }
        for (int j = 0; j < k; ++j) {
            const uint32_t hk = key[0];
            const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
            const bool have = hk == mk && hk != 0u;
            const unsigned holders = __ballot_sync(0xffffffffu, have);
            uint32_t win;
            if ((holders & (holders - 1u)) == 0u) {
                const int wl = holders ? __ffs(holders) - 1 : 0;
                win = static_cast<uint32_t>(__shfl_sync(0xffffffffu, idx[0], wl) * 32 + wl);
            } else {
                win = __reduce_min_sync(0xffffffffu, have ? static_cast<uint32_t>(idx[0] * 32 + lane) : 0xFFFFFFFFu);
            }
            if (static_cast<int>(win & 31u) == lane) {
#pragma unroll
                for (int i = 0; i + 1 < PER_LANE; ++i) {
                    key[i] = key[i + 1];
                    idx[i] = idx[i + 1];
                }
                key[PER_LANE - 1] = 0u;
            }
            if (lane == j) {
                my_l = topk_unkey(mk);
                my_e = static_cast<int>(win);
            }
        }
        slot_e = my_e;
        slot_l = my_l;
        return;
    }
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
    slot_e = my_e;
    slot_l = my_l;
}

// The renormalised weight of slot `lane` from the selected logits (slot 0
// holds the maximum).  All 32 lanes call it.
__device__ __forceinline__ float topk_weight(float slot_l, int k, int lane)
{
    const float mx = __shfl_sync(0xffffffffu, slot_l, 0);
    const float p = lane < k ? expf(slot_l - mx) : 0.f;
    const float z = warp_sum(p);
    return lane < k ? p / z : 0.f;
}

// Lane j < k receives slot j: its expert id and renormalised weight.
template <int PER_LANE, typename Hook>
__device__ __forceinline__ void topk_warp(const float *__restrict__ l, int E, int k, int lane, int &slot_e,
                                          float &slot_w, Hook hook)
{
    float slot_l;
    topk_select<PER_LANE>(l, E, k, lane, slot_e, slot_l, hook);
    slot_w = topk_weight(slot_l, k, lane);
}

template <int PER_LANE>
__device__ __forceinline__ void topk_warp(const float *__restrict__ l, int E, int k, int lane, int &slot_e,
                                          float &slot_w)
{
    topk_warp<PER_LANE>(l, E, k, lane, slot_e, slot_w, [] {});
}

}  // namespace moe
