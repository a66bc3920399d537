// topk.cu -- top-k softmax routing (one warp per token).
//
// "Warp decode", section on the conventional MoE path: every token selects
// k of E experts (8 of 128 in the page's layer).  Selection is by logit,
// which orders experts exactly as the softmax probabilities do; ties go to
// the lower expert id and slots come out in descending order.  The k weights
// are the softmax probabilities renormalised over the chosen experts, i.e.
// exp(l_j - l_max) / sum_{chosen} exp(l_i - l_max), computed in FP32.
#include "common.cuh"

namespace moe {

constexpr int kTopkMaxPerLane = 128;   // E <= 4096
constexpr int kTopkWarps = 4;

// Order: larger logit first, then lower expert id.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib)
{
    return a > b || (a == b && ia < ib);
}

template <int PER_LANE>
__global__ void __launch_bounds__(kTopkWarps * 32)
topk_softmax_kernel(const float *__restrict__ logits, int M, int E, int k,
                    int32_t *__restrict__ ids, float *__restrict__ wts)
{
    // let the next kernel (the layer) get resident; it waits for us itself
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (t >= M)
        return;
    const float *l = logits + static_cast<int64_t>(t) * E;
    float v[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) {
        const int e = i * 32 + lane;
        v[i] = e < E ? __ldcg(l + e) : -INFINITY;
    }
    uint32_t taken[(PER_LANE + 31) / 32];
#pragma unroll
    for (int i = 0; i < (PER_LANE + 31) / 32; ++i)
        taken[i] = 0;
    float my_l = -INFINITY;     // slot j = lane keeps its (logit, id)
    int my_e = -1;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int e = i * 32 + lane;
            const bool free_ = e < E && !((taken[i >> 5] >> (i & 31)) & 1u);
            if (free_ && (be == 0x7fffffff || better(v[i], e, bv, be))) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || better(ov, oe, bv, be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) {           // the owner marks the entry as taken
            const int i = be >> 5;
#pragma unroll
            for (int ii = 0; ii < PER_LANE; ++ii)
                if (ii == i)
                    taken[ii >> 5] |= 1u << (ii & 31);
        }
        if (lane == j) {
            my_l = bv;
            my_e = be;
        }
    }
    const float mx = __shfl_sync(0xffffffffu, my_l, 0);
    const float p = lane < k ? expf(my_l - mx) : 0.f;
    const float z = warp_sum(p);
    if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = my_e;
        wts[static_cast<int64_t>(t) * k + lane] = p / z;
    }
}

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_topk_softmax(const float *logits, int32_t M, int32_t E, int32_t k,
                                      int32_t *topk_ids, float *topk_w, void *stream)
{
    if (M < 0 || E < 1 || E > 32 * kTopkMaxPerLane || k < 1 || k > 32 || k > E)
        return MOE_ERR_INVALID_ARG;
    if (M == 0)
        return MOE_OK;
    if (!logits || !topk_ids || !topk_w)
        return MOE_ERR_INVALID_ARG;
    dim3 grid((M + kTopkWarps - 1) / kTopkWarps), block(kTopkWarps * 32);
    cudaStream_t s = as_stream(stream);
    int per_lane = (E + 31) / 32;
    if (per_lane <= 4)
        topk_softmax_kernel<4><<<grid, block, 0, s>>>(logits, M, E, k, topk_ids, topk_w);
    else if (per_lane <= 16)
        topk_softmax_kernel<16><<<grid, block, 0, s>>>(logits, M, E, k, topk_ids, topk_w);
    else if (per_lane <= 32)
        topk_softmax_kernel<32><<<grid, block, 0, s>>>(logits, M, E, k, topk_ids, topk_w);
    else
        topk_softmax_kernel<kTopkMaxPerLane><<<grid, block, 0, s>>>(logits, M, E, k, topk_ids, topk_w);
    return launch_status();
}
