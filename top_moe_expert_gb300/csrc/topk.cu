// topk.cu -- top-k softmax routing (one warp per token); the selection
// itself is topk_warp (topk.cuh).
#include "common.cuh"
#include "topk.cuh"

namespace moe {

constexpr int kTopkMaxPerLane = 128;   // E <= 4096
constexpr int kTopkWarps = 4;

template <int PER_LANE>
__global__ void __launch_bounds__(kTopkWarps * 32)
topk_softmax_kernel(const float *__restrict__ logits, int M, int E, int k,
                    int32_t *__restrict__ ids, float *__restrict__ wts)
{
    // the logits may come from the previous kernel; the next kernel may get
    // resident now (it waits for this one itself)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (t >= M)
        return;
    int e;
    float w;
    topk_warp<PER_LANE>(logits + static_cast<int64_t>(t) * E, E, k, lane, e, w);
    if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = e;
        wts[static_cast<int64_t>(t) * k + lane] = w;
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
    cudaError_t e;
    if (per_lane <= 4)
        e = launch_pdl(topk_softmax_kernel<4>, grid, block, 0, s, logits, M, E, k, topk_ids, topk_w);
    else if (per_lane <= 16)
        e = launch_pdl(topk_softmax_kernel<16>, grid, block, 0, s, logits, M, E, k, topk_ids, topk_w);
    else if (per_lane <= 32)
        e = launch_pdl(topk_softmax_kernel<32>, grid, block, 0, s, logits, M, E, k, topk_ids, topk_w);
    else
        e = launch_pdl(topk_softmax_kernel<kTopkMaxPerLane>, grid, block, 0, s, logits, M, E, k, topk_ids, topk_w);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
