// ep.cu -- expert-parallel sharding of the routing.
//
// "Hardware-Native Joint Sparse-Quantization for Trillion-Scale Mixture-of-
// Experts", App. D.3, serves the layer with the experts sharded over the
// ranks of an expert-parallel group.  A rank that owns experts [e_lo, e_hi)
// runs the layer on its own expert weights (indexed 0 .. e_hi - e_lo - 1)
// with every route of another rank's experts made invalid: the layer skips
// invalid routes, so the rank's output is its experts' share of y, and the
// shares of all ranks add up to the full layer.
#include "common.cuh"

namespace moe {

__global__ void ep_local_routes_kernel(const int32_t *__restrict__ ids, int64_t n, int32_t e_lo, int32_t e_hi,
                                       int32_t *__restrict__ out)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int32_t e = ids[i];
        out[i] = (e >= e_lo && e < e_hi) ? e - e_lo : -1;
    }
}

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_ep_local_routes(const int32_t *topk_ids, int64_t n, int32_t e_lo, int32_t e_hi,
                                         int32_t *local_ids, void *stream)
{
    if (n < 0 || e_lo < 0 || e_hi < e_lo)
        return MOE_ERR_INVALID_ARG;
    if (n == 0)
        return MOE_OK;
    if (!topk_ids || !local_ids)
        return MOE_ERR_INVALID_ARG;
    const int threads = 256;
    const int64_t blocks64 = (n + threads - 1) / threads;
    const int blocks = static_cast<int>(blocks64 < 4096 ? blocks64 : 4096);
    ep_local_routes_kernel<<<blocks, threads, 0, as_stream(stream)>>>(topk_ids, n, e_lo, e_hi, local_ids);
    return launch_status();
}
