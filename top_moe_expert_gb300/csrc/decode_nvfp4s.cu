// decode_nvfp4s.cu -- output-centric decode of the routed expert layer on
// paired 4:8 sparse NVFP4 weights.
//
// The two kernels of "Warp decode" (cursor.com blog, section on how the two
// kernels work), on the weight format of "Hardware-Native Joint Sparse-
// Quantization for Trillion-Scale Mixture-of-Experts", App. A (2.75 bits per
// weight, a third of MXFP8's 8.25):
//   gate/up: one warp per (route, intermediate neuron); lanes stride over
//            64-weight chunks (16 bytes of kept codes, 4 of patterns, 2 of
//            scales), decode the kept values on the fly against x[t] staged
//            in shared memory as FP32, butterfly sum, h = SiLU(g) * u (FP32);
//   down:    one warp per (token, output); h[t] staged in shared memory; the
//            routing weight and the expert's constant fold into the down
//            accumulation, slots added in slot order.
// Every output's summation order depends only on the shapes, so repeats are
// bit-identical and a token's result does not depend on the other tokens.
#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "nvfp4s.cuh"

namespace moe {
namespace dn4 {

constexpr int kWarps = 8;

struct Packed {
    const uint8_t *v;       // kept E2M1 codes [E][N][K/4]
    const uint8_t *m;       // pattern nibbles [E][N][K/16]
    const uint8_t *s;       // UE4M3 scales    [E][N][K/32]
    const float *alpha;     // [E]
};

template <typename XT>
__device__ __forceinline__ float to_f32(XT v);
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

// Chunk c (64 weights) of row `row` of a [rows][K] projection dotted with x
// (the chunk's 64 activations), without the expert's constant.
__device__ __forceinline__ float row_chunk(const Packed &w, int64_t row, int K, int c, const float *x)
{
    const uint4 vv = ld_stream_u4(w.v + row * (K / 4) + 16 * static_cast<int64_t>(c));
    const uint32_t v[4] = {vv.x, vv.y, vv.z, vv.w};
    const uint32_t meta = __ldg(reinterpret_cast<const uint32_t *>(w.m + row * (K / 16)) + c);
    const uint32_t sc2 = __ldg(reinterpret_cast<const uint16_t *>(w.s + row * (K / 32)) + c);
    return nv4::chunk_dot(v, meta, sc2, x);
}

// h[r][n] = SiLU(g) * u, g and u the gate and up rows of route r's expert
// dotted with x[t]; grid (M*k, ceil(I / kWarps)).
template <typename XT>
__global__ void __launch_bounds__(kWarps * 32)
gate_up_kernel(const XT *__restrict__ x, int d, int I, const int32_t *__restrict__ ids, int k, int E, Packed w13,
               float *__restrict__ h, int32_t *__restrict__ dev_status)
{
    extern __shared__ float xs[];                             // [d]
    asm volatile("griddepcontrol.wait;" ::: "memory");       // ids / x may come from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x;
    const int n = blockIdx.y * kWarps + (threadIdx.x >> 5);
    const int t = r / k;
    const int e = ids[r];
    float *hout = h + static_cast<int64_t>(r) * I;
    if (e < 0 || e >= E) {                                    // invalid route: h = 0, counted once
        if (n < I && lane == 0)
            hout[n] = 0.f;
        if (blockIdx.y == 0 && threadIdx.x == 0 && dev_status)
            atomicAdd(dev_status, 1);
        return;
    }
    for (int i = threadIdx.x; i < d; i += kWarps * 32)
        xs[i] = to_f32<XT>(x[static_cast<int64_t>(t) * d + i]);
    __syncthreads();
    if (n >= I)
        return;
    const int64_t grow = static_cast<int64_t>(e) * (2 * I) + n, urow = grow + I;
    float ag = 0.f, au = 0.f;
    for (int c = lane; c < d / 64; c += 32) {
        ag += row_chunk(w13, grow, d, c, xs + 64 * c);
        au += row_chunk(w13, urow, d, c, xs + 64 * c);
    }
    const float a = w13.alpha[e];
    ag = warp_sum(ag) * a;
    au = warp_sum(au) * a;
    if (lane == 0)
        hout[n] = silu_mul(ag, au);
}

// y[t][o] = sum over slots j in order of w[t][j] * alpha[e_j] * (W2_{e_j}[o] . h[t][j]);
// grid (ceil(d / kWarps), M).
template <typename YT>
__global__ void __launch_bounds__(kWarps * 32)
down_kernel(const float *__restrict__ h, int d, int I, const int32_t *__restrict__ ids,
            const float *__restrict__ wts, int k, int E, Packed w2, YT *__restrict__ y)
{
    extern __shared__ float hs[];                             // [k][I]
    asm volatile("griddepcontrol.wait;" ::: "memory");       // h comes from the gate/up kernel
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.y;
    const int o = blockIdx.x * kWarps + (threadIdx.x >> 5);
    for (int i = threadIdx.x; i < k * I; i += kWarps * 32)
        hs[i] = h[static_cast<int64_t>(t) * k * I + i];
    __syncthreads();
    if (o >= d)
        return;
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
        const int e = ids[static_cast<int64_t>(t) * k + j];
        if (e < 0 || e >= E)
            continue;
        float s = 0.f;
        for (int c = lane; c < I / 64; c += 32)
            s += row_chunk(w2, static_cast<int64_t>(e) * d + o, I, c, hs + j * I + 64 * c);
        s = warp_sum(s);
        acc = fmaf(wts[static_cast<int64_t>(t) * k + j] * w2.alpha[e], s, acc);
    }
    if (lane == 0) {
        if constexpr (sizeof(YT) == 4)
            y[static_cast<int64_t>(t) * d + o] = acc;
        else
            y[static_cast<int64_t>(t) * d + o] = __float2bfloat16_rn(acc);
    }
}

}  // namespace dn4

bool decode_nvfp4s_eligible(int k, int d, int I)
{
    return d % 64 == 0 && I % 64 == 0 && d >= 64 && I >= 64 && static_cast<size_t>(d) * sizeof(float) <= 200 * 1024 &&
           static_cast<size_t>(k) * I * sizeof(float) <= 200 * 1024 && (I + dn4::kWarps - 1) / dn4::kWarps <= 65535;
}

moe_status_t decode_nvfp4s_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                  const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                  void *y, bool y_f32, float *h, int32_t *dev_status, cudaStream_t s)
{
    using namespace dn4;
    if (!decode_nvfp4s_eligible(k, d, I))
        return MOE_ERR_UNSUPPORTED;
    for (const moe_weights_t *w : {w13, w2})
        if (!w->alpha || !aligned(w->q, 16) || !aligned(w->zero, 4) || !aligned(w->scale, 2))
            return MOE_ERR_INVALID_ARG;
    const Packed p13{static_cast<const uint8_t *>(w13->q), static_cast<const uint8_t *>(w13->zero),
                     static_cast<const uint8_t *>(w13->scale), w13->alpha};
    const Packed p2{static_cast<const uint8_t *>(w2->q), static_cast<const uint8_t *>(w2->zero),
                    static_cast<const uint8_t *>(w2->scale), w2->alpha};
    const size_t smem_a = static_cast<size_t>(d) * sizeof(float);
    const size_t smem_b = static_cast<size_t>(k) * I * sizeof(float);
    const void *ka = x_bf16 ? reinterpret_cast<const void *>(gate_up_kernel<__nv_bfloat16>)
                            : reinterpret_cast<const void *>(gate_up_kernel<__half>);
    const void *kb = y_f32 ? reinterpret_cast<const void *>(down_kernel<float>)
                           : reinterpret_cast<const void *>(down_kernel<__nv_bfloat16>);
    if ((smem_a > 48 * 1024 && !smem_attr(ka, 200 * 1024)) || (smem_b > 48 * 1024 && !smem_attr(kb, 200 * 1024)))
        return MOE_ERR_CUDA;
    const dim3 ga(static_cast<unsigned>(M * k), static_cast<unsigned>((I + kWarps - 1) / kWarps));
    cudaError_t err;
    if (x_bf16)
        err = launch_pdl(gate_up_kernel<__nv_bfloat16>, ga, dim3(kWarps * 32), smem_a, s,
                         static_cast<const __nv_bfloat16 *>(x), d, I, ids, k, E, p13, h, dev_status);
    else
        err = launch_pdl(gate_up_kernel<__half>, ga, dim3(kWarps * 32), smem_a, s, static_cast<const __half *>(x), d,
                         I, ids, k, E, p13, h, dev_status);
    if (err != cudaSuccess)
        return MOE_ERR_CUDA;
    const dim3 gb(static_cast<unsigned>((d + kWarps - 1) / kWarps), static_cast<unsigned>(M));
    if (y_f32)
        err = launch_pdl(down_kernel<float>, gb, dim3(kWarps * 32), smem_b, s, static_cast<const float *>(h), d, I,
                         ids, wts, k, E, p2, static_cast<float *>(y));
    else
        err = launch_pdl(down_kernel<__nv_bfloat16>, gb, dim3(kWarps * 32), smem_b, s, static_cast<const float *>(h),
                         d, I, ids, wts, k, E, p2, static_cast<__nv_bfloat16 *>(y));
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
