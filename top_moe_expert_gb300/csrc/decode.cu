// decode.cu -- output-centric small-batch path of the routed expert FFN.
//
// "Warp decode" (cursor.com blog), sections on what changed and how the two
// kernels work: parallelism is organised around outputs instead of experts.
//   gate/up kernel: one warp per intermediate neuron n of one (token, routed
//     expert) pair; it streams the gate row and the up row of that neuron,
//     converts MXFP8 to FP32 on the fly, keeps two FP32 accumulators, reduces
//     with a warp butterfly and writes SiLU(g) * u.
//   down kernel: one warp per output dimension o of one token; it loops over
//     the k routed experts, streams the down row and the intermediate h, and
//     folds the routing weight of each expert into a single FP32 accumulator;
//     a __shfl_xor_sync butterfly produces the output scalar.
// There is no alignment, padding, scatter or combine buffer; the only
// intermediate is h (FP32, [M*k][I]) in the caller's workspace.
//
// GB300 specifics: weights are streamed with 16-byte L1::no_allocate loads,
// four chunks per lane in flight per row; the down kernel is launched with
// programmatic dependent launch and prefetches its W2 rows into L2 before it
// waits for the gate/up grid, so the W2 stream overlaps the gate/up tail.
// Per-output summation order depends only on (d, I, k) and the lane layout,
// never on M, on other tokens or on the grid, so results are bit-stable.
#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"

namespace moe {

constexpr int kDecWarps = 8;              // warps per CTA (as on the page)
constexpr int kDecBatch = 4;              // 16-byte chunks per lane in flight

struct DecWeights {
    const uint8_t *q;       // MXFP8 codes / AWQ packed nibbles (as bytes)
    const uint8_t *s;       // E8M0 bytes / fp16 scales (as bytes)
    const int32_t *z;       // AWQ zeros or null
    int N, K;
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---- activation chunk -> floats -------------------------------------------------
template <typename XT>
__device__ __forceinline__ void x_to_float(uint32_t w, float &a, float &b);
template <>
__device__ __forceinline__ void x_to_float<__nv_bfloat16>(uint32_t w, float &a, float &b) { bf16x2_to_float(w, a, b); }
template <>
__device__ __forceinline__ void x_to_float<__half>(uint32_t w, float &a, float &b) { f16x2_to_float(w, a, b); }

// ---- one 16-byte weight chunk dotted with its activation slice -----------------
// MXFP8: 16 elements, scale byte index = chunk/2.  Returns scale * sum(q*x).
template <typename XT>
__device__ __forceinline__ float mx_chunk_dot(uint4 wq, float scale, const XT *xs)
{
    const uint4 xa = __ldg(reinterpret_cast<const uint4 *>(xs));
    const uint4 xb = __ldg(reinterpret_cast<const uint4 *>(xs) + 1);
    const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w};
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float q0, q1, q2, q3, x0, x1, x2, x3;
        e4m3x4_to_float(ww[i], q0, q1, q2, q3);
        x_to_float<XT>(xw[2 * i], x0, x1);
        x_to_float<XT>(xw[2 * i + 1], x2, x3);
        acc = fmaf(q0, x0, acc);
        acc = fmaf(q1, x1, acc);
        acc = fmaf(q2, x2, acc);
        acc = fmaf(q3, x3, acc);
    }
    return acc * scale;
}

// AWQ: 32 elements (4 words of 8 nibbles), one (scale, zero) per 128.
// Returns scale * (sum(q*x) - zero * sum(x)).
template <typename XT>
__device__ __forceinline__ float awq_chunk_dot(uint4 wq, float scale, float zero, const XT *xs)
{
    const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w};
    float acc = 0.f, xsum = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(xs) + i);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            float x0, x1;
            x_to_float<XT>(xw[p], x0, x1);
            const float q0 = static_cast<float>((ww[i] >> (8 * p)) & 0xFu);
            const float q1 = static_cast<float>((ww[i] >> (8 * p + 4)) & 0xFu);
            acc = fmaf(q0, x0, acc);
            acc = fmaf(q1, x1, acc);
            xsum += x0 + x1;
        }
    }
    return scale * fmaf(-zero, xsum, acc);
}

// ---- gate/up ---------------------------------------------------------------------
template <int FMT, typename XT>
__global__ void __launch_bounds__(kDecWarps * 32)
decode_gate_up_kernel(const XT *__restrict__ x, int d, int I, const int32_t *__restrict__ ids,
                      int k, int E, DecWeights w13, float *__restrict__ h,
                      int32_t *__restrict__ dev_status)
{
    constexpr int EPC = FMT == MOE_W_MXFP8 ? 16 : 32;        // elements per chunk
    pdl_wait();                  // ids / x may come from the previous kernel
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x;                                 // route t*k + j
    const int n = blockIdx.y * kDecWarps + (threadIdx.x >> 5);
    const int t = r / k;
    const int e = ids[r];
    float *hout = h + static_cast<int64_t>(r) * I;
    if (e < 0 || e >= E) {
        if (n < I && lane == 0)
            hout[n] = 0.f;
        if (blockIdx.y == 0 && threadIdx.x == 0 && dev_status)
            atomicAdd(dev_status, 1);
        return;
    }
    if (n >= I)
        return;
    const int nchunk = d / EPC;                               // multiple of 32
    const int64_t grow = static_cast<int64_t>(e) * (2 * I) + n;
    const int64_t urow = grow + I;
    const int64_t rowbytes = FMT == MOE_W_MXFP8 ? d : d / 2;
    const uint8_t *gq = w13.q + grow * rowbytes;
    const uint8_t *uq = w13.q + urow * rowbytes;
    const XT *xt = x + static_cast<int64_t>(t) * d;
    float ag = 0.f, au = 0.f;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * kDecBatch) {
        uint4 g[kDecBatch], u[kDecBatch];
#pragma unroll
        for (int i = 0; i < kDecBatch; ++i) {
            const int c = c0 + i * 32 + lane;
            if (c < nchunk) {
                g[i] = ld_stream_u4(gq + static_cast<int64_t>(c) * 16);
                u[i] = ld_stream_u4(uq + static_cast<int64_t>(c) * 16);
            }
        }
#pragma unroll
        for (int i = 0; i < kDecBatch; ++i) {
            const int c = c0 + i * 32 + lane;
            if (c < nchunk) {
                const XT *xs = xt + static_cast<int64_t>(c) * EPC;
                if constexpr (FMT == MOE_W_MXFP8) {
                    const float sg = e8m0_to_float(__ldg(w13.s + grow * (d / 32) + (c >> 1)));
                    const float su = e8m0_to_float(__ldg(w13.s + urow * (d / 32) + (c >> 1)));
                    ag += mx_chunk_dot<XT>(g[i], sg, xs);
                    au += mx_chunk_dot<XT>(u[i], su, xs);
                } else {
                    const __half *sc = reinterpret_cast<const __half *>(w13.s);
                    const int grp = c >> 2, G = d / 128;
                    const float sg = __half2float(sc[grow * G + grp]);
                    const float su = __half2float(sc[urow * G + grp]);
                    const int64_t zr = static_cast<int64_t>(e) * (2 * I / 8);
                    const float zg = static_cast<float>((static_cast<uint32_t>(__ldg(w13.z + (zr + n / 8) * G + grp)) >> (4 * (n & 7))) & 0xFu);
                    const float zu = static_cast<float>((static_cast<uint32_t>(__ldg(w13.z + (zr + (I + n) / 8) * G + grp)) >> (4 * ((I + n) & 7))) & 0xFu);
                    ag += awq_chunk_dot<XT>(g[i], sg, zg, xs);
                    au += awq_chunk_dot<XT>(u[i], su, zu, xs);
                }
            }
        }
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    if (lane == 0)
        hout[n] = silu_mul(ag, au);
}

// ---- down + combine ----------------------------------------------------------------
// One CTA = kDecWarps consecutive outputs of one token; h[t] (k x I floats)
// is staged once in shared memory.
template <int FMT, typename YT>
__global__ void __launch_bounds__(kDecWarps * 32)
decode_down_kernel(const float *__restrict__ h, int d, int I, const int32_t *__restrict__ ids,
                   const float *__restrict__ wts, int k, int E, DecWeights w2, YT *__restrict__ y)
{
    constexpr int EPC = FMT == MOE_W_MXFP8 ? 16 : 32;
    extern __shared__ float hs[];                             // [k][I]
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.y;
    const int o = blockIdx.x * kDecWarps + (threadIdx.x >> 5);
    const int rowbytes = FMT == MOE_W_MXFP8 ? I : I / 2;
    const int nc_row = I / EPC;                               // chunks per row
    const int total = k * nc_row;

    // Before the dependency wait: W2 rows depend only on the routing inputs,
    // so pull them towards L2 while the gate/up grid is still running.
    if (o < d) {
        for (int j = 0; j < k; ++j) {
            const int e = ids[static_cast<int64_t>(t) * k + j];
            if (e < 0 || e >= E)
                continue;
            const uint8_t *row = w2.q + (static_cast<int64_t>(e) * d + o) * rowbytes;
            for (int off = lane * 128; off < rowbytes; off += 32 * 128)
                prefetch_l2(row + off);
        }
    }
    pdl_wait();
    pdl_launch_dependents();

    const float *ht = h + static_cast<int64_t>(t) * k * I;
    for (int i = threadIdx.x * 4; i < k * I; i += blockDim.x * 4)
        *reinterpret_cast<float4 *>(hs + i) = *reinterpret_cast<const float4 *>(ht + i);
    __syncthreads();
    if (o >= d)
        return;

    float acc = 0.f;
    for (int c0 = 0; c0 < total; c0 += 32 * kDecBatch) {
        uint4 wv[kDecBatch];
        int jj[kDecBatch], ch[kDecBatch], ee[kDecBatch];
#pragma unroll
        for (int i = 0; i < kDecBatch; ++i) {
            const int c = c0 + i * 32 + lane;
            ee[i] = -1;
            if (c < total) {
                jj[i] = c / nc_row;
                ch[i] = c - jj[i] * nc_row;
                const int e = ids[static_cast<int64_t>(t) * k + jj[i]];
                if (e >= 0 && e < E) {
                    ee[i] = e;
                    wv[i] = ld_stream_u4(w2.q + (static_cast<int64_t>(e) * d + o) * rowbytes + ch[i] * 16);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kDecBatch; ++i) {
            if (ee[i] < 0)
                continue;
            const int e = ee[i];
            const float wj = wts[static_cast<int64_t>(t) * k + jj[i]];
            const float *hv = hs + jj[i] * I + ch[i] * EPC;
            const int64_t row = static_cast<int64_t>(e) * d + o;
            if constexpr (FMT == MOE_W_MXFP8) {
                const float sc = e8m0_to_float(__ldg(w2.s + row * (I / 32) + (ch[i] >> 1)));
                const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
                float p = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float q0, q1, q2, q3;
                    e4m3x4_to_float(ww[q], q0, q1, q2, q3);
                    const float4 hh = *reinterpret_cast<const float4 *>(hv + 4 * q);
                    p = fmaf(q0, hh.x, p);
                    p = fmaf(q1, hh.y, p);
                    p = fmaf(q2, hh.z, p);
                    p = fmaf(q3, hh.w, p);
                }
                acc = fmaf(wj * sc, p, acc);
            } else {
                const __half *scp = reinterpret_cast<const __half *>(w2.s);
                const int G = I / 128, grp = ch[i] >> 2;
                const float sc = __half2float(scp[row * G + grp]);
                const float z = static_cast<float>((static_cast<uint32_t>(__ldg(w2.z + (static_cast<int64_t>(e) * (d / 8) + o / 8) * G + grp)) >> (4 * (o & 7))) & 0xFu);
                const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
                float p = 0.f, hsum = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 ha = *reinterpret_cast<const float4 *>(hv + 8 * q);
                    const float4 hb = *reinterpret_cast<const float4 *>(hv + 8 * q + 4);
                    const float hh[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
                    for (int b = 0; b < 8; ++b) {
                        p = fmaf(static_cast<float>((ww[q] >> (4 * b)) & 0xFu), hh[b], p);
                        hsum += hh[b];
                    }
                }
                acc = fmaf(wj * sc, fmaf(-z, hsum, p), acc);
            }
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) {
        if constexpr (sizeof(YT) == 4)
            y[static_cast<int64_t>(t) * d + o] = acc;
        else
            y[static_cast<int64_t>(t) * d + o] = __float2bfloat16_rn(acc);
    }
}

template <int FMT, typename XT, typename YT>
moe_status_t decode_launch(const void *x, int M, int d, const int32_t *ids, const float *wts, int k,
                           const moe_weights_t *w13, const moe_weights_t *w2, void *y, float *h,
                           int32_t *dev_status, cudaStream_t s)
{
    const int I = w2->K, E = w13->E;
    DecWeights a{static_cast<const uint8_t *>(w13->q), static_cast<const uint8_t *>(w13->scale),
                 static_cast<const int32_t *>(w13->zero), w13->N, w13->K};
    DecWeights b{static_cast<const uint8_t *>(w2->q), static_cast<const uint8_t *>(w2->scale),
                 static_cast<const int32_t *>(w2->zero), w2->N, w2->K};
    dim3 g1(M * k, (I + kDecWarps - 1) / kDecWarps);
    if (launch_pdl(decode_gate_up_kernel<FMT, XT>, g1, dim3(kDecWarps * 32), 0, s,
                   static_cast<const XT *>(x), d, I, ids, k, E, a, h, dev_status) != cudaSuccess)
        return MOE_ERR_CUDA;
    const size_t smem = static_cast<size_t>(k) * I * sizeof(float);
    auto kd = decode_down_kernel<FMT, YT>;
    if (smem > 48 * 1024 && !smem_attr(reinterpret_cast<const void *>(kd), 200 * 1024))
        return MOE_ERR_CUDA;
    dim3 g2((d + kDecWarps - 1) / kDecWarps, M);
    if (launch_pdl(kd, g2, dim3(kDecWarps * 32), smem, s, static_cast<const float *>(h), d, I, ids, wts,
                   k, E, b, static_cast<YT *>(y)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_ffn_decode_workspace_size(int32_t M, int32_t k, int32_t d, int32_t I, size_t *bytes)
{
    if (M < 0 || k < 1 || d < 1 || I < 1 || !bytes)
        return MOE_ERR_INVALID_ARG;
    // The first kWsReserved bytes belong to the one-kernel single-token path
    // (its CTA count and its h exchange words); every other path starts its
    // data after them, so one workspace serves calls of any batch size in
    // turn without disturbing them.
    const size_t h = kWsReserved + ws_round(static_cast<size_t>(M) * k * I * sizeof(float));
    *bytes = h;
    return MOE_OK;
}

static moe_status_t check_weights(const moe_weights_t *w, int N, int K)
{
    if (!w || !w->q || !w->scale || w->N != N || w->K != K || w->E < 1)
        return MOE_ERR_INVALID_ARG;
    if (w->fmt == MOE_W_MXFP8) {
        if (K % 32 != 0)
            return MOE_ERR_INVALID_ARG;
    } else if (w->fmt == MOE_W_AWQ4) {
        if (!w->zero || K % 128 != 0 || N % 8 != 0)
            return MOE_ERR_INVALID_ARG;
    } else if (w->fmt == MOE_W_NVFP4S) {
        if (!w->zero || !w->alpha || K % 64 != 0)
            return MOE_ERR_INVALID_ARG;
    } else {
        return MOE_ERR_INVALID_ARG;
    }
    if (!aligned(w->q, 16))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// the single-token NVFP4S kernel's bulk copies want 16-byte aligned code,
// pattern and gate/up scale arrays; its down scales are read 8 bytes at a time
static bool nv4_pipe_aligned(const moe_weights_t *w13, const moe_weights_t *w2)
{
    return aligned(w13->q, 16) && aligned(w13->zero, 16) && aligned(w13->scale, 16) && aligned(w2->q, 16) &&
           aligned(w2->zero, 16) && aligned(w2->scale, 8) && w13->alpha && w2->alpha;
}

MOE_API moe_status_t moe_ffn_decode(const void *x, int32_t xdt, int32_t M, int32_t d,
                                    const int32_t *topk_ids, const float *topk_w, int32_t k,
                                    const moe_weights_t *w13, const moe_weights_t *w2,
                                    void *y, int32_t ydt, void *ws, size_t ws_bytes,
                                    int32_t *dev_status, void *stream)
{
    if (M < 0 || d < 1 || k < 1 || k > 32 || !w13 || !w2)
        return MOE_ERR_INVALID_ARG;
    const int I = w2->K;
    moe_status_t st;
    if ((st = check_weights(w13, 2 * I, d)) != MOE_OK || (st = check_weights(w2, d, I)) != MOE_OK)
        return st;
    if (w13->E != w2->E)
        return MOE_ERR_INVALID_ARG;
    if (w13->fmt != w2->fmt)
        return MOE_ERR_INVALID_ARG;
    const int fmt = w13->fmt;
    if (fmt == MOE_W_MXFP8 && (d % 512 != 0 || I % 32 != 0))
        return MOE_ERR_UNSUPPORTED;
    if (fmt == MOE_W_AWQ4 && (d % 1024 != 0 || I % 128 != 0))
        return MOE_ERR_UNSUPPORTED;
    if (fmt == MOE_W_NVFP4S && !decode_nvfp4s_eligible(k, d, I))
        return MOE_ERR_UNSUPPORTED;
    if (ydt != MOE_BF16 && ydt != MOE_FP32)
        return MOE_ERR_UNSUPPORTED;
    if (fmt == MOE_W_MXFP8 ? xdt != MOE_BF16 : (xdt != MOE_BF16 && xdt != MOE_FP16))
        return MOE_ERR_UNSUPPORTED;
    if (static_cast<size_t>(k) * I * sizeof(float) > 200 * 1024)
        return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(M) * k > INT32_MAX || M > 65535)
        return MOE_ERR_UNSUPPORTED;
    if (M == 0)
        return MOE_OK;
    if (!x || !topk_ids || !topk_w || !y || !aligned(x, 16))
        return MOE_ERR_INVALID_ARG;
    size_t need;
    moe_ffn_decode_workspace_size(M, k, d, I, &need);
    if (!ws || ws_bytes < need || !aligned(ws, 256))
        return MOE_ERR_WORKSPACE;
    // past the reserved bytes: h of the two-kernel and per-scalar paths
    float *h = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kWsReserved);
    cudaStream_t s = as_stream(stream);
    if (fmt == MOE_W_NVFP4S && decode_pipe_nv4_eligible(M, k, d, I, w13->E) && nv4_pipe_aligned(w13, w2)) {
        // one token, paired 4:8 sparse NVFP4: one kernel (gate/up, SwiGLU, down)
        return decode_pipe_nv4_launch(x, xdt == MOE_BF16, d, I, w13->E, topk_ids, topk_w, nullptr, nullptr, nullptr, k,
                                      w13, w2, y, ydt == MOE_FP32, ws, dev_status, s);
    }
    if (fmt == MOE_W_NVFP4S)
        return decode_nvfp4s_launch(x, xdt == MOE_BF16, M, d, I, w13->E, topk_ids, topk_w, k, w13, w2, y,
                                    ydt == MOE_FP32, h, dev_status, s);
    if (fmt == MOE_W_MXFP8 && decode_pipe_eligible(M, k, d, I, w13->E) && aligned(w13->scale, 16) &&
        aligned(w2->q, 16) && aligned(w2->scale, 8)) {
        // one token on the standard layout: one kernel (gate/up, SwiGLU, down)
        return decode_pipe_launch(static_cast<const __nv_bfloat16 *>(x), d, I, w13->E, topk_ids, topk_w, nullptr,
                                  nullptr, nullptr, k, static_cast<const uint8_t *>(w13->q),
                                  static_cast<const uint8_t *>(w13->scale), static_cast<const uint8_t *>(w2->q),
                                  static_cast<const uint8_t *>(w2->scale), y, ydt == MOE_FP32, ws, dev_status, s);
    }
    if (fmt == MOE_W_AWQ4 && decode_pipe_awq_eligible(M, k, d, I, w13->E) && aligned(w13->q, 16) &&
        aligned(w2->q, 16) && aligned(w13->scale, 16) && aligned(w13->zero, 16)) {
        // one token, 4-bit AWQ: one kernel (gate/up, SwiGLU, down)
        return decode_pipe_awq_launch(x, xdt == MOE_BF16, d, I, w13->E, topk_ids, topk_w, nullptr, nullptr, nullptr, k,
                                      w13, w2, y, ydt == MOE_FP32, ws, dev_status, s);
    }
    if (fmt == MOE_W_MXFP8 && decode_stream_eligible(M, k, d, I, w13->E, w13->q, w13->scale, w2->q, w2->scale)) {
        const moe_status_t st2 = decode_stream_launch(static_cast<const __nv_bfloat16 *>(x), M, d, I, w13->E, topk_ids, topk_w, k,
                                    static_cast<const uint8_t *>(w13->q), static_cast<const uint8_t *>(w13->scale),
                                    static_cast<const uint8_t *>(w2->q), static_cast<const uint8_t *>(w2->scale),
                                    y, ydt == MOE_FP32, h, dev_status, s);
        if (st2 != MOE_ERR_UNSUPPORTED)      // shapes it cannot stage take the general kernels
            return st2;
    }
    if (fmt == MOE_W_MXFP8) {
        return ydt == MOE_FP32
                   ? decode_launch<MOE_W_MXFP8, __nv_bfloat16, float>(x, M, d, topk_ids, topk_w, k, w13, w2, y, h, dev_status, s)
                   : decode_launch<MOE_W_MXFP8, __nv_bfloat16, __nv_bfloat16>(x, M, d, topk_ids, topk_w, k, w13, w2, y, h, dev_status, s);
    }
    if (xdt == MOE_FP16)
        return ydt == MOE_FP32
                   ? decode_launch<MOE_W_AWQ4, __half, float>(x, M, d, topk_ids, topk_w, k, w13, w2, y, h, dev_status, s)
                   : decode_launch<MOE_W_AWQ4, __half, __nv_bfloat16>(x, M, d, topk_ids, topk_w, k, w13, w2, y, h, dev_status, s);
    return ydt == MOE_FP32
               ? decode_launch<MOE_W_AWQ4, __nv_bfloat16, float>(x, M, d, topk_ids, topk_w, k, w13, w2, y, h, dev_status, s)
               : decode_launch<MOE_W_AWQ4, __nv_bfloat16, __nv_bfloat16>(x, M, d, topk_ids, topk_w, k, w13, w2, y, h, dev_status, s);
}

MOE_API moe_status_t moe_ffn_decode_logits(const float *logits, const void *x, int32_t xdt, int32_t M, int32_t d,
                                           int32_t k, const moe_weights_t *w13, const moe_weights_t *w2,
                                           int32_t *topk_ids, float *topk_w, void *y, int32_t ydt, void *ws,
                                           size_t ws_bytes, int32_t *dev_status, void *stream)
{
    if (M < 0 || d < 1 || k < 1 || k > 32 || !w13 || !w2)
        return MOE_ERR_INVALID_ARG;
    if (M == 0)
        return MOE_OK;
    if (!logits || !topk_ids || !topk_w)
        return MOE_ERR_INVALID_ARG;
    const int I = w2->K, E = w13->E;
    // one token on the standard layout: one kernel with the routing inside
    if (M == 1 && w2->fmt == MOE_W_MXFP8 && w13->fmt == MOE_W_MXFP8 && xdt == MOE_BF16 &&
        (ydt == MOE_BF16 || ydt == MOE_FP32) && check_weights(w13, 2 * I, d) == MOE_OK &&
        check_weights(w2, d, I) == MOE_OK && w2->E == E && decode_pipe_eligible(1, k, d, I, E) &&
        decode_pipe_route_eligible(E, k) && aligned(w13->scale, 16) && aligned(w2->q, 16) &&
        aligned(w2->scale, 8) && x && y && aligned(x, 16)) {
        size_t need;
        moe_ffn_decode_workspace_size(M, k, d, I, &need);
        if (!ws || ws_bytes < need || !aligned(ws, 256))
            return MOE_ERR_WORKSPACE;
        return decode_pipe_launch(static_cast<const __nv_bfloat16 *>(x), d, I, E, nullptr, nullptr, logits,
                                  topk_ids, topk_w, k, static_cast<const uint8_t *>(w13->q),
                                  static_cast<const uint8_t *>(w13->scale), static_cast<const uint8_t *>(w2->q),
                                  static_cast<const uint8_t *>(w2->scale), y, ydt == MOE_FP32, ws, dev_status,
                                  as_stream(stream));
    }
    // one token, 4-bit AWQ: one kernel with the routing inside
    if (M == 1 && w2->fmt == MOE_W_AWQ4 && w13->fmt == MOE_W_AWQ4 && (xdt == MOE_BF16 || xdt == MOE_FP16) &&
        (ydt == MOE_BF16 || ydt == MOE_FP32) && check_weights(w13, 2 * I, d) == MOE_OK &&
        check_weights(w2, d, I) == MOE_OK && w2->E == E && decode_pipe_awq_eligible(1, k, d, I, E) &&
        decode_pipe_awq_route_eligible(E, k) && aligned(w13->q, 16) && aligned(w2->q, 16) &&
        aligned(w13->scale, 16) && aligned(w13->zero, 16) && x && y &&
        aligned(x, 16)) {
        size_t need;
        moe_ffn_decode_workspace_size(M, k, d, I, &need);
        if (!ws || ws_bytes < need || !aligned(ws, 256))
            return MOE_ERR_WORKSPACE;
        return decode_pipe_awq_launch(x, xdt == MOE_BF16, d, I, E, nullptr, nullptr, logits, topk_ids, topk_w, k,
                                      w13, w2, y, ydt == MOE_FP32, ws, dev_status, as_stream(stream));
    }
    // one token, paired 4:8 sparse NVFP4: one kernel with the routing inside
    if (M == 1 && w2->fmt == MOE_W_NVFP4S && w13->fmt == MOE_W_NVFP4S && (xdt == MOE_BF16 || xdt == MOE_FP16) &&
        (ydt == MOE_BF16 || ydt == MOE_FP32) && check_weights(w13, 2 * I, d) == MOE_OK &&
        check_weights(w2, d, I) == MOE_OK && w2->E == E && decode_pipe_nv4_eligible(1, k, d, I, E) &&
        decode_pipe_nv4_route_eligible(E, k) && nv4_pipe_aligned(w13, w2) && x && y && aligned(x, 16)) {
        size_t need;
        moe_ffn_decode_workspace_size(M, k, d, I, &need);
        if (!ws || ws_bytes < need || !aligned(ws, 256))
            return MOE_ERR_WORKSPACE;
        return decode_pipe_nv4_launch(x, xdt == MOE_BF16, d, I, E, nullptr, nullptr, logits, topk_ids, topk_w, k,
                                      w13, w2, y, ydt == MOE_FP32, ws, dev_status, as_stream(stream));
    }
    // otherwise: routing, then the layer
    moe_status_t st = moe_topk_softmax(logits, M, E, k, topk_ids, topk_w, stream);
    if (st != MOE_OK)
        return st;
    return moe_ffn_decode(x, xdt, M, d, topk_ids, topk_w, k, w13, w2, y, ydt, ws, ws_bytes, dev_status, stream);
}
