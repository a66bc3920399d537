// grouped_awq_mma.cu -- expert-centric grouped path for 4-bit AWQ weights
// with MoE blocks of b <= 16 rows, on mma.sync.
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic" (opening paragraph):
// the packed-AWQ expert GEMMs applied to the aligned rows, one MoE block of b
// rows of one expert at a time.  With b <= 16 a block is one M-tile of
// mma.sync m16n8k16, and each expert's weights stream through once per block
// as the B operand in the raw-code form of decode_awq_m1.cuh: the f16 pair
// (1024 + q) from one AND-OR, the zero and the offset folded out in FP32 once
// per group of 128, s (D - (1024 + z) sum a).
//
// One CTA per SM, 16 warps, one kernel for both GEMMs:
//  * Phase 1 (gate/up): units (block, 8 rows of W13) are split evenly over
//    the CTAs in block order.  A CTA stages the A operand of each block it
//    touches -- the block's rows of x, scaled per row by an exact power of two
//    into f16 range, in the MMA's K order, with per-group sums -- and its
//    warps split the block's units; a warp keeps the next items' loads in
//    flight while one item's eight MMAs run.  A unit writes the FP32 gate or
//    up values of the block's routes and bumps the block's counter.
//  * Phase 2 (down): units (block, 8 rows of W2) in the same way.  A CTA waits
//    (bounded) until its block's counter shows every gate/up unit done, forms
//    h = w SiLU(g) u of the block's routes, scales each row by a power of two
//    and splits it into f16 hi + lo (staged like x), then runs 2 x 8 MMAs per
//    group and writes each route's FP32 down-projection row to Yr.
//  * The routing-weighted sum over each token's slots is the grouped path's
//    combine kernel (slot order), chained by programmatic dependent launch.
// Every value has one owner and a fixed summation order, so results do not
// depend on the grid, the block membership of other routes, or timing.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "grouped_awq_mma.cuh"
#include "grouped_internal.h"

namespace moe {
namespace gsm {

__device__ __forceinline__ void set_err(int32_t *st, int code)
{
    if (st)
        atomicCAS(st + 1, 0, code);
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ int f16_sigma(float m)
{
    if (!(m > 0.f))
        return 0;
    int ex;
    frexpf(m, &ex);
    return 15 - ex;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float load_x(const Args &a, int64_t i)
{
    return a.x_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.x)[i])
                    : __half2float(reinterpret_cast<const __half *>(a.x)[i]);
}

// The eight MMAs of one item (A from the staged operand, B from the chunk).
__device__ __forceinline__ void item_mma(float (&dd)[4], const uint8_t *abase, int rs, int off, const Ld &ld,
                                         int lane)
{
    uint32_t bb[8][2];
    chunk_b(ld.c, bb);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        uint32_t aa[4];
        a_regs(abase, rs, off, lane, t, aa);
        mma16816(dd, aa, bb[t][0], bb[t][1]);
    }
}

__global__ void __launch_bounds__(kThreads, 1) awq_mma_kernel(const Args a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int d = a.d, I = a.I, b = a.b, k = a.k;
    const int NG1 = d / 128, NG2 = I / 128, RB1 = 2 * I / 8, RB2 = d / 8;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q4 = lane & 3, gl = lane >> 2;
    const int G = gridDim.x, cta = blockIdx.x;
    const Smem L{d, I};
    uint8_t *A = smem + L.a();
    float *sums = reinterpret_cast<float *>(smem + L.sums());
    int *r_route = reinterpret_cast<int *>(smem + L.rows());
    int *r_sig = r_route + kRows;
    __shared__ int s_abort;

    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0)
        s_abort = 0;
    const int nblk = min(max(__ldg(a.npp), 0) / b, a.cap_blocks);

    // ---------------------------------------------------------------- phase 1
    {
        const int T = nblk * RB1;
        const int c0 = static_cast<int>(static_cast<int64_t>(T) * cta / G);
        const int c1 = static_cast<int>(static_cast<int64_t>(T) * (cta + 1) / G);
        const int rs = L.xrow();
        for (int u = c0; u < c1;) {
            const int blk = u / RB1, seg_end = min(c1, (blk + 1) * RB1);
            __syncthreads();                                   // the previous block's operand is no longer read
            // the block's rows: route, scale exponent, x in f16 (MMA order), group sums
            const int e_raw = __ldg(a.expert_ids + blk);
            const bool e_ok = e_raw >= 0 && e_raw < a.E;           // a block of an invalid expert writes nothing
            const int e = e_ok ? e_raw : 0;
            if (tid < kRows) {
                const int route = tid < b ? __ldg(a.sorted + static_cast<int64_t>(blk) * b + tid) : a.mk;
                r_route[tid] = e_ok && route >= 0 && route < a.mk ? route : -1;
            }
            // the warps split the block's units [u, seg_end); items (unit, group).
            // Their first weight loads go out before the operand is staged.
            const int n = seg_end - u;
            const int v0 = u + n * warp / kWarps, v1 = u + n * (warp + 1) / kWarps;
            const int items = (v1 - v0) * NG1;
            Ld ring[kPF];
#pragma unroll
            for (int s = 0; s < kPF; ++s)
                if (s < items) {
                    const int v = v0 + s / NG1, g = s % NG1;
                    load_item(a.q13, a.s13, a.z13, static_cast<int64_t>(e) * 2 * I + (v - blk * RB1) * 8, d, g,
                              lane, ring[s]);
                }
            __syncthreads();
            for (int r = warp; r < kRows; r += kWarps) {
                const int route = r_route[r];
                float m = 0.f;
                if (route >= 0)
                    for (int i = lane; i < d; i += 32)
                        m = fmaxf(m, fabsf(load_x(a, static_cast<int64_t>(route / k) * d + i)));
                m = warp_max(m);
                const int sig = f16_sigma(m);
                if (lane == 0)
                    r_sig[r] = sig;
                __half *row = reinterpret_cast<__half *>(A + r * rs);
                for (int i = lane; i < d; i += 32) {
                    const float v = route >= 0
                                        ? load_x(a, static_cast<int64_t>(route / k) * d + (i & ~7) + interleave(i & 7))
                                        : 0.f;
                    row[i] = __float2half_rn(ldexpf(v, sig));
                }
                __syncwarp();
                for (int g = 0; g < NG1; ++g) {
                    float v = 0.f;
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        v += __half2float(row[g * 128 + t * 32 + lane]);
                    v = warp_sum(v);
                    if (lane == 0)
                        sums[r * NG1 + g] = v;
                }
            }
            __syncthreads();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int ib = 0; ib < items; ib += kPF) {
#pragma unroll
                for (int s = 0; s < kPF; ++s) {
                    const int it = ib + s;
                    if (it < items) {
                        const int v = v0 + it / NG1, g = it % NG1;
                        const Ld cur = ring[s];
                        if (it + kPF < items) {
                            const int vn = v0 + (it + kPF) / NG1, gn = (it + kPF) % NG1;
                            load_item(a.q13, a.s13, a.z13, static_cast<int64_t>(e) * 2 * I + (vn - blk * RB1) * 8,
                                      d, gn, lane, ring[s]);
                        }
                        float dd[4] = {0.f, 0.f, 0.f, 0.f};
                        item_mma(dd, A, rs, g * 128 + 32 * q4, cur, lane);
                        fold4(acc, dd, cur, lane, sums[gl * NG1 + g], sums[(gl + 8) * NG1 + g]);
                        if (g == NG1 - 1) {
                            // unit done: gate/up values of the block's routes
                            const int col = (v - blk * RB1) * 8 + 2 * q4;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int r = gl + 8 * h, route = r_route[r];
                                if (r < b && route >= 0) {
                                    const float un = ldexpf(1.0f, -r_sig[r]);
                                    float2 *dst = reinterpret_cast<float2 *>(a.gu + static_cast<int64_t>(route) * 2 * I +
                                                                             col);
                                    __stcg(dst, make_float2(acc[2 * h] * un, acc[2 * h + 1] * un));
                                }
                            }
                            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                            __syncwarp();
                            if (lane == 0) {
                                __threadfence();
                                atomicAdd(a.done + blk, 1);
                            }
                        }
                    }
                }
            }
            u = seg_end;
        }
    }

    // ---------------------------------------------------------------- phase 2
    {
        const int T = nblk * RB2;
        const int c0 = static_cast<int>(static_cast<int64_t>(T) * cta / G);
        const int c1 = static_cast<int>(static_cast<int64_t>(T) * (cta + 1) / G);
        const int rs = L.hrow();
        uint8_t *Ahi = A, *Alo = A + kRows * rs;
        for (int u = c0; u < c1;) {
            const int blk = u / RB2, seg_end = min(c1, (blk + 1) * RB2);
            __syncthreads();
            const int e_raw = __ldg(a.expert_ids + blk);
            const bool e_ok = e_raw >= 0 && e_raw < a.E;
            const int e = e_ok ? e_raw : 0;
            // the warps split the block's units; their first weight loads go
            // out before the wait for the block's gate/up values
            const int n = seg_end - u;
            const int v0 = u + n * warp / kWarps, v1 = u + n * (warp + 1) / kWarps;
            const int items = (v1 - v0) * NG2;
            Ld ring[kPF];
#pragma unroll
            for (int s = 0; s < kPF; ++s)
                if (s < items) {
                    const int v = v0 + s / NG2, g = s % NG2;
                    load_item(a.q2, a.s2, a.z2, static_cast<int64_t>(e) * d + (v - blk * RB2) * 8, I, g, lane,
                              ring[s]);
                }
            if (tid == 0) {
                // every gate/up unit of the block has written its values
                const long long t0 = clock64(), limit = static_cast<long long>(kWaitNs) * 5 / 2;
                int v;
                for (;;) {
                    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(a.done + blk) : "memory");
                    if (v >= RB1)
                        break;
                    if (clock64() - t0 > limit) {
                        s_abort = 1;
                        set_err(a.dev_status, MOE_ERR_TIMEOUT);
                        break;
                    }
                }
            }
            if (tid < kRows) {
                const int route = tid < b ? __ldg(a.sorted + static_cast<int64_t>(blk) * b + tid) : a.mk;
                r_route[tid] = e_ok && route >= 0 && route < a.mk ? route : -1;
            }
            __syncthreads();
            if (s_abort)
                return;
            for (int r = warp; r < kRows; r += kWarps) {
                const int route = r_route[r];
                const float w = route >= 0 ? __ldg(a.wts + route) : 0.f;
                const float *g_row = a.gu + static_cast<int64_t>(route >= 0 ? route : 0) * 2 * I;
                float m = 0.f;
                if (route >= 0)
                    for (int n2 = lane; n2 < I; n2 += 32)
                        m = fmaxf(m, fabsf(w * silu_mul(__ldcg(g_row + n2), __ldcg(g_row + I + n2))));
                m = warp_max(m);
                const int sig = f16_sigma(m);
                if (lane == 0)
                    r_sig[r] = sig;
                __half *hi = reinterpret_cast<__half *>(Ahi + r * rs);
                __half *lo = reinterpret_cast<__half *>(Alo + r * rs);
                for (int i = lane; i < I; i += 32) {
                    float v = 0.f;
                    if (route >= 0) {
                        const int n2 = (i & ~7) + interleave(i & 7);
                        v = ldexpf(w * silu_mul(__ldcg(g_row + n2), __ldcg(g_row + I + n2)), sig);
                    }
                    const __half h = __float2half_rn(v);
                    hi[i] = h;
                    lo[i] = __float2half_rn(v - __half2float(h));
                }
                __syncwarp();
                for (int g = 0; g < NG2; ++g) {
                    float v = 0.f;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int i = g * 128 + t * 32 + lane;
                        v += __half2float(hi[i]) + __half2float(lo[i]);
                    }
                    v = warp_sum(v);
                    if (lane == 0)
                        sums[r * NG2 + g] = v;
                }
            }
            __syncthreads();
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int ib = 0; ib < items; ib += kPF) {
#pragma unroll
                for (int s = 0; s < kPF; ++s) {
                    const int it = ib + s;
                    if (it < items) {
                        const int v = v0 + it / NG2, g = it % NG2;
                        const Ld cur = ring[s];
                        if (it + kPF < items) {
                            const int vn = v0 + (it + kPF) / NG2, gn = (it + kPF) % NG2;
                            load_item(a.q2, a.s2, a.z2, static_cast<int64_t>(e) * d + (vn - blk * RB2) * 8, I, gn,
                                      lane, ring[s]);
                        }
                        float dd[4] = {0.f, 0.f, 0.f, 0.f};
                        item_mma(dd, Ahi, rs, g * 128 + 32 * q4, cur, lane);
                        item_mma(dd, Alo, rs, g * 128 + 32 * q4, cur, lane);
                        fold4(acc, dd, cur, lane, sums[gl * NG2 + g], sums[(gl + 8) * NG2 + g]);
                        if (g == NG2 - 1) {
                            const int col = (v - blk * RB2) * 8 + 2 * q4;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int r = gl + 8 * h, route = r_route[r];
                                if (r < b && route >= 0) {
                                    const float un = ldexpf(1.0f, -r_sig[r]);
                                    float2 *dst = reinterpret_cast<float2 *>(a.yr + static_cast<int64_t>(route) * d +
                                                                             col);
                                    __stcg(dst, make_float2(acc[2 * h] * un, acc[2 * h + 1] * un));
                                }
                            }
                            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                        }
                    }
                }
            }
            u = seg_end;
        }
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

}  // namespace gsm

// Workspace of this path: [done: cap_rows / b int32 | gu: M*k*2I f32 | yr: M*k*d f32].
size_t grouped_awq_mma_workspace(int M, int k, int d, int I, int b, int cap_rows)
{
    const size_t mk = static_cast<size_t>(M) * k;
    return ws_round(static_cast<size_t>(cap_rows / b) * 4) + ws_round(mk * 2 * I * 4) + ws_round(mk * d * 4);
}

bool grouped_awq_mma_eligible(int b, int d, int I)
{
    const gsm::Smem L{d, I};
    return b >= 1 && b <= gsm::kRows && d % 128 == 0 && I % 128 == 0 && L.bytes() <= 220 * 1024;
}

moe_status_t grouped_awq_mma_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                    const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                    const int32_t *sorted, const int32_t *expert_ids, const int32_t *npp, int b,
                                    int cap_rows, void *y, bool y_f32, void *ws, int32_t *dev_status, cudaStream_t s)
{
    if (!grouped_awq_mma_eligible(b, d, I))
        return MOE_ERR_UNSUPPORTED;
    const size_t mk = static_cast<size_t>(M) * k;
    uint8_t *w = static_cast<uint8_t *>(ws);
    int32_t *done = reinterpret_cast<int32_t *>(w);
    float *gu = reinterpret_cast<float *>(w + ws_round(static_cast<size_t>(cap_rows / b) * 4));
    float *yr = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(gu) + ws_round(mk * 2 * I * 4));
    const gsm::Smem L{d, I};
    static std::atomic<uint64_t> attr_done{0};
    if (!smem_attr_once(attr_done, reinterpret_cast<const void *>(gsm::awq_mma_kernel), 220 * 1024))
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(done, 0, static_cast<size_t>(cap_rows / b) * 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const gsm::Args a{x, wts, sorted, expert_ids, npp, static_cast<const uint32_t *>(w13->q),
                      static_cast<const uint16_t *>(w13->scale), static_cast<const int32_t *>(w13->zero),
                      static_cast<const uint32_t *>(w2->q), static_cast<const uint16_t *>(w2->scale),
                      static_cast<const int32_t *>(w2->zero), done, gu, yr, dev_status, x_bf16 ? 1 : 0,
                      M, k, d, I, E, b, static_cast<int>(mk), cap_rows / b};
    if (launch_pdl(gsm::awq_mma_kernel, dim3(device_sm_count()), dim3(gsm::kThreads),
                   static_cast<size_t>(L.bytes()), s, a) != cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, ids, M, k, d, E, y, y_f32, s);
}

bool decode_awq_small_eligible(int M, int k, int d, int I, int E)
{
    return M >= 2 && M <= 64 && k >= 1 && k <= 32 && E >= 1 && grouped_awq_mma_eligible(gsm::kRows, d, I) &&
           static_cast<int64_t>(M) * k * (2 * I + d) * 4 < (int64_t(1) << 31);
}

moe_status_t decode_awq_small_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                     const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                     void *y, bool y_f32, void *ws, size_t ws_bytes, int32_t *dev_status,
                                     cudaStream_t s)
{
    if (!decode_awq_small_eligible(M, k, d, I, E) || !aligned(ws, 256) || !aligned(w13->q, 16) ||
        !aligned(w2->q, 16))
        return MOE_ERR_UNSUPPORTED;
    const SmallWs W = small_ws_layout(M, k, d, I, E);
    if (ws_bytes < W.total)
        return MOE_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    int32_t *sorted = reinterpret_cast<int32_t *>(w + W.sorted);
    int32_t *expert = reinterpret_cast<int32_t *>(w + W.expert);
    int32_t *npp = reinterpret_cast<int32_t *>(w + W.npp);
    int32_t *done = reinterpret_cast<int32_t *>(w + W.done);
    float *gu = reinterpret_cast<float *>(w + W.gu);
    float *yr = reinterpret_cast<float *>(w + W.yr);
    static std::atomic<uint64_t> attr_done{0};
    if (!smem_attr_once(attr_done, reinterpret_cast<const void *>(gsm::awq_mma_kernel), 220 * 1024))
        return MOE_ERR_CUDA;
    // the routes in blocks of 16 rows per expert (invalid ids are counted here)
    const moe_status_t st = moe_align_block_size(ids, M, k, E, gsm::kRows, sorted, expert, npp, W.cap_rows,
                                                 W.cap_blocks, w + W.align_ws, W.sorted - W.align_ws, dev_status,
                                                 s);
    if (st != MOE_OK)
        return st;
    if (cudaMemsetAsync(done, 0, static_cast<size_t>(W.cap_blocks) * 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const gsm::Smem L{d, I};
    const size_t mk = static_cast<size_t>(M) * k;
    const gsm::Args a{x, wts, sorted, expert, npp, static_cast<const uint32_t *>(w13->q),
                      static_cast<const uint16_t *>(w13->scale), static_cast<const int32_t *>(w13->zero),
                      static_cast<const uint32_t *>(w2->q), static_cast<const uint16_t *>(w2->scale),
                      static_cast<const int32_t *>(w2->zero), done, gu, yr, dev_status, x_bf16 ? 1 : 0,
                      M, k, d, I, E, gsm::kRows, static_cast<int>(mk), W.cap_blocks};
    if (launch_pdl(gsm::awq_mma_kernel, dim3(device_sm_count()), dim3(gsm::kThreads),
                   static_cast<size_t>(L.bytes()), s, a) != cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, ids, M, k, d, E, y, y_f32, s);
}

}  // namespace moe
