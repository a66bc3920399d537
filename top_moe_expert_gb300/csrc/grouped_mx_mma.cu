// grouped_mx_mma.cu -- the MXFP8 layer for 2 <= M <= 64 tokens through
// moe_ffn_decode: route alignment into blocks of 16 rows, one kernel for both
// expert GEMMs on mma.sync, then the slot-ordered combine.
//
// Output-centric decode ("Warp decode", sections on what changed and how the
// two kernels work) keeps activations and h unquantized and accumulates in
// FP32.  Here each routed expert's weights stream once per MoE block of up to
// 16 of its routes ("Route-Block Membership Selects Packed-AWQ Arithmetic",
// opening paragraph: the aligned blocks), so a block is one M-tile of
// mma.sync m16n8k16: B = eight weight rows, each E4M3 pair converted exactly
// to f16; A = the block's rows of x (an exact per-row power of two into f16
// range) or of h (an f16 hi + lo pair); every 32-value block's FP32 sum is
// multiplied by its E8M0 scale.
//
// One CTA per SM, 16 warps, one kernel for both GEMMs:
//  * Phase 1 (gate/up): units (block, 8 rows of W13) are split evenly over
//    the CTAs in block order; a CTA stages the A operand of each block it
//    touches and its warps split the block's units, with the first weight
//    loads issued before the staging.  A unit writes the FP32 gate or up
//    values of the block's routes and bumps the block's counter.
//  * Phase 2 (down): units (block, 8 rows of W2).  A CTA waits (bounded)
//    until its block's counter shows every gate/up unit done, forms
//    h = w SiLU(g) u of the block's routes, splits it into f16 hi + lo, and
//    writes each route's FP32 down-projection row to Yr.
//  * The combine kernel of the grouped path adds each token's slots in order.
// Every value has one owner and a fixed summation order: a route's result
// depends on neither the other rows of its block nor the grid.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "grouped_internal.h"
#include "grouped_mx_mma.cuh"

namespace moe {
namespace gmx {

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

__device__ __forceinline__ float load_x(const Args &a, int64_t i) { return __bfloat162float(a.x[i]); }

// One item (64 K values): per piece (scale block) two MMAs into a fresh D,
// then the block's scale into the lane's four accumulators.
__device__ __forceinline__ void item(float (&acc)[4], const uint8_t *abase, int rs, int base, const Ld &ld,
                                     int lane)
{
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float dd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            uint32_t aa[4], b0, b1;
            a_regs(abase, rs, base, p, t, lane, aa);
            mx_b(ld, p, t, b0, b1);
            mma16816(dd, aa, b0, b1);
        }
        fold4(acc, dd, ld, p);
    }
}

// A 16-row item with both halves of h (hi, lo) as A: D accumulates both.
__device__ __forceinline__ void item2(float (&acc)[4], const uint8_t *ahi, const uint8_t *alo, int rs, int base,
                                      const Ld &ld, int lane)
{
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float dd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            uint32_t aa[4], b0, b1;
            mx_b(ld, p, t, b0, b1);
            a_regs(ahi, rs, base, p, t, lane, aa);
            mma16816(dd, aa, b0, b1);
            a_regs(alo, rs, base, p, t, lane, aa);
            mma16816(dd, aa, b0, b1);
        }
        fold4(acc, dd, ld, p);
    }
}

__global__ void __launch_bounds__(kThreads, 1) mx_mma_kernel(const Args a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int d = a.d, I = a.I, b = kRows, k = a.k;
    const int NG1 = d / 64, NG2 = I / 64, RB1 = 2 * I / 8, RB2 = d / 8;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q4 = lane & 3, gl = lane >> 2;
    const int G = gridDim.x, cta = blockIdx.x;
    const Smem L{d, I};
    uint8_t *A = smem + L.a();
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
            // the block's rows: route, scale exponent, x in f16
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
                    mx_load(a.q13, a.s13, static_cast<int64_t>(e) * 2 * I + (v - blk * RB1) * 8, d, g, lane,
                            ring[s]);
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
                                        ? load_x(a, static_cast<int64_t>(route / k) * d + i)
                                        : 0.f;
                    row[i] = __float2half_rn(ldexpf(v, sig));
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
                            mx_load(a.q13, a.s13, static_cast<int64_t>(e) * 2 * I + (vn - blk * RB1) * 8, d, gn,
                                    lane, ring[s]);
                        }
                        item(acc, A, rs, g * 64, cur, lane);
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
                    mx_load(a.q2, a.s2, static_cast<int64_t>(e) * d + (v - blk * RB2) * 8, I, g, lane, ring[s]);
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
                        v = ldexpf(w * silu_mul(__ldcg(g_row + i), __ldcg(g_row + I + i)), sig);
                    }
                    const __half h = __float2half_rn(v);
                    hi[i] = h;
                    lo[i] = __float2half_rn(v - __half2float(h));
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
                            mx_load(a.q2, a.s2, static_cast<int64_t>(e) * d + (vn - blk * RB2) * 8, I, gn, lane,
                                    ring[s]);
                        }
                        item2(acc, Ahi, Alo, rs, g * 64, cur, lane);
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

}  // namespace gmx


SmallWs small_ws_layout(int M, int k, int d, int I, int E)
{
    SmallWs w{};
    int32_t cr = 0, cb = 0;
    size_t na = 0;
    moe_align_capacity(M, k, E, gmx::kRows, &cr, &cb);
    moe_align_workspace_size(M, k, E, gmx::kRows, &na);
    const size_t mk = static_cast<size_t>(M) * k;
    size_t off = 0;
    w.align_ws = off; off += ws_round(na);
    w.sorted = off;   off += ws_round(static_cast<size_t>(cr) * 4);
    w.expert = off;   off += ws_round(static_cast<size_t>(cb) * 4);
    w.npp = off;      off += 256;
    w.done = off;     off += ws_round(static_cast<size_t>(cb) * 4);
    w.gu = off;       off += ws_round(mk * 2 * I * 4);
    w.yr = off;       off += ws_round(mk * d * 4);
    w.total = off;
    w.cap_rows = cr;
    w.cap_blocks = cb;
    return w;
}

bool decode_mx_small_eligible(int M, int k, int d, int I, int E)
{
    const gmx::Smem L{d, I};
    return M >= 2 && M <= 64 && k >= 1 && k <= 32 && E >= 1 && d % 64 == 0 && I % 64 == 0 &&
           L.bytes() <= 220 * 1024 && static_cast<int64_t>(M) * k * (2 * I + d) * 4 < (int64_t(1) << 31);
}

size_t decode_mx_small_workspace(int M, int k, int d, int I, int E)
{
    return small_ws_layout(M, k, d, I, E).total;
}

moe_status_t decode_mx_small_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                    const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                    const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32, void *ws,
                                    size_t ws_bytes, int32_t *dev_status, cudaStream_t s)
{
    if (!decode_mx_small_eligible(M, k, d, I, E) || !aligned(ws, 256) || !aligned(q13, 8) || !aligned(q2, 8) ||
        !aligned(s13, 2) || !aligned(s2, 2))
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
    if (!smem_attr_once(attr_done, reinterpret_cast<const void *>(gmx::mx_mma_kernel), 220 * 1024))
        return MOE_ERR_CUDA;
    // the routes in blocks of 16 rows per expert (invalid ids are counted here)
    const moe_status_t st = moe_align_block_size(ids, M, k, E, gmx::kRows, sorted, expert, npp, W.cap_rows,
                                                 W.cap_blocks, w + W.align_ws, W.sorted - W.align_ws, dev_status,
                                                 s);
    if (st != MOE_OK)
        return st;
    if (cudaMemsetAsync(done, 0, static_cast<size_t>(W.cap_blocks) * 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const gmx::Smem L{d, I};
    const gmx::Args a{x, wts, sorted, expert, npp, q13, s13, q2, s2, done, gu, yr, dev_status,
                      M, k, d, I, E, M * k, W.cap_blocks};
    if (launch_pdl(gmx::mx_mma_kernel, dim3(device_sm_count()), dim3(gmx::kThreads), static_cast<size_t>(L.bytes()),
                   s, a) != cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, ids, M, k, d, E, y, y_f32, s);
}

}  // namespace moe
