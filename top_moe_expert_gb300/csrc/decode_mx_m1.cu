// decode_mx_m1.cu -- single-token (M = 1) decode of the routed MXFP8 expert
// layer in one kernel, on the standard (K-contiguous) layout of both
// projections, with the routing optionally inside.
//
// Output-centric decode ("Warp decode", cursor.com blog, sections on what
// changed and how the two kernels work): for each routed expert
//     h_j = w_j SiLU(Wg_{e_j} x) (Wu_{e_j} x),   y = sum_j W2_{e_j} h_j,
// weights streamed once, converted on the fly, FP32 sums; no alignment,
// padding or combine buffers.  The routing weight is applied to h (equal, in
// exact arithmetic, to applying it in the down accumulation).  Dot products
// run on mma.sync with the operands of decode_mx_m1.cuh.
//
// One CTA per SM, 16 warps:
//  * Prologue: the routing -- top-k softmax of the logits by warp 0 of every
//    CTA (CTA 0 writes the ids and weights out), or the given ids and
//    weights -- with the valid routes compacted in slot order; x scaled by an
//    exact power of two into f16 range and staged; warp 0 starts
//    cp.async.bulk copies of this CTA's W2 rows (its blocks of 8 outputs,
//    every valid slot) into shared memory.
//  * Phase 1: items (unit = 8 rows of W13 of one slot; chunk of 64 K values)
//    split evenly over the CTAs and their warps; four items' loads in flight
//    per warp.  A unit's partial sums are combined in a fixed order: within
//    the CTA through shared memory, across CTAs as pieces in the workspace.
//  * The CTA stages its W2 scale bytes; grid barrier (one arrival per CTA on
//    a never-reset 64-bit counter in ws[0..8); bounded spin).
//  * Phase 2: h from the pieces in a fixed order; per slot an exact power of
//    two into f16 range and an f16 hi + lo split; units (slot, block of 8
//    outputs) over the warps, 2 x 2 MMAs per scale block with W2 from shared
//    memory; y = the slots' results added in slot order.
// Every output's summation order depends only on the shapes and the grid,
// so repeats are bit-identical.  The grid is one CTA per SM, all resident
// together; dependent launches start after the barrier.
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "decode_mx_m1.cuh"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {
namespace dx1 {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kPF = 8;                  // phase-1 items in flight per warp (16 bytes each per lane)
constexpr int kPF2 = 4;                 // phase-2 items in flight per warp

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

// The lane's two accumulators over one item: per piece (scale block) two
// MMAs into a fresh D, then the block's scale.
__device__ __forceinline__ void item(float (&acc)[2], const Ld &ld, const uint32_t *a32, int base, int lane)
{
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float dd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            uint32_t aa[4], b0, b1;
            mx_a(a32, base, p, t, lane, aa);
            mx_b(ld, p, t, b0, b1);
            mma16816(dd, aa, b0, b1);
        }
        mx_fold(acc, dd, ld, p);
    }
}

template <int ROUTE_PL, bool STAGE_W2>
__global__ void __launch_bounds__(kThreads, 1) mx_m1_kernel(const Args a)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int d = a.d, I = a.I, NG = d / 64, NG2 = I / 64, RB = 2 * I / 8;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q = lane & 3, gl = lane >> 2;
    const int G = gridDim.x, b = blockIdx.x;
    const int B2 = d / 8, blk0 = split_lo(B2, b, G), nb = split_lo(B2, b + 1, G) - blk0;
    const Smem L{d, I, a.k, nb, STAGE_W2 ? 1 : 0};
    __half *xp = reinterpret_cast<__half *>(smem + L.xp());
    int *r_e = reinterpret_cast<int *>(smem + L.route());
    float *r_w = reinterpret_cast<float *>(r_e + kMaxK);
    int *r_sig = reinterpret_cast<int *>(r_w + kMaxK);
    const uint32_t mbar = tc::smem_u32(smem + L.mbar());
    float *p1v = reinterpret_cast<float *>(smem + L.part1());           // [16][4][8]
    int *p1u = reinterpret_cast<int *>(p1v + kWarps * 4 * 8);          // [16][4]
    uint8_t *w2s = smem + L.w2();
    uint8_t *s2s = smem + L.s2();
    float *hf = reinterpret_cast<float *>(smem + L.hf());
    __half *hp = reinterpret_cast<__half *>(smem + L.hp());            // [2][k][I]
    float *part2 = reinterpret_cast<float *>(smem + L.part2());
    __shared__ int s_nv, s_ok, s_abort, s_sigx;
    __shared__ unsigned long long s_epoch;
    __shared__ float s_wmax[kWarps];

    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        unsigned long long v;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
        s_epoch = v;
        s_abort = 0;
        tc::mbar_init(mbar, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        int e;
        float w;
        if constexpr (ROUTE_PL > 0) {
            topk_warp<ROUTE_PL>(a.logits, a.E, a.k, lane, e, w);
            if (b == 0 && lane < a.k) {
                a.ids_out[lane] = e;
                a.wts_out[lane] = w;
            }
            if (lane >= a.k)
                e = -1;
        } else {
            e = lane < a.k ? a.ids[lane] : -1;
            w = lane < a.k ? a.wts[lane] : 0.f;
        }
        const bool ok = lane < a.k && e >= 0 && e < a.E;
        const unsigned vm = __ballot_sync(0xffffffffu, ok);
        if (ok) {
            const int i = __popc(vm & ((1u << lane) - 1u));
            r_e[i] = e;
            r_w[i] = w;
        }
        if (lane == 0) {
            s_nv = __popc(vm);
            if (b == 0 && a.k > __popc(vm) && a.dev_status)
                atomicAdd(a.dev_status, a.k - __popc(vm));
        }
    }
    float xm = 0.f;
    for (int i = tid; i < d; i += kThreads)
        xm = fmaxf(xm, fabsf(__bfloat162float(a.x[i])));
    xm = warp_max(xm);
    if (lane == 0)
        s_wmax[warp] = xm;
    for (int i = tid; i < kWarps * 4; i += kThreads)
        p1u[i] = -1;
    __syncthreads();
    const int nv = s_nv;
    if (tid == 0) {
        float m = 0.f;
        for (int w = 0; w < kWarps; ++w)
            m = fmaxf(m, s_wmax[w]);
        s_sigx = f16_sigma(m);
    }
    // W2 rows of this CTA (I bytes each): into shared memory, or (rows that
    // do not fit) into L2 for phase 2 to read
    if (warp == 0) {
        if (lane == 0)
            tc::mbar_arrive_expect_tx(mbar, STAGE_W2 ? static_cast<uint32_t>(nv * nb * 8 * I) : 0u);
        __syncwarp();
        for (int r = lane; r < nv * nb * 8; r += 32) {
            const int j = r / (nb * 8), o = blk0 * 8 + (r - j * nb * 8);
            const uint8_t *src = a.q2 + (static_cast<int64_t>(r_e[j]) * d + o) * I;
            if constexpr (STAGE_W2)
                tc::bulk_load(tc::smem_u32(w2s) + r * I, src, I, mbar);
            else
                tc::bulk_prefetch_l2(src, I);
        }
    }
    __syncthreads();
    const int sigx = s_sigx;
    for (int i = tid; i < d; i += kThreads)
        xp[i] = __float2half_rn(ldexpf(__bfloat162float(a.x[i]), sigx));
    __syncthreads();

    // ---- phase 1
    const int T = nv * RB * NG;
    const int c0 = split_lo(T, b, G), c1 = split_lo(T, b + 1, G);
    {
        const int n = c1 - c0;
        const int i0 = c0 + split_lo(n, warp, kWarps), i1 = c0 + split_lo(n, warp + 1, kWarps);
        const uint32_t *x32 = reinterpret_cast<const uint32_t *>(xp);
        auto load = [&](int i, Ld &o) {
            const int u = i / NG, c = i - u * NG;
            const int j = u / RB, rb = u - j * RB;
            mx_load(a.q13, a.s13, static_cast<int64_t>(r_e[j]) * 2 * I + rb * 8, d, c, lane, o);
        };
        Ld ring[kPF];
#pragma unroll
        for (int s = 0; s < kPF; ++s)
            if (i0 + s < i1)
                load(i0 + s, ring[s]);
        float acc[2] = {0.f, 0.f};
        int cur = i0 < i1 ? i0 / NG : -1, slot = 0;
        for (int ib = i0; ib < i1; ib += kPF) {
#pragma unroll
            for (int s = 0; s < kPF; ++s) {
                const int i = ib + s;
                if (i < i1) {
                    const int u = i / NG, c = i - u * NG;
                    if (u != cur) {
                        // at most 4 units per warp (the host's size check)
                        if (gl == 0 && slot < 4) {
                            p1v[(warp * 4 + slot) * 8 + 2 * q] = acc[0];
                            p1v[(warp * 4 + slot) * 8 + 2 * q + 1] = acc[1];
                        }
                        if (lane == 0 && slot < 4)
                            p1u[warp * 4 + slot] = cur;
                        ++slot;
                        cur = u;
                        acc[0] = acc[1] = 0.f;
                    }
                    const Ld ld = ring[s];
                    if (i + kPF < i1)
                        load(i + kPF, ring[s]);
                    item(acc, ld, x32, c * 64, lane);
                }
            }
        }
        if (cur >= 0 && slot < 4) {
            if (gl == 0) {
                p1v[(warp * 4 + slot) * 8 + 2 * q] = acc[0];
                p1v[(warp * 4 + slot) * 8 + 2 * q + 1] = acc[1];
            }
            if (lane == 0)
                p1u[warp * 4 + slot] = cur;
        }
        if (slot >= 4 && lane == 0)
            set_err(a.dev_status, MOE_ERR_UNSUPPORTED);
    }
    __syncthreads();
    if (c1 > c0) {
        const int u0 = c0 / NG, u1 = (c1 - 1) / NG;
        const float unscale = ldexpf(1.0f, -sigx);
        for (int t = tid; t < (u1 - u0 + 1) * 8; t += kThreads) {
            const int u = u0 + t / 8, r = t % 8;
            float v = 0.f;
            for (int w = 0; w < kWarps * 4; ++w)
                if (p1u[w] == u)
                    v += p1v[w * 8 + r];
            const int piece = b - owner(u * NG, T, G);
            __stcg(a.gp + (static_cast<int64_t>(u) * kMaxPieces + piece) * 8 + r, v * unscale);
        }
    }
    // W2 scale bytes of this CTA's rows
    for (int i = tid; STAGE_W2 && i < nv * nb * 8 * (I / 32); i += kThreads) {
        const int r = i / (I / 32), c = i - r * (I / 32);
        const int j = r / (nb * 8), o = blk0 * 8 + (r - j * nb * 8);
        s2s[i] = __ldg(a.s2 + (static_cast<int64_t>(r_e[j]) * d + o) * (I / 32) + c);
    }

    // ---- grid barrier: every piece is visible before any is read
    __syncthreads();
    if (tid == 0) {
        const unsigned long long GG = G, target = (s_epoch / GG + 1) * GG;
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(a.bar) : "memory");
        const long long t0 = clock64(), limit = static_cast<long long>(kWaitNs) * 5 / 2;
        int ok = 1;
        unsigned long long v;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
            if (v >= target)
                break;
            if (clock64() - t0 > limit) {
                ok = 0;
                break;
            }
        }
        s_ok = ok;
        if (!ok)
            set_err(a.dev_status, MOE_ERR_TIMEOUT);
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;");
    if (!s_ok) {
        if (!tc::mbar_wait(mbar, 0, &s_abort, kWaitNs))
            set_err(a.dev_status, MOE_ERR_TIMEOUT);
        return;
    }

    // ---- phase 2: h of every slot
    for (int t = tid; t < nv * I; t += kThreads) {
        const int j = t / I, n2 = t - j * I;
        const int ug = j * RB + n2 / 8, uu = j * RB + (I + n2) / 8, r = n2 % 8;
        float gv = 0.f, uv = 0.f;
        const int pg = owner(ug * NG + NG - 1, T, G) - owner(ug * NG, T, G) + 1;
        const int pu = owner(uu * NG + NG - 1, T, G) - owner(uu * NG, T, G) + 1;
        for (int p = 0; p < pg; ++p)
            gv += __ldcg(a.gp + (static_cast<int64_t>(ug) * kMaxPieces + p) * 8 + r);
        for (int p = 0; p < pu; ++p)
            uv += __ldcg(a.gp + (static_cast<int64_t>(uu) * kMaxPieces + p) * 8 + r);
        hf[t] = r_w[j] * silu_mul(gv, uv);
    }
    __syncthreads();
    for (int j = warp; j < nv; j += kWarps) {
        float m = 0.f;
        for (int n2 = lane; n2 < I; n2 += 32)
            m = fmaxf(m, fabsf(hf[j * I + n2]));
        m = warp_max(m);
        if (lane == 0)
            r_sig[j] = f16_sigma(m);
    }
    __syncthreads();
    for (int t = tid; t < nv * I; t += kThreads) {
        const int j = t / I;
        const float v = ldexpf(hf[t], r_sig[j]);
        const __half hi = __float2half_rn(v);
        hp[t] = hi;
        hp[nv * I + t] = __float2half_rn(v - __half2float(hi));
    }
    if (!tc::mbar_wait(mbar, 0, &s_abort, kWaitNs))
        set_err(a.dev_status, MOE_ERR_TIMEOUT);
    __syncthreads();
    if (s_abort)
        return;

    // ---- phase 2: units (slot j, output block) over the warps: warp w takes
    // units w, w + 16, ...; its items (unit, chunk) run with kPF2 in flight
    const uint32_t *h32 = reinterpret_cast<const uint32_t *>(hp);
    {
        const int nunits = nv * nb;
        const int my_units = nunits > warp ? (nunits - warp + kWarps - 1) / kWarps : 0;
        const int items = my_units * NG2;
        auto load2 = [&](int it, Ld &o) {
            const int v = warp + kWarps * (it / NG2), c = it % NG2;
            const int j = v / nb, bl = v - j * nb;
            if constexpr (STAGE_W2)
                mx_load(w2s, s2s, j * nb * 8 + bl * 8, I, c, lane, o);
            else
                mx_load(a.q2, a.s2, static_cast<int64_t>(r_e[j]) * d + (blk0 + bl) * 8, I, c, lane, o);
        };
        Ld ring[kPF2];
#pragma unroll
        for (int s = 0; s < kPF2; ++s)
            if (s < items)
                load2(s, ring[s]);
        float acc[2] = {0.f, 0.f};
        for (int ib = 0; ib < items; ib += kPF2) {
#pragma unroll
            for (int s = 0; s < kPF2; ++s) {
                const int it = ib + s;
                if (it < items) {
                    const int v = warp + kWarps * (it / NG2), c = it % NG2;
                    const int j = v / nb, bl = v - j * nb;
                    const Ld ld = ring[s];
                    if (it + kPF2 < items)
                        load2(it + kPF2, ring[s]);
                    item(acc, ld, h32 + j * I / 2, c * 64, lane);
                    item(acc, ld, h32 + (nv + j) * I / 2, c * 64, lane);
                    if (c == NG2 - 1) {
                        if (gl == 0) {
                            const float un = ldexpf(1.0f, -r_sig[j]);
                            part2[(j * nb + bl) * 8 + 2 * q] = acc[0] * un;
                            part2[(j * nb + bl) * 8 + 2 * q + 1] = acc[1] * un;
                        }
                        acc[0] = acc[1] = 0.f;
                    }
                }
            }
        }
    }
    __syncthreads();
    for (int t = tid; t < nb * 8; t += kThreads) {
        float yo = 0.f;
        for (int j = 0; j < nv; ++j)
            yo += part2[(j * nb + t / 8) * 8 + t % 8];
        const int o = blk0 * 8 + t;
        if (a.y_f32)
            reinterpret_cast<float *>(a.y)[o] = yo;
        else
            reinterpret_cast<__nv_bfloat16 *>(a.y)[o] = __float2bfloat16_rn(yo);
    }
}

}  // namespace dx1

// Whether the phase-1 item split of this grid keeps every unit within
// kMaxPieces CTAs and every warp within 4 units (see decode_awq_m1.cu).
static bool mx_split_fits(int nv, int d, int I, int G)
{
    const int NG = d / 64, T = nv * (2 * I / 8) * NG;
    const int min_cta = T / G;
    if (min_cta == 0)
        return NG == 1;
    if ((NG - 1 + min_cta - 1) / min_cta + 1 > dx1::kMaxPieces)
        return false;
    const int max_cta = (T + G - 1) / G;
    const int max_warp = (max_cta + dx1::kWarps - 1) / dx1::kWarps;
    return (max_warp - 1 + NG - 1) / NG + 1 <= 4;
}

bool decode_mx_m1_eligible(int M, int k, int d, int I, int E)
{
    const int G = device_sm_count();
    if (M != 1 || k < 1 || k > dx1::kMaxK || E < 1 || d % 64 || d < 64 || I % 64 || I < 64 || G > 1024 ||
        static_cast<int64_t>(k) * 2 * I / 8 * (d / 64) > INT32_MAX / 2)
        return false;
    const dx1::Smem L{d, I, k, (d / 8 + G - 1) / G, 0};         // W2 read from global if it does not fit
    if (L.bytes() > 220 * 1024)
        return false;
    for (int nv = 1; nv <= k; ++nv)
        if (!mx_split_fits(nv, d, I, G))
            return false;
    return true;
}

size_t decode_mx_m1_workspace(int k, int I)
{
    return 256 + ws_round(static_cast<size_t>(k) * (2 * I / 8) * dx1::kMaxPieces * 8 * sizeof(float));
}

moe_status_t decode_mx_m1_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                                 const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                                 const uint8_t *s13, const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32,
                                 void *ws, int32_t *dev_status, cudaStream_t stream)
{
    const int G = device_sm_count();
    if (!decode_mx_m1_eligible(1, k, d, I, E) || !aligned(q2, 16) || !aligned(ws, 256) || !aligned(q13, 8) ||
        !aligned(s13, 2) ||
        (logits && (E > 512 || E < k)))
        return MOE_ERR_UNSUPPORTED;
    const dx1::Smem Ls{d, I, k, (d / 8 + G - 1) / G, 1}, Lg{d, I, k, (d / 8 + G - 1) / G, 0};
    const bool stage = Ls.bytes() <= 220 * 1024;
    const int smem = stage ? Ls.bytes() : Lg.bytes();
    uint8_t *w = static_cast<uint8_t *>(ws);
    const dx1::Args a{x, ids, wts, logits, ids_out, wts_out, q13, s13, q2, s2,
                      reinterpret_cast<unsigned long long *>(w), reinterpret_cast<float *>(w + 256), y, dev_status,
                      y_f32 ? 1 : 0, k, d, I, E};
    auto go = [&](auto kern) -> moe_status_t {
        if (!smem_attr(reinterpret_cast<const void *>(kern), 220 * 1024))
            return MOE_ERR_CUDA;
        return launch_pdl(kern, dim3(G), dim3(dx1::kThreads), static_cast<size_t>(smem), stream, a) == cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    };
    const int pl = !logits ? 0 : (E + 31) / 32 <= 4 ? 4 : (E + 31) / 32 <= 8 ? 8 : 16;
    if (stage)
        return pl == 0 ? go(dx1::mx_m1_kernel<0, true>) : pl == 4 ? go(dx1::mx_m1_kernel<4, true>)
               : pl == 8 ? go(dx1::mx_m1_kernel<8, true>) : go(dx1::mx_m1_kernel<16, true>);
    return pl == 0 ? go(dx1::mx_m1_kernel<0, false>) : pl == 4 ? go(dx1::mx_m1_kernel<4, false>)
           : pl == 8 ? go(dx1::mx_m1_kernel<8, false>) : go(dx1::mx_m1_kernel<16, false>);
}

}  // namespace moe
