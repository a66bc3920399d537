// grouped.cu -- expert-centric grouped path for larger batches (MXFP8).
//
// "Hardware-Native Joint Sparse-Quantization for Trillion-Scale MoE"
// (arXiv 2610.02241), Sec. 3.4 and App. D.1: a routed MoE layer evaluates
// the expert products Y_e = X_e W_e^T as one grouped GEMM; the weights go on
// the MMA's left operand (Y_e^T = W_e X_e^T), which needs no copy because
// row-major X_e is the column-major B operand; activations are quantized at
// run time into 32-element scale blocks before the first GEMM, and the
// SwiGLU output is requantized for the second.  Rows are the aligned routes
// of "Route-Block Membership Selects Packed-AWQ Arithmetic" (stable
// construction), one MMA N-tile per MoE block of b rows.
//
// Kernels:
//   act_quant_kernel : x[t] of every aligned row -> MXFP8 codes + E8M0 atoms
//   gemm_kernel      : both GEMMs, one CTA per SM, persistent over tiles --
//                      first-GEMM tiles [g;u] = W13_e Xq^T on tcgen05
//                      kind::mxf8f6f4 with block scaling, epilogue
//                      h = SiLU(g) * u -> MXFP8; then second-GEMM tiles
//                      W2_e Hq^T, epilogue Yr[route] = w_route * acc
//   combine_kernel   : y[t] = sum over slots j (in order) of Yr[t*k + j]
// K-reduction order: every output element accumulates its K-tiles in
// ascending order in one TMEM accumulator; no split-K, no atomics, so the
// bits of a route's row do not depend on its block membership or the grid.
//
// GEMM roles: warp 0 issues TMA (operand tiles, 128-byte swizzled) and bulk
// copies (scale atoms) into a ring of as many stages as shared memory holds
// (up to 12); warp 1 owns TMEM and issues
// tcgen05.cp (scales -> TMEM) and tcgen05.mma from one thread; warps 2..5
// drain the TMEM accumulator with tcgen05.ld.  Every mbarrier wait is
// bounded; an expired wait records MOE_ERR_TIMEOUT in dev_status[1].
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "attr.h"
#include "common.cuh"
#include "grouped_internal.h"
#include "tc.cuh"

namespace moe {
namespace gg {

constexpr int kMaxStages = 12;         // operand ring depth: as many stages as shared memory holds
constexpr int kHeaderBytes = 256;      // mbarriers, TMEM address, abort flag
constexpr int kThreads = 192;          // 6 warps
constexpr uint32_t kTmemCols = 512;    // accumulator: columns 0..255; scales from 256
constexpr uint64_t kWaitNs = 2000000000ull;

struct Args {
    const uint8_t *sfa;       // A scale atoms  [E][n_mt][KT][512]
    const uint8_t *sfb;       // B scale atoms  [cap_blocks][KT][nsf][512]
    const int32_t *expert_ids;
    const int32_t *brow;      // first row of each block (fixed-capacity layout), or null: block j at j * b
    const int32_t *npp;       // num_rows_post_pad
    const int32_t *sorted;    // sorted_route_ids
    const float *wts;         // topk_w flattened [MK]
    uint8_t *hq;              // kind 1: [cap_rows][I] codes
    uint8_t *hs;              // kind 1: [cap_blocks][I/128][nsf][512] atoms
    float *yr;                // kind 2: [MK][d]
    int32_t *dev_status;
    int b, n_mma, nsf, n_mt, KT, I, d, MK;
    int a_rows;               // rows of one expert in the A tensor (2I or d)
    int stages;               // ring depth (<= kMaxStages)
    int E, cap_blocks;        // experts, and the row-blocks the operands hold (debug bounds checks)
};

// Scale-atom byte offset of (row m of a 128-row group, k-block kb of 4):
// 32 rows x 16 bytes; row m0 = m % 32 holds, for each 32-row group
// m1 = m / 32, the four k-blocks' bytes.  tcgen05.cp .32x128b.warpx4 copies
// it into TMEM (4 columns, every 32-lane quadrant).
__host__ __device__ __forceinline__ int atom_off(int m, int kb) { return (m & 31) * 16 + (m >> 5) * 4 + kb; }

__device__ __forceinline__ int mx_exp(uint32_t amax_bits)
{
    const int ef = static_cast<int>((amax_bits >> 23) & 0xFFu);
    if (ef == 0)
        return -127;
    int X = ef - 127 - 8;
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}

__device__ __forceinline__ float mx_inv(int X)
{
    return X <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - X) << 23) : __uint_as_float(0x00400000u);
}

// SiLU(g) * u with the fast exponential and division: no branches, so
// independent columns pipeline (relative error a few ulp of fp32).
__device__ __forceinline__ float silu_mul_fast(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ uint32_t to_e4m3(float u)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(u));
    return r & 0xFFu;
}

// ---------------------------------------------------------------- act quant
// One warp per aligned row; lane l quantizes 32-element blocks l, l+32, ...
// with 16-byte loads and stores (the block's amax stays in the lane).
__global__ void __launch_bounds__(256) act_quant_kernel(const __nv_bfloat16 *__restrict__ x, int d, int k, int MK,
                                                        const int32_t *__restrict__ sorted,
                                                        const int32_t *__restrict__ npp,
                                                        const int32_t *__restrict__ brow, int b, int nsf,
                                                        int cap_rows, uint8_t *__restrict__ xq,
                                                        uint8_t *__restrict__ xs, int32_t *__restrict__ done,
                                                        int32_t *__restrict__ dev_status)
{
    // chained by programmatic dependent launch: the alignment must be done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    int rows = *npp;                              // b * active blocks
    if (!MOE_IN_BOUNDS(rows >= 0 && rows <= cap_rows, dev_status))
        rows = 0;
    // the GEMM's per-block counters of finished first-GEMM tiles start at 0
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < rows / b; j += gridDim.x * blockDim.x) {
        const int jb = brow ? brow[j] / b : j;
        if (MOE_IN_BOUNDS(jb >= 0 && jb < cap_rows / b, dev_status))
            done[jb] = 0;
    }
    const int nblk = d / 32, KT = d / 128;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int cr = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); cr < rows; cr += nw) {
        // the cr-th row of the active blocks: row rho of row-block jb
        const int j = cr / b, m = cr - j * b;
        const int jb = brow ? brow[j] / b : j, rho = jb * b + m;
        if (!MOE_IN_BOUNDS(jb >= 0 && jb < cap_rows / b, dev_status))
            continue;
        int r = sorted[rho];
        if (!MOE_IN_BOUNDS(r >= 0 && r <= MK, dev_status))
            r = MK;                                   // read as padding
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(r < MK ? r / k : 0) * d);
        uint4 *qr = reinterpret_cast<uint4 *>(xq + static_cast<int64_t>(rho) * d);
        for (int blk = lane; blk < nblk; blk += 32) {
            float v[32];
            if (r < MK) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 w = __ldg(xr + blk * 4 + i);
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[i * 8 + 2 * j] = __uint_as_float(ww[j] << 16);
                        v[i * 8 + 2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = 0.f;
            }
            uint32_t amax = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                amax = max(amax, __float_as_uint(fabsf(v[i])));
            const int X = mx_exp(amax);
            const float inv = mx_inv(X);
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                packed[i] = to_e4m3(v[4 * i] * inv) | (to_e4m3(v[4 * i + 1] * inv) << 8) |
                            (to_e4m3(v[4 * i + 2] * inv) << 16) | (to_e4m3(v[4 * i + 3] * inv) << 24);
            qr[blk * 2] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            qr[blk * 2 + 1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            xs[((static_cast<int64_t>(jb) * KT + blk / 4) * nsf + m / 128) * 512 + atom_off(m & 127, blk & 3)] =
                static_cast<uint8_t>(X + 127);
        }
    }
}

// ---------------------------------------------------------------- prepare
// A-operand scale atoms of all experts.  kind 1 (W13, N = 2I): m-tile mt
// holds gate rows 64mt..64mt+63 then up rows I+64mt..; kind 2 (W2, N = d):
// rows 128mt..128mt+127.
__global__ void prepare_sfa_kernel(const uint8_t *__restrict__ s, int E, int N, int K, int kind, int I,
                                   uint8_t *__restrict__ atoms)
{
    const int KT = K / 128, n_mt = kind == 1 ? I / 64 : N / 128;
    const int64_t total = static_cast<int64_t>(E) * n_mt * KT * 512;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int byte = static_cast<int>(i % 512);
        const int64_t atom = i / 512;
        const int kt = static_cast<int>(atom % KT);
        const int mt = static_cast<int>((atom / KT) % n_mt);
        const int e = static_cast<int>(atom / (static_cast<int64_t>(KT) * n_mt));
        // invert atom_off: byte = m0*16 + m1*4 + kb
        const int m0 = byte / 16, m1 = (byte % 16) / 4, kb = byte % 4;
        const int m = m1 * 32 + m0;
        int row;
        if (kind == 1)
            row = m < 64 ? 64 * mt + m : I + 64 * mt + (m - 64);
        else
            row = 128 * mt + m;
        atoms[i] = s[(static_cast<int64_t>(e) * N + row) * (K / 32) + kt * 4 + kb];
    }
}

// ---------------------------------------------------------------- the GEMMs
// Both expert GEMMs in one persistent kernel.  The tile list is every
// first-GEMM tile (W13 against the quantized activations; epilogue SwiGLU and
// requantization into Hq/Hs), block-major, then every second-GEMM tile (W2
// against Hq; epilogue w_route * acc per route).  CTA c takes tiles c,
// c + grid, ..., so it finishes its first-GEMM tiles before any second-GEMM
// tile.  A second-GEMM tile of block jb waits until all first-GEMM tiles of
// jb have published Hq/Hs (a per-block counter, release/acquire, plus proxy
// fences because TMA reads what generic stores wrote).  SMs that run out of
// first-GEMM tiles start on the second GEMM instead of idling at a kernel
// boundary.  Progress needs every CTA resident: the grid is one CTA per SM.
// A tile's block: its expert and row-block, and (debug build) whether both
// lie inside their buffers; every role takes the same decision for a tile.
__device__ __forceinline__ bool block_ok(const Args &a, int jb, int &e, int &rb)
{
    e = a.expert_ids[jb];
    rb = a.brow ? a.brow[jb] / a.b : jb;
    return MOE_IN_BOUNDS(e >= 0 && e < a.E && rb >= 0 && rb < a.cap_blocks, a.dev_status);
}

__device__ __forceinline__ int tile_kind(int t, int total1, int n_mt1, int n_mt2, int &jb, int &mt)
{
    if (t < total1) {
        jb = t / n_mt1;
        mt = t - jb * n_mt1;
        return 1;
    }
    t -= total1;
    jb = t / n_mt2;
    mt = t - jb * n_mt2;
    return 2;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
            const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, const Args a1,
            const Args a2, int32_t *done)
{
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1024-byte aligned base for the 128-byte swizzled tiles
    const uint32_t raw = tc::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int n_mma = a1.n_mma, nsf = a1.nsf;                      // the same for both GEMMs
    const int NB = n_mma * 128;                                    // B tile bytes
    const int stage_bytes = (16384 + NB + 512 + nsf * 512 + 1023) & ~1023;
    const int kStages = a1.stages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * stage_bytes);
    const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8 * kStages;
    const uint32_t accf0 = full0 + 16 * kStages, acce0 = accf0 + 16, fin = acce0 + 16;   // accf[2], acce[2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // 16-byte aligned after the 128-byte barrier header
    float *ubuf = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + kHeaderBytes);   // [2 bufs][2 pairs][32][33]
    int *t_route = reinterpret_cast<int *>(ubuf + 4 * 32 * 33);    // [256] routes of the tile's rows
    float *t_w = reinterpret_cast<float *>(t_route + 256);         // [256] their weights
    // two accumulator buffers (columns 0 and 128) when a tile fits in 128
    // columns, so the MMA of the next tile overlaps this tile's epilogue
    const int nbuf = n_mma <= 128 ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(accf0 + 8 * i, 1);
            tc::mbar_init(acce0 + 8 * i, 4);
        }
        tc::mbar_init(fin, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmA1);
        tc::prefetch_tmap(&tmB1);
        tc::prefetch_tmap(&tmA2);
        tc::prefetch_tmap(&tmB2);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // set-up above overlapped the previous kernel; its outputs are read below
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    int n_blocks = *a1.npp / a1.b;
    if (!MOE_IN_BOUNDS(n_blocks >= 0 && n_blocks <= a1.cap_blocks, a1.dev_status))
        n_blocks = 0;
    const int n_mt1 = a1.n_mt, n_mt2 = a2.n_mt;
    const int total1 = n_blocks * n_mt1, total = total1 + n_blocks * n_mt2;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0, issued = 0;
            uint32_t ph = 0;
            const uint32_t tx = 16384u + NB + 512u + nsf * 512u;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                int jb, mt;
                const int kind = tile_kind(t, total1, n_mt1, n_mt2, jb, mt);
                int e, rb;                                          // the block's expert and row-block
                if (!block_ok(a1, jb, e, rb))
                    continue;
                const int KT = kind == 1 ? a1.KT : a2.KT;
                const int n_mt = kind == 1 ? n_mt1 : n_mt2;
                const int a_rows = kind == 1 ? a1.a_rows : a2.a_rows;
                const CUtensorMap *tA = kind == 1 ? &tmA1 : &tmA2;
                const CUtensorMap *tB = kind == 1 ? &tmB1 : &tmB2;
                const uint8_t *sfa = kind == 1 ? a1.sfa : a2.sfa;
                const uint8_t *sfb = kind == 1 ? a1.sfb : a2.sfb;
                if (kind == 2) {
                    // block jb's Hq/Hs: every first-GEMM tile of jb published
                    const long long t0 = clock64();
                    const long long limit = static_cast<long long>(kWaitNs) * 5 / 2;
                    int v;
                    for (;;) {
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(done + rb) : "memory");
                        if (v >= n_mt1)
                            break;
                        if (*abort_flag || clock64() - t0 > limit) {
                            *abort_flag = 1;
                            break;
                        }
                    }
                    if (v < n_mt1)
                        break;
                    // the tensor-memory-access proxy reads what generic stores wrote
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                for (int kt = 0; kt < KT; ++kt, ++issued) {
                    if (!tc::mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, kWaitNs))
                        break;
                    uint8_t *st = smem + s * stage_bytes;
                    const uint32_t fb = full0 + 8 * s;
                    tc::mbar_arrive_expect_tx(fb, tx);
                    const int x = kt * 128;
                    if (kind == 1) {
                        tc::tma_load_2d(tc::smem_u32(st), tA, x, e * a_rows + 64 * mt, fb);
                        tc::tma_load_2d(tc::smem_u32(st + 8192), tA, x, e * a_rows + a1.I + 64 * mt, fb);
                    } else {
                        tc::tma_load_2d(tc::smem_u32(st), tA, x, e * a_rows + 128 * mt, fb);
                    }
                    tc::tma_load_2d(tc::smem_u32(st + 16384), tB, x, rb * a1.b, fb);
                    tc::bulk_load(tc::smem_u32(st + 16384 + NB),
                                  sfa + ((static_cast<int64_t>(e) * n_mt + mt) * KT + kt) * 512, 512, fb);
                    tc::bulk_load(tc::smem_u32(st + 16384 + NB + 512),
                                  sfb + (static_cast<int64_t>(rb) * KT + kt) * nsf * 512, nsf * 512, fb);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // every issued copy must land before the CTA may finish
            volatile int never = 0;
            const int n = issued < kStages ? issued : kStages;
            for (int i = 1; i <= n; ++i) {
                int st = s - i;
                uint32_t pp = ph;
                if (st < 0) {
                    st += kStages;
                    pp ^= 1u;
                }
                tc::mbar_wait(full0 + 8 * st, pp, &never, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, ti = 0;
            uint32_t ph = 0;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                int jb, mt, e, rb;
                tile_kind(t, total1, n_mt1, n_mt2, jb, mt);
                if (!block_ok(a1, jb, e, rb))
                    continue;
                const int tix = ti++;                           // this CTA's tiles that run
                const int KT = t < total1 ? a1.KT : a2.KT;
                const int buf = nbuf == 2 ? (tix & 1) : 0;
                const uint32_t use = static_cast<uint32_t>(nbuf == 2 ? (tix >> 1) : tix);
                if (!tc::mbar_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, abort_flag, kWaitNs))
                    break;
                tc::tc_fence_after();
                const uint32_t acc = tmem + 128 * buf;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(full0 + 8 * s, ph, abort_flag, kWaitNs))
                        break;
                    tc::tc_fence_after();
                    const uint32_t sa = tc::smem_u32(smem + s * stage_bytes);
                    const uint32_t sb = sa + 16384;
                    const uint32_t ssfa = sb + NB, ssfb = ssfa + 512;
                    const uint32_t tsfa = tmem + 256 + s * 16, tsfb = tsfa + 4;
                    tc::tc_cp_32x128b_x4(tsfa, tc::smem_desc(ssfa, 0, 128, tc::kLayoutNone));
                    for (int q = 0; q < nsf; ++q)
                        tc::tc_cp_32x128b_x4(tsfb + 4 * q, tc::smem_desc(ssfb + 512 * q, 0, 128, tc::kLayoutNone));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::smem_desc(sa + 32 * kk, 16, 1024, tc::kLayoutSw128);
                        const uint64_t bd = tc::smem_desc(sb + 32 * kk, 16, 1024, tc::kLayoutSw128);
                        tc::mma_mxf8(acc, ad, bd, tc::idesc_mxf8(128, n_mma, kk, kk), tsfa, tsfb,
                                     (kt | kk) != 0 ? 1u : 0u);
                    }
                    tc::tc_commit(empty0 + 8 * s);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                tc::tc_commit(accf0 + 8 * buf);
            }
            // all MMAs of this CTA complete before TMEM is released
            tc::tc_commit(fin);
            volatile int never = 0;
            tc::mbar_wait(fin, 0, &never, kWaitNs);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                       // TMEM lane quadrant
        const int etid = threadIdx.x - 64;
        int ti = 0;
        const int b = a1.b;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int jb, mt, e, rb;                                        // the block's expert and row-block
            const int kind = tile_kind(t, total1, n_mt1, n_mt2, jb, mt);
            if (!block_ok(a1, jb, e, rb))
                continue;
            const int tix = ti++;                                     // this CTA's tiles that run
            const int buf = nbuf == 2 ? (tix & 1) : 0;
            const uint32_t use = static_cast<uint32_t>(nbuf == 2 ? (tix >> 1) : tix);
            const int rho0 = rb * b;
            if (kind == 2) {
                // routes and routing weights of the tile's rows, loaded once
                for (int c = etid; c < b; c += 128) {
                    int r = a2.sorted[rho0 + c];
                    if (!MOE_IN_BOUNDS(r >= 0 && r <= a2.MK, a2.dev_status))
                        r = a2.MK;                                // read as padding
                    t_route[c] = r;
                    t_w[c] = r < a2.MK ? a2.wts[r] : 0.f;
                }
            }
            if (!tc::mbar_wait(accf0 + 8 * buf, use & 1u, abort_flag, kWaitNs) && a1.dev_status)
                atomicCAS(a1.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
            tc::tc_fence_after();
            tc::named_bar(1, 128);
            for (int c0 = 0, chunk = 0; c0 < b; c0 += 32, ++chunk) {
                uint32_t v[32];
                tc::tmem_ld_32x32b_x32(tmem + 128 * buf + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
                tc::tmem_ld_wait();
                const int ncol = min(32, b - c0);
                if (kind == 1) {
                    // Lanes 0..63 of the tile are gate rows, 64..127 up rows:
                    // quadrant q pairs with q ^ 2 (same 32 neurons).  The
                    // gate quadrant finishes columns 0..15 of the chunk, the
                    // up quadrant columns 16..31; each hands the other half
                    // of its values over through a double-buffered exchange.
                    const bool is_gate = q < 2;
                    float *ub = ubuf + ((chunk & 1) * 2 + (q & 1)) * 32 * 33 + lane * 33;
                    const int keep = is_gate ? 0 : 16;
                    // register indices stay compile-time constants (a
                    // runtime index would move v to local memory)
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        ub[16 - keep + c] = __uint_as_float(is_gate ? v[16 + c] : v[c]);
                    tc::named_bar(1, 128);
                    // the 16 columns are independent: SiLU, block amax and
                    // code conversion each run as 16 parallel chains
                    float hv[16];
                    uint32_t am[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float mine = __uint_as_float(is_gate ? v[c] : v[16 + c]);
                        const float other = ub[keep + c];
                        hv[c] = is_gate ? silu_mul_fast(mine, other) : silu_mul_fast(other, mine);
                    }
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        am[c] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[c])));
                    const int n = 64 * mt + 32 * (q & 1) + lane;     // neuron of this lane
                    const int kblk = 2 * mt + (q & 1);                // its 32-neuron block
                    uint8_t *hrow = a1.hq + static_cast<int64_t>(rho0 + c0 + keep) * a1.I + n;
                    uint8_t *hsa = a1.hs + ((static_cast<int64_t>(rb) * (a1.I / 128) + kblk / 4) * nsf) * 512;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int X = mx_exp(am[c]);
                        if (keep + c < ncol) {
                            hrow[static_cast<int64_t>(c) * a1.I] = static_cast<uint8_t>(to_e4m3(hv[c] * mx_inv(X)));
                            if (lane == 0) {
                                const int m = c0 + keep + c;
                                hsa[(m / 128) * 512 + atom_off(m & 127, kblk & 3)] = static_cast<uint8_t>(X + 127);
                            }
                        }
                    }
                } else {
                    const int o = 128 * mt + 32 * q + lane;          // output row of this lane
                    // the chunk's routes and weights into registers first
                    // (broadcast 16-byte loads), then 32 independent stores
                    int rr[32];
                    float ww[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int4 r4 = reinterpret_cast<const int4 *>(t_route + c0)[i];
                        const float4 w4 = reinterpret_cast<const float4 *>(t_w + c0)[i];
                        rr[4 * i] = r4.x;
                        rr[4 * i + 1] = r4.y;
                        rr[4 * i + 2] = r4.z;
                        rr[4 * i + 3] = r4.w;
                        ww[4 * i] = w4.x;
                        ww[4 * i + 1] = w4.y;
                        ww[4 * i + 2] = w4.z;
                        ww[4 * i + 3] = w4.w;
                    }
                    float *yo = a2.yr + o;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (c < ncol && rr[c] < a2.MK)
                            yo[static_cast<int64_t>(rr[c]) * a2.d] = ww[c] * __uint_as_float(v[c]);
                    }
                }
            }
            if (kind == 1)
                asm volatile("fence.proxy.async.global;" ::: "memory");   // Hq/Hs are read by TMA
            tc::tc_fence_before();
            tc::named_bar(1, 128);                    // t_route / t_w reuse by the next tile
            if (lane == 0)
                tc::mbar_arrive(acce0 + 8 * buf);
            if (kind == 1 && etid == 0)                // every epilogue thread's stores are ordered before this
                asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(done + rb) : "memory");
        }
        (void)etid;
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- combine
// Four consecutive outputs per thread (d is a multiple of 128): 16-byte
// loads of the k route rows, summed in slot order.  The slot ids of a group
// of 8 slots are loaded together, then all their rows, so a thread waits for
// two memory round trips per 8 slots instead of two per slot.
template <typename YT>
__global__ void combine_kernel(const float *__restrict__ yr, const int32_t *__restrict__ ids, int M, int k, int d,
                               int E, YT *__restrict__ y)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int d4 = d >> 2;
    const int total = M * d4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / d4, o4 = i - t * d4;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < k; j0 += 8) {
            int e[8];
            float4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                e[jj] = j0 + jj < k ? __ldg(ids + t * k + j0 + jj) : -1;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                v[jj] = e[jj] >= 0 && e[jj] < E
                            ? __ldcs(reinterpret_cast<const float4 *>(yr + static_cast<int64_t>(t * k + j0 + jj) * d) + o4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (e[jj] >= 0 && e[jj] < E) {
                    s.x += v[jj].x;
                    s.y += v[jj].y;
                    s.z += v[jj].z;
                    s.w += v[jj].w;
                }
            }
        }
        if constexpr (sizeof(YT) == 4) {
            reinterpret_cast<float4 *>(y)[i] = s;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t *>(&lo);
            pk.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(y)[i] = pk;
        }
    }
}

// ---------------------------------------------------------------- host helpers

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D uint8 tensor [rows][inner] (row stride = inner bytes), box
// 128 bytes x box_rows, 128-byte swizzle.
static bool tmap_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct WsLayout {
    size_t xq, xs, hq, hs, yr, done, total;
};

static WsLayout ws_layout(int M, int k, int d, int I, int b, int cap_rows)
{
    const int n_mma = (b + 15) / 16 * 16;
    const int nsf = (n_mma + 127) / 128;
    const int cap_blocks = cap_rows / b;
    WsLayout L;
    size_t off = 0;
    L.xq = off;
    off += ws_round(static_cast<size_t>(cap_rows) * d);
    L.xs = off;
    off += ws_round(static_cast<size_t>(cap_blocks) * (d / 128) * nsf * 512);
    L.hq = off;
    off += ws_round(static_cast<size_t>(cap_rows) * I);
    L.hs = off;
    off += ws_round(static_cast<size_t>(cap_blocks) * (I / 128) * nsf * 512);
    L.yr = off;
    off += ws_round(static_cast<size_t>(M) * k * d * sizeof(float));
    L.done = off;
    off += ws_round(static_cast<size_t>(cap_blocks) * sizeof(int32_t));
    L.total = off;
    return L;
}

}  // namespace gg

bool grouped_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, int elem_bytes, const void *base, uint64_t inner,
                     uint64_t rows, uint32_t box_inner, uint32_t box_rows, bool sw128)
{
    auto fn = gg::encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * static_cast<cuuint64_t>(elem_bytes)};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int grouped_sm_count() { return device_sm_count(); }

moe_status_t grouped_combine_launch(const float *yr, const int32_t *ids, int M, int k, int d, int E, void *y,
                                    bool y_f32, cudaStream_t s)
{
    const int64_t n = static_cast<int64_t>(M) * (d / 4);
    const int cb = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    const cudaError_t e = y_f32 ? launch_pdl(gg::combine_kernel<float>, dim3(cb), dim3(256), 0, s, yr, ids, M, k, d, E,
                                             static_cast<float *>(y))
                                : launch_pdl(gg::combine_kernel<__nv_bfloat16>, dim3(cb), dim3(256), 0, s, yr, ids, M, k,
                                             d, E, static_cast<__nv_bfloat16 *>(y));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

using namespace moe;
using namespace moe::gg;

MOE_API moe_status_t moe_grouped_prepare_size(const moe_weights_t *w13, const moe_weights_t *w2, size_t *sfa13_bytes,
                                              size_t *sfa2_bytes)
{
    if (!w13 || !w2 || !sfa13_bytes || !sfa2_bytes)
        return MOE_ERR_INVALID_ARG;
    const bool nv4 = w13->fmt == MOE_W_NVFP4S && w2->fmt == MOE_W_NVFP4S;
    if (!nv4 && (w13->fmt != MOE_W_MXFP8 || w2->fmt != MOE_W_MXFP8))
        return MOE_ERR_INVALID_ARG;
    const int I = w2->K, d = w13->K, E = w13->E;
    if (w13->N != 2 * I || w2->N != d || d % 128 || I % 128)
        return MOE_ERR_UNSUPPORTED;
    if (nv4) {
        if (d % 256)
            return MOE_ERR_UNSUPPORTED;
        *sfa13_bytes = grouped_nv4_prepare_bytes(E, 2 * I, d);
        *sfa2_bytes = grouped_nv4_prepare_bytes(w2->E, d, I);
        return MOE_OK;
    }
    *sfa13_bytes = static_cast<size_t>(E) * (I / 64) * (d / 128) * 512;
    *sfa2_bytes = static_cast<size_t>(E) * (d / 128) * (I / 128) * 512;
    return MOE_OK;
}

MOE_API moe_status_t moe_grouped_prepare(const moe_weights_t *w13, const moe_weights_t *w2, void *sfa13, void *sfa2,
                                         void *stream)
{
    size_t b13, b2;
    moe_status_t st = moe_grouped_prepare_size(w13, w2, &b13, &b2);
    if (st != MOE_OK)
        return st;
    if (w13->fmt != MOE_W_MXFP8)
        return MOE_ERR_INVALID_ARG;              // NVFP4S: moe_grouped_prepare_nvfp4s
    if (!w13->scale || !w2->scale || !sfa13 || !sfa2)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    prepare_sfa_kernel<<<1024, 256, 0, s>>>(static_cast<const uint8_t *>(w13->scale), w13->E, w13->N, w13->K, 1,
                                            w2->K, static_cast<uint8_t *>(sfa13));
    if (launch_status() != MOE_OK)
        return MOE_ERR_CUDA;
    prepare_sfa_kernel<<<1024, 256, 0, s>>>(static_cast<const uint8_t *>(w2->scale), w2->E, w2->N, w2->K, 2, w2->K,
                                            static_cast<uint8_t *>(sfa2));
    return launch_status();
}

MOE_API moe_status_t moe_grouped_prepare_nvfp4s(const moe_weights_t *w13, const moe_weights_t *w2, float alpha_x,
                                                float alpha_h, void *p13, void *p2, void *stream)
{
    size_t b13, b2;
    if (!w13 || !w2 || w13->fmt != MOE_W_NVFP4S || w2->fmt != MOE_W_NVFP4S)
        return MOE_ERR_INVALID_ARG;
    moe_status_t st = moe_grouped_prepare_size(w13, w2, &b13, &b2);
    if (st != MOE_OK)
        return st;
    if (w2->E != w13->E || !w13->zero || !w2->zero || !w13->scale || !w2->scale || !w13->alpha || !w2->alpha ||
        !p13 || !p2 || !aligned(p13, 256) || !aligned(p2, 256) || !aligned(w13->zero, 16) || !aligned(w2->zero, 16) ||
        !aligned(w13->scale, 16) || !aligned(w2->scale, 16))
        return MOE_ERR_INVALID_ARG;
    if (!(alpha_x > 0.f) || !(alpha_h > 0.f) || !std::isfinite(alpha_x) || !std::isfinite(alpha_h))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    st = grouped_nv4_prepare(w13, alpha_x, p13, s);
    if (st != MOE_OK)
        return st;
    return grouped_nv4_prepare(w2, alpha_h, p2, s);
}

MOE_API moe_status_t moe_ffn_grouped_workspace_size(int32_t M, int32_t k, int32_t d, int32_t I, int32_t b,
                                                    int32_t cap_rows, size_t *bytes)
{
    if (M < 0 || k < 1 || d < 1 || I < 1 || b < 1 || cap_rows < 0 || !bytes)
        return MOE_ERR_INVALID_ARG;
    // one size for both weight formats: the larger of the MXFP8 and AWQ layouts
    const size_t mx = ws_layout(M, k, d, I, b, cap_rows).total, aw = grouped_awq_workspace(M, k, d, I, b, cap_rows);
    *bytes = mx > aw ? mx : aw;
    return MOE_OK;
}

// The grouped layer on aligned rows (block_rows null: block j is rows j*b ..)
// or on the fixed-capacity layout (block j starts at row block_rows[j]).
static moe_status_t grouped_impl(const void *x, int32_t xdt, int32_t M, int32_t d, const int32_t *topk_ids,
                                 const float *topk_w, int32_t k, const moe_weights_t *w13, const moe_weights_t *w2,
                                 const void *sfa13, const void *sfa2, const int32_t *sorted_route_ids,
                                 const int32_t *expert_ids, const int32_t *block_rows,
                                 const int32_t *num_rows_post_pad, int32_t b, int32_t cap_rows, void *y, int32_t ydt,
                                 void *ws, size_t ws_bytes, int32_t *dev_status, void *stream)
{
    if (M < 0 || d < 1 || k < 1 || !w13 || !w2)
        return MOE_ERR_INVALID_ARG;
    const bool awq = w13->fmt == MOE_W_AWQ4 && w2->fmt == MOE_W_AWQ4;
    const bool nv4 = w13->fmt == MOE_W_NVFP4S && w2->fmt == MOE_W_NVFP4S;
    if (!awq && !nv4 && (w13->fmt != MOE_W_MXFP8 || w2->fmt != MOE_W_MXFP8 || xdt != MOE_BF16))
        return MOE_ERR_UNSUPPORTED;
    if ((awq || nv4) && xdt != MOE_FP16 && xdt != MOE_BF16)
        return MOE_ERR_UNSUPPORTED;
    if (ydt != MOE_BF16 && ydt != MOE_FP32)
        return MOE_ERR_UNSUPPORTED;
    const int I = w2->K, E = w13->E;
    if (w13->N != 2 * I || w13->K != d || w2->N != d || w2->E != E || E < 1)
        return MOE_ERR_INVALID_ARG;
    if (d % 128 || I % 128 || b < 8 || b > 256 || b % 8)
        return MOE_ERR_UNSUPPORTED;
    const int64_t mk = static_cast<int64_t>(M) * k;
    if (block_rows) {
        // fixed capacity: any multiple of b holds the layout it was built for
        if (cap_rows < b || cap_rows % b)
            return MOE_ERR_CAPACITY;
        if (awq || nv4)
            return MOE_ERR_UNSUPPORTED;
    } else {
        int32_t need_rows, need_blocks;
        if (moe_align_capacity(M, k, E, b, &need_rows, &need_blocks) != MOE_OK)
            return MOE_ERR_UNSUPPORTED;
        if (cap_rows < need_rows || cap_rows % b)
            return MOE_ERR_CAPACITY;
    }
    if (M == 0)
        return MOE_OK;
    if (nv4) {
        if (!x || !topk_ids || !topk_w || !y || !sfa13 || !sfa2 || !sorted_route_ids || !expert_ids ||
            !num_rows_post_pad || !w13->q || !w2->q)
            return MOE_ERR_INVALID_ARG;
        if (!aligned(w13->q, 16) || !aligned(w2->q, 16) || !aligned(sfa13, 256) || !aligned(sfa2, 256) ||
            !aligned(x, 16) || !aligned(y, 16))
            return MOE_ERR_INVALID_ARG;
        if (static_cast<int64_t>(M) * (d / 4) > INT32_MAX || d % 256)
            return MOE_ERR_UNSUPPORTED;
        size_t need = 0;
        moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows, &need);
        if (!ws || ws_bytes < need || !aligned(ws, 256))
            return MOE_ERR_WORKSPACE;
        return grouped_nv4_launch(x, xdt == MOE_BF16, M, d, I, E, topk_ids, topk_w, k, w13, w2, sfa13, sfa2,
                                  sorted_route_ids, expert_ids, num_rows_post_pad, b, cap_rows, y, ydt == MOE_FP32, ws,
                                  dev_status, as_stream(stream));
    }
    if (awq) {
        if (!x || !topk_ids || !topk_w || !y || !sorted_route_ids || !expert_ids || !num_rows_post_pad ||
            !w13->q || !w2->q || !w13->scale || !w2->scale || !w13->zero || !w2->zero)
            return MOE_ERR_INVALID_ARG;
        if (!aligned(w13->q, 16) || !aligned(w2->q, 16) || !aligned(w13->scale, 16) || !aligned(w2->scale, 16) ||
            !aligned(w13->zero, 16) || !aligned(w2->zero, 16) || !aligned(x, 16) || !aligned(y, 16))
            return MOE_ERR_INVALID_ARG;
        if (static_cast<int64_t>(M) * (d / 4) > INT32_MAX || d > 8192 || I > 8192)
            return MOE_ERR_UNSUPPORTED;
        size_t need = 0;
        moe_ffn_grouped_workspace_size(M, k, d, I, b, cap_rows, &need);
        if (!ws || ws_bytes < need || !aligned(ws, 256))
            return MOE_ERR_WORKSPACE;
        return grouped_awq_launch(x, xdt == MOE_BF16, M, d, I, E, topk_ids, topk_w, k, w13, w2, sorted_route_ids,
                                  expert_ids, num_rows_post_pad, b, cap_rows, y, ydt == MOE_FP32, ws, dev_status,
                                  as_stream(stream));
    }
    if (!x || !topk_ids || !topk_w || !y || !sfa13 || !sfa2 || !sorted_route_ids || !expert_ids ||
        !num_rows_post_pad || !w13->q || !w2->q)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(w13->q, 16) || !aligned(w2->q, 16) || !aligned(sfa13, 16) || !aligned(sfa2, 16) ||
        !aligned(x, 16) || !aligned(y, 16))
        return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(M) * (d / 4) > INT32_MAX)
        return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(M, k, d, I, b, cap_rows);
    if (!ws || ws_bytes < L.total || !aligned(ws, 256))
        return MOE_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint8_t *xq = w + L.xq, *xs = w + L.xs, *hq = w + L.hq, *hs = w + L.hs;
    float *yr = reinterpret_cast<float *>(w + L.yr);
    int32_t *done = reinterpret_cast<int32_t *>(w + L.done);
    const int n_mma = (b + 15) / 16 * 16;
    const int nsf = (n_mma + 127) / 128;
    cudaStream_t s = as_stream(stream);

    // tensor maps: A = weights [E*N][K], B = activations [cap_rows][K]
    CUtensorMap tA1, tB1, tA2, tB2;
    if (!tmap_u8(&tA1, w13->q, d, static_cast<uint64_t>(E) * 2 * I, 64) ||
        !tmap_u8(&tB1, xq, d, cap_rows, n_mma) ||
        !tmap_u8(&tA2, w2->q, I, static_cast<uint64_t>(E) * d, 128) ||
        !tmap_u8(&tB2, hq, I, cap_rows, n_mma))
        return MOE_ERR_CUDA;

    if (launch_pdl(act_quant_kernel, dim3(device_sm_count() * 4), dim3(256), 0, s, static_cast<const __nv_bfloat16 *>(x), d,
                   k, static_cast<int>(mk), sorted_route_ids, num_rows_post_pad, block_rows, b, nsf, cap_rows, xq,
                   xs, done, dev_status) != cudaSuccess)
        return MOE_ERR_CUDA;

    const int stage_bytes = (16384 + n_mma * 128 + 512 + nsf * 512 + 1023) & ~1023;
    const size_t fixed = 1024 + kHeaderBytes + 4 * 32 * 33 * sizeof(float) + 512 * 4;
    const int stages = static_cast<int>((227 * 1024 - fixed) / stage_bytes) < kMaxStages
                           ? static_cast<int>((227 * 1024 - fixed) / stage_bytes)
                           : kMaxStages;
    const size_t smem = fixed + static_cast<size_t>(stages) * stage_bytes;
    static std::atomic<uint64_t> attr_done{0};
    if (stages < 2 || smem > 227 * 1024 ||
        !smem_attr_once(attr_done, reinterpret_cast<const void *>(gemm_kernel), 227 * 1024))
        return MOE_ERR_CUDA;
    const int grid = device_sm_count();

    Args a1{static_cast<const uint8_t *>(sfa13), xs, expert_ids, block_rows, num_rows_post_pad, sorted_route_ids, topk_w,
            hq, hs, nullptr, dev_status, b, n_mma, nsf, I / 64, d / 128, I, d, static_cast<int>(mk), 2 * I, stages,
            E, cap_rows / b};
    Args a2{static_cast<const uint8_t *>(sfa2), hs, expert_ids, block_rows, num_rows_post_pad, sorted_route_ids, topk_w,
            nullptr, nullptr, yr, dev_status, b, n_mma, nsf, d / 128, I / 128, I, d, static_cast<int>(mk), d, stages,
            E, cap_rows / b};
    if (launch_pdl(gemm_kernel, dim3(grid), dim3(kThreads), smem, s, tA1, tB1, tA2, tB2, a1, a2, done) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, topk_ids, M, k, d, E, y, ydt == MOE_FP32, s);
}

MOE_API moe_status_t moe_ffn_grouped(const void *x, int32_t xdt, int32_t M, int32_t d, const int32_t *topk_ids,
                                     const float *topk_w, int32_t k, const moe_weights_t *w13,
                                     const moe_weights_t *w2, const void *sfa13, const void *sfa2,
                                     const int32_t *sorted_route_ids, const int32_t *expert_ids,
                                     const int32_t *num_rows_post_pad, int32_t b, int32_t cap_rows, void *y,
                                     int32_t ydt, void *ws, size_t ws_bytes, int32_t *dev_status, void *stream)
{
    return grouped_impl(x, xdt, M, d, topk_ids, topk_w, k, w13, w2, sfa13, sfa2, sorted_route_ids, expert_ids,
                        nullptr, num_rows_post_pad, b, cap_rows, y, ydt, ws, ws_bytes, dev_status, stream);
}

MOE_API moe_status_t moe_ffn_grouped_batched(const void *x, int32_t xdt, int32_t M, int32_t d,
                                             const int32_t *topk_ids, const float *topk_w, int32_t k,
                                             const moe_weights_t *w13, const moe_weights_t *w2, const void *sfa13,
                                             const void *sfa2, const int32_t *sorted_route_ids,
                                             const int32_t *expert_ids, const int32_t *block_rows,
                                             const int32_t *num_rows_post_pad, int32_t b, int32_t cap_rows,
                                             void *y, int32_t ydt, void *ws, size_t ws_bytes, int32_t *dev_status,
                                             void *stream)
{
    if (!block_rows)
        return MOE_ERR_INVALID_ARG;
    return grouped_impl(x, xdt, M, d, topk_ids, topk_w, k, w13, w2, sfa13, sfa2, sorted_route_ids, expert_ids,
                        block_rows, num_rows_post_pad, b, cap_rows, y, ydt, ws, ws_bytes, dev_status, stream);
}
