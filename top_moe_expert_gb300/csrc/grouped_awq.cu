// grouped_awq.cu -- expert-centric grouped path for 4-bit AWQ weights.
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic" (arXiv 2607.26316),
// opening paragraph: packed-AWQ MoE GEMMs (4-bit values, group 128 along K,
// fp16 scale and 4-bit zero per group) applied to the aligned rows, one MoE
// block of b rows at a time; its schedule paragraphs show that a split-K
// schedule with a global reduction makes a route's bits depend on its block
// membership.  Here every output element accumulates its K-tiles in one
// fixed ascending order in one TMEM accumulator -- no split-K, no atomics --
// so the result depends on neither membership nor grid, and repeats are
// bit-identical.
//
// The tensor cores take fp16 x fp16 (tcgen05 kind::f16, FP32 accumulate):
//   gather_kernel   : Xg[rho] = x[route(rho) / k] as fp16 (zero for padding)
//   gemm_kernel<1>  : [g;u] = W13_e Xg^T; epilogue h = SiLU(g) * u -> fp16 Hg
//   gemm_kernel<2>  : W2_e Hg^T; epilogue Yr[route] = w_route * acc
//   combine         : y[t] = sum over slots j (in order) of Yr[t*k + j]
// The A operand is dequantized on chip: TMA brings each stage's packed tile
// (128 rows x 64 values = 32 bytes per row) and the activation tile into
// shared memory; eight dequantizing warps turn the nibbles into fp16
// w = (q - z) * s -- (q - z) exactly through the 0x6400 exponent trick, one
// rounding in the multiply -- written in the 128-byte-swizzled K-major layout
// the MMA reads; a proxy fence then hands the tile to the MMA warp.
//
// Roles (one CTA per SM, persistent over tiles): warp 0 TMA, warp 1 TMEM and
// MMA issue, warps 2..5 epilogue, warps 6..13 dequantization.  Every
// mbarrier wait is bounded; an expired wait records MOE_ERR_TIMEOUT in
// dev_status[1].
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "grouped_internal.h"
#include "tc.cuh"

namespace moe {
namespace ga {

constexpr int kMaxStages = 12;
constexpr int kDqWarps = 8;
constexpr int kThreads = (6 + kDqWarps) * 32;   // 448
constexpr uint32_t kTmemCols = 256;
constexpr int kHeaderBytes = 512;
constexpr int kMaxG = 64;                        // K <= 8192
constexpr uint64_t kWaitNs = 2000000000ull;

struct Args {
    const uint16_t *s;        // scales [E*N][K/128] fp16 bits
    const int32_t *z;         // zeros  [E][N/8][K/128]
    const int32_t *expert_ids;
    const int32_t *npp;
    const int32_t *sorted;
    const float *wts;
    __half *hg;               // kind 1: [cap_rows][I]
    float *yr;                // kind 2: [MK][d]
    int32_t *dev_status;
    int b, n_mma, n_mt, KT, I, d, MK, N, G, stages;
};

// Stage: A tile (fp16 [128][64], swizzled) | B tile (fp16 [n_mma][64],
// swizzled) | packed A [128][32 bytes]
struct Geo {
    int n_mma;
    __host__ __device__ int a_off() const { return 0; }
    __host__ __device__ int b_off() const { return 16384; }
    __host__ __device__ int raw_off() const { return 16384 + n_mma * 128; }
    __host__ __device__ int bytes() const { return (16384 + n_mma * 128 + 4096 + 1023) & ~1023; }
};

// row of expert e's weight matrix held by row m of an m-tile: kind 1 pairs
// 64 gate rows with the same 64 neurons' up rows
__device__ __forceinline__ int tile_row(int kind, int mt, int m, int I)
{
    return kind == 1 ? (m < 64 ? 64 * mt + m : I + 64 * mt + (m - 64)) : 128 * mt + m;
}

// Two 4-bit values (bits 0..3 and 4..7 of `byte`) minus zero, times scale,
// as an fp16 pair: 0x6400 | n is exactly 1024 + n in fp16.
__device__ __forceinline__ uint32_t dq_pair(uint32_t byte, __half2 zb, __half2 sc)
{
    const uint32_t v = 0x64006400u | (byte & 0xFu) | ((byte & 0xF0u) << 12);
    const __half2 q = *reinterpret_cast<const __half2 *>(&v);
    const __half2 r = __hmul2(__hsub2(q, zb), sc);
    return *reinterpret_cast<const uint32_t *>(&r);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmB, const Args a)
{
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t raw = tc::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const Geo geo{a.n_mma};
    const int S = a.stages, SB = geo.bytes();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * SB);
    const uint32_t rfull0 = tc::smem_u32(bars), afull0 = rfull0 + 8 * S, empty0 = afull0 + 8 * S;
    const uint32_t accf0 = empty0 + 8 * S, acce0 = accf0 + 16, fin = acce0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * S + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *ubuf = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(bars) + kHeaderBytes);   // [2][2][32][33]
    int *t_route = reinterpret_cast<int *>(ubuf + 4 * 32 * 33);                               // [256]
    float *t_w = reinterpret_cast<float *>(t_route + 256);                                    // [256]
    __half *sc_s = reinterpret_cast<__half *>(t_w + 256);                                     // [128][G]
    uint8_t *zs_s = reinterpret_cast<uint8_t *>(sc_s + 128 * a.G);                            // [128][G]
    const int nbuf = a.n_mma <= 128 ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(rfull0 + 8 * s, 1);
            tc::mbar_init(afull0 + 8 * s, kDqWarps);
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
        tc::prefetch_tmap(&tmQ);
        tc::prefetch_tmap(&tmB);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    const int n_blocks = *a.npp / a.b;
    const int total = n_blocks * a.n_mt;
    const int KT = a.KT;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0, issued = 0;
            uint32_t ph = 0;
            const uint32_t tx = 128u * 32u + static_cast<uint32_t>(a.n_mma) * 128u;
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x) {
                const int jb = t / a.n_mt, mt = t % a.n_mt;
                const int e = a.expert_ids[jb];
                const int row0 = e * a.N;
                for (int kt = 0; kt < KT; ++kt, ++issued) {
                    if (!tc::mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, kWaitNs))
                        break;
                    uint8_t *st = smem + s * SB;
                    const uint32_t fb = rfull0 + 8 * s;
                    tc::mbar_arrive_expect_tx(fb, tx);
                    // packed A rows: 32 bytes (64 values) of each, x in bytes
                    if (KIND == 1) {
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off()), &tmQ, kt * 32, row0 + 64 * mt, fb);
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off() + 64 * 32), &tmQ, kt * 32,
                                        row0 + a.I + 64 * mt, fb);
                    } else {
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off()), &tmQ, kt * 32, row0 + 128 * mt, fb);
                    }
                    // B tile: n_mma rows of 64 fp16, x in elements
                    tc::tma_load_2d(tc::smem_u32(st + geo.b_off()), &tmB, kt * 64, jb * a.b, fb);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            volatile int never = 0;
            const int n = issued < S ? issued : S;
            for (int i = 1; i <= n; ++i) {
                int st = s - i;
                uint32_t pp = ph;
                if (st < 0) {
                    st += S;
                    pp ^= 1u;
                }
                tc::mbar_wait(rfull0 + 8 * st, pp, &never, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, ti = 0;
            uint32_t ph = 0;
            const uint32_t idesc = tc::idesc_f16(128, a.n_mma, false);
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++ti) {
                const int buf = nbuf == 2 ? (ti & 1) : 0;
                const uint32_t use = static_cast<uint32_t>(nbuf == 2 ? (ti >> 1) : ti);
                if (!tc::mbar_wait(acce0 + 8 * buf, (use & 1u) ^ 1u, abort_flag, kWaitNs))
                    break;
                tc::tc_fence_after();
                const uint32_t acc = tmem + 128 * buf;
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(rfull0 + 8 * s, ph, abort_flag, kWaitNs) ||
                        !tc::mbar_wait(afull0 + 8 * s, ph, abort_flag, kWaitNs))
                        break;
                    tc::tc_fence_after();
                    const uint32_t sa = tc::smem_u32(smem + s * SB + geo.a_off());
                    const uint32_t sb = tc::smem_u32(smem + s * SB + geo.b_off());
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::smem_desc(sa + 32 * kk, 16, 1024, tc::kLayoutSw128);
                        const uint64_t bd = tc::smem_desc(sb + 32 * kk, 16, 1024, tc::kLayoutSw128);
                        tc::mma_f16(acc, ad, bd, idesc, (kt | kk) != 0 ? 1u : 0u);
                    }
                    tc::tc_commit(empty0 + 8 * s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                tc::tc_commit(accf0 + 8 * buf);
            }
            tc::tc_commit(fin);
            volatile int never = 0;
            tc::mbar_wait(fin, 0, &never, kWaitNs);
        }
    } else if (warp < 6) {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                       // TMEM lane quadrant
        const int etid = threadIdx.x - 64;
        int ti = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++ti) {
            const int jb = t / a.n_mt, mt = t % a.n_mt;
            const int buf = nbuf == 2 ? (ti & 1) : 0;
            const uint32_t use = static_cast<uint32_t>(nbuf == 2 ? (ti >> 1) : ti);
            const int rho0 = jb * a.b;
            if (KIND == 2) {
                for (int c = etid; c < a.b; c += 128) {
                    const int r = a.sorted[rho0 + c];
                    t_route[c] = r;
                    t_w[c] = r < a.MK ? a.wts[r] : 0.f;
                }
            }
            if (!tc::mbar_wait(accf0 + 8 * buf, use & 1u, abort_flag, kWaitNs) && a.dev_status)
                atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
            tc::tc_fence_after();
            tc::named_bar(1, 128);
            for (int c0 = 0, chunk = 0; c0 < a.b; c0 += 32, ++chunk) {
                uint32_t v[32];
                tc::tmem_ld_32x32b_x32(tmem + 128 * buf + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
                tc::tmem_ld_wait();
                const int ncol = min(32, a.b - c0);
                if (KIND == 1) {
                    // gate quadrant q pairs with up quadrant q ^ 2 (same 32
                    // neurons); each finishes half of the chunk's columns
                    const bool is_gate = q < 2;
                    float *ub = ubuf + ((chunk & 1) * 2 + (q & 1)) * 32 * 33 + lane * 33;
                    const int keep = is_gate ? 0 : 16;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        ub[16 - keep + c] = __uint_as_float(is_gate ? v[16 + c] : v[c]);
                    tc::named_bar(1, 128);
                    const int n = 64 * mt + 32 * (q & 1) + lane;
                    __half *hrow = a.hg + static_cast<int64_t>(rho0 + c0 + keep) * a.I + n;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float mine = __uint_as_float(is_gate ? v[c] : v[16 + c]);
                        const float other = ub[keep + c];
                        const float hv = is_gate ? silu_mul(mine, other) : silu_mul(other, mine);
                        if (keep + c < ncol)
                            hrow[static_cast<int64_t>(c) * a.I] = __float2half_rn(hv);
                    }
                } else {
                    const int o = 128 * mt + 32 * q + lane;
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
                    float *yo = a.yr + o;
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c < ncol && rr[c] < a.MK)
                            yo[static_cast<int64_t>(rr[c]) * a.d] = ww[c] * __uint_as_float(v[c]);
                }
            }
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            if (lane == 0)
                tc::mbar_arrive(acce0 + 8 * buf);
        }
    } else {
        // ------------------------------------------------ dequantization (warps 6..13)
        const int dt = threadIdx.x - 6 * 32;           // 0 .. 255
        const int m = dt >> 1, half = dt & 1;          // row of the tile, 32-value half of its 64
        int s = 0;
        uint32_t ph = 0;
        // every dequantizing thread walks all tiles (the named barriers below
        // need all of them); after a timeout the waits return at once
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            const int jb = t / a.n_mt, mt = t % a.n_mt;
            const int e = a.expert_ids[jb];
            // the tile's scales and zeros: row m's G groups
            tc::named_bar(2, kDqWarps * 32);           // previous tile's values no longer read
            {
                const int row = tile_row(KIND, mt, m, a.I);
                const int64_t gr = static_cast<int64_t>(e) * a.N + row;
                const int64_t zr = (static_cast<int64_t>(e) * (a.N / 8) + row / 8) * a.G;
                for (int g = half; g < a.G; g += 2) {
                    sc_s[m * a.G + g] = __ushort_as_half(a.s[gr * a.G + g]);
                    zs_s[m * a.G + g] = static_cast<uint8_t>((static_cast<uint32_t>(a.z[zr + g]) >> (4 * (row & 7))) & 0xFu);
                }
            }
            tc::named_bar(2, kDqWarps * 32);
            for (int kt = 0; kt < KT; ++kt) {
                if (!tc::mbar_wait(rfull0 + 8 * s, ph, abort_flag, kWaitNs) && a.dev_status)
                    atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
                uint8_t *st = smem + s * SB;
                const uint4 w = *reinterpret_cast<const uint4 *>(st + geo.raw_off() + m * 32 + half * 16);
                const int g = kt >> 1;                 // a 64-value k-tile lies in one group of 128
                const __half sv = sc_s[m * a.G + g];
                const __half zv = __float2half_rn(1024.0f + static_cast<float>(zs_s[m * a.G + g]));
                const __half2 sc2 = __halves2half2(sv, sv), zb2 = __halves2half2(zv, zv);
                const uint32_t ws_[4] = {w.x, w.y, w.z, w.w};
                uint8_t *arow = st + geo.a_off() + m * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // word c: values 8c .. 8c + 7 of this half -> 16-byte chunk 4 half + c
                    const uint32_t wd = ws_[c];
                    uint4 out;
                    out.x = dq_pair(wd & 0xFFu, zb2, sc2);
                    out.y = dq_pair((wd >> 8) & 0xFFu, zb2, sc2);
                    out.z = dq_pair((wd >> 16) & 0xFFu, zb2, sc2);
                    out.w = dq_pair(wd >> 24, zb2, sc2);
                    const int chunk = 4 * half + c;
                    *reinterpret_cast<uint4 *>(arow + ((chunk ^ (m & 7)) << 4)) = out;
                }
                // generic-proxy writes become visible to the tensor core
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(afull0 + 8 * s);
                if (++s == a.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// Xg[rho] = x[route / k] as fp16 (zero rows for padding); 8 values per thread
template <typename XT>
__global__ void gather_kernel(const XT *__restrict__ x, int d, int k, int MK, const int32_t *__restrict__ sorted,
                              const int32_t *__restrict__ npp, __half *__restrict__ xg)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int rows = *npp;
    const int d8 = d / 8;
    const int64_t total = static_cast<int64_t>(rows) * d8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int rho = static_cast<int>(i / d8), c = static_cast<int>(i - static_cast<int64_t>(rho) * d8);
        const int r = sorted[rho];
        uint4 out = make_uint4(0, 0, 0, 0);
        if (r < MK) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(r / k) * d) + c);
            if constexpr (sizeof(XT) == 2 && std::is_same<XT, __half>::value) {
                out = v;
            } else {
                const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 h = __floats2half2_rn(__uint_as_float(vv[j] << 16), __uint_as_float(vv[j] & 0xFFFF0000u));
                    o[j] = *reinterpret_cast<const uint32_t *>(&h);
                }
                out = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        reinterpret_cast<uint4 *>(xg + static_cast<int64_t>(rho) * d)[c] = out;
    }
}

struct WsLayout {
    size_t xg, hg, yr, total;
};

static WsLayout ws_layout(int M, int k, int d, int I, int cap_rows)
{
    WsLayout L;
    size_t off = 0;
    L.xg = off;
    off += ws_round(static_cast<size_t>(cap_rows) * d * 2);
    L.hg = off;
    off += ws_round(static_cast<size_t>(cap_rows) * I * 2);
    L.yr = off;
    off += ws_round(static_cast<size_t>(M) * k * d * sizeof(float));
    L.total = off;
    return L;
}

}  // namespace ga

size_t grouped_awq_workspace(int M, int k, int d, int I, int cap_rows)
{
    return ga::ws_layout(M, k, d, I, cap_rows).total;
}

moe_status_t grouped_awq_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                const int32_t *sorted, const int32_t *expert_ids, const int32_t *npp, int b,
                                int cap_rows, void *y, bool y_f32, void *ws, int32_t *dev_status, cudaStream_t s)
{
    using namespace ga;
    const int64_t mk = static_cast<int64_t>(M) * k;
    const int n_mma = (b + 15) / 16 * 16;
    const WsLayout L = ws_layout(M, k, d, I, cap_rows);
    uint8_t *w = static_cast<uint8_t *>(ws);
    __half *xg = reinterpret_cast<__half *>(w + L.xg);
    __half *hg = reinterpret_cast<__half *>(w + L.hg);
    float *yr = reinterpret_cast<float *>(w + L.yr);

    // tensor maps: packed weights as bytes [E*N][K/2]; activations fp16 [cap_rows][K]
    CUtensorMap tQ1, tB1, tQ2, tB2;
    if (!grouped_tmap_2d(&tQ1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w13->q, d / 2, static_cast<uint64_t>(E) * 2 * I, 32,
                         64, false) ||
        !grouped_tmap_2d(&tB1, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xg, d, cap_rows, 64, n_mma, true) ||
        !grouped_tmap_2d(&tQ2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w2->q, I / 2, static_cast<uint64_t>(E) * d, 32, 128,
                         false) ||
        !grouped_tmap_2d(&tB2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hg, I, cap_rows, 64, n_mma, true))
        return MOE_ERR_CUDA;

    const int gblocks = grouped_sm_count() * 4;
    const cudaError_t ge =
        x_bf16 ? launch_pdl(gather_kernel<__nv_bfloat16>, dim3(gblocks), dim3(256), 0, s,
                            static_cast<const __nv_bfloat16 *>(x), d, k, static_cast<int>(mk), sorted, npp, xg)
               : launch_pdl(gather_kernel<__half>, dim3(gblocks), dim3(256), 0, s, static_cast<const __half *>(x), d, k,
                            static_cast<int>(mk), sorted, npp, xg);
    if (ge != cudaSuccess)
        return MOE_ERR_CUDA;

    const int G1 = d / 128, G2 = I / 128, Gmax = G1 > G2 ? G1 : G2;
    if (Gmax > kMaxG)
        return MOE_ERR_UNSUPPORTED;
    const int stage_bytes = Geo{n_mma}.bytes();
    const size_t fixed = 1024 + kHeaderBytes + 4 * 32 * 33 * sizeof(float) + 512 * 4 + static_cast<size_t>(128) * Gmax * 3;
    int stages = static_cast<int>((227 * 1024 - fixed) / stage_bytes);
    stages = stages > kMaxStages ? kMaxStages : stages;
    const size_t smem = fixed + static_cast<size_t>(stages) * stage_bytes;
    static std::once_flag once;
    static bool attr_ok = false;
    std::call_once(once, [] {
        attr_ok = cudaFuncSetAttribute(gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) ==
                      cudaSuccess &&
                  cudaFuncSetAttribute(gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) ==
                      cudaSuccess;
    });
    if (!attr_ok || stages < 2 || smem > 227 * 1024)
        return MOE_ERR_CUDA;
    const int grid = grouped_sm_count();
    Args a1{static_cast<const uint16_t *>(w13->scale), static_cast<const int32_t *>(w13->zero), expert_ids, npp, sorted,
            wts, hg, nullptr, dev_status, b, n_mma, I / 64, d / 64, I, d, static_cast<int>(mk), 2 * I, G1, stages};
    if (launch_pdl(gemm_kernel<1>, dim3(grid), dim3(kThreads), smem, s, tQ1, tB1, a1) != cudaSuccess)
        return MOE_ERR_CUDA;
    Args a2{static_cast<const uint16_t *>(w2->scale), static_cast<const int32_t *>(w2->zero), expert_ids, npp, sorted,
            wts, nullptr, yr, dev_status, b, n_mma, d / 128, I / 64, I, d, static_cast<int>(mk), d, G2, stages};
    if (launch_pdl(gemm_kernel<2>, dim3(grid), dim3(kThreads), smem, s, tQ2, tB2, a2) != cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, ids, M, k, d, E, y, y_f32, s);
}

}  // namespace moe
