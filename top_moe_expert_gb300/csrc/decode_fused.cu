// decode_fused.cu -- single-pass streaming decode for small batches (M <= 4).
//
// Same mathematics as the two-kernel output-centric decode of "Warp decode"
// (cursor.com blog, sections on what changed and how the two kernels work):
// per routed expert g = W_gate x, u = W_up x, h = SiLU(g) * u, and
// y = sum_j w_j * W2_{e_j} h_j with the routing weight folded into the down
// accumulation, FP32 accumulation, MXFP8 weights converted on the fly, no
// alignment / padding / scatter / combine buffers.
//
// GB300 design.  The decode layer at M <= 4 is a pure HBM stream; the cost
// that remains after streaming is every dependency between kernels.  So the
// whole layer is one pass over the bytes:
//   * CTA c (one per SM) owns an exactly balanced range of neurons of the
//     distinct routed experts, and a producer warp streams, per stage of up
//     to 4 neurons, their gate rows, up rows (d bytes each) and -- from the
//     neuron-major packed W2 -- their down-projection columns (d bytes each)
//     with cp.async.bulk into a ring of shared-memory stages.
//   * Compute warps form h for those neurons (dot products, warp butterfly)
//     and immediately apply them to the down columns as outer products,
//     accumulating a per-CTA partial y in registers (deferred per 32-neuron
//     MX block, where the E8M0 scale row is applied once).  h never leaves
//     the SM.
//   * A small second kernel, launched with programmatic dependent launch,
//     sums the per-CTA partial outputs in CTA order (deterministic).
// Activations are carried as fp16 after an exact power-of-two per-token
// rescale, so the inner product uses the mixed-precision fma.rn.f32.f16
// (FP32 accumulate); the rescale is exact for every element within 2^28 of
// the token's largest magnitude (bf16 carries 8 significant bits).
#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "tc.cuh"

namespace moe {
namespace df {

constexpr int kDotWarps = 8;
constexpr int kOuterWarps = 8;
constexpr int kProducerWarp = kDotWarps + kOuterWarps;
constexpr int kThreads = (kProducerWarp + 1) * 32;
constexpr int kMaxStages = 4;
constexpr int kMaxM = 4;
constexpr int kMaxRoutes = 8;               // routes per expert handled per batch (res buffer)
constexpr uint64_t kWaitNs = 2000000000ull;

struct Args {
    const __nv_bfloat16 *x;
    const int32_t *ids;
    const float *wts;
    const uint8_t *q13, *s13;   // [E][2I][d], [E][2I][d/32]
    const uint8_t *q2t, *s2t;   // [E][I][d],  [E][I/32][d]  (neuron-major down projection)
    float *partial;             // [gridDim][M][d]
    int32_t *dev_status;
    int M, k, d, I, E;
    int R;                      // neurons per stage (<= 4)
    int stages;
};

// ---- plan: distinct experts ascending, routes of each ordered by route id
struct Plan {
    int *cnt, *dist, *rstart, *rlist, *n_dist, *n_invalid;
};

__device__ __forceinline__ Plan plan_carve(int *base, int E, int MK)
{
    Plan p;
    p.cnt = base;
    p.dist = base + E;
    p.rstart = p.dist + MK;
    p.rlist = p.rstart + MK + 1;
    p.n_dist = p.rlist + MK;
    p.n_invalid = p.n_dist + 1;
    return p;
}

__device__ void plan_build(const Plan &p, const int32_t *ids, int MK, int E)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int e = tid; e < E; e += nt)
        p.cnt[e] = 0;
    if (tid == 0)
        *p.n_invalid = 0;
    __syncthreads();
    int inval = 0;
    for (int r = tid; r < MK; r += nt) {
        const int e = __ldcg(ids + r);
        if (e >= 0 && e < E)
            atomicAdd(&p.cnt[e], 1);
        else
            ++inval;
    }
    if (inval)
        atomicAdd(p.n_invalid, inval);
    __syncthreads();
    if (tid < 32) {
        const int lane = tid;
        int run_off = 0, run_slot = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? p.cnt[e] : 0;
            const int f = c > 0;
            int ic = c, iff = f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, ic, o);
                const int b = __shfl_up_sync(0xffffffffu, iff, o);
                if (lane >= o) {
                    ic += a;
                    iff += b;
                }
            }
            const int off = run_off + ic - c, slot = run_slot + iff - f;
            if (f) {
                p.dist[slot] = e;
                p.rstart[slot] = off;
            }
            if (e < E)
                p.cnt[e] = off;
            run_off += __shfl_sync(0xffffffffu, ic, 31);
            run_slot += __shfl_sync(0xffffffffu, iff, 31);
        }
        if (lane == 0) {
            *p.n_dist = run_slot;
            p.rstart[run_slot] = run_off;
        }
        __syncwarp();
        for (int base = 0; base < MK; base += 32) {
            const int r = base + lane;
            const int e = r < MK ? __ldcg(ids + r) : -1;
            const bool ok = r < MK && e >= 0 && e < E;
            const unsigned key = ok ? static_cast<unsigned>(e) : 0xffffffffu;
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            const unsigned lt = (1u << lane) - 1u;
            int pos = 0;
            if (ok)
                pos = p.cnt[e] + __popc(peers & lt);
            __syncwarp();
            if (ok) {
                p.rlist[pos] = r;
                if ((peers & lt) == 0)
                    p.cnt[e] += __popc(peers);
            }
            __syncwarp();
        }
    }
    __syncthreads();
}


// One-warp routing plan for M*k <= 64 (the single-pass path's batches): one
// global round trip for the ids and weights, then shuffles, a 1024-bit expert
// mask and shared-memory counters.  Fills dist / rstart / rlist like
// plan_build, plus the token and routing weight of every rlist entry.
// Executed by all 32 lanes of one warp.
__device__ void plan_build_warp(const Plan &p, int *mask, int *scnt, int *rtok, float *rwt,
                                const int32_t *ids, const float *wts, int MK, int k, int E)
{
    const int lane = threadIdx.x & 31;
    int e[2];
    float w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h * 32 + lane;
        e[h] = r < MK ? __ldcg(ids + r) : -1;
        w[h] = r < MK ? __ldcg(wts + r) : 0.f;
    }
    mask[lane] = 0;
    scnt[lane] = 0;
    scnt[lane + 32] = 0;
    __syncwarp();
    int inval = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h * 32 + lane;
        if (r < MK) {
            if (e[h] >= 0 && e[h] < E)
                atomicOr(&mask[e[h] >> 5], 1 << (e[h] & 31));
            else
                ++inval;
        }
    }
    __syncwarp();
    // distinct experts ascending: slot = (#set bits in earlier words) + (#set bits below in the word)
    const int words = (E + 31) / 32;
    int pc = lane < words ? __popc(mask[lane]) : 0;
    int incl = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    const int n_dist = __shfl_sync(0xffffffffu, incl, 31);
    const int wordbase_lane = incl - pc;
    int slot[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        slot[h] = -1;
        const int r = h * 32 + lane;
        const bool ok = r < MK && e[h] >= 0 && e[h] < E;
        const int wi = ok ? (e[h] >> 5) : 0;
        const int wb = __shfl_sync(0xffffffffu, wordbase_lane, wi);
        if (ok) {
            slot[h] = wb + __popc(mask[wi] & ((1u << (e[h] & 31)) - 1u));
            p.dist[slot[h]] = e[h];
            atomicAdd(&scnt[slot[h]], 1);
        }
    }
    __syncwarp();
    // exclusive prefix of the per-slot counts (n_dist <= 64: two per lane)
    const int c0 = scnt[2 * lane], c1 = scnt[2 * lane + 1];
    int s2 = c0 + c1, inc2 = s2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc2, o);
        if (lane >= o)
            inc2 += t;
    }
    const int ex = inc2 - s2;
    __syncwarp();
    if (2 * lane < n_dist)
        p.rstart[2 * lane] = ex;
    if (2 * lane + 1 < n_dist)
        p.rstart[2 * lane + 1] = ex + c0;
    if (lane == 31)
        p.rstart[n_dist] = inc2;        // number of valid routes
    scnt[2 * lane] = ex;                // running positions
    scnt[2 * lane + 1] = ex + c0;
    __syncwarp();
    // stable placement, routes ascending within each expert
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = h * 32 + lane;
        const bool ok = slot[h] >= 0;
        const unsigned key = ok ? static_cast<unsigned>(slot[h]) : 0xffffffffu;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const unsigned lt = (1u << lane) - 1u;
        int pos = 0;
        if (ok)
            pos = scnt[slot[h]] + __popc(peers & lt);
        __syncwarp();
        if (ok) {
            p.rlist[pos] = r;
            rtok[pos] = r / k;
            rwt[pos] = w[h];
            if ((peers & lt) == 0)
                scnt[slot[h]] += __popc(peers);
        }
        __syncwarp();
    }
    inval = __reduce_add_sync(0xffffffffu, inval);
    if (lane == 0) {
        *p.n_dist = n_dist;
        *p.n_invalid = inval;
    }
    __syncwarp();
}

// ---- arithmetic helpers

__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two)));
    return r;
}

// d = a * b + c with a, b fp16 (exact in fp32) and c, d fp32: one rounding.
__device__ __forceinline__ float fma_h(__half a, __half b, float c)
{
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;"
        : "=f"(d) : "h"(__half_as_ushort(a)), "h"(__half_as_ushort(b)), "f"(c));
    return d;
}

// sum_{i<16} w_i * x_i for 16 E4M3 codes and 16 fp16 activations (as 8
// half2 words), FP32 accumulation in two chains.
__device__ __forceinline__ float dot16_h(uint4 q, uint4 xa, uint4 xb)
{
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
    const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = e4m3x2_f16x2(qw[i] & 0xFFFFu);
        const uint32_t hi = e4m3x2_f16x2(qw[i] >> 16);
        const __half2 wl = *reinterpret_cast<const __half2 *>(&lo);
        const __half2 wh = *reinterpret_cast<const __half2 *>(&hi);
        const __half2 xl = *reinterpret_cast<const __half2 *>(&xw[2 * i]);
        const __half2 xh = *reinterpret_cast<const __half2 *>(&xw[2 * i + 1]);
        a0 = fma_h(__low2half(wl), __low2half(xl), a0);
        a1 = fma_h(__high2half(wl), __high2half(xl), a1);
        a0 = fma_h(__low2half(wh), __low2half(xh), a0);
        a1 = fma_h(__high2half(wh), __high2half(xh), a1);
    }
    return a0 + a1;
}

__device__ __forceinline__ float e8m0f(uint32_t s)
{
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

__device__ __forceinline__ void drain_copies(uint32_t full0, int s, uint32_t ph, int issued, int nstages)
{
    volatile int never = 0;
    const int n = issued < nstages ? issued : nstages;
    for (int i = 1; i <= n; ++i) {
        int st = s - i;
        uint32_t pp = ph;
        if (st < 0) {
            st += nstages;
            pp ^= 1u;
        }
        tc::mbar_wait(full0 + 8 * st, pp, &never, kWaitNs);
    }
}

// ---- stage geometry (same arithmetic on host and device)
struct Geo {
    int d, R;
    __host__ __device__ int row() const { return d; }
    __host__ __device__ int gate_off() const { return 0; }
    __host__ __device__ int up_off() const { return R * d; }
    __host__ __device__ int w2_off() const { return 2 * R * d; }
    __host__ __device__ int gs_off() const { return 3 * R * d; }
    __host__ __device__ int us_off() const { return 3 * R * d + R * (d / 32); }
    __host__ __device__ int bytes() const { return 3 * R * d + 2 * R * (d / 32); }
};

// Range [p, p+nr) of the flattened (distinct expert, neuron) space that the
// next stage covers: at most R neurons, never across an expert or a
// 32-neuron MX block of the down projection.
__device__ __forceinline__ int stage_rows(int n, int left, int I, int R)
{
    int nr = R;
    const int to_blk = 32 - (n & 31);
    if (nr > to_blk)
        nr = to_blk;
    if (nr > I - n)
        nr = I - n;
    if (left < nr)
        nr = left;
    return nr;
}

// Warp roles: warps 0..7 ("dot" warps) form h for the stage's neurons,
// warps 8..15 ("outer" warps) apply it to the down-projection columns, warp
// 16 streams the weights.  The two compute groups hand the routing-weighted
// coefficients over through a double-buffered mbarrier pair, so the dot
// products of one stage overlap the outer products of the previous one.
// Template parameters: CPL = 16-byte chunks per lane of one warp's part of
// a weight row; NJ = 4-output chunks per outer thread (ceil(d / 1024));
// RB = routes accumulated in registers; XREG = one token whose activation
// slice the dot warps keep in registers.
template <int CPL, int NJ, int RB, bool XREG>
__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int MK = a.M * a.k, d = a.d, I = a.I, R = a.R;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Geo geo{d, R};

    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    // ---- shared memory carve-up
    uint8_t *stages = smem;
    uint8_t *s2row = stages + a.stages * geo.bytes();                       // [2][d] E8M0 rows
    __half *xh = reinterpret_cast<__half *>(s2row + 2 * d);                 // [M][d]
    float *acc = reinterpret_cast<float *>(xh + a.M * d);                   // [M][d]
    float *res = acc + a.M * d;                                             // [8][2][4][kMaxRoutes] partial dots
    float *coef = res + kDotWarps * 2 * 4 * kMaxRoutes;                     // [2][8][kMaxRoutes]
    float *xinv = coef + 2 * 8 * kMaxRoutes;                                // [4]
    // barriers: full[S], empty[S], scale full[2], scale empty[2], coef full[2], coef empty[2]
    uint64_t *bars = reinterpret_cast<uint64_t *>(xinv + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * kMaxStages + 8);
    int *plan_base = reinterpret_cast<int *>(bars + 2 * kMaxStages + 9);
    const Plan P = plan_carve(plan_base, a.E, MK);
    int *pmask = plan_base + a.E + 3 * MK + 4;                              // [32]
    int *pscnt = pmask + 32;                                                // [64]
    int *rtok = pscnt + 64;                                                 // [MK] token of rlist[i]
    float *rwt = reinterpret_cast<float *>(rtok + MK);                      // [MK] weight of rlist[i]
    const uint32_t full0 = tc::smem_u32(bars), empty0 = tc::smem_u32(bars + kMaxStages);
    const uint32_t sfull0 = tc::smem_u32(bars + 2 * kMaxStages);
    const uint32_t sempty0 = sfull0 + 16;
    const uint32_t cfull0 = sfull0 + 32;
    const uint32_t cempty0 = sfull0 + 48;

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, kDotWarps + kOuterWarps);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(sfull0 + 8 * b, 1);
            tc::mbar_init(sempty0 + 8 * b, kOuterWarps);
            tc::mbar_init(cfull0 + 8 * b, kDotWarps);
            tc::mbar_init(cempty0 + 8 * b, kOuterWarps);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    const int ND = kDotWarps * 32;
    if (warp == kProducerWarp) {
        // the producer warp builds the routing plan while the dot warps
        // convert the activations
        plan_build_warp(P, pmask, pscnt, rtok, rwt, a.ids, a.wts, MK, a.k, a.E);
    } else if (warp < kDotWarps) {
        // activations -> fp16 with an exact power-of-two per-token rescale
        for (int t = 0; t < a.M; ++t) {
            const __nv_bfloat16 *xt = a.x + static_cast<int64_t>(t) * d;
            uint32_t m = 0;
            for (int i = tid; i < d; i += ND)
                m = max(m, __float_as_uint(fabsf(__bfloat162float(xt[i]))));
            m = __reduce_max_sync(0xffffffffu, m);
            if (lane == 0)
                reinterpret_cast<uint32_t *>(res)[warp] = m;
            tc::named_bar(1, ND);
            uint32_t amax = 0;
            for (int w = 0; w < kDotWarps; ++w)
                amax = max(amax, reinterpret_cast<uint32_t *>(res)[w]);
            // scale 2^p with amax * 2^p in [2^14, 2^15)
            int pw = 0;
            if (amax != 0) {
                const int ef = static_cast<int>(amax >> 23);
                pw = ef == 0 ? 100 : 14 - (ef - 127);
                pw = pw < -100 ? -100 : (pw > 100 ? 100 : pw);
            }
            const float sc = ldexpf(1.0f, pw);
            for (int i = tid; i < d; i += ND)
                xh[t * d + i] = __float2half_rn(__bfloat162float(xt[i]) * sc);
            if (tid == 0)
                xinv[t] = ldexpf(1.0f, -pw);
            tc::named_bar(1, ND);
        }
    } else {
        // outer warps own the partial outputs: 4-output chunks tid_o + 256 j
        const int to = tid - ND;
        for (int t = 0; t < a.M; ++t)
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const int cj = to + kOuterWarps * 32 * j;
                if (cj < d / 4)
                    *reinterpret_cast<float4 *>(acc + t * d + cj * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
    }
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0 && *P.n_invalid && a.dev_status)
        atomicAdd(a.dev_status, *P.n_invalid);
    const int nd = *P.n_dist;
    const int Ptot = nd * I;
    const int p0 = static_cast<int>(static_cast<long long>(Ptot) * blockIdx.x / gridDim.x);
    const int p1 = static_cast<int>(static_cast<long long>(Ptot) * (blockIdx.x + 1) / gridDim.x);

    if (warp == kProducerWarp) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            int s = 0, issued = 0, nblk = 0;
            uint32_t ph = 0;
            int u = p0 / I, n = p0 % I;
            for (int p = p0; p < p1; ++issued) {
                const int nr = stage_rows(n, p1 - p, I, R);
                const int e = P.dist[u];
                if (p == p0 || (n & 31) == 0) {
                    // first stage of a 32-neuron block: its E8M0 row of the down
                    // projection goes to scale buffer (nblk & 1) once the outer
                    // warps released that buffer's previous block
                    const int buf = nblk & 1;
                    const uint32_t use = static_cast<uint32_t>(nblk >> 1);
                    if (!tc::mbar_wait(sempty0 + 8 * buf, (use & 1u) ^ 1u, abort_flag, kWaitNs))
                        break;
                    tc::mbar_arrive_expect_tx(sfull0 + 8 * buf, d);
                    tc::bulk_load(tc::smem_u32(s2row + buf * d),
                                  a.s2t + (static_cast<int64_t>(e) * (I / 32) + n / 32) * d, d, sfull0 + 8 * buf);
                    ++nblk;
                }
                if (!tc::mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, kWaitNs))
                    break;
                uint8_t *st = stages + s * geo.bytes();
                const uint32_t b = full0 + 8 * s;
                tc::mbar_arrive_expect_tx(b, nr * (3 * d + 2 * (d / 32)));
                const int64_t grow = static_cast<int64_t>(e) * 2 * I + n;
                tc::bulk_load(tc::smem_u32(st + geo.gate_off()), a.q13 + grow * d, nr * d, b);
                tc::bulk_load(tc::smem_u32(st + geo.up_off()), a.q13 + (grow + I) * d, nr * d, b);
                tc::bulk_load(tc::smem_u32(st + geo.w2_off()), a.q2t + (static_cast<int64_t>(e) * I + n) * d,
                              nr * d, b);
                tc::bulk_load(tc::smem_u32(st + geo.gs_off()), a.s13 + grow * (d / 32), nr * (d / 32), b);
                tc::bulk_load(tc::smem_u32(st + geo.us_off()), a.s13 + (grow + I) * (d / 32), nr * (d / 32), b);
                p += nr;
                n += nr;
                if (n == I) {
                    n = 0;
                    ++u;
                }
                if (++s == a.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            drain_copies(full0, s, ph, issued, a.stages);
            volatile int never = 0;
            for (int i = 1; i <= (nblk < 2 ? nblk : 2); ++i) {
                const int b = nblk - i;
                tc::mbar_wait(sfull0 + 8 * (b & 1), static_cast<uint32_t>((b >> 1) & 1), &never, kWaitNs);
            }
        }
        return;
    }

    if (warp < kDotWarps) {
        // ------------------------------------------------ dot warps
        // wpn warps per neuron: one warp does both rows (wpn == 1), else the
        // gate and up rows are split into wpn / 2 parts each
        const int wpn = kDotWarps / R;
        const int wpr = wpn > 1 ? wpn / 2 : 1;
        const int dnn = warp / wpn, sub = warp % wpn;
        const int drow0 = wpn > 1 ? sub / wpr : 0;          // first row: 0 gate, 1 up
        const int drow1 = wpn > 1 ? drow0 : 1;              // last row
        const int dpart = wpn > 1 ? sub % wpr : 0;
        uint32_t xr[XREG ? CPL * 8 : 1];
        if constexpr (XREG) {
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = (i * wpr + dpart) * 32 + lane;
                const bool in = c < d / 16;
                const uint4 xa = in ? *reinterpret_cast<const uint4 *>(xh + c * 16) : make_uint4(0, 0, 0, 0);
                const uint4 xb = in ? *reinterpret_cast<const uint4 *>(xh + c * 16 + 8) : make_uint4(0, 0, 0, 0);
                xr[i * 8 + 0] = xa.x; xr[i * 8 + 1] = xa.y; xr[i * 8 + 2] = xa.z; xr[i * 8 + 3] = xa.w;
                xr[i * 8 + 4] = xb.x; xr[i * 8 + 5] = xb.y; xr[i * 8 + 6] = xb.z; xr[i * 8 + 7] = xb.w;
            }
        }
        int s = 0, hix = 0;
        uint32_t ph = 0;
        int u = p0 / I, n = p0 % I;
        for (int p = p0; p < p1;) {
            const int nr = stage_rows(n, p1 - p, I, R);
            if (!tc::mbar_wait(full0 + 8 * s, ph, abort_flag, kWaitNs) && a.dev_status)
                atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
            const uint8_t *st = stages + s * geo.bytes();
            const int rs = P.rstart[u], re = P.rstart[u + 1];
            for (int r0 = rs; r0 < re; r0 += kMaxRoutes, ++hix) {
                const int nb = min(kMaxRoutes, re - r0);
                const int cb = hix & 1;
                if (dnn < nr) {
                    for (int row = drow0; row <= drow1; ++row) {
                        const uint8_t *wrow = st + (row == 0 ? geo.gate_off() : geo.up_off()) + dnn * d;
                        const uint8_t *srow = st + (row == 0 ? geo.gs_off() : geo.us_off()) + dnn * (d / 32);
                        uint4 qv[CPL];
                        float sv[CPL];
#pragma unroll
                        for (int i = 0; i < CPL; ++i) {
                            const int c = (i * wpr + dpart) * 32 + lane;
                            const bool in = c < d / 16;
                            qv[i] = in ? *reinterpret_cast<const uint4 *>(wrow + c * 16) : make_uint4(0, 0, 0, 0);
                            sv[i] = in ? e8m0f(srow[c >> 1]) : 0.f;
                        }
                        for (int ri = 0; ri < nb; ++ri) {
                            const int t = rtok[r0 + ri];
                            float part[CPL];
#pragma unroll
                            for (int i = 0; i < CPL; ++i) {
                                uint4 xa, xb;
                                if constexpr (XREG) {
                                    xa = make_uint4(xr[i * 8 + 0], xr[i * 8 + 1], xr[i * 8 + 2], xr[i * 8 + 3]);
                                    xb = make_uint4(xr[i * 8 + 4], xr[i * 8 + 5], xr[i * 8 + 6], xr[i * 8 + 7]);
                                } else {
                                    const int c = (i * wpr + dpart) * 32 + lane;
                                    const __half *xt = xh + t * d;
                                    const bool in = c < d / 16;
                                    xa = in ? *reinterpret_cast<const uint4 *>(xt + c * 16) : make_uint4(0, 0, 0, 0);
                                    xb = in ? *reinterpret_cast<const uint4 *>(xt + c * 16 + 8) : make_uint4(0, 0, 0, 0);
                                }
                                part[i] = dot16_h(qv[i], xa, xb) * sv[i];
                            }
                            float dacc = 0.f;
#pragma unroll
                            for (int i = 0; i < CPL; ++i)
                                dacc += part[i];
                            dacc = warp_sum(dacc);
                            if (lane == 0)
                                res[((dnn * 2 + row) * 4 + dpart) * kMaxRoutes + ri] = dacc;
                        }
                    }
                }
                // partial dots of split rows meet in shared memory
                if (wpn > 1)
                    tc::named_bar(2 + dnn, 32 * wpn);
                else
                    __syncwarp();
                // the coefficient buffer of two handovers ago must be free
                if (!tc::mbar_wait(cempty0 + 8 * cb, static_cast<uint32_t>(((hix >> 1) & 1) ^ 1), abort_flag,
                                   kWaitNs) && a.dev_status)
                    atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
                if (sub == 0 && lane < nb && dnn < nr) {
                    const int ri = lane;
                    float g = 0.f, uu = 0.f;
                    for (int q = 0; q < wpr; ++q) {              // parts in fixed order
                        g += res[((dnn * 2 + 0) * 4 + q) * kMaxRoutes + ri];
                        uu += res[((dnn * 2 + 1) * 4 + q) * kMaxRoutes + ri];
                    }
                    const float xi = xinv[rtok[r0 + ri]];
                    coef[(cb * 8 + dnn) * kMaxRoutes + ri] = rwt[r0 + ri] * silu_mul(g * xi, uu * xi);
                }
                if (wpn > 1)
                    tc::named_bar(2 + dnn, 32 * wpn);        // res reuse
                else
                    __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(cfull0 + 8 * cb);
            }
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(empty0 + 8 * s);
            p += nr;
            n += nr;
            if (n == I) {
                n = 0;
                ++u;
            }
            if (++s == a.stages) {
                s = 0;
                ph ^= 1u;
            }
        }
        return;
    }

    // ------------------------------------------------ outer warps
    const int to = tid - ND;
    const int NO = kOuterWarps * 32;
    float2 ablk[RB][NJ][2];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            ablk[r][j][0] = ablk[r][j][1] = make_float2(0.f, 0.f);
    int s = 0, nblk = -1, hix = 0;
    uint32_t ph = 0;
    bool blk_scale_ready = false;
    int u = p0 / I, n = p0 % I;
    for (int p = p0; p < p1;) {
        const int nr = stage_rows(n, p1 - p, I, R);
        const bool blk_start = (p == p0) || ((n & 31) == 0);
        const bool blk_end = ((n + nr) & 31) == 0 || p + nr == p1;
        if (blk_start) {
            ++nblk;
            blk_scale_ready = false;
        }
        const int blk_parity = nblk & 1;
        if (!tc::mbar_wait(full0 + 8 * s, ph, abort_flag, kWaitNs) && a.dev_status)
            atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
        const uint8_t *w2 = stages + s * geo.bytes() + geo.w2_off();
        const int rs = P.rstart[u], re = P.rstart[u + 1];
        const bool many = re - rs > RB;       // flush after every route group
        for (int r0 = rs; r0 < re; r0 += kMaxRoutes, ++hix) {
            const int nb = min(kMaxRoutes, re - r0);
            const int cb = hix & 1;
            if (!tc::mbar_wait(cfull0 + 8 * cb, static_cast<uint32_t>((hix >> 1) & 1), abort_flag, kWaitNs) &&
                a.dev_status)
                atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
            const float *cf = coef + cb * 8 * kMaxRoutes;
            for (int g0 = 0; g0 < nb; g0 += RB) {
                // outer products of this route group with the stage's columns
                for (int nn = 0; nn < nr; ++nn) {
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const int cj = to + NO * j;
                        if (NJ * NO * 4 == d || cj < d / 4) {
                            const uint32_t q4 = *reinterpret_cast<const uint32_t *>(w2 + nn * d + cj * 4);
                            const uint32_t lp = e4m3x2_f16x2(q4 & 0xFFFFu);
                            const uint32_t hp = e4m3x2_f16x2(q4 >> 16);
                            const float2 w01 = __half22float2(*reinterpret_cast<const __half2 *>(&lp));
                            const float2 w23 = __half22float2(*reinterpret_cast<const __half2 *>(&hp));
#pragma unroll
                            for (int ri = 0; ri < RB; ++ri) {
                                if (g0 + ri < nb) {
                                    const float c = cf[nn * kMaxRoutes + g0 + ri];
                                    const float2 cc = make_float2(c, c);
                                    ablk[ri][j][0] = __ffma2_rn(w01, cc, ablk[ri][j][0]);
                                    ablk[ri][j][1] = __ffma2_rn(w23, cc, ablk[ri][j][1]);
                                }
                            }
                        }
                    }
                }
                // flush into the per-token partial with the block's E8M0 row
                if (blk_end || many) {
                    if (!blk_scale_ready) {
                        if (!tc::mbar_wait(sfull0 + 8 * blk_parity, static_cast<uint32_t>((nblk >> 1) & 1),
                                           abort_flag, kWaitNs) && a.dev_status)
                            atomicCAS(a.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
                        blk_scale_ready = true;
                    }
                    const uint8_t *srw = s2row + blk_parity * d;
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const int cj = to + NO * j;
                        if (NJ * NO * 4 == d || cj < d / 4) {
                            const uint32_t s4 = *reinterpret_cast<const uint32_t *>(srw + cj * 4);
#pragma unroll
                            for (int ri = 0; ri < RB; ++ri) {
                                if (g0 + ri < nb) {
                                    const int t = rtok[r0 + g0 + ri];
                                    float4 *ap = reinterpret_cast<float4 *>(acc + t * d + cj * 4);
                                    float4 v = *ap;
                                    v.x = fmaf(e8m0f(s4 & 0xFFu), ablk[ri][j][0].x, v.x);
                                    v.y = fmaf(e8m0f((s4 >> 8) & 0xFFu), ablk[ri][j][0].y, v.y);
                                    v.z = fmaf(e8m0f((s4 >> 16) & 0xFFu), ablk[ri][j][1].x, v.z);
                                    v.w = fmaf(e8m0f(s4 >> 24), ablk[ri][j][1].y, v.w);
                                    *ap = v;
                                    ablk[ri][j][0] = ablk[ri][j][1] = make_float2(0.f, 0.f);
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(cempty0 + 8 * cb);
        }
        __syncwarp();
        if (lane == 0) {
            tc::mbar_arrive(empty0 + 8 * s);
            if (blk_end)                         // the block's scale row is no longer needed
                tc::mbar_arrive(sempty0 + 8 * blk_parity);
        }
        p += nr;
        n += nr;
        if (n == I) {
            n = 0;
            ++u;
        }
        if (++s == a.stages) {
            s = 0;
            ph ^= 1u;
        }
    }
    // each outer thread writes the outputs it owns
    float *out = a.partial + static_cast<int64_t>(blockIdx.x) * a.M * d;
    for (int t = 0; t < a.M; ++t)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int cj = to + NO * j;
            if (cj < d / 4)
                __stcg(reinterpret_cast<float4 *>(out + t * d + cj * 4),
                       *reinterpret_cast<const float4 *>(acc + t * d + cj * 4));
        }
}

// y[t][o] = sum over CTAs c (ascending) of partial[c][t][o].  A CTA covers
// 32 consecutive outputs; warp w adds CTAs [G*w/8, G*(w+1)/8) with four
// independent accumulators, then warp 0 adds the eight group sums in order.
template <typename YT>
__global__ void __launch_bounds__(256) reduce_kernel(const float *__restrict__ partial, int G, int n, YT *y)
{
    __shared__ float gs[8][33];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int o = blockIdx.x * 32 + lane;
    const int c0 = G * w / 8, c1 = G * (w + 1) / 8;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    if (o < n) {
        int c = c0;
        for (; c + 4 <= c1; c += 4) {
            a0 += __ldcg(partial + static_cast<int64_t>(c) * n + o);
            a1 += __ldcg(partial + static_cast<int64_t>(c + 1) * n + o);
            a2 += __ldcg(partial + static_cast<int64_t>(c + 2) * n + o);
            a3 += __ldcg(partial + static_cast<int64_t>(c + 3) * n + o);
        }
        for (; c < c1; ++c)
            a0 += __ldcg(partial + static_cast<int64_t>(c) * n + o);
    }
    gs[w][lane] = (a0 + a1) + (a2 + a3);
    __syncthreads();
    if (w == 0 && o < n) {
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            sum += gs[i][lane];
        if constexpr (sizeof(YT) == 4)
            y[o] = sum;
        else
            y[o] = __float2bfloat16_rn(sum);
    }
}

}  // namespace df

// ---------------------------------------------------------------- host side

size_t decode_fused_workspace(int M, int d)
{
    return ws_round(static_cast<size_t>(device_sm_count()) * M * d * sizeof(float));
}

bool decode_fused_eligible(int M, int k, int d, int I, int E)
{
    return M >= 1 && M <= df::kMaxM && M * k <= 64 && E <= 1024 && d % 1024 == 0 && d <= 8192 && I % 32 == 0;
}

moe_status_t decode_fused_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                 const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                 const uint8_t *q2t, const uint8_t *s2t, void *y, bool y_f32, float *partial,
                                 int32_t *dev_status, cudaStream_t stream)
{
    using namespace df;
    const int G = device_sm_count();
    const int MK = M * k;
    // neurons per stage: as many as keep three stages within ~150 KB (at most
    // one per dot warp); wpn = 8 / R dot warps per neuron split its rows
    int R = 8;
    size_t stage = static_cast<size_t>(Geo{d, R}.bytes());
    while (R > 1 && 3 * stage > 150 * 1024) {
        R /= 2;
        stage = static_cast<size_t>(Geo{d, R}.bytes());
    }
    const int wpn = kDotWarps / R;
    const int wpr = wpn > 1 ? wpn / 2 : 1;
    const int CPL = (d / 16 + 32 * wpr - 1) / (32 * wpr);
    int stages = static_cast<int>((150 * 1024) / stage);
    stages = stages < 2 ? 2 : (stages > kMaxStages ? kMaxStages : stages);
    const size_t smem = stages * stage + 2 * d + static_cast<size_t>(M) * d * 2 + static_cast<size_t>(M) * d * 4 +
                        (kDotWarps * 2 * 4 * kMaxRoutes + 2 * 8 * kMaxRoutes + 4) * sizeof(float) +
                        (2 * kMaxStages + 9) * sizeof(uint64_t) + (static_cast<size_t>(E) + 3 * MK + 4 + 96 + 2 * MK) * sizeof(int);
    if (smem > 220 * 1024)
        return MOE_ERR_UNSUPPORTED;
    Args a{x, ids, wts, q13, s13, q2t, s2t, partial, dev_status, M, k, d, I, E, R, stages};
    auto pick = [&](auto kern) -> moe_status_t {
        if (!smem_attr(reinterpret_cast<const void *>(kern), 220 * 1024))
            return MOE_ERR_CUDA;
        return launch_pdl(kern, dim3(G), dim3(kThreads), smem, stream, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };
    const int NJ = (d + 1023) / 1024;
    moe_status_t st = MOE_ERR_UNSUPPORTED;
    if (M == 1) {
        if (CPL == 4 && NJ == 2) st = pick(fused_kernel<4, 2, 1, true>);          // d = 2048
        else if (CPL == 2 && NJ == 1) st = pick(fused_kernel<2, 1, 1, true>);     // d = 1024
        else if (CPL == 7 && NJ == 7) st = pick(fused_kernel<7, 7, 1, false>);    // d = 7168
        else return MOE_ERR_UNSUPPORTED;
    } else {
        if (CPL == 4 && NJ == 2) st = pick(fused_kernel<4, 2, 4, false>);
        else if (CPL == 2 && NJ == 1) st = pick(fused_kernel<2, 1, 4, false>);
        else return MOE_ERR_UNSUPPORTED;
    }
    if (st != MOE_OK)
        return st;
    const int n = M * d;
    const int blocks = (n + 31) / 32;
    cudaError_t e = y_f32 ? launch_pdl(reduce_kernel<float>, dim3(blocks), dim3(256), 0, stream,
                                       static_cast<const float *>(partial), G, n, static_cast<float *>(y))
                          : launch_pdl(reduce_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, stream,
                                       static_cast<const float *>(partial), G, n, static_cast<__nv_bfloat16 *>(y));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
