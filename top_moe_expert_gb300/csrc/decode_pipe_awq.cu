// decode_pipe_awq.cu -- single-token decode of the routed expert layer on
// 4-bit AWQ weights (group 128) as one kernel, optionally with the top-k
// routing inside.
//
// The method is the output-centric decode of "Warp decode" (cursor.com
// blog, sections on what changed and on how the two kernels work), on the
// packed-AWQ weights of "Route-Block Membership Selects Packed-AWQ
// Arithmetic" (AWQ g128): w = (q - z) * s.  The structure is the MXFP8
// single-token kernel's (one CTA per SM; warp 0 streams this CTA's gate/up
// rows and then its down rows through one ring of bulk copies; four groups
// of four warps form h = SiLU(g) * u and publish it as (value, launch tag)
// words; every CTA reads all of h back once the words carry the launch's
// tag and forms its d / G output rows of every route's down projection).
//
// Dequantization, exact: a word holds 8 nibbles, element 8c + i in bits
// 4i..4i+3; (word >> 4j) & 0x000F000F | 0x64006400 is the fp16 pair
// (1024 + n_j, 1024 + n_{j+4}), and subtracting the fp16 pair (1024 + z) gives
// (q - z) in [-15, 15] exactly.  Those multiply the activations (fp16 after an
// exact power-of-two rescale, in the same pair order) with fp16 x fp16 -> FP32
// FMAs, exact products; each lane's partial covers one group of 128 (8
// elements per word, 128 % 8 == 0) and is multiplied by that group's fp16
// scale s in FP32.  h is exchanged in FP32 and taken by the down projection
// as fp16 after an exact per-lane power-of-two rescale.
//
// The launch tag and the exchange words use the same reserved start of the
// decode workspace as the MXFP8 single-token kernel (one count of CTAs over
// every launch of either), so one workspace serves both.  Every output's
// summation order depends only on the shapes and the grid.
#include <atomic>
#include <type_traits>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "pipe_common.cuh"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {
namespace dpa {

constexpr int kMaxK = 32;
constexpr int kGW = 4;                                // warps of a gate/up group (they split K)
constexpr int kGroups = 4;                            // gate/up groups
constexpr int kPS = 8;                                // neurons per gate/up stage
constexpr int kMaxSlots = 11;                         // ring slots, at most
constexpr int kMinSlots = 4;
constexpr int kTW = 8;                                // warps of the scale-staging role
constexpr int kWarpGU0 = 2;
constexpr int kWarpT0 = kWarpGU0 + kGW * kGroups;     // 18
constexpr int kWarps = kWarpT0 + kTW;                 // 26
constexpr int kThreads = kWarps * 32;                 // 832
constexpr int kCW = kWarps - kWarpGU0;                // compute warps of the exchange and tail: 24
constexpr int kMaxPerLane = 32;                       // exchange words per lane, at most
constexpr uint64_t kWaitNs = 2000000000ull;           // 2 s
constexpr int kBarRoutes = 1;                         // named barriers: routes published (all warps but 1)
constexpr int kBarTail = 2;                           //   the compute warps
constexpr int kBarGroup0 = 3;                         //   gate/up group g: kBarGroup0 + g
constexpr int kBarRank = kBarGroup0 + kGroups;        //   the compute warps ranking the logits
constexpr int kBarScales = kBarRank + 1;              //   gate/up scales and zeros staged, launch tag formed
                                                      //   (staging warps and warp 1 arrive)
constexpr int kSmemMax = 227 * 1024;
constexpr int kMaxG2 = 8;                             // groups of a down row (I / 128), at most

struct Args {
    const void *x;               // [d] fp16 or bf16
    const int32_t *ids;          // given routing: ids / weights [k]
    const float *wts;
    const float *logits;         // or routed here: router logits [E] ...
    int32_t *ids_out;            // ... and the chosen ids / weights written by CTA 0
    float *wts_out;
    const uint8_t *q13;          // packed codes [E][2I][d/8] int32 words
    const uint16_t *s13;         // fp16 scales [E][2I][d/128]
    const uint32_t *z13;         // packed zeros [E][2I/8][d/128]
    const uint8_t *q2;           // [E][d][I/8] words
    const uint16_t *s2;          // [E][d][I/128]
    const uint32_t *z2;          // [E][d/8][I/128]
    unsigned long long *ctr;     // CTA count over all launches
    unsigned long long *xh;      // exchange words [k][I]: value bits | tag << 32
    void *y;
    int32_t *dev_status;
    int y_f32, k, d, I, E;
    int stall;                   // readers expect a tag nobody writes (failure-detection test)
};

// Shared-memory plan (bytes), identical on host and device.  A ring slot is
// kPS gate rows then kPS up rows of packed codes (d / 2 bytes a row); the
// down rows of every route reuse the ring after the gate/up stages.
struct Plan {
    int d, I, k, G;
    __host__ __device__ int rows_max() const { return (d + G - 1) / G; }
    __host__ __device__ int s1() const { return kPS * 2 * (d / 2); }            // slot: gate rows | up rows
    __host__ __device__ int pmax() const { return (k * I + G - 1) / G; }        // pairs of a CTA, at most
    __host__ __device__ int s2() const { return rows_max() * (I / 2); }         // one route's down rows
    __host__ __device__ int rps() const { return s1() / s2(); }                 // routes per down stage
    __host__ __device__ int w2_stages() const { return (k + rps() - 1) / rps(); }
    __host__ __device__ static int up16(int v) { return (v + 15) & ~15; }
    // everything but the ring: h, down scale|zero words, gate/up scale|zero
    // words, partials, barriers, the route table
    __host__ __device__ int fixed() const
    {
        return up16(k * I * 4) + up16(k * rows_max() * (I / 128) * 4) + up16(pmax() * 2 * (d / 128) * 4) +
               kGroups * 2 * kGW * 2 * kPS * 4 + up16(k * rows_max() * 4) + 2 * kMaxSlots * 8 + 3 * kMaxK * 4 + 32;
    }
    __host__ __device__ int slots() const
    {
        const int n = (kSmemMax - fixed()) / s1();
        return n > kMaxSlots ? kMaxSlots : n;
    }
    __host__ __device__ int o_h() const { return slots() * s1(); }             // h [k][I] f32
    __host__ __device__ int o_s2z() const { return o_h() + up16(k * I * 4); }
    __host__ __device__ int o_gsz() const { return o_s2z() + up16(k * rows_max() * (I / 128) * 4); }
    __host__ __device__ int o_gpart() const { return o_gsz() + up16(pmax() * 2 * (d / 128) * 4); }
    __host__ __device__ int o_dpart() const { return o_gpart() + kGroups * 2 * kGW * 2 * kPS * 4; }
    __host__ __device__ int o_bars() const { return o_dpart() + up16(k * rows_max() * 4); }
    __host__ __device__ int o_route() const { return o_bars() + 2 * kMaxSlots * 8; }
    // route data: r_e[kMaxK] | r_w[kMaxK] | r_l[kMaxK] | tag, nv, abort, tabort (32 bytes kept)
    __host__ __device__ int bytes() const { return o_route() + 3 * kMaxK * 4 + 32; }
    __host__ __device__ bool fits() const
    {
        // every CTA's gate/up stages within the ring's first lap: a group then
        // never waits (by barrier parity) on a slot that another group's
        // stage, possibly not landed yet, held one lap earlier
        return s2() > 0 && s2() <= s1() && slots() >= kMinSlots && w2_stages() <= slots() &&
               (pmax() + kPS - 1) / kPS <= slots() && bytes() <= kSmemMax &&
               static_cast<size_t>(k) * I * 8 <= kWsTagBytes && k * I <= kCW * 32 * kMaxPerLane &&
               I / 128 <= kMaxG2 && (I / 128) % 2 == 0;
    }
};

using namespace pipe;

// The (q - z) pairs of one packed word, exact, as fp16x2: o[j] holds
// (n_j - z, n_{j+4} - z); zz2 is the fp16 pair (1024 + z, 1024 + z).
__device__ __forceinline__ void awq_pairs(uint32_t w, uint32_t zz2, uint32_t (&o)[4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t p = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;     // (1024 + n_j, 1024 + n_{j+4})
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(p), "r"(zz2));
    }
}

// a staged (scale, zero) word: fp16 scale bits | (0x6400 | z) << 16
__device__ __forceinline__ uint32_t sz_word(uint16_t s, uint32_t z) { return s | ((0x6400u | z) << 16); }

__device__ __forceinline__ float sz_scale(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t sz_zz2(uint32_t w) { return (w >> 16) | (w & 0xFFFF0000u); }

template <bool XBF>
__device__ __forceinline__ float x_at(const void *x, int i)
{
    if constexpr (XBF)
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(x)[i]);
    else
        return __half2float(static_cast<const __half *>(x)[i]);
}

// KPL: gate/up elements per lane of a warp's K slice (d = 32 * kGW * KPL,
// KPL % 8 == 0); HPL: down elements per lane (I = 32 * HPL, HPL % 8 == 0);
// ROUTE: the kernel routes the token itself; XBF: x is bf16 (else fp16).
template <int KPL, int HPL, bool ROUTE, bool XBF>
__global__ void __launch_bounds__(kThreads, 1) pipe_kernel(const Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int d = a.d, I = a.I, k = a.k, G = gridDim.x, c = blockIdx.x;
    const Plan pl{d, I, k, G};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int RM = pl.rows_max(), S1 = pl.s1(), S2 = pl.s2(), NS = pl.slots(), RPS = pl.rps();
    const int G13 = d / 128, G2 = I / 128;                               // groups of a gate/up, a down row
    uint8_t *ring = smem;
    float *hbuf = reinterpret_cast<float *>(smem + pl.o_h());           // [nv][I] h of every route
    uint32_t *s2z = reinterpret_cast<uint32_t *>(smem + pl.o_s2z());     // [k][RM][G2] down scale|zero
    uint32_t *gsz = reinterpret_cast<uint32_t *>(smem + pl.o_gsz());     // [P][2][G13] gate/up scale|zero
    float *gpart = reinterpret_cast<float *>(smem + pl.o_gpart());       // [grp][2][kGW][2 kPS]
    float *dpart = reinterpret_cast<float *>(smem + pl.o_dpart());       // [k][RM]
    const uint32_t full = tc::smem_u32(smem + pl.o_bars());
    const uint32_t empty = full + 8 * kMaxSlots;
    int *r_e = reinterpret_cast<int *>(smem + pl.o_route());
    float *r_w = reinterpret_cast<float *>(r_e + kMaxK);
    float *r_l = r_w + kMaxK;                                            // logits of the chosen routes
    uint32_t *s_tag = reinterpret_cast<uint32_t *>(r_l + kMaxK);
    int *s_nv = reinterpret_cast<int *>(s_tag + 1);
    volatile int *s_abort = s_nv + 1;
    volatile int *tabort = s_nv + 2;                                     // decided before the first tail barrier

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---------------------------------------------------------------- set-up
    // This CTA's split is formed before the routes barrier wherever the
    // number of valid routes is known there (routing here: all k are valid;
    // given routes: warp 0 counts them), so the producer can stream as soon
    // as the routes are out.
    pipe::Split sp{};
    if (warp == 0) {
        if constexpr (ROUTE)
            sp = pipe::cta_split<kPS>(k, I, d, c, G, RPS);
        if (lane == 0) {
            for (int i = 0; i < NS; ++i) {
                tc::mbar_init(full + 8 * i, 1);
                tc::mbar_init(empty + 8 * i, kGW);
            }
            *s_abort = 0;
            *tabort = 0;
            if constexpr (ROUTE)
                *s_nv = k;                                         // E >= k: every chosen route is valid
            tc::fence_mbar_init();
        }
        if constexpr (!ROUTE) {
            const int e = lane < k ? __ldcg(a.ids + lane) : -1;
            const float w = lane < k ? __ldcg(a.wts + lane) : 0.f;
            // the valid routes (0 <= id < E), compacted in slot order
            const bool ok = lane < k && e >= 0 && e < a.E;
            const unsigned vm = __ballot_sync(0xffffffffu, ok);
            const int vi = __popc(vm & ((1u << lane) - 1u));
            if (ok) {
                r_e[vi] = e;
                r_w[vi] = w;
            }
            sp = pipe::cta_split<kPS>(__popc(vm), I, d, c, G, RPS);
            if (lane == 0) {
                *s_nv = __popc(vm);
                if (c == 0 && k > __popc(vm) && a.dev_status)
                    atomicAdd(a.dev_status, k - __popc(vm));
            }
        }
    } else if (warp == 1) {
        // this launch's tag, from the count read before this CTA adds its
        // one; the gate/up warps read it after the staging barrier (it is not
        // needed before, so this warp stays off the routes barrier)
        if (lane == 0) {
            const unsigned long long v = ld_relaxed_u64(a.ctr);
            *s_tag = static_cast<uint32_t>(v / static_cast<unsigned>(G)) + 1u;
            red_relaxed_add(a.ctr);
        }
        __syncwarp();
        tc::named_arrive(kBarScales, kCW * 32 + 32);
        return;
    } else if constexpr (ROUTE) {
        // top-k of the router logits by rank: thread e (of the 24 compute
        // warps) holds expert e's order-preserving key; its slot is the
        // number of experts ahead of it -- larger logit, or equal logit and
        // lower id -- which is the order the top-k routing defines.  The
        // keys sit in the ring, idle until the routes are out.
        uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
        const int e = tid - kWarpGU0 * 32, Ep = (a.E + 3) & ~3;
        float l = 0.f;
        if (e < a.E)
            l = __ldcg(a.logits + e);
        sp = pipe::cta_split<kPS>(k, I, d, c, G, RPS);
        if (e < Ep)
            keys[e] = e < a.E ? topk_key(l) : 0u;
        tc::named_bar(kBarRank, kCW * 32);
        if (e < a.E) {
            const uint32_t me = keys[e];
            int rank = 0;
            const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
            for (int j = 0; j < Ep; j += 4) {
                const uint4 v = k4[j >> 2];
                rank += (v.x > me || (v.x == me && j < e)) + (v.y > me || (v.y == me && j + 1 < e)) +
                        (v.z > me || (v.z == me && j + 2 < e)) + (v.w > me || (v.w == me && j + 3 < e));
            }
            if (rank < k) {
                r_e[rank] = e;
                r_l[rank] = l;
            }
        }
    }
    tc::named_bar(kBarRoutes, kThreads - 32);

    const int nv = *s_nv;
    if constexpr (!ROUTE) {
        if (warp != 0)
            sp = pipe::cta_split<kPS>(nv, I, d, c, G, RPS);
    }
    // this CTA's (route, neuron) pairs: a contiguous range of q = r * I + n,
    // the whole space split evenly over the CTAs (h[q] is formed here)
    const int q_lo = sp.q_lo, P = sp.P, S = sp.S;                     // S gate/up stages
    const int o0 = sp.o0, nrows = sp.nrows, SW = sp.SW;               // SW down stages

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            const int64_t rowb = d / 2, row2 = I / 2;      // bytes of a gate/up row, of a down row
            tc::fence_proxy_async_smem();                  // the ring held the routing's keys
            int t = 0;
            for (; t < S + SW; ++t) {
                const int sl = t % NS;
                const uint32_t ph = (t / NS) & 1u;
                if (!tc::mbar_wait(empty + 8 * sl, ph ^ 1u, s_abort, kWaitNs))
                    break;
                uint8_t *st = ring + sl * S1;
                const uint32_t bar = full + 8 * sl;
                if (t < S) {
                    // gate/up stage t: runs of neurons of one route, gate rows then up rows
                    const int q0 = q_lo + t * kPS, q1 = q_lo + min(t * kPS + kPS, P);
                    tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(q1 - q0) * (2 * rowb));
                    for (int q = q0; q < q1;) {
                        const int r = q / I, n = q - r * I, len = min(q1 - q, I - n), i = q - q0;
                        const int64_t grow = static_cast<int64_t>(r_e[r]) * 2 * I + n;
                        tc::bulk_load(tc::smem_u32(st + i * rowb), a.q13 + grow * rowb, len * rowb, bar);
                        tc::bulk_load(tc::smem_u32(st + (kPS + i) * rowb), a.q13 + (grow + I) * rowb, len * rowb,
                                      bar);
                        q += len;
                    }
                } else {
                    // down stage: this CTA's rows of routes r0 .. r1-1, S2 bytes apart
                    const int r0 = (t - S) * RPS, r1 = min(nv, r0 + RPS);
                    tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>((r1 - r0) * nrows * row2));
                    for (int r = r0; r < r1; ++r)
                        tc::bulk_load(tc::smem_u32(st + (r - r0) * S2),
                                      a.q2 + (static_cast<int64_t>(r_e[r]) * d + o0) * row2, nrows * row2, bar);
                }
            }
            // every issued copy lands before the CTA may finish (the stages
            // before t - NS were consumed, so they have landed)
            volatile int never = 0;
            for (int u = max(0, t - NS); u < t; ++u)
                tc::mbar_wait(full + 8 * (u % NS), (u / NS) & 1u, &never, kWaitNs);
        }
        return;
    }
    const int cw = warp - kWarpGU0;                      // compute warp 0..23
    if (warp < kWarpT0) {
        // ------------------------------------------------ gate/up warps
        const int grp = cw / kGW, om = cw % kGW;
        const int kbase = om * (d / kGW) + lane * KPL;     // this lane's K slice of every row: one group
        const int gk = kbase / 128;
        // x slice as fp16 after an exact power-of-two rescale of the warp's
        // slice, pairs (x_8w+j, x_8w+j+4) to match the packed words
        uint32_t xw[KPL / 2];
        float xinv;
        {
            float xv[KPL];
#pragma unroll
            for (int i = 0; i < KPL; ++i)
                xv[i] = x_at<XBF>(a.x, kbase + i);
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < KPL; ++i)
                m = fmaxf(m, fabsf(xv[i]));
            const int pw = f16_shift(warp_max(m));
            const float sc = ldexpf(1.0f, pw);
            xinv = ldexpf(1.0f, -pw);
#pragma unroll
            for (int w = 0; w < KPL / 8; ++w)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 h2 = __floats2half2_rn(xv[8 * w + j] * sc, xv[8 * w + j + 4] * sc);
                    xw[4 * w + j] = *reinterpret_cast<const uint32_t *>(&h2);
                }
        }
        tc::named_bar(kBarScales, kCW * 32 + 32);         // the scales and zeros are staged, the tag formed
        const uint32_t tag = *s_tag;
        for (int s = grp, m = 0; s < S; s += kGroups, ++m) {
            const int sl = s % NS, buf = m & 1;
            const uint32_t ph = (s / NS) & 1u;
            const bool got = tc::mbar_wait(full + 8 * sl, ph, s_abort, kWaitNs);
            const int npairs = min(kPS, P - s * kPS);
            if (got) {
                const uint8_t *st = ring + sl * S1;
                float v[2 * kPS];
#pragma unroll
                for (int i = 0; i < 2 * kPS; ++i) {
                    v[i] = 0.f;
                    if (i % kPS < npairs) {
                        const uint8_t *rp = st + i * (d / 2) + kbase / 2;
                        uint32_t wq[KPL / 8];
                        if constexpr (KPL == 8) {
                            wq[0] = *reinterpret_cast<const uint32_t *>(rp);
                        } else {
                            const uint2 u2 = *reinterpret_cast<const uint2 *>(rp);
                            wq[0] = u2.x; wq[1] = u2.y;
                        }
                        // scale|zero of pair s*kPS + i%kPS, gate (i < kPS) or up row, group gk
                        const uint32_t szw = gsz[((s * kPS + i % kPS) * 2 + i / kPS) * G13 + gk];
                        const uint32_t zz2 = sz_zz2(szw);
                        float acc = 0.f;
#pragma unroll
                        for (int w = 0; w < KPL / 8; ++w) {
                            uint32_t dq[4];
                            awq_pairs(wq[w], zz2, dq);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                acc = fma2(dq[j], xw[4 * w + j], acc);
                        }
                        v[i] = acc * sz_scale(szw);
                    }
                }
                // 8 rows' sums at a time (gate rows, then up rows)
#pragma unroll
                for (int h8 = 0; h8 < 2 * kPS / 8; ++h8) {
                    float v8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v8[i] = v[8 * h8 + i];
                    const float tot = reduce8(v8, lane) * xinv;
                    if ((lane & 3) == 0) {
                        const int vi = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                        gpart[((grp * 2 + buf) * kGW + om) * 2 * kPS + 8 * h8 + vi] = tot;
                    }
                }
            }
            if (tc::named_bar_or(kBarGroup0 + grp, kGW * 32, !got)) {
                *tabort = 1;                               // the stage never landed: the group stops together
                break;
            }
            if (lane == 0)
                tc::mbar_arrive(empty + 8 * sl);
            if (om == 0 && lane < npairs) {
                // h of neuron `lane` of the stage: partials added in warp order,
                // published with this launch's tag
                const float *gp = gpart + (grp * 2 + buf) * kGW * 2 * kPS;
                float g = gp[lane], u = gp[kPS + lane];
#pragma unroll
                for (int w2 = 1; w2 < kGW; ++w2) {
                    g += gp[w2 * 2 * kPS + lane];
                    u += gp[w2 * 2 * kPS + kPS + lane];
                }
                const unsigned long long word =
                    static_cast<unsigned long long>(__float_as_uint(silu_mul(g, u))) |
                    (static_cast<unsigned long long>(tag) << 32);
                st_relaxed_u64(a.xh + q_lo + s * kPS + lane, word);
            }
        }
    } else {
        // ------------------------------------------------ scale-staging warps
        const int tw = warp - kWarpT0, tt = tid - kWarpT0 * 32;
        // scale|zero words of this CTA's gate and up rows, every group: one
        // thread per (pair, gate or up, 8 groups), 16-byte loads of the 8
        // scales and of the 8 zero words (each word holds 8 rows' zeros)
        const int h8 = G13 / 8;
        for (int i = tt; i < P * 2 * h8; i += kTW * 32) {
            const int pr = i / (2 * h8), rem = i - pr * 2 * h8, up = rem / h8, hf = rem - up * h8;
            const int q = q_lo + pr, r = q / I, n = q - r * I, nr = n + (up ? I : 0);
            const int64_t row = static_cast<int64_t>(r_e[r]) * 2 * I + nr;
            const int64_t zrow = static_cast<int64_t>(r_e[r]) * (2 * I / 8) + nr / 8;
            const uint4 sv = __ldg(reinterpret_cast<const uint4 *>(a.s13 + row * G13) + hf);
            const uint4 za = __ldg(reinterpret_cast<const uint4 *>(a.z13 + zrow * G13) + 2 * hf);
            const uint4 zb = __ldg(reinterpret_cast<const uint4 *>(a.z13 + zrow * G13) + 2 * hf + 1);
            const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
            const uint32_t zw[8] = {za.x, za.y, za.z, za.w, zb.x, zb.y, zb.z, zb.w};
            const int sh = 4 * (nr & 7);
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = sz_word(static_cast<uint16_t>(sw[j >> 1] >> (16 * (j & 1))), (zw[j] >> sh) & 0xFu);
            uint4 *dst = reinterpret_cast<uint4 *>(gsz + (pr * 2 + up) * G13 + 8 * hf);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        tc::named_arrive(kBarScales, kCW * 32 + 32);
        if constexpr (ROUTE) {
            if (tw == 0) {
                // the renormalised weights of the chosen routes (needed only at the end)
                const float w = topk_weight(lane < k ? r_l[lane] : 0.f, k, lane);
                if (lane < k) {
                    r_w[lane] = w;
                    if (c == 0) {
                        a.ids_out[lane] = r_e[lane];
                        a.wts_out[lane] = w;
                    }
                }
            }
        }
        // scale|zero words of this CTA's down rows of every route: one thread
        // per (route, row), every load of the row issued before any is used
        for (int i = tt; i < nv * nrows; i += kTW * 32) {
            const int r = i / nrows, rho = i - r * nrows, o = o0 + rho;
            const int64_t row = static_cast<int64_t>(r_e[r]) * d + o;
            const int64_t zrow = static_cast<int64_t>(r_e[r]) * (d / 8) + o / 8;
            const uint32_t *sp = reinterpret_cast<const uint32_t *>(a.s2 + row * G2);   // G2 even: 4-byte pairs
            const uint32_t *zp = a.z2 + zrow * G2;
            uint32_t sw[kMaxG2 / 2], zw[kMaxG2];
#pragma unroll
            for (int j = 0; j < kMaxG2 / 2; ++j)
                if (2 * j < G2)
                    sw[j] = __ldg(sp + j);
#pragma unroll
            for (int j = 0; j < kMaxG2; ++j)
                if (j < G2)
                    zw[j] = __ldg(zp + j);
            const int sh = 4 * (o & 7);
#pragma unroll
            for (int j = 0; j < kMaxG2; ++j)
                if (j < G2)
                    s2z[(r * RM + rho) * G2 + j] =
                        sz_word(static_cast<uint16_t>(sw[j >> 1] >> (16 * (j & 1))), (zw[j] >> sh) & 0xFu);
        }
    }

    // ---------------------------------------------------------------- exchange
    // every compute warp is done with its own gate/up work and staging: read
    // all of h, warp cw taking words (j * kCW + cw) * 64 + 2 * lane (+1),
    // until each carries this launch's tag
    tc::named_bar(kBarTail, kCW * 32);
    const bool work = !*tabort && nv > 0 && nrows > 0;
    if (work) {
        const int NP = nv * I;                                      // words; NP % 64 == 0 (I % 64 == 0)
        const int nj = (NP / 64 + kCW - 1) / kCW;                   // 16-byte loads per lane
        const uint32_t tag = *s_tag;                                // formed before the staging barrier
        const uint32_t want = a.stall ? tag ^ 0x80000000u : tag;
        uint32_t pend = 0;
        for (int j = 0; j < nj; ++j)
            if ((j * kCW + cw) * 64 < NP)
                pend |= 1u << j;
        const uint64_t t0 = tc::globaltimer_ns();
        for (uint32_t it = 0; pend; ++it) {
            for (int j0 = 0; j0 < nj; j0 += 4) {
                unsigned long long v0[4], v1[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    v0[u] = v1[u] = 0;
                    if ((pend >> (j0 + u)) & 1u)
                        ld_relaxed_u64x2(a.xh + ((j0 + u) * kCW + cw) * 64 + 2 * lane, v0[u], v1[u]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = j0 + u;
                    if (((pend >> j) & 1u) && static_cast<uint32_t>(v0[u] >> 32) == want &&
                        static_cast<uint32_t>(v1[u] >> 32) == want) {
                        *reinterpret_cast<float2 *>(hbuf + (j * kCW + cw) * 64 + 2 * lane) =
                            make_float2(__uint_as_float(static_cast<uint32_t>(v0[u])),
                                        __uint_as_float(static_cast<uint32_t>(v1[u])));
                        pend &= ~(1u << j);
                    }
                }
            }
            if (!pend)
                break;
            __nanosleep(64);
            if ((it & 15u) == 15u && (*s_abort || tc::globaltimer_ns() - t0 > kWaitNs)) {
                *s_abort = 1;
                *tabort = 1;
                set_err(a.dev_status, MOE_ERR_TIMEOUT);
                break;
            }
        }
    }
    tc::named_bar(kBarTail, kCW * 32);
    if (cw == 0 && lane == 0 && !*tabort)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---------------------------------------------------------------- tail
    if (work && !*tabort) {
        // the (route, row) units of this CTA, a contiguous block per warp
        const int U = nv * nrows;
        const int u0 = U * cw / kCW, u1 = U * (cw + 1) / kCW;
        int cur = -1;
        uint32_t hh[HPL / 2];
        float inv = 1.f;
        const uint8_t *w2r = ring;
        for (int u = u0; u < u1;) {
            const int r = u / nrows, rho = u - r * nrows;
            if (r != cur) {
                cur = r;
                const int t = S + r / RPS;                         // the down stage holding route r
                if (!tc::mbar_wait(full + 8 * (t % NS), (t / NS) & 1u, s_abort, kWaitNs)) {
                    set_err(a.dev_status, MOE_ERR_TIMEOUT);
                    break;
                }
                w2r = ring + (t % NS) * S1 + (r % RPS) * S2;
                // this lane's HPL values of h_r as fp16 after an exact
                // power-of-two rescale of the lane's largest magnitude into
                // [2^14, 2^15), in the packed words' pair order
                float hv[HPL];
                const float4 *hp = reinterpret_cast<const float4 *>(hbuf + r * I + HPL * lane);
#pragma unroll
                for (int i = 0; i < HPL / 4; ++i) {
                    const float4 f = hp[i];
                    hv[4 * i] = f.x; hv[4 * i + 1] = f.y; hv[4 * i + 2] = f.z; hv[4 * i + 3] = f.w;
                }
                float mx = 0.f;
#pragma unroll
                for (int i = 0; i < HPL; ++i)
                    mx = fmaxf(mx, fabsf(hv[i]));
                const int pw = f16_shift(mx);
                const float sc = ldexpf(1.0f, pw);
                inv = ldexpf(1.0f, -pw);
#pragma unroll
                for (int w = 0; w < HPL / 8; ++w)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const __half2 h2 = __floats2half2_rn(hv[8 * w + j] * sc, hv[8 * w + j + 4] * sc);
                        hh[4 * w + j] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
            }
            // two rows of the same route at once when the block has them
            const bool two = u + 1 < u1 && rho + 1 < nrows;
            const int rho1 = two ? rho + 1 : rho;
            const uint32_t *w0 = reinterpret_cast<const uint32_t *>(w2r + rho * (I / 2)) + HPL / 8 * lane;
            const uint32_t *w1 = reinterpret_cast<const uint32_t *>(w2r + rho1 * (I / 2)) + HPL / 8 * lane;
            const uint32_t *z0 = s2z + (r * RM + rho) * G2;
            const uint32_t *z1 = s2z + (r * RM + rho1) * G2;
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int w = 0; w < HPL / 8; ++w) {
                const int g = (HPL * lane + 8 * w) >> 7;          // a word lies in one group
                const uint32_t sz0 = z0[g], sz1 = z1[g];
                uint32_t da[4], db[4];
                awq_pairs(w0[w], sz_zz2(sz0), da);
                awq_pairs(w1[w], sz_zz2(sz1), db);
                float pa = 0.f, pb = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    pa = fma2(da[j], hh[4 * w + j], pa);
                    pb = fma2(db[j], hh[4 * w + j], pb);
                }
                acc0 = fmaf(pa, sz_scale(sz0), acc0);
                acc1 = fmaf(pb, sz_scale(sz1), acc1);
            }
            acc0 *= inv;
            acc1 *= inv;
            // both sums at once: lanes 0..15 end with row rho's, 16..31 with rho1's
            const bool up = lane & 16;
            float tsum = (up ? acc1 : acc0) + __shfl_xor_sync(0xffffffffu, up ? acc0 : acc1, 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
            if (lane == 0)
                dpart[r * RM + rho] = tsum;
            if (two && lane == 16)
                dpart[r * RM + rho1] = tsum;
            u += two ? 2 : 1;
        }
    }
    tc::named_bar(kBarTail, kCW * 32);
    const int ct = tid - kWarpGU0 * 32;
    if (ct < nrows && !*tabort) {
        // y = sum over routes in slot order of w_j * (W2_j h_j)
        float acc = 0.f;
        for (int r = 0; r < nv; ++r)
            acc += r_w[r] * dpart[r * RM + ct];
        if (a.y_f32)
            static_cast<float *>(a.y)[o0 + ct] = acc;
        else
            static_cast<__nv_bfloat16 *>(a.y)[o0 + ct] = __float2bfloat16_rn(acc);
    }
}

template <int KPL, int HPL, bool ROUTE, bool XBF>
moe_status_t launch_t(const Args &a, int G, int smem, cudaStream_t s)
{
    auto kern = pipe_kernel<KPL, HPL, ROUTE, XBF>;
    if (!smem_attr(reinterpret_cast<const void *>(kern), kSmemMax))
        return MOE_ERR_CUDA;
    return launch_pdl(kern, dim3(G), dim3(kThreads), static_cast<size_t>(smem), s, a) == cudaSuccess ? MOE_OK
                                                                                                   : MOE_ERR_CUDA;
}

template <int KPL, int HPL>
moe_status_t launch_shape(const Args &a, bool x_bf16, int G, int smem, cudaStream_t s)
{
    if (a.logits)
        return x_bf16 ? launch_t<KPL, HPL, true, true>(a, G, smem, s) : launch_t<KPL, HPL, true, false>(a, G, smem, s);
    return x_bf16 ? launch_t<KPL, HPL, false, true>(a, G, smem, s) : launch_t<KPL, HPL, false, false>(a, G, smem, s);
}

// the (d, I) pairs built: gate/up elements per lane KPL = d / 128, down
// elements per lane HPL = I / 32
inline bool shape_ok(int d, int I)
{
    return (d == 1024 && (I == 256 || I == 512)) || (d == 2048 && (I == 512 || I == 768));
}

}  // namespace dpa

bool decode_pipe_awq_shape_fits(int k, int d, int I, int G)
{
    return k >= 1 && k <= dpa::kMaxK && G >= 1 && dpa::shape_ok(d, I) && dpa::Plan{d, I, k, G}.fits();
}

bool decode_pipe_awq_eligible(int M, int k, int d, int I, int E)
{
    return M == 1 && E >= 1 && decode_pipe_awq_shape_fits(k, d, I, device_sm_count());
}

bool decode_pipe_awq_route_eligible(int E, int k) { return E >= k && E <= dpa::kCW * 32; }

moe_status_t decode_pipe_awq_launch(const void *x, bool x_bf16, int d, int I, int E, const int32_t *ids,
                                    const float *wts, const float *logits, int32_t *ids_out, float *wts_out, int k,
                                    const moe_weights_t *w13, const moe_weights_t *w2, void *y, bool y_f32, void *ws,
                                    int32_t *dev_status, cudaStream_t s)
{
    using namespace dpa;
    const int G = device_sm_count();
    const Plan pl{d, I, k, G};
    if (!pl.fits() || !shape_ok(d, I))
        return MOE_ERR_UNSUPPORTED;
    Args a{};
    a.x = x;
    a.ids = ids;
    a.wts = wts;
    a.logits = logits;
    a.ids_out = ids_out;
    a.wts_out = wts_out;
    a.q13 = static_cast<const uint8_t *>(w13->q);
    a.s13 = static_cast<const uint16_t *>(w13->scale);
    a.z13 = static_cast<const uint32_t *>(w13->zero);
    a.q2 = static_cast<const uint8_t *>(w2->q);
    a.s2 = static_cast<const uint16_t *>(w2->scale);
    a.z2 = static_cast<const uint32_t *>(w2->zero);
    a.ctr = static_cast<unsigned long long *>(ws);
    a.xh = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(ws) + kWsCounterBytes);
    a.y = y;
    a.dev_status = dev_status;
    a.y_f32 = y_f32 ? 1 : 0;
    a.k = k;
    a.d = d;
    a.I = I;
    a.E = E;
    a.stall = decode_exchange_stall();
    const int smem = pl.bytes();
    switch (d * 10000 + I) {
    case 1024 * 10000 + 256: return launch_shape<8, 8>(a, x_bf16, G, smem, s);
    case 1024 * 10000 + 512: return launch_shape<8, 16>(a, x_bf16, G, smem, s);
    case 2048 * 10000 + 512: return launch_shape<16, 16>(a, x_bf16, G, smem, s);
    case 2048 * 10000 + 768: return launch_shape<16, 24>(a, x_bf16, G, smem, s);
    default: return MOE_ERR_UNSUPPORTED;
    }
}

}  // namespace moe
