// decode_pipe_nv4.cu -- single-token decode of the routed expert layer on
// paired 4:8 sparse NVFP4 weights as one kernel, optionally with the top-k
// routing inside.
//
// The method is the output-centric decode of "Warp decode" (cursor.com
// blog, sections on what changed and on how the two kernels work), on the
// weight format of "Hardware-Native Joint Sparse-Quantization for
// Trillion-Scale Mixture-of-Experts", App. A: in every group of 8 weights
// two adjacent pairs are kept (E2M1 codes), one UE4M3 scale per 32 weights,
// one FP32 constant alpha per expert and matrix.  The structure is the
// single-token AWQ kernel's (one CTA per SM; warp 0 streams the kept codes
// of this CTA's gate/up rows and then its down rows through one ring, while
// eight staging warps load the gate/up rows' patterns and scales; four
// groups of four warps form
// h = SiLU(g) * u and publish it as (value, launch tag) words; every CTA
// reads all of h back once the words carry the launch's tag and forms its
// d / G output rows of every route's down projection).
//
// Arithmetic, exact up to the FP32 sums: a kept pair of E2M1 codes becomes an
// fp16 pair (cvt.rn.f16x2.e2m1x2), which multiplies the fp16 pair of x (or
// h) at the pair's position in the group (fma.rn.f32.f16: exact products);
// each lane's partial over its 16 weights (one scale block) is multiplied
// by the block's UE4M3 scale in FP32; alpha multiplies the row's total.  x
// and h enter as fp16 after an exact power-of-two rescale (as in the other
// single-token kernels).  Every output's summation order depends only on
// the shapes and the grid.
#include <atomic>
#include <type_traits>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "pipe_common.cuh"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {
namespace dpn {

using namespace pipe;

constexpr int kMaxK = 32;
constexpr int kGW = 4;                                // warps of a gate/up group (they split K)
constexpr int kGroups = 4;                            // gate/up groups
constexpr int kPS = 8;                                // neurons per gate/up stage
constexpr int kMaxSlots = 11;                         // ring slots, at most
constexpr int kMinSlots = 4;
constexpr int kTW = 8;                                // warps of the staging role
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
constexpr int kBarSide = kBarRank + 1;                //   gate/up patterns, scales and constants staged,
                                                      //   launch tag formed (staging warps and warp 1 arrive)
constexpr int kSmemMax = 227 * 1024;

struct Args {
    const void *x;               // [d] fp16 or bf16
    const int32_t *ids;          // given routing: ids / weights [k]
    const float *wts;
    const float *logits;         // or routed here: router logits [E] ...
    int32_t *ids_out;            // ... and the chosen ids / weights written by CTA 0
    float *wts_out;
    const uint8_t *v13, *m13, *s13;   // W13: kept codes [E][2I][d/4], patterns [E][2I][d/16], scales [E][2I][d/32]
    const float *a13;                 // [E]
    const uint8_t *v2, *m2, *s2;      // W2: [E][d][I/4], [E][d][I/16], [E][d][I/32]
    const float *a2;
    unsigned long long *ctr;     // CTA count over all launches
    unsigned long long *xh;      // exchange words [k][I]: value bits | tag << 32
    void *y;
    int32_t *dev_status;
    int y_f32, k, d, I, E;
    int stall;                   // readers expect a tag nobody writes (failure-detection test)
};

// Shared-memory plan (bytes), identical on host and device.  A ring slot is
// kPS gate rows then kPS up rows of kept codes; the down rows of every route
// reuse the ring after the gate/up stages (codes of the CTA's rows, then
// their patterns).  The gate/up rows' patterns and scales (side records,
// d/16 + d/32 bytes a row) and the down rows' scales (I/32 bytes a row, 24
// at I = 768, not 16-byte aligned) are staged by plain loads.
struct Plan {
    int d, I, k, G;
    __host__ __device__ int rows_max() const { return (d + G - 1) / G; }
    __host__ __device__ int s1() const { return 2 * kPS * (d / 4); }
    __host__ __device__ int pmax() const { return (k * I + G - 1) / G; }
    __host__ __device__ int side() const { return d / 16 + d / 32; }            // side record of a gate/up row
    __host__ __device__ int s2() const { return rows_max() * (I / 4 + I / 16); }  // one route's down rows
    __host__ __device__ int rps() const { return s1() / s2(); }
    __host__ __device__ int w2_stages() const { return (k + rps() - 1) / rps(); }
    __host__ __device__ static int up16(int v) { return (v + 15) & ~15; }
    // everything but the ring: h, gate/up side records, down scales, partials, barriers, the route table
    __host__ __device__ int fixed() const
    {
        return up16(k * I * 4) + pmax() * 2 * side() + up16(k * rows_max() * (I / 32)) +
               kGroups * 2 * kGW * 2 * kPS * 4 + up16(k * rows_max() * 4) + 2 * kMaxSlots * 8 + 5 * kMaxK * 4 + 32;
    }
    __host__ __device__ int slots() const
    {
        const int n = (kSmemMax - fixed()) / s1();
        return n > kMaxSlots ? kMaxSlots : n;
    }
    __host__ __device__ int o_h() const { return slots() * s1(); }              // h [k][I] f32
    __host__ __device__ int o_gs() const { return o_h() + up16(k * I * 4); }    // side records [P][2][side]
    __host__ __device__ int o_s2s() const { return o_gs() + pmax() * 2 * side(); }   // down scales [k][RM][I/32]
    __host__ __device__ int o_gpart() const { return o_s2s() + up16(k * rows_max() * (I / 32)); }
    __host__ __device__ int o_dpart() const { return o_gpart() + kGroups * 2 * kGW * 2 * kPS * 4; }
    __host__ __device__ int o_bars() const { return o_dpart() + up16(k * rows_max() * 4); }
    __host__ __device__ int o_route() const { return o_bars() + 2 * kMaxSlots * 8; }
    // route data: r_e | r_w | r_l | r_a13 | r_a2 [kMaxK each] | tag, nv, abort, tabort (32 bytes kept)
    __host__ __device__ int bytes() const { return o_route() + 5 * kMaxK * 4 + 32; }
    __host__ __device__ bool fits() const
    {
        // every CTA's gate/up stages within the ring's first lap: a group then
        // never waits (by barrier parity) on a slot that another group's
        // stage, possibly not landed yet, held one lap earlier
        return s2() > 0 && s2() <= s1() && slots() >= kMinSlots && w2_stages() <= slots() &&
               (pmax() + kPS - 1) / kPS <= slots() && bytes() <= kSmemMax &&
               static_cast<size_t>(k) * I * 8 <= kWsTagBytes && k * I <= kCW * 32 * kMaxPerLane;
    }
};

// Two E2M1 codes (low nibble first) -> the fp16 pair of their values (exact).
__device__ __forceinline__ uint32_t e2m1x2(uint32_t byte)
{
    uint32_t r;
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "r"(byte));
    return r;
}

// A UE4M3 scale code (sign bit clear) -> its value (exact).
__device__ __forceinline__ float ue4m3(uint32_t s)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(s & 0xFFu)));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(r & 0xFFFFu)));
}

// One group of 8 weights against the 8 activations of its positions (four
// fp16 pairs a0..a3, natural order): the kept codes (16 bits: pair p0's two
// values, then pair p1's, low nibble first) times the activation pairs at
// p0 and p1 (pattern nibble p0 | p1 << 2), added to acc.
__device__ __forceinline__ float group_dot(uint32_t codes16, uint32_t nib, uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, float acc)
{
    // the pairs at p0 (0..2) and p1 (1..3), chosen without branches (lanes differ in patterns)
    uint32_t xa, xb;
    asm("{\n .reg .pred q0, q1, q2, q3;\n"
        " and.b32 %0, %2, 3;\n shr.b32 %1, %2, 2;\n"
        " setp.eq.u32 q0, %0, 0;\n setp.eq.u32 q1, %0, 1;\n"
        " setp.eq.u32 q2, %1, 3;\n setp.eq.u32 q3, %1, 2;\n"
        " selp.b32 %0, %4, %5, q1;\n selp.b32 %0, %3, %0, q0;\n"
        " selp.b32 %1, %5, %4, q3;\n selp.b32 %1, %6, %1, q2;\n}"
        : "=&r"(xa), "=&r"(xb)
        : "r"(nib), "r"(a0), "r"(a1), "r"(a2), "r"(a3));
    acc = fma2(e2m1x2(codes16 & 0xFFu), xa, acc);
    return fma2(e2m1x2(codes16 >> 8), xb, acc);
}

template <bool XBF>
__device__ __forceinline__ float x_at(const void *x, int i)
{
    if constexpr (XBF)
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(x)[i]);
    else
        return __half2float(static_cast<const __half *>(x)[i]);
}

// KPL: gate/up weights per lane of a warp's K slice (d = 32 * kGW * KPL; 8
// or 16, one or two groups, inside one scale block); HG: down groups per
// lane (I = 256 * HG), group lane + 32 j; ROUTE: the kernel routes the token
// itself; XBF: x is bf16 (else fp16).
template <int KPL, int HG, bool ROUTE, bool XBF>
__global__ void __launch_bounds__(kThreads, 1) pipe_kernel(const Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int d = a.d, I = a.I, k = a.k, G = gridDim.x, c = blockIdx.x;
    const Plan pl{d, I, k, G};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int RM = pl.rows_max(), S1 = pl.s1(), S2 = pl.s2(), NS = pl.slots(), RPS = pl.rps();
    uint8_t *ring = smem;
    float *hbuf = reinterpret_cast<float *>(smem + pl.o_h());           // [nv][I] h of every route
    uint8_t *gs = smem + pl.o_gs();                                      // [P][2][side] gate/up patterns | scales
    uint8_t *s2s = smem + pl.o_s2s();                                    // [k][RM][I/32] down scales
    float *gpart = reinterpret_cast<float *>(smem + pl.o_gpart());       // [grp][2][kGW][2 kPS]
    float *dpart = reinterpret_cast<float *>(smem + pl.o_dpart());       // [k][RM]
    const uint32_t full = tc::smem_u32(smem + pl.o_bars());
    const uint32_t empty = full + 8 * kMaxSlots;
    int *r_e = reinterpret_cast<int *>(smem + pl.o_route());
    float *r_w = reinterpret_cast<float *>(r_e + kMaxK);
    float *r_l = r_w + kMaxK;                                            // logits of the chosen routes
    float *r_a13 = r_l + kMaxK, *r_a2 = r_a13 + kMaxK;                   // the routes' experts' constants
    uint32_t *s_tag = reinterpret_cast<uint32_t *>(r_a2 + kMaxK);
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
        tc::named_arrive(kBarSide, kCW * 32 + 32);
        return;
    } else if constexpr (ROUTE) {
        // top-k of the router logits by rank, as in the other single-token
        // kernels: expert e's slot is the number of experts ahead of it
        // (larger logit, or equal logit and lower id); the keys sit in the
        // ring, idle until the routes are out.
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
            const int cbw = d / 4;                               // code bytes of a gate/up row
            const int cb2 = I / 4, mb2 = I / 16;                 // of a down row: codes, patterns
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
                    tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(q1 - q0) * 2 * cbw);
                    for (int q = q0; q < q1;) {
                        const int r = q / I, n = q - r * I, len = min(q1 - q, I - n), i = q - q0;
                        const int64_t g0 = static_cast<int64_t>(r_e[r]) * 2 * I + n, g1 = g0 + I;
                        tc::bulk_load(tc::smem_u32(st + i * cbw), a.v13 + g0 * cbw, len * cbw, bar);
                        tc::bulk_load(tc::smem_u32(st + (kPS + i) * cbw), a.v13 + g1 * cbw, len * cbw, bar);
                        q += len;
                    }
                } else {
                    // down stage: this CTA's rows of routes r0 .. r1-1, S2 bytes apart (codes, then patterns)
                    const int r0 = (t - S) * RPS, r1 = min(nv, r0 + RPS);
                    tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>((r1 - r0) * nrows * (cb2 + mb2)));
                    for (int r = r0; r < r1; ++r) {
                        const int64_t row = static_cast<int64_t>(r_e[r]) * d + o0;
                        uint8_t *dst = st + (r - r0) * S2;
                        tc::bulk_load(tc::smem_u32(dst), a.v2 + row * cb2, nrows * cb2, bar);
                        tc::bulk_load(tc::smem_u32(dst + RM * cb2), a.m2 + row * mb2, nrows * mb2, bar);
                    }
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
        const int kbase = om * (d / kGW) + lane * KPL;     // this lane's K slice of every row: KPL / 8 groups
        // x slice as fp16 pairs (natural order) after an exact power-of-two
        // rescale of the warp's slice
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
            for (int i = 0; i < KPL / 2; ++i) {
                const __half2 h2 = __floats2half2_rn(xv[2 * i] * sc, xv[2 * i + 1] * sc);
                xw[i] = *reinterpret_cast<const uint32_t *>(&h2);
            }
        }
        const int SD = pl.side();
        tc::named_bar(kBarSide, kCW * 32 + 32);           // the side records and constants are staged, the tag formed
        const uint32_t tag = *s_tag;
        for (int s = grp, m = 0; s < S; s += kGroups, ++m) {
            const int sl = s % NS, buf = m & 1;
            const uint32_t ph = (s / NS) & 1u;
            const bool got = tc::mbar_wait(full + 8 * sl, ph, s_abort, kWaitNs);
            const int npairs = min(kPS, P - s * kPS);
            if (got) {
                const uint8_t *st = ring + sl * S1;
                // 8 rows at a time (gate rows, then up rows): this lane's KPL
                // weights of each (KPL / 4 code bytes, KPL / 16 pattern bytes,
                // one scale), then the 8 sums across the lanes
#pragma unroll
                for (int h8 = 0; h8 < 2 * kPS / 8; ++h8) {
                    float v8[8];
#pragma unroll
                    for (int ii = 0; ii < 8; ++ii) {
                        const int i = 8 * h8 + ii;
                        v8[ii] = 0.f;
                        if (i % kPS < npairs) {
                            // this row's side record: pair s * kPS + i % kPS, gate (i < kPS) or up
                            const uint8_t *sr = gs + ((s * kPS + i % kPS) * 2 + i / kPS) * SD;
                            float acc = 0.f;
                            if constexpr (KPL == 16) {
                                const uint32_t cw4 =
                                    *reinterpret_cast<const uint32_t *>(st + i * (d / 4) + kbase / 4);
                                const uint32_t mb = sr[kbase / 16];
                                acc = group_dot(cw4 & 0xFFFFu, mb & 0xFu, xw[0], xw[1], xw[2], xw[3], acc);
                                acc = group_dot(cw4 >> 16, mb >> 4, xw[4], xw[5], xw[6], xw[7], acc);
                            } else {
                                const uint32_t cw2 =
                                    *reinterpret_cast<const uint16_t *>(st + i * (d / 4) + kbase / 4);
                                const uint32_t mb = sr[kbase / 16];
                                acc = group_dot(cw2, (mb >> (4 * ((kbase >> 3) & 1))) & 0xFu, xw[0], xw[1], xw[2],
                                                xw[3], acc);
                            }
                            v8[ii] = acc * ue4m3(sr[d / 16 + kbase / 32]);
                        }
                    }
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
                // scaled by the expert's constant, published with this launch's tag
                const float *gp = gpart + (grp * 2 + buf) * kGW * 2 * kPS;
                float g = gp[lane], u = gp[kPS + lane];
#pragma unroll
                for (int w2 = 1; w2 < kGW; ++w2) {
                    g += gp[w2 * 2 * kPS + lane];
                    u += gp[w2 * 2 * kPS + kPS + lane];
                }
                const int q = q_lo + s * kPS + lane;
                const float al = r_a13[q / I];
                const unsigned long long word =
                    static_cast<unsigned long long>(__float_as_uint(silu_mul(g * al, u * al))) |
                    (static_cast<unsigned long long>(tag) << 32);
                st_relaxed_u64(a.xh + q, word);
            }
        }
    } else {
        // ------------------------------------------------ staging warps
        const int tw = warp - kWarpT0, tt = tid - kWarpT0 * 32;
        // the side records of this CTA's gate and up rows (patterns d/16
        // bytes, then scales d/32 bytes), 16-byte loads, and the routes'
        // experts' constants
        {
            const int SD = pl.side(), nm = d / 256, n16 = SD / 16;   // 16-byte pieces: patterns, all
            for (int i = tt; i < P * 2 * n16; i += kTW * 32) {
                const int pr = i / (2 * n16), rem = i - pr * 2 * n16, up = rem / n16, j = rem - up * n16;
                const int q = q_lo + pr, r = q / I, n = q - r * I;
                const int64_t row = static_cast<int64_t>(r_e[r]) * 2 * I + n + (up ? I : 0);
                const uint4 v = j < nm ? __ldg(reinterpret_cast<const uint4 *>(a.m13 + row * (d / 16)) + j)
                                       : __ldg(reinterpret_cast<const uint4 *>(a.s13 + row * (d / 32)) + (j - nm));
                *reinterpret_cast<uint4 *>(gs + (pr * 2 + up) * SD + 16 * j) = v;
            }
            if (tt < nv) {
                r_a13[tt] = __ldg(a.a13 + r_e[tt]);
                r_a2[tt] = __ldg(a.a2 + r_e[tt]);
            }
        }
        tc::named_arrive(kBarSide, kCW * 32 + 32);
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
        // the scales of this CTA's down rows of every route: one thread per
        // (route, row), I / 32 bytes as 8-byte loads, all issued before use
        constexpr int kS8 = HG * 8 / 8;                    // I / 32 bytes = HG * 8 bytes
        for (int i = tt; i < nv * nrows; i += kTW * 32) {
            const int r = i / nrows, rho = i - r * nrows;
            const int64_t row = static_cast<int64_t>(r_e[r]) * d + o0 + rho;
            const uint2 *sp = reinterpret_cast<const uint2 *>(a.s2 + row * (I / 32));
            uint2 sv[kS8];
#pragma unroll
            for (int j = 0; j < kS8; ++j)
                sv[j] = __ldg(sp + j);
            uint2 *dst = reinterpret_cast<uint2 *>(s2s + (r * RM + rho) * (I / 32));
#pragma unroll
            for (int j = 0; j < kS8; ++j)
                dst[j] = sv[j];
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
        const int cb2 = I / 4, mb2 = I / 16, sb2 = I / 32;
        int cur = -1;
        uint32_t hh[4 * HG];                                  // groups lane + 32 j: 8 values each, as 4 pairs
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
                // this lane's 8 HG values of h_r as fp16 after an exact
                // power-of-two rescale of the lane's largest magnitude into
                // [2^14, 2^15), natural pairs
                float hv[8 * HG];
#pragma unroll
                for (int j = 0; j < HG; ++j) {
                    const float4 *hp = reinterpret_cast<const float4 *>(hbuf + r * I + 8 * (lane + 32 * j));
                    const float4 f0 = hp[0], f1 = hp[1];
                    hv[8 * j] = f0.x; hv[8 * j + 1] = f0.y; hv[8 * j + 2] = f0.z; hv[8 * j + 3] = f0.w;
                    hv[8 * j + 4] = f1.x; hv[8 * j + 5] = f1.y; hv[8 * j + 6] = f1.z; hv[8 * j + 7] = f1.w;
                }
                float mx = 0.f;
#pragma unroll
                for (int i = 0; i < 8 * HG; ++i)
                    mx = fmaxf(mx, fabsf(hv[i]));
                const int pw = f16_shift(mx);
                const float sc = ldexpf(1.0f, pw);
                inv = ldexpf(1.0f, -pw);
#pragma unroll
                for (int i = 0; i < 4 * HG; ++i) {
                    const __half2 h2 = __floats2half2_rn(hv[2 * i] * sc, hv[2 * i + 1] * sc);
                    hh[i] = *reinterpret_cast<const uint32_t *>(&h2);
                }
            }
            // two rows of the same route at once when the block has them
            const bool two = u + 1 < u1 && rho + 1 < nrows;
            const int rho1 = two ? rho + 1 : rho;
            const uint8_t *c0 = w2r + rho * cb2, *c1 = w2r + rho1 * cb2;
            const uint8_t *m0 = w2r + RM * cb2 + rho * mb2, *m1 = w2r + RM * cb2 + rho1 * mb2;
            const uint8_t *s0 = s2s + (r * RM + rho) * sb2, *s1 = s2s + (r * RM + rho1) * sb2;
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int j = 0; j < HG; ++j) {
                const int g = lane + 32 * j;
                const uint32_t ca = *reinterpret_cast<const uint16_t *>(c0 + 2 * g);
                const uint32_t cb = *reinterpret_cast<const uint16_t *>(c1 + 2 * g);
                const int sh = 4 * (g & 1);
                const uint32_t na = (m0[g >> 1] >> sh) & 0xFu, nb = (m1[g >> 1] >> sh) & 0xFu;
                const float pa = group_dot(ca, na, hh[4 * j], hh[4 * j + 1], hh[4 * j + 2], hh[4 * j + 3], 0.f);
                const float pb = group_dot(cb, nb, hh[4 * j], hh[4 * j + 1], hh[4 * j + 2], hh[4 * j + 3], 0.f);
                acc0 = fmaf(pa, ue4m3(s0[g >> 2]), acc0);
                acc1 = fmaf(pb, ue4m3(s1[g >> 2]), acc1);
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
        // y = sum over routes in slot order of w_j * alpha_j * (W2_j h_j)
        float acc = 0.f;
        for (int r = 0; r < nv; ++r)
            acc += r_w[r] * r_a2[r] * dpart[r * RM + ct];
        if (a.y_f32)
            static_cast<float *>(a.y)[o0 + ct] = acc;
        else
            static_cast<__nv_bfloat16 *>(a.y)[o0 + ct] = __float2bfloat16_rn(acc);
    }
}

template <int KPL, int HG, bool ROUTE, bool XBF>
moe_status_t launch_t(const Args &a, int G, int smem, cudaStream_t s)
{
    auto kern = pipe_kernel<KPL, HG, ROUTE, XBF>;
    if (!smem_attr(reinterpret_cast<const void *>(kern), kSmemMax))
        return MOE_ERR_CUDA;
    return launch_pdl(kern, dim3(G), dim3(kThreads), static_cast<size_t>(smem), s, a) == cudaSuccess ? MOE_OK
                                                                                                   : MOE_ERR_CUDA;
}

template <int KPL, int HG>
moe_status_t launch_shape(const Args &a, bool x_bf16, int G, int smem, cudaStream_t s)
{
    if (a.logits)
        return x_bf16 ? launch_t<KPL, HG, true, true>(a, G, smem, s) : launch_t<KPL, HG, true, false>(a, G, smem, s);
    return x_bf16 ? launch_t<KPL, HG, false, true>(a, G, smem, s) : launch_t<KPL, HG, false, false>(a, G, smem, s);
}

// the (d, I) pairs built: gate/up weights per lane KPL = d / 128, down
// groups per lane HG = I / 256
inline bool shape_ok(int d, int I)
{
    return (d == 1024 && (I == 256 || I == 512)) || (d == 2048 && (I == 512 || I == 768));
}

}  // namespace dpn

bool decode_pipe_nv4_shape_fits(int k, int d, int I, int G)
{
    return k >= 1 && k <= dpn::kMaxK && G >= 1 && dpn::shape_ok(d, I) && dpn::Plan{d, I, k, G}.fits();
}

bool decode_pipe_nv4_eligible(int M, int k, int d, int I, int E)
{
    return M == 1 && E >= 1 && decode_pipe_nv4_shape_fits(k, d, I, device_sm_count());
}

bool decode_pipe_nv4_route_eligible(int E, int k) { return E >= k && E <= dpn::kCW * 32; }

moe_status_t decode_pipe_nv4_launch(const void *x, bool x_bf16, int d, int I, int E, const int32_t *ids,
                                    const float *wts, const float *logits, int32_t *ids_out, float *wts_out, int k,
                                    const moe_weights_t *w13, const moe_weights_t *w2, void *y, bool y_f32, void *ws,
                                    int32_t *dev_status, cudaStream_t s)
{
    using namespace dpn;
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
    a.v13 = static_cast<const uint8_t *>(w13->q);
    a.m13 = static_cast<const uint8_t *>(w13->zero);
    a.s13 = static_cast<const uint8_t *>(w13->scale);
    a.a13 = w13->alpha;
    a.v2 = static_cast<const uint8_t *>(w2->q);
    a.m2 = static_cast<const uint8_t *>(w2->zero);
    a.s2 = static_cast<const uint8_t *>(w2->scale);
    a.a2 = w2->alpha;
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
    case 1024 * 10000 + 256: return launch_shape<8, 1>(a, x_bf16, G, smem, s);
    case 1024 * 10000 + 512: return launch_shape<8, 2>(a, x_bf16, G, smem, s);
    case 2048 * 10000 + 512: return launch_shape<16, 2>(a, x_bf16, G, smem, s);
    case 2048 * 10000 + 768: return launch_shape<16, 3>(a, x_bf16, G, smem, s);
    default: return MOE_ERR_UNSUPPORTED;
    }
}

}  // namespace moe
