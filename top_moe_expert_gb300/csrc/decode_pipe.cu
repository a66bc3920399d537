// decode_pipe.cu -- single-token decode of the routed MXFP8 expert layer as
// one kernel on the standard (K-contiguous) layout of both projections,
// optionally with the top-k routing inside.
//
// Output-centric decode ("Warp decode", cursor.com blog, sections on what
// changed and on how the two kernels work): for each routed expert e_j
//     h_j = SiLU(Wg_{e_j} x) * (Wu_{e_j} x),    y = sum_j w_j * (W2_{e_j} h_j),
// the weights streamed once and converted on the fly, FP32 sums reduced with
// shuffle butterflies, the routing weight folded into the down projection's
// sum over routes; no alignment, padding, scatter or combine buffer.
//
// At one token the layer is an HBM stream of the k routed experts' weights
// (38.9 MB at d = 2048, I = 768, k = 8).  One CTA per SM, with warp roles:
//   * warp 0, producer: routes the token (or reads the given routing),
//     publishes the valid routes in slot order, then streams through one
//     ring of up to 11 slots (176 KB in flight per SM at d = 2048): first
//     this CTA's gate and up rows, 4 neurons per stage, then this CTA's rows
//     of every routed expert's down projection, one or more routes per
//     stage, each issued as soon as its slot is free.
//   * warp 1: reads the launch's epoch from the call counter and advances it.
//   * warps 2..17, gate/up: 4 groups of 4 warps.  Group g takes stages g,
//     g+4, g+8, ...; its warps split K, each holding its slice of x in
//     registers (fp16 after an exact power-of-two rescale), and form the
//     slice's partial dot products with mixed fp16 x fp16 -> FP32 FMAs.  The
//     group adds the partials in a fixed order, forms h = SiLU(g) * u in
//     FP32 and publishes it as one 8-byte (value, launch tag) word.
//   * warps 18..25: load the E8M0 rows of this CTA's gate/up neurons (before
//     the first stage is consumed) and of its down-projection rows.
// Exchange: the 24 compute warps read every route's h words until each
// carries this launch's tag, into shared memory.  No flag, fence or barrier
// across CTAs: a word is written once per launch and read atomically, so a
// value is taken only when its own tag says it belongs to this launch.
// Tail: each warp forms (route, row) units of this CTA's output rows of the
// down projection, two rows at a time, from the down rows in the ring and
// h converted per lane to fp16 after an exact power-of-two rescale; y is the
// routing-weighted sum over routes in slot order.  The (route, neuron) space
// is split evenly over the CTAs and each CTA owns d / G output rows, so no
// output is reduced across CTAs.
//
// Launch tag: the first 8 bytes of the workspace count CTAs over all
// launches (zero before the first use).  Every launch adds exactly one per
// CTA, and a launch starts only after the previous one has completed, so
// every CTA of launch n reads a count in [nG, nG + G) and takes n + 1 as
// its tag.  The exchange words sit in the workspace's reserved area, which
// no other path writes, so a word's stale tag is that of an earlier launch
// of this kernel.  Every output's summation order depends only on the
// shapes and the grid, so repeats are bit-identical.
#include <atomic>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "pipe_common.cuh"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {
namespace dp {

constexpr int kMaxK = 32;
constexpr int kGW = 4;                                // warps of a gate/up group (they split K)
constexpr int kGroups = 4;                            // gate/up groups
constexpr int kPS = 4;                                // neurons per gate/up stage (4 or 8)
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
constexpr int kBarScales = kBarRank + 1;              //   gate/up E8M0 rows staged, launch tag formed
                                                      //   (staging warps and warp 1 arrive)
constexpr int kSmemMax = 227 * 1024;

struct Args {
    const __nv_bfloat16 *x;      // [d]
    const int32_t *ids;          // given routing: ids / weights [k]
    const float *wts;
    const float *logits;         // or routed here: router logits [E] ...
    int32_t *ids_out;            // ... and the chosen ids / weights written by CTA 0
    float *wts_out;
    const uint8_t *q13, *s13;    // [E][2I][d], [E][2I][d/32]
    const uint8_t *q2, *s2;      // [E][d][I],  [E][d][I/32]
    unsigned long long *ctr;     // CTA count over all launches
    unsigned long long *xh;      // exchange words [k][I]: value bits | tag << 32
    void *y;
    int32_t *dev_status;
    int y_f32, k, d, I, E;
    int stall;                   // readers expect a tag nobody writes (failure-detection test)
};

// Shared-memory plan (bytes), identical on host and device.
struct Plan {
    int d, I, k, G;
    __host__ __device__ int rows_max() const { return (d + G - 1) / G; }
    __host__ __device__ int s1() const { return kPS * 2 * d; }                   // slot: gate rows | up rows
    __host__ __device__ int pmax() const { return (k * I + G - 1) / G; }        // pairs of a CTA, at most
    __host__ __device__ int s2() const { return rows_max() * I; }               // one route's down rows
    __host__ __device__ int rps() const { return s1() / s2(); }                 // routes per down stage
    __host__ __device__ int w2_stages() const { return (k + rps() - 1) / rps(); }
    __host__ __device__ static int up16(int v) { return (v + 15) & ~15; }
    // everything but the ring
    __host__ __device__ int fixed() const
    {
        return up16(k * I * 4) + k * rows_max() * (I / 32) * 4 + up16(pmax() * 2 * (d / 32)) +
               kGroups * 2 * kGW * 2 * kPS * 4 + up16(k * rows_max() * 4) + 2 * kMaxSlots * 8 + 3 * kMaxK * 4 + 32;
    }
    __host__ __device__ int slots() const
    {
        const int n = (kSmemMax - fixed()) / s1();
        return n > kMaxSlots ? kMaxSlots : n;
    }
    __host__ __device__ int o_h() const { return slots() * s1(); }             // h [k][I] f32
    __host__ __device__ int o_s2s() const { return o_h() + up16(k * I * 4); }
    __host__ __device__ int o_gsc() const { return o_s2s() + k * rows_max() * (I / 32) * 4; }
    __host__ __device__ int o_gpart() const { return o_gsc() + up16(pmax() * 2 * (d / 32)); }
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
               static_cast<size_t>(k) * I * 8 <= kWsTagBytes && k * I <= kCW * 32 * kMaxPerLane;
    }
};

// set_err, fma2, reduce8, f16_shift, warp_max and the relaxed exchange loads
// and stores come from pipe_common.cuh, shared with the 4-bit single-token
// kernels.
using namespace pipe;

__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two)));
    return r;
}

// four E4M3 codes (one word, byte order) -> two f16x2 words, exactly; the
// word is split into its 16-bit halves without integer instructions
__device__ __forceinline__ void cvt_e4m3x4(uint32_t q, uint32_t &w01, uint32_t &w23)
{
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n"
        " cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
        : "=r"(w01), "=r"(w23) : "r"(q));
}

// sum over 4 E4M3 codes (one word, byte order) times 4 fp16 (two f16x2 words)
__device__ __forceinline__ float dot4(uint32_t q, uint32_t a01, uint32_t a23, float acc)
{
    uint32_t w01, w23;
    cvt_e4m3x4(q, w01, w23);
    acc = fma2(w01, a01, acc);
    return fma2(w23, a23, acc);
}

// KPL bytes at p (16-byte aligned for KPL >= 16, KPL-aligned otherwise) into words
template <int KPL>
__device__ __forceinline__ void lds_codes(const uint8_t *p, uint32_t (&w)[KPL / 4])
{
    if constexpr (KPL == 4) {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    } else if constexpr (KPL == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < KPL / 16; ++i) {
            const uint4 v = *reinterpret_cast<const uint4 *>(p + 16 * i);
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    }
}

// KPL: gate/up elements per lane of a warp's K slice (d = 32 * kGW * KPL);
// HPL: down elements per lane (I = 32 * HPL); ROUTE: the kernel routes the
// token itself from its E <= kCW * 32 router logits.
template <int KPL, int HPL, bool ROUTE>
__global__ void __launch_bounds__(kThreads, 1) pipe_kernel(const Args a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int d = a.d, I = a.I, k = a.k, G = gridDim.x, c = blockIdx.x;
    const Plan pl{d, I, k, G};
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int RM = pl.rows_max(), S1 = pl.s1(), S2 = pl.s2(), NS = pl.slots(), RPS = pl.rps();
    uint8_t *ring = smem;
    float *hbuf = reinterpret_cast<float *>(smem + pl.o_h());           // [nv][I] h of every route
    float *s2s = reinterpret_cast<float *>(smem + pl.o_s2s());           // [k][RM][I/32] down scales
    uint8_t *gsc = smem + pl.o_gsc();                                    // [P][2][d/32] gate/up E8M0 rows
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
        // one; the gate/up warps read it after the scale barrier (it is not
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
            const int64_t rowb = d;
            tc::fence_proxy_async_smem();          // the ring held the routing's keys
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
                    tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(q1 - q0) * (2 * d));
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
                    tc::mbar_arrive_expect_tx(bar, static_cast<uint32_t>((r1 - r0) * nrows * I));
                    for (int r = r0; r < r1; ++r)
                        tc::bulk_load(tc::smem_u32(st + (r - r0) * S2),
                                      a.q2 + (static_cast<int64_t>(r_e[r]) * d + o0) * I, nrows * I, bar);
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
        const int kbase = om * (d / kGW) + lane * KPL;     // this lane's K slice of every row
        // x slice as fp16 after an exact power-of-two rescale of the warp's slice
        uint32_t xw[KPL / 2];
        float xinv;
        {
            uint32_t raw[KPL / 2];
            const uint8_t *xp = reinterpret_cast<const uint8_t *>(a.x) + 2 * kbase;
            if constexpr (KPL == 4) {
                const uint2 v = __ldg(reinterpret_cast<const uint2 *>(xp));
                raw[0] = v.x; raw[1] = v.y;
            } else {
#pragma unroll
                for (int i = 0; i < KPL / 8; ++i) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xp) + i);
                    raw[4 * i] = v.x; raw[4 * i + 1] = v.y; raw[4 * i + 2] = v.z; raw[4 * i + 3] = v.w;
                }
            }
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < KPL / 2; ++i)
                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(raw[i] << 16)), fabsf(__uint_as_float(raw[i] & 0xFFFF0000u))));
            const int pw = f16_shift(warp_max(m));
            const float sc = ldexpf(1.0f, pw);
            xinv = ldexpf(1.0f, -pw);
#pragma unroll
            for (int i = 0; i < KPL / 2; ++i) {
                const __half2 h2 = __floats2half2_rn(__uint_as_float(raw[i] << 16) * sc,
                                                     __uint_as_float(raw[i] & 0xFFFF0000u) * sc);
                xw[i] = *reinterpret_cast<const uint32_t *>(&h2);
            }
        }
        const int sclb = d / 32;
        tc::named_bar(kBarScales, kCW * 32 + 32);          // the E8M0 rows are staged, the tag formed
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
                        uint32_t wq[KPL / 4];
                        lds_codes<KPL>(st + i * d + kbase, wq);
                        float acc = 0.f;
#pragma unroll
                        for (int u = 0; u < KPL / 4; ++u)
                            acc = dot4(wq[u], xw[2 * u], xw[2 * u + 1], acc);
                        // E8M0 of pair s*kPS + i%kPS, gate (i < kPS) or up row, this lane's block
                        v[i] = acc * e8m0_to_float(gsc[((s * kPS + i % kPS) * 2 + i / kPS) * sclb + (kbase >> 5)]);
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
        const int nb2 = I / 32;
        {
            // the gate and up E8M0 rows of this CTA's pairs, 16 bytes per load
            const int nb1 = d / 32, w16 = nb1 / 16;            // d % 512 == 0: whole 16-byte pieces
            for (int i = tt; i < P * 2 * w16; i += kTW * 32) {
                const int pr = i / (2 * w16), rem = i - pr * 2 * w16, up = rem / w16, wv = rem - up * w16;
                const int q = q_lo + pr, r = q / I, n = q - r * I;
                const int64_t row = static_cast<int64_t>(r_e[r]) * 2 * I + n + (up ? I : 0);
                reinterpret_cast<uint4 *>(gsc + (pr * 2 + up) * nb1)[wv] =
                    __ldg(reinterpret_cast<const uint4 *>(a.s13 + row * nb1) + wv);
            }
            tc::named_arrive(kBarScales, kCW * 32 + 32);
        }
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
        // the E8M0 bytes of this CTA's rows of every route
        for (int i = tt; i < nv * nrows * nb2; i += kTW * 32) {
            const int r = i / (nrows * nb2), rem = i - r * nrows * nb2, rho = rem / nb2, b = rem - rho * nb2;
            s2s[(r * RM + rho) * nb2 + b] =
                e8m0_to_float(__ldg(a.s2 + (static_cast<int64_t>(r_e[r]) * d + o0 + rho) * nb2 + b));
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
        const uint32_t tag = *s_tag;                                // formed before the scale barrier
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
        const int U = nv * nrows, nb2 = I / 32;
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
                // [2^14, 2^15) (relative rounding at most 2^-12 each)
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
                for (int i = 0; i < HPL / 2; ++i) {
                    const __half2 h2 = __floats2half2_rn(hv[2 * i] * sc, hv[2 * i + 1] * sc);
                    hh[i] = *reinterpret_cast<const uint32_t *>(&h2);
                }
            }
            // two rows of the same route at once when the block has them
            const bool two = u + 1 < u1 && rho + 1 < nrows;
            const int rho1 = two ? rho + 1 : rho;
            const uint8_t *w0 = w2r + rho * I + HPL * lane;
            const uint8_t *w1 = w2r + rho1 * I + HPL * lane;
            const float *sr0 = s2s + (r * RM + rho) * nb2 + ((HPL * lane) >> 5);
            const float *sr1 = s2s + (r * RM + rho1) * nb2 + ((HPL * lane) >> 5);
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < HPL / 8; ++c8) {
                const uint2 q0 = *reinterpret_cast<const uint2 *>(w0 + 8 * c8);
                const uint2 q1 = *reinterpret_cast<const uint2 *>(w1 + 8 * c8);
                const int sb = (((HPL * lane) & 31) + 8 * c8) >> 5;
                float p0 = 0.f, p1 = 0.f;
                uint32_t wa[4], wb[4];
                cvt_e4m3x4(q0.x, wa[0], wa[1]);
                cvt_e4m3x4(q0.y, wa[2], wa[3]);
                cvt_e4m3x4(q1.x, wb[0], wb[1]);
                cvt_e4m3x4(q1.y, wb[2], wb[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p0 = fma2(wa[i], hh[4 * c8 + i], p0);
                    p1 = fma2(wb[i], hh[4 * c8 + i], p1);
                }
                acc0 = fmaf(p0, sr0[sb], acc0);
                acc1 = fmaf(p1, sr1[sb], acc1);
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

template <int KPL, int HPL, bool ROUTE>
moe_status_t launch_t(const Args &a, int G, int smem, cudaStream_t s)
{
    auto kern = pipe_kernel<KPL, HPL, ROUTE>;
    if (!smem_attr(reinterpret_cast<const void *>(kern), kSmemMax))
        return MOE_ERR_CUDA;
    return launch_pdl(kern, dim3(G), dim3(kThreads), static_cast<size_t>(smem), s, a) == cudaSuccess ? MOE_OK
                                                                                                   : MOE_ERR_CUDA;
}

template <int KPL, int HPL>
moe_status_t launch_route(const Args &a, int G, int smem, cudaStream_t s)
{
    return a.logits ? launch_t<KPL, HPL, true>(a, G, smem, s) : launch_t<KPL, HPL, false>(a, G, smem, s);
}

// the (d, I) pairs built: gate/up elements per lane KPL = d / 128, down
// elements per lane HPL = I / 32
inline bool shape_ok(int d, int I)
{
    return (d == 512 && I == 256) || (d == 1024 && I == 512) || (d == 2048 && (I == 512 || I == 768 || I == 1024));
}

}  // namespace dp

// When set, the next launches' exchange waits for a tag that no CTA writes:
// the wait gives up after its time limit and reports MOE_ERR_TIMEOUT, which
// lets a test exercise the failure path without faulting or hanging the GPU.
static std::atomic<int> g_stall{0};

int decode_exchange_stall() { return g_stall.load(std::memory_order_relaxed); }

bool decode_pipe_shape_fits(int k, int d, int I, int G)
{
    return k >= 1 && k <= dp::kMaxK && G >= 1 && dp::shape_ok(d, I) && dp::Plan{d, I, k, G}.fits();
}

bool decode_pipe_eligible(int M, int k, int d, int I, int E)
{
    return M == 1 && E >= 1 && decode_pipe_shape_fits(k, d, I, device_sm_count());
}

bool decode_pipe_route_eligible(int E, int k) { return E >= k && E <= dp::kCW * 32; }

moe_status_t decode_pipe_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                                const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                                const uint8_t *s13, const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32,
                                void *ws, int32_t *dev_status, cudaStream_t s)
{
    using namespace dp;
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
    a.q13 = q13;
    a.s13 = s13;
    a.q2 = q2;
    a.s2 = s2;
    a.ctr = static_cast<unsigned long long *>(ws);
    a.xh = reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(ws) + kWsCounterBytes);
    a.y = y;
    a.dev_status = dev_status;
    a.y_f32 = y_f32 ? 1 : 0;
    a.k = k;
    a.d = d;
    a.I = I;
    a.E = E;
    a.stall = g_stall.load(std::memory_order_relaxed);
    const int smem = pl.bytes();
    switch (d * 10000 + I) {
    case 512 * 10000 + 256: return launch_route<4, 8>(a, G, smem, s);
    case 1024 * 10000 + 512: return launch_route<8, 16>(a, G, smem, s);
    case 2048 * 10000 + 768: return launch_route<16, 24>(a, G, smem, s);
    case 2048 * 10000 + 512: return launch_route<16, 16>(a, G, smem, s);
    case 2048 * 10000 + 1024: return launch_route<16, 32>(a, G, smem, s);
    default: return MOE_ERR_UNSUPPORTED;
    }
}

}  // namespace moe

MOE_API moe_status_t moe_debug_exchange_stall(int32_t on)
{
    if (on != 0 && on != 1)
        return MOE_ERR_INVALID_ARG;
    moe::g_stall.store(on, std::memory_order_relaxed);
    return MOE_OK;
}
