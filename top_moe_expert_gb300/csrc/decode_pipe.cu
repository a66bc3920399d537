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
//     publishes the valid routes in slot order, then streams this CTA's gate
//     and up rows with cp.async.bulk through a ring of 12 slots of 4 neurons
//     each (192 KB in flight per SM at d = 2048).  Once its last gate/up
//     stage has landed it sends this CTA's rows of every routed expert's down
//     projection to L2 (a bulk prefetch), and once the ring is drained it
//     copies them from L2 into the idle ring.
//   * warp 1: reads the arrival counter's epoch (below) before this CTA can
//     arrive; a CTA with no (route, neuron) pair arrives at once.
//   * warps 2..17, gate/up: 4 groups of 4 warps.  Group g takes stages g,
//     g+4, g+8, ...; its warps split K, each holding its slice of x in
//     registers (fp16 after an exact power-of-two rescale), and form the
//     slice's partial dot products with mixed fp16 x fp16 -> FP32 FMAs.  The
//     group adds the partials in a fixed order, forms h = SiLU(g) * u in
//     FP32 and writes it to the workspace; the CTA's last h arrives on the
//     counter.
//   * warps 18..25: load the E8M0 rows of this CTA's gate/up neurons (before
//     the first stage is consumed) and of its down-projection rows, then one
//     lane waits until every CTA has arrived and copies all of h into
//     shared memory in one bulk copy.
// Tail: the 24 compute warps form this CTA's output rows of every route's
// down projection (h as fp16 after an exact power-of-two rescale per route,
// one warp per (route, row), butterfly sums); y is the
// routing-weighted sum over routes in slot order.  The (route, neuron) space
// is split evenly over the CTAs and each CTA owns d / G output rows, so no
// output is reduced across CTAs.
//
// Arrival counter (the first 8 bytes of the workspace, zero before the first
// use): it only grows; every launch adds exactly one per CTA, so between
// launches it is a multiple of the grid size.  A CTA reads it before it
// arrives; the count rounded down to a multiple of the grid is the epoch, and
// every CTA has arrived once the count reaches the epoch plus the grid size.
// All CTAs must be resident together: the grid is one CTA per SM, and
// dependent launches start only after this CTA has seen every arrival.
// Every output's summation order depends only on the shapes and the grid,
// so repeats are bit-identical.
#include <atomic>

#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {
namespace dp {

constexpr int kMaxK = 32;
constexpr int kGW = 4;                                // warps of a gate/up group (they split K)
constexpr int kGroups = 4;                            // gate/up groups
constexpr int kPS = 4;                                // neurons per gate/up stage
constexpr int kSlots = 3 * kGroups;                   // gate/up ring: three slots per group
constexpr int kTW = 8;                                // warps of the wait/copy role
constexpr int kWarpGU0 = 2;
constexpr int kWarpT0 = kWarpGU0 + kGW * kGroups;     // 18
constexpr int kWarps = kWarpT0 + kTW;                 // 26
constexpr int kThreads = kWarps * 32;                 // 832
constexpr int kCW = kWarps - kWarpGU0;                // compute warps of the tail: 24
constexpr uint64_t kWaitNs = 2000000000ull;           // 2 s
constexpr int kBarRoutes = 1;                         // named barriers: routes published (all warps)
constexpr int kBarTail = 2;                           //   the compute warps
constexpr int kBarGroup0 = 3;                         //   gate/up group g: kBarGroup0 + g
constexpr int kBarRank = kBarGroup0 + kGroups;        //   the compute warps ranking the logits
constexpr int kBarScales = kBarRank + 1;              //   gate/up E8M0 rows staged (wait/copy warps arrive)
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
    unsigned long long *ctr;     // arrival counter
    float *h;                    // [kMaxK][I]
    void *y;
    int32_t *dev_status;
    int y_f32, k, d, I, E;
    int shortfall;               // arrivals the counter wait expects beyond the grid (failure-detection test)
};

// Shared-memory plan (bytes), identical on host and device.  The tail's h and
// down-projection rows reuse the gate/up ring, which is idle by then.
struct Plan {
    int d, I, k, G;
    __host__ __device__ int rows_max() const { return (d + G - 1) / G; }
    __host__ __device__ int s1() const { return kPS * 2 * d; }                   // gate rows | up rows
    __host__ __device__ int pmax() const { return (k * I + G - 1) / G; }        // pairs of a CTA, at most
    __host__ __device__ int s2() const { return rows_max() * I; }
    __host__ __device__ static int up16(int v) { return (v + 15) & ~15; }
    __host__ __device__ int o_w2() const { return up16(k * I * 4); }            // in the ring, after h
    __host__ __device__ int o_hh() const { return o_w2() + k * s2(); }          // in the ring: h as fp16
    __host__ __device__ int o_s2s() const { return kSlots * s1(); }
    __host__ __device__ int o_gsc() const { return o_s2s() + k * rows_max() * (I / 32) * 4; }
    __host__ __device__ int o_gpart() const { return o_gsc() + up16(pmax() * 2 * (d / 32)); }
    __host__ __device__ int o_dpart() const { return o_gpart() + kGroups * 2 * kGW * 2 * kPS * 4; }
    __host__ __device__ int o_bars() const { return o_dpart() + up16(k * rows_max() * 4 + k * 4); }  // + 1/scale of h
    __host__ __device__ int o_route() const { return o_bars() + (2 * kSlots + k + 1) * 8; }
    // route data: r_e[kMaxK] | r_w[kMaxK] | r_l[kMaxK] | target u64 | nv, done, abort, tabort, gabort[kGroups]
    __host__ __device__ int bytes() const { return o_route() + 3 * kMaxK * 4 + 8 + 16 + kGroups * 4; }
    __host__ __device__ bool fits() const { return bytes() <= kSmemMax && o_hh() + k * I * 2 <= kSlots * s1(); }
};

__device__ __forceinline__ void set_err(int32_t *st, int code)
{
    if (st)
        atomicCAS(st + 1, 0, code);
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(uint32_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two)));
    return r;
}

// acc + w.lo * a.lo + w.hi * a.hi: fp16 products exact in FP32, one rounding each
__device__ __forceinline__ float fma2(uint32_t w, uint32_t a, float acc)
{
    asm("{\n .reg .f16 w0, w1, a0, a1;\n mov.b32 {w0, w1}, %1;\n mov.b32 {a0, a1}, %2;\n"
        " fma.rn.f32.f16 %0, w0, a0, %0;\n fma.rn.f32.f16 %0, w1, a1, %0;\n}"
        : "+f"(acc) : "r"(w), "r"(a));
    return acc;
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

// Sum over 8 values of 32 lanes at once: lane l ends with the total of value
// v_index(l) = 4 * bit4(l) + 2 * bit3(l) + bit2(l) in every lane of its quad.
__device__ __forceinline__ float reduce8(const float (&v)[8], int lane)
{
    float u[4], t[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? v[i] : v[i + 4];
        u[i] = (b4 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? u[i] : u[i + 2];
        t[i] = (b3 ? u[i + 2] : u[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float r = (b2 ? t[1] : t[0]) + __shfl_xor_sync(0xffffffffu, b2 ? t[0] : t[1], 4);
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}

// exponent p with m * 2^p in [2^14, 2^15) for a finite m > 0 (the largest
// magnitude of a vector); 0 for m == 0
__device__ __forceinline__ int f16_shift(float m)
{
    if (!(m > 0.f))
        return 0;
    int ex;
    frexpf(m, &ex);            // m = f * 2^ex, f in [0.5, 1)
    const int p = 15 - ex;
    return p < -100 ? -100 : (p > 100 ? 100 : p);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(unsigned long long *p)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

__device__ __forceinline__ void red_relaxed_add(unsigned long long *p)
{
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_cta(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
                 : "=r"(old) : "r"(tc::smem_u32(p)), "r"(v) : "memory");
    return old;
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
    const int RM = pl.rows_max(), S1 = pl.s1(), S2 = pl.s2();
    uint8_t *slot1 = smem;
    float *hbuf = reinterpret_cast<float *>(smem);                       // [nv][I], the tail's h
    uint8_t *slot2 = smem + pl.o_w2();                                   // the tail's [k][RM][I] down rows
    float *s2s = reinterpret_cast<float *>(smem + pl.o_s2s());           // [k][RM][I/32] down scales
    uint8_t *gsc = smem + pl.o_gsc();                                    // [P][2][d/32] gate/up E8M0 rows
    float *gpart = reinterpret_cast<float *>(smem + pl.o_gpart());       // [grp][2][kGW][2 kPS]
    float *dpart = reinterpret_cast<float *>(smem + pl.o_dpart());       // [k][RM]
    const uint32_t full1 = tc::smem_u32(smem + pl.o_bars());
    const uint32_t empty1 = full1 + 8 * kSlots, full2 = empty1 + 8 * kSlots, hbar = full2 + 8 * k;
    int *r_e = reinterpret_cast<int *>(smem + pl.o_route());
    float *r_w = reinterpret_cast<float *>(r_e + kMaxK);
    float *r_l = r_w + kMaxK;                                            // logits of the chosen routes
    unsigned long long *target = reinterpret_cast<unsigned long long *>(r_l + kMaxK);
    int *s_nv = reinterpret_cast<int *>(target + 1);
    uint32_t *s_done = reinterpret_cast<uint32_t *>(s_nv + 1);            // neurons of this CTA with h written
    volatile int *s_abort = s_nv + 2;
    volatile int *tabort = s_nv + 3;                                     // decided before the first tail barrier
    volatile int *gabort = s_nv + 4;                                     // [kGroups]

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---------------------------------------------------------------- set-up
    if (warp == 0) {
        if (lane == 0) {
            for (int i = 0; i < kSlots; ++i) {
                tc::mbar_init(full1 + 8 * i, 1);
                tc::mbar_init(empty1 + 8 * i, kGW);
            }
            for (int i = 0; i <= k; ++i)
                tc::mbar_init(full2 + 8 * i, 1);                   // k down slots, then h of the tail
            *s_abort = 0;
            *tabort = 0;
            *s_done = 0;
            for (int g = 0; g < kGroups; ++g)
                gabort[g] = 0;
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
            if (lane == 0) {
                *s_nv = __popc(vm);
                if (c == 0 && k > __popc(vm) && a.dev_status)
                    atomicAdd(a.dev_status, k - __popc(vm));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // the arrival counter's epoch, read before this CTA arrives
            const unsigned long long v = ld_relaxed_u64(a.ctr);
            *target = v / static_cast<unsigned>(G) * static_cast<unsigned>(G) + static_cast<unsigned>(G) +
                  static_cast<unsigned>(a.shortfall);
        }
    } else if constexpr (ROUTE) {
        // top-k of the router logits by rank: thread e (of the 24 compute
        // warps) holds expert e's order-preserving key; its slot is the
        // number of experts ahead of it -- larger logit, or equal logit and
        // lower id -- which is the order the top-k routing defines.  The
        // keys sit in the gate/up ring, idle until the routes are out.
        uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
        const int e = tid - kWarpGU0 * 32, Ep = (a.E + 3) & ~3;
        float l = 0.f;
        if (e < a.E)
            l = __ldcg(a.logits + e);
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
    tc::named_bar(kBarRoutes, kThreads);

    const int nv = *s_nv;
    // this CTA's (route, neuron) pairs: a contiguous range of q = r * I + n,
    // the whole space split evenly over the CTAs (h[q] is written here)
    const int q_lo = static_cast<int>(static_cast<int64_t>(nv) * I * c / G);
    const int P = static_cast<int>(static_cast<int64_t>(nv) * I * (c + 1) / G) - q_lo;
    const int S = (P + kPS - 1) / kPS;                                              // gate/up stages
    const int o0 = static_cast<int>(static_cast<int64_t>(d) * c / G);
    const int nrows = static_cast<int>(static_cast<int64_t>(d) * (c + 1) / G) - o0;

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            const int64_t rowb = d;
            tc::fence_proxy_async_smem();          // the ring held the routing's keys
            bool go = true;
            int s = 0;
            for (; s < S; ++s) {
                const int sl = s % kSlots;
                const uint32_t ph = (s / kSlots) & 1u;
                if (!tc::mbar_wait(empty1 + 8 * sl, ph ^ 1u, s_abort, kWaitNs)) {
                    go = false;
                    break;
                }
                const int q0 = q_lo + s * kPS, q1 = q_lo + min(s * kPS + kPS, P);
                tc::mbar_arrive_expect_tx(full1 + 8 * sl, static_cast<uint32_t>(q1 - q0) * (2 * d));
                uint8_t *st = slot1 + sl * S1;
                const uint32_t bar = full1 + 8 * sl;
                for (int q = q0; q < q1;) {
                    // a run of neurons of one route: gate rows, up rows
                    const int r = q / I, n = q - r * I, len = min(q1 - q, I - n), i = q - q0;
                    const int64_t grow = static_cast<int64_t>(r_e[r]) * 2 * I + n;
                    tc::bulk_load(tc::smem_u32(st + i * rowb), a.q13 + grow * rowb, len * rowb, bar);
                    tc::bulk_load(tc::smem_u32(st + (kPS + i) * rowb), a.q13 + (grow + I) * rowb, len * rowb, bar);
                    q += len;
                }
            }
            // this CTA's down-projection rows of every routed expert go to L2
            // once its last gate/up stage has landed: they stream while h is
            // formed and exchanged, and do not slow the gate/up stream
            if (go && S > 0)
                go = tc::mbar_wait(full1 + 8 * ((S - 1) % kSlots), ((S - 1) / kSlots) & 1u, s_abort, kWaitNs);
            if (go && nrows > 0)
                for (int r = 0; r < nv; ++r)
                    tc::bulk_prefetch_l2(a.q2 + (static_cast<int64_t>(r_e[r]) * d + o0) * I, nrows * I);
            // once every gate/up stage is consumed the ring is idle: the down
            // rows move from L2 into it while the grid's last CTAs finish
            for (int t = max(0, s - kSlots); t < s && go; ++t)
                go = tc::mbar_wait(empty1 + 8 * (t % kSlots), (t / kSlots) & 1u, s_abort, kWaitNs);
            if (go && nrows > 0) {
                tc::fence_proxy_async_smem();
                for (int r = 0; r < nv; ++r) {
                    tc::mbar_arrive_expect_tx(full2 + 8 * r, static_cast<uint32_t>(nrows * I));
                    tc::bulk_load(tc::smem_u32(slot2 + r * S2), a.q2 + (static_cast<int64_t>(r_e[r]) * d + o0) * I,
                                  nrows * I, full2 + 8 * r);
                }
            }
            // every issued copy lands before the CTA may finish
            volatile int never = 0;
            for (int t = max(0, s - kSlots); t < s; ++t)
                tc::mbar_wait(full1 + 8 * (t % kSlots), (t / kSlots) & 1u, &never, kWaitNs);
            if (go && nrows > 0)
                for (int r = 0; r < nv; ++r)
                    tc::mbar_wait(full2 + 8 * r, 0, &never, kWaitNs);
        }
        return;
    }
    if (warp == 1) {
        // nothing to compute here: arrive at once
        if (lane == 0 && P == 0)
            red_release_add(a.ctr);
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
        tc::named_bar(kBarScales, kCW * 32);               // the E8M0 rows are staged
        for (int s = grp, m = 0; s < S; s += kGroups, ++m) {
            const int sl = s % kSlots, buf = m & 1;
            const uint32_t ph = (s / kSlots) & 1u;
            const bool got = tc::mbar_wait(full1 + 8 * sl, ph, s_abort, kWaitNs);
            if (!got)
                gabort[grp] = 1;
            const int npairs = min(kPS, P - s * kPS);
            if (got) {
                const uint8_t *st = slot1 + sl * S1;
                float v[2 * kPS];
#pragma unroll
                for (int i = 0; i < 2 * kPS; ++i) {
                    v[i] = 0.f;
                    if (i % kPS < npairs) {
                        uint32_t wq[KPL / 4];
                        lds_codes<KPL>(st + i * d + kbase, wq);
                        float acc = 0.f;
#pragma unroll
                        for (int t = 0; t < KPL / 4; ++t)
                            acc = dot4(wq[t], xw[2 * t], xw[2 * t + 1], acc);
                        // E8M0 of pair s*kPS + i%kPS, gate (i < kPS) or up row, this lane's block
                        v[i] = acc * e8m0_to_float(gsc[((s * kPS + i % kPS) * 2 + i / kPS) * sclb + (kbase >> 5)]);
                    }
                }
                const float tot = reduce8(v, lane) * xinv;
                if ((lane & 3) == 0) {
                    const int vi = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                    gpart[((grp * 2 + buf) * kGW + om) * 2 * kPS + vi] = tot;
                }
            }
            tc::named_bar(kBarGroup0 + grp, kGW * 32);
            if (gabort[grp]) {
                *tabort = 1;
                break;
            }
            if (lane == 0)
                tc::mbar_arrive(empty1 + 8 * sl);
            if (om == 0 && lane < npairs) {
                // h of neuron `lane` of the stage: partials added in warp order
                const float *gp = gpart + (grp * 2 + buf) * kGW * 2 * kPS;
                float g = gp[lane], u = gp[kPS + lane];
#pragma unroll
                for (int w2 = 1; w2 < kGW; ++w2) {
                    g += gp[w2 * 2 * kPS + lane];
                    u += gp[w2 * 2 * kPS + kPS + lane];
                }
                __stcg(a.h + q_lo + s * kPS + lane, silu_mul(g, u));
                if (atom_add_acq_rel_cta(s_done, 1u) + 1u == static_cast<uint32_t>(P))
                    // every h of this CTA is written (the CTA-scope acquire above
                    // orders the other lanes' stores before this release): arrive
                    red_release_add(a.ctr);
            }
        }
    } else {
        // ------------------------------------------------ wait/copy warps
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
            tc::named_arrive(kBarScales, kCW * 32);
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
        if (tw == 0 && lane == 0) {
            // every CTA has written its share of h (one lane polls, with a
            // short back-off, so that the L2 slice holding the counter keeps
            // serving the stream), then h comes to shared memory in one copy
            const unsigned long long want = *target;
            const uint64_t t0 = tc::globaltimer_ns();
            bool ok = true;
            for (uint32_t it = 0; ld_relaxed_u64(a.ctr) < want; ++it) {
                __nanosleep(64);
                if ((it & 15u) == 15u && (*s_abort || tc::globaltimer_ns() - t0 > kWaitNs)) {
                    ok = false;
                    break;
                }
            }
            if (ok) {
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
                if (nv > 0 && nrows > 0) {
                    tc::fence_proxy_async_smem();
                    tc::mbar_arrive_expect_tx(hbar, static_cast<uint32_t>(nv * I * 4));
                    tc::bulk_load(tc::smem_u32(hbuf), a.h, nv * I * 4, hbar);
                }
            } else {
                *s_abort = 1;
                *tabort = 1;
                set_err(a.dev_status, MOE_ERR_TIMEOUT);
            }
        }
    }

    // ---------------------------------------------------------------- tail
    tc::named_bar(kBarTail, kCW * 32);
    const bool work = !*tabort && nv > 0 && nrows > 0;
    const bool got = work && tc::mbar_wait(hbar, 0, s_abort, kWaitNs);
    if (work && !got)
        set_err(a.dev_status, MOE_ERR_TIMEOUT);
    // h of every route once, by one warp per route: fp16 after an exact
    // power-of-two rescale that puts the route's largest magnitude in
    // [2^14, 2^15) (relative rounding at most 2^-12 of each element)
    __half2 *h16 = reinterpret_cast<__half2 *>(slot1 + pl.o_hh());        // [nv][I/2]
    float *hinv = dpart + pl.k * RM;                                     // [nv]
    for (int r = cw; got && r < nv; r += kCW) {
        float hv[HPL];
        const float4 *hp = reinterpret_cast<const float4 *>(hbuf + r * I + HPL * lane);
#pragma unroll
        for (int i = 0; i < HPL / 4; ++i) {
            const float4 f = hp[i];
            hv[4 * i] = f.x; hv[4 * i + 1] = f.y; hv[4 * i + 2] = f.z; hv[4 * i + 3] = f.w;
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < HPL; ++i)
            m = fmaxf(m, fabsf(hv[i]));
        const int pw = f16_shift(warp_max(m));
        const float sc = ldexpf(1.0f, pw);
        if (lane == 0)
            hinv[r] = ldexpf(1.0f, -pw);
#pragma unroll
        for (int i = 0; i < HPL / 2; ++i)
            h16[(r * I + HPL * lane) / 2 + i] = __floats2half2_rn(hv[2 * i] * sc, hv[2 * i + 1] * sc);
    }
    tc::named_bar(kBarTail, kCW * 32);
    if (got) {
        // the (route, row) units of this CTA, a contiguous block per warp
        const int U = nv * nrows, nb2 = I / 32;
        const int u0 = U * cw / kCW, u1 = U * (cw + 1) / kCW;
        int cur = -1;
        uint32_t hh[HPL / 2];
        float inv = 1.f;
        for (int u = u0; u < u1;) {
            const int r = u / nrows, rho = u - r * nrows;
            if (r != cur) {
                cur = r;
                if (!tc::mbar_wait(full2 + 8 * r, 0, s_abort, kWaitNs)) {
                    set_err(a.dev_status, MOE_ERR_TIMEOUT);
                    break;
                }
                const uint4 *ph = reinterpret_cast<const uint4 *>(h16 + (r * I + HPL * lane) / 2);
#pragma unroll
                for (int i = 0; i < HPL / 8; ++i) {
                    const uint4 v = ph[i];
                    hh[4 * i] = v.x; hh[4 * i + 1] = v.y; hh[4 * i + 2] = v.z; hh[4 * i + 3] = v.w;
                }
                inv = hinv[r];
            }
            // two rows of the same route at once when the block has them
            const bool two = u + 1 < u1 && rho + 1 < nrows;
            const int rho1 = two ? rho + 1 : rho;
            const uint8_t *w0 = slot2 + r * S2 + rho * I + HPL * lane;
            const uint8_t *w1 = slot2 + r * S2 + rho1 * I + HPL * lane;
            const float *sr0 = s2s + (r * RM + rho) * nb2 + ((HPL * lane) >> 5);
            const float *sr1 = s2s + (r * RM + rho1) * nb2 + ((HPL * lane) >> 5);
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < HPL / 8; ++c8) {
                const uint2 q0 = *reinterpret_cast<const uint2 *>(w0 + 8 * c8);
                const uint2 q1 = *reinterpret_cast<const uint2 *>(w1 + 8 * c8);
                const int sb = (((HPL * lane) & 31) + 8 * c8) >> 5;
                float p0 = 0.f, p1 = 0.f;
                uint32_t a[4], b[4];
                cvt_e4m3x4(q0.x, a[0], a[1]);
                cvt_e4m3x4(q0.y, a[2], a[3]);
                cvt_e4m3x4(q1.x, b[0], b[1]);
                cvt_e4m3x4(q1.y, b[2], b[3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p0 = fma2(a[i], hh[4 * c8 + i], p0);
                    p1 = fma2(b[i], hh[4 * c8 + i], p1);
                }
                acc0 = fmaf(p0, sr0[sb], acc0);
                acc1 = fmaf(p1, sr1[sb], acc1);
            }
            // both sums at once: lanes 0..15 end with row rho's, 16..31 with rho1's
            const bool up = lane & 16;
            float t = (up ? acc1 : acc0) + __shfl_xor_sync(0xffffffffu, up ? acc0 : acc1, 16);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                t += __shfl_xor_sync(0xffffffffu, t, o);
            if (lane == 0)
                dpart[r * RM + rho] = t * inv;
            if (two && lane == 16)
                dpart[r * RM + rho1] = t * inv;
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

// Arrivals the next launches' counter wait expects beyond the grid size: 0
// in normal use; moe_debug_arrival_shortfall sets it so that a test can make
// the wait run out (it gives up after its time limit and reports
// MOE_ERR_TIMEOUT) without faulting or hanging the GPU.
static std::atomic<int> g_shortfall{0};

bool decode_pipe_shape_fits(int k, int d, int I, int G)
{
    return k >= 1 && k <= dp::kMaxK && G >= 1 && dp::shape_ok(d, I) && dp::Plan{d, I, k, G}.fits();
}

bool decode_pipe_eligible(int M, int k, int d, int I, int E)
{
    return M == 1 && E >= 1 && decode_pipe_shape_fits(k, d, I, device_sm_count());
}

bool decode_pipe_route_eligible(int E, int k) { return E >= k && E <= dp::kCW * 32; }

size_t decode_pipe_workspace(int k, int I)
{
    return kWsReserved + ws_round(static_cast<size_t>(k) * I * sizeof(float));
}

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
    a.h = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kWsReserved);
    a.y = y;
    a.dev_status = dev_status;
    a.y_f32 = y_f32 ? 1 : 0;
    a.k = k;
    a.d = d;
    a.I = I;
    a.E = E;
    a.shortfall = g_shortfall.load(std::memory_order_relaxed);
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

MOE_API moe_status_t moe_debug_arrival_shortfall(int32_t n)
{
    if (n < 0 || n > 1024)
        return MOE_ERR_INVALID_ARG;
    moe::g_shortfall.store(n, std::memory_order_relaxed);
    return MOE_OK;
}
