// decode_m1.cu -- single-token decode (M = 1) as one streaming kernel.
//
// The mathematics is the output-centric decode of "Warp decode" (cursor.com
// blog, sections on what changed and how the two kernels work): for each
// routed expert g = W_gate x, u = W_up x, h = SiLU(g) * u, and
// y = sum_j w_j * W2_{e_j} h_j with the routing weight folded in, MXFP8
// weights converted on the fly, FP32 accumulation, no alignment, padding,
// scatter or combine buffers.
//
// At M = 1 the layer is a pure HBM stream of k experts' weights (38.9 MB at
// d = 2048, I = 768, k = 8).  Design:
//   * One CTA per SM owns an exactly balanced range of the (route, neuron)
//     space.  A producer warp issues, per stage of up to 8 neurons, their
//     gate rows, up rows, down-projection columns (neuron-major W2), the
//     E8M0 rows of gate and up, and -- when the stage opens a 32-neuron
//     block -- the block's E8M0 row of the down projection, with
//     cp.async.bulk into a ring of 4 stages (about 200 KB): most of a CTA's
//     share is requested at once.
//   * 16 compute warps.  Dot phase: warp w forms one row's dot product
//     (gate row of neuron w, or up row of neuron w - 8) with the token's
//     activation slice held in registers (fp16 after an exact power-of-two
//     rescale; mixed fma.rn.f32.f16 products, FP32 sums) and a butterfly.
//     One barrier among the compute warps hands g and u over through shared
//     memory.  Outer phase: warp w owns outputs [w d/16, (w+1) d/16); each
//     lane forms h of one of the stage's neurons, the warp broadcasts them
//     and adds h_n * W2[o][n] for the stage's neurons into per-lane FP32
//     accumulators of the current block; the block's E8M0 scales are applied
//     once, when the block closes.
//   * Each CTA writes its partial of y; a grid-wide barrier (bounded spin
//     on a 64-bit arrival counter in the workspace) then lets each CTA
//     reduce a slice of outputs over all CTAs in a fixed order and write y.
//     The counter is never reset: every launch adds exactly one arrival per
//     CTA, so a CTA that draws arrival number a waits for the count to reach
//     the next multiple of the grid size above a (the counter starts at 0).
// The CTAs of the grid must be resident together: the grid is one CTA per SM
// and the kernel lets dependent launches start only after the barrier.
#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "tc.cuh"
#include "topk.cuh"

namespace moe {
namespace dm {

constexpr int kR = 8;                           // neurons per stage
constexpr int kWarps = 2 * kR;                  // compute warps: one row (gate or up) each per stage
constexpr int kThreads = (kWarps + 1) * 32;     // + producer warp
constexpr int kStages = 4;
constexpr int kMaxK = 32;
constexpr uint64_t kWaitNs = 2000000000ull;     // 2 s

struct Args {
    const __nv_bfloat16 *x;
    const int32_t *ids;          // routes given: ids / weights [k]
    const float *wts;
    const float *logits;         // or routed here: router logits [E] ...
    int32_t *ids_out;            // ... and the chosen ids / weights written by CTA 0
    float *wts_out;
    const uint8_t *q13, *s13;    // [E][2I][d], [E][2I][d/32]
    const uint8_t *q2t, *s2t;    // [E][I][d],  [E][I/32][d]
    unsigned long long *bar;     // arrivals: every launch adds one per CTA (starts at 0)
    float *partial;              // [G][d]
    void *y;
    int32_t *dev_status;
    int y_f32, k, d, I, E;
};

// stage layout: gate rows | up rows | W2 columns | gate E8M0 | up E8M0 |
// W2 E8M0 row of the block the stage opens | of the block it crosses into
struct Geo {
    int d;
    __host__ __device__ int gate_off() const { return 0; }
    __host__ __device__ int up_off() const { return kR * d; }
    __host__ __device__ int w2_off() const { return 2 * kR * d; }
    __host__ __device__ int gs_off() const { return 3 * kR * d; }
    __host__ __device__ int us_off() const { return 3 * kR * d + kR * (d / 32); }
    __host__ __device__ int s2_off() const { return 3 * kR * d + 2 * kR * (d / 32); }
    __host__ __device__ int bytes() const { return 3 * kR * d + 2 * kR * (d / 32) + 2 * d; }
};

__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(two)));
    return r;
}

// d = a * b + c, a and b fp16 (exact in fp32), c and d fp32: one rounding
__device__ __forceinline__ float fma_h(uint16_t a, uint16_t b, float c)
{
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}

// sum of 16 products: E4M3 codes q with fp16 activations (8 half2 words)
__device__ __forceinline__ float dot16(const uint4 q, const uint32_t *xw)
{
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;     // four short chains
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = e4m3x2_f16x2(qw[i] & 0xFFFFu), hi = e4m3x2_f16x2(qw[i] >> 16);
        a0 = fma_h(static_cast<uint16_t>(lo), static_cast<uint16_t>(xw[2 * i]), a0);
        a1 = fma_h(static_cast<uint16_t>(lo >> 16), static_cast<uint16_t>(xw[2 * i] >> 16), a1);
        a2 = fma_h(static_cast<uint16_t>(hi), static_cast<uint16_t>(xw[2 * i + 1]), a2);
        a3 = fma_h(static_cast<uint16_t>(hi >> 16), static_cast<uint16_t>(xw[2 * i + 1] >> 16), a3);
    }
    return (a0 + a1) + (a2 + a3);
}

// SiLU(g) * u with the fast exponential and divide (a few ulp of fp32)
__device__ __forceinline__ float silu_mul_fast(float g, float u)
{
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ float e8m0f(uint32_t s)
{
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t h2)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// neurons [n, n + nr) of the next stage: at most kR, never across a route,
// never past the CTA's range (a stage may straddle one 32-neuron scale block
// boundary: kR < 32)
__device__ __forceinline__ int stage_rows(int n, int left, int I)
{
    int nr = kR;
    nr = nr < I - n ? nr : I - n;
    return nr < left ? nr : left;
}

__device__ __forceinline__ void set_status(int32_t *dev_status, int code)
{
    if (dev_status)
        atomicCAS(dev_status + 1, 0, code);
}

// The stage sequence of a CTA, walked identically by the producer and the
// compute warps.
struct StageIt {
    int p, n, r, nr, s;
    uint32_t ph;
    bool opens;      // the stage's first neuron starts a 32-neuron block in this CTA
    int cross;       // > 0: neuron `cross` of the stage starts the next block
    __device__ __forceinline__ void init(int p0, int p1, int I)
    {
        p = p0;
        r = p0 / I;
        n = p0 - r * I;
        s = 0;
        ph = 0;
        opens = true;
        // the range's remainder rows (beyond a multiple of kR) form the first
        // stage: that short stage lands early and frees its slot for a full
        // one, so a CTA with one row more than its neighbours does not wait
        // an extra stage round trip at the end
        const int f = (p1 - p0) % kR;
        nr = p < p1 ? stage_rows(n, f ? f : kR, I) : 0;
        cross = (n & 31) + nr > 32 ? 32 - (n & 31) : 0;
    }
    __device__ __forceinline__ void next(int p1, int I)
    {
        p += nr;
        n += nr;
        if (n == I) {
            n = 0;
            ++r;
        }
        if (++s == kStages) {
            s = 0;
            ph ^= 1u;
        }
        opens = (n & 31) == 0;
        nr = p < p1 ? stage_rows(n, p1 - p, I) : 0;
        cross = (n & 31) + nr > 32 ? 32 - (n & 31) : 0;
    }
};

// OPL outputs per lane of a compute warp (d = 512 * OPL); the dot phase uses
// OPL 16-byte chunks per lane of a d-byte row as well.  ROUTE_PL > 0: the
// kernel routes the token itself from its logits (top-k softmax, ROUTE_PL
// logits per lane) instead of reading ids and weights.
template <int OPL, int ROUTE_PL>
__global__ void __launch_bounds__(kThreads, 1) m1_kernel(const Args a)
{
    constexpr int CPL = OPL;
    extern __shared__ __align__(128) uint8_t smem[];
    const int d = a.d, I = a.I;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Geo geo{d};
    uint8_t *stages = smem;
    float *hbuf = reinterpret_cast<float *>(smem + kStages * geo.bytes());  // [2][2][kR] g, u per stage parity
    uint64_t *bars = reinterpret_cast<uint64_t *>(hbuf + 4 * kR);
    int *r_e = reinterpret_cast<int *>(bars + 2 * kStages);       // [kMaxK] expert of valid route i
    float *r_w = reinterpret_cast<float *>(r_e + kMaxK);          // [kMaxK] its routing weight
    int *n_valid = reinterpret_cast<int *>(r_w + kMaxK);          // [1]
    volatile int *abort_flag = n_valid + 1;                       // [1]
    __shared__ int passed;
    const uint32_t full0 = tc::smem_u32(bars), empty0 = full0 + 8 * kStages;

    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the grid barrier's epoch: the arrival counter is a multiple of the grid
    // size between launches, and this CTA has not arrived yet, so the count
    // read now rounds down to the arrivals of earlier launches
    unsigned long long bar_epoch = 0;
    if (tid == 0)
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(bar_epoch) : "l"(a.bar) : "memory");

    if (warp == kWarps) {
        // ------------------------------------------------ producer warp
        int e;
        float w = 0.f, sl = 0.f;
        if constexpr (ROUTE_PL > 0) {
            // the logits are the first bytes the step needs: their loads go
            // out first, the barriers are set up while they arrive; the
            // weights are computed after the first copies are out
            topk_select<ROUTE_PL>(a.logits, a.E, a.k, lane, e, sl, [&] {
                if (lane == 0) {
                    for (int s = 0; s < kStages; ++s) {
                        tc::mbar_init(full0 + 8 * s, 1);
                        tc::mbar_init(empty0 + 8 * s, kWarps);
                    }
                    *abort_flag = 0;
                    tc::fence_mbar_init();
                }
            });
        } else {
            e = lane < a.k ? __ldcg(a.ids + lane) : -1;
            w = lane < a.k ? __ldcg(a.wts + lane) : 0.f;
            if (lane == 0) {
                for (int s = 0; s < kStages; ++s) {
                    tc::mbar_init(full0 + 8 * s, 1);
                    tc::mbar_init(empty0 + 8 * s, kWarps);
                }
                *abort_flag = 0;
                tc::fence_mbar_init();
            }
        }
        const bool ok = lane < a.k && e >= 0 && e < a.E;
        const unsigned vm = __ballot_sync(0xffffffffu, ok);
        const int vi = __popc(vm & ((1u << lane) - 1u));
        if (ok)
            r_e[vi] = e;
        const int nv = __popc(vm);
        if (lane == 0) {
            *n_valid = nv;
            if (blockIdx.x == 0 && a.k > nv && a.dev_status)
                atomicAdd(a.dev_status, a.k - nv);
        }
        __syncwarp();
        // the routing weights, then the compute warps go: done once the
        // first ring-full of copies is out (those need only the expert ids)
        bool released = false;
        auto release = [&] {
            if constexpr (ROUTE_PL > 0) {
                w = topk_weight(sl, a.k, lane);
                if (blockIdx.x == 0 && lane < a.k) {
                    if (a.ids_out)
                        a.ids_out[lane] = e;
                    if (a.wts_out)
                        a.wts_out[lane] = w;
                }
            }
            if (ok)
                r_w[vi] = w;
            __syncwarp();
            tc::named_arrive(2, kThreads);
            released = true;
        };
        const unsigned Ptot = static_cast<unsigned>(nv) * I;
        const int p0 = static_cast<int>(Ptot * blockIdx.x / gridDim.x);
        const int p1 = static_cast<int>(Ptot * (blockIdx.x + 1) / gridDim.x);
        StageIt it;
        it.init(p0, p1, I);
        int issued = 0;
        for (; it.p < p1; it.next(p1, I), ++issued) {
            if (issued == kStages && !released)
                release();
            int go = 1;
            if (lane == 0) {
                go = tc::mbar_wait(empty0 + 8 * it.s, it.ph ^ 1u, abort_flag, kWaitNs) ? 1 : 0;
                if (go)
                    tc::mbar_arrive_expect_tx(full0 + 8 * it.s, static_cast<uint32_t>(it.nr) * (3 * d + 2 * (d / 32)) +
                                                                    (it.opens ? d : 0) + (it.cross ? d : 0));
            }
            if (!__shfl_sync(0xffffffffu, go, 0))
                break;
            if (issued == kStages && lane == 0) {
                // the ring is full: pull every later stage's bytes into L2 now
                // (the TMA prefetch takes no shared memory), so that the copies
                // that refill the ring hit L2
                StageIt pf = it;
                for (; pf.p < p1; pf.next(p1, I)) {
                    const int ex = r_e[pf.r];
                    const int64_t grow = static_cast<int64_t>(ex) * 2 * I + pf.n;
                    tc::bulk_prefetch_l2(a.q13 + grow * d, pf.nr * d);
                    tc::bulk_prefetch_l2(a.q13 + (grow + I) * d, pf.nr * d);
                    tc::bulk_prefetch_l2(a.q2t + (static_cast<int64_t>(ex) * I + pf.n) * d, pf.nr * d);
                    tc::bulk_prefetch_l2(a.s13 + grow * (d / 32), pf.nr * (d / 32));
                    tc::bulk_prefetch_l2(a.s13 + (grow + I) * (d / 32), pf.nr * (d / 32));
                    if (pf.opens)
                        tc::bulk_prefetch_l2(a.s2t + (static_cast<int64_t>(ex) * (I / 32) + (pf.n >> 5)) * d, d);
                    if (pf.cross)
                        tc::bulk_prefetch_l2(a.s2t + (static_cast<int64_t>(ex) * (I / 32) + (pf.n >> 5) + 1) * d, d);
                }
            }
            // gate rows, up rows, W2 columns, gate E8M0, up E8M0, and the
            // block's W2 E8M0 row when the stage opens a block
            if (lane == 0) {
                const int ex = r_e[it.r];
                uint8_t *st = stages + it.s * geo.bytes();
                const uint32_t b = full0 + 8 * it.s;
                const int64_t grow = static_cast<int64_t>(ex) * 2 * I + it.n;
                tc::bulk_load(tc::smem_u32(st + geo.gate_off()), a.q13 + grow * d, it.nr * d, b);
                tc::bulk_load(tc::smem_u32(st + geo.up_off()), a.q13 + (grow + I) * d, it.nr * d, b);
                tc::bulk_load(tc::smem_u32(st + geo.w2_off()), a.q2t + (static_cast<int64_t>(ex) * I + it.n) * d,
                              it.nr * d, b);
                tc::bulk_load(tc::smem_u32(st + geo.gs_off()), a.s13 + grow * (d / 32), it.nr * (d / 32), b);
                tc::bulk_load(tc::smem_u32(st + geo.us_off()), a.s13 + (grow + I) * (d / 32), it.nr * (d / 32), b);
                if (it.opens)
                    tc::bulk_load(tc::smem_u32(st + geo.s2_off()),
                                  a.s2t + (static_cast<int64_t>(ex) * (I / 32) + (it.n >> 5)) * d, d, b);
                if (it.cross)
                    tc::bulk_load(tc::smem_u32(st + geo.s2_off() + d),
                                  a.s2t + (static_cast<int64_t>(ex) * (I / 32) + (it.n >> 5) + 1) * d, d, b);
            }
            __syncwarp();
        }
        if (!released)
            release();
        // every issued copy lands before the CTA may finish
        if (lane == 0) {
            volatile int never = 0;
            const int nq = issued < kStages ? issued : kStages;
            for (int i = 1; i <= nq; ++i) {
                int st = it.s - i;
                uint32_t pp = it.ph;
                if (st < 0) {
                    st += kStages;
                    pp ^= 1u;
                }
                tc::mbar_wait(full0 + 8 * st, pp, &never, kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------ compute warps
        // the token's activations: lane chunk i covers x[16 c .. 16 c + 16),
        // c = 32 i + lane; every warp holds all of x
        uint32_t xw[CPL * 8];
        float xinv;
        {
            uint32_t raw[CPL * 8];
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.x) + 2 * (32 * i + lane);
                const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                raw[i * 8 + 0] = v0.x; raw[i * 8 + 1] = v0.y; raw[i * 8 + 2] = v0.z; raw[i * 8 + 3] = v0.w;
                raw[i * 8 + 4] = v1.x; raw[i * 8 + 5] = v1.y; raw[i * 8 + 6] = v1.z; raw[i * 8 + 7] = v1.w;
            }
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < CPL * 8; ++i)
                m = max(m, max(raw[i] & 0x7FFFu, (raw[i] >> 16) & 0x7FFFu));
            m = __reduce_max_sync(0xffffffffu, m);
            // scale 2^p with amax * 2^p in [2^14, 2^15): exact in fp16 for
            // every element within 2^28 of the largest magnitude
            int pw = 0;
            if (m != 0) {
                const int ef = static_cast<int>(m >> 7);
                pw = ef == 0 ? 100 : 14 - (ef - 127);
                pw = pw < -100 ? -100 : (pw > 100 ? 100 : pw);
            }
            const float sc = ldexpf(1.0f, pw);
            xinv = ldexpf(1.0f, -pw);
#pragma unroll
            for (int i = 0; i < CPL * 8; ++i) {
                const float lo = __uint_as_float(raw[i] << 16) * sc, hi = __uint_as_float(raw[i] & 0xFFFF0000u) * sc;
                const __half2 h2 = __floats2half2_rn(lo, hi);
                xw[i] = *reinterpret_cast<const uint32_t *>(&h2);
            }
        }
        tc::named_bar(2, kThreads);          // routes and barriers from the producer
        const int nv = *n_valid;
        const unsigned Ptot = static_cast<unsigned>(nv) * I;
        const int p0 = static_cast<int>(Ptot * blockIdx.x / gridDim.x);
        const int p1 = static_cast<int>(Ptot * (blockIdx.x + 1) / gridDim.x);

        const int row = warp >> 3;           // 0 gate, 1 up
        const int wn = warp & 7;             // neuron of a stage whose row this warp takes
        const int obase = warp * (d / kWarps) + OPL * lane;
        float yacc[OPL], tacc[OPL];          // outputs obase + j: total, and the current block unscaled
        uint32_t sblk = 0;                   // E8M0 bytes of the current block for this lane's outputs
#pragma unroll
        for (int j = 0; j < OPL; ++j)
            yacc[j] = tacc[j] = 0.f;

        // dot product of this warp's row in stage `it`, into hbuf[par]
        auto dot_phase = [&](const StageIt &it, int par, bool store) {
            const uint8_t *st = stages + it.s * geo.bytes();
            const uint8_t *wrow = st + (row ? geo.up_off() : geo.gate_off()) + wn * d;
            const uint8_t *srow = st + (row ? geo.us_off() : geo.gs_off()) + wn * (d / 32);
            float part[CPL];
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                const int c = 32 * i + lane;
                const uint4 q = *reinterpret_cast<const uint4 *>(wrow + 16 * c);
                part[i] = dot16(q, xw + 8 * i) * e8m0f(srow[c >> 1]);
            }
            float acc = part[0];
#pragma unroll
            for (int i = 1; i < CPL; ++i)
                acc += part[i];
            acc = warp_sum(acc);
            if (store && lane == 0)
                hbuf[par * 2 * kR + row * kR + wn] = acc;
        };
        // close the current block: its products times its E8M0 scales
        auto close_block = [&]() {
#pragma unroll
            for (int j = 0; j < OPL; ++j) {
                yacc[j] = fmaf(e8m0f((sblk >> (8 * j)) & 0xFFu), tacc[j], yacc[j]);
                tacc[j] = 0.f;
            }
        };
        // this lane's E8M0 bytes of scale row `slot` of stage `it`
        auto scale_row = [&](const StageIt &it, int slot) -> uint32_t {
            const uint8_t *sr = stages + it.s * geo.bytes() + geo.s2_off() + slot * d + obase;
            if constexpr (OPL == 4)
                return *reinterpret_cast<const uint32_t *>(sr);
            else
                return *reinterpret_cast<const uint16_t *>(sr);
        };

        StageIt it;
        it.init(p0, p1, I);
        bool have = false;
        for (int si = 0; it.p < p1; it.next(p1, I), ++si) {
            if (!tc::mbar_wait(full0 + 8 * it.s, it.ph, abort_flag, kWaitNs))
                set_status(a.dev_status, MOE_ERR_TIMEOUT);
            dot_phase(it, si & 1, wn < it.nr);
            if (it.opens) {
                if (have)
                    close_block();
                sblk = scale_row(it, 0);
                have = true;
            }
            const uint32_t sblk_next = it.cross ? scale_row(it, 1) : 0u;
            tc::named_bar(1, kWarps * 32);
            // outer phase: h of neuron `lane` of the stage, then the stage's
            // columns applied to this warp's outputs
            const float *hb = hbuf + (si & 1) * 2 * kR;
            const float hl = lane < it.nr ? r_w[it.r] * silu_mul_fast(hb[lane] * xinv, hb[kR + lane] * xinv) : 0.f;
            const uint8_t *w2 = stages + it.s * geo.bytes() + geo.w2_off() + obase;
            uint32_t qv[kR];
#pragma unroll
            for (int nn = 0; nn < kR; ++nn) {
                if constexpr (OPL == 4)
                    qv[nn] = nn < it.nr ? *reinterpret_cast<const uint32_t *>(w2 + nn * d) : 0u;
                else
                    qv[nn] = nn < it.nr ? *reinterpret_cast<const uint16_t *>(w2 + nn * d) : 0u;
            }
            // the stage's bytes are all in registers or consumed: release it
            __syncwarp();
            if (lane == 0)
                tc::mbar_arrive(empty0 + 8 * it.s);
#pragma unroll
            for (int nn = 0; nn < kR; ++nn) {
                const float h = __shfl_sync(0xffffffffu, hl, nn);
                const float2 hh = make_float2(h, h);
                if (nn > 0 && nn == it.cross) {      // neuron nn starts the next block
                    close_block();
                    sblk = sblk_next;
                }
                if constexpr (OPL == 4) {
                    const float2 lo = half2_to_float2(e4m3x2_f16x2(qv[nn] & 0xFFFFu));
                    const float2 hi = half2_to_float2(e4m3x2_f16x2(qv[nn] >> 16));
                    const float2 t0 = __ffma2_rn(lo, hh, make_float2(tacc[0], tacc[1]));
                    const float2 t1 = __ffma2_rn(hi, hh, make_float2(tacc[2], tacc[3]));
                    tacc[0] = t0.x;
                    tacc[1] = t0.y;
                    tacc[2] = t1.x;
                    tacc[3] = t1.y;
                } else {
                    const float2 lo = half2_to_float2(e4m3x2_f16x2(qv[nn]));
                    const float2 t0 = __ffma2_rn(lo, hh, make_float2(tacc[0], tacc[1]));
                    tacc[0] = t0.x;
                    tacc[1] = t0.y;
                }
            }
        }
        if (have) {
#pragma unroll
            for (int j = 0; j < OPL; ++j)
                yacc[j] = fmaf(e8m0f((sblk >> (8 * j)) & 0xFFu), tacc[j], yacc[j]);
        }
        // this CTA's partial of y
        float *dst = a.partial + static_cast<int64_t>(blockIdx.x) * d + obase;
        if constexpr (OPL == 4)
            __stcg(reinterpret_cast<float4 *>(dst), make_float4(yacc[0], yacc[1], yacc[2], yacc[3]));
        else
            __stcg(reinterpret_cast<float2 *>(dst), make_float2(yacc[0], yacc[1]));
    }

    // ---- grid barrier: every CTA's partial is visible before any is read
    __syncthreads();
    if (tid == 0) {
        // a release add needs no reply: the CTA's partial (ordered before it
        // by the barrier above) is visible to whoever sees the new count
        const unsigned long long G = gridDim.x;
        const unsigned long long target = (bar_epoch / G + 1) * G;
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(a.bar) : "memory");
        const long long t0 = clock64();
        const long long limit = static_cast<long long>(kWaitNs) * 5 / 2;
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
        __threadfence();
        passed = ok;
        if (!ok)
            set_status(a.dev_status, MOE_ERR_TIMEOUT);
    }
    __syncthreads();
    // dependents may start now: every CTA of this grid is resident
    asm volatile("griddepcontrol.launch_dependents;");
    if (passed) {
        // outputs [4 c0, 4 c1): one warp per 4-output chunk; lane l adds the
        // partials of CTAs [G l / 32, G (l+1) / 32) in order, then a fixed
        // butterfly adds the lanes
        const int nch = d / 4;
        const int c0 = static_cast<int>(static_cast<unsigned>(nch) * blockIdx.x / gridDim.x);
        const int c1 = static_cast<int>(static_cast<unsigned>(nch) * (blockIdx.x + 1) / gridDim.x);
        const int G = gridDim.x;
        const int g0 = G * lane / 32, g1 = G * (lane + 1) / 32;
        constexpr int kMaxPer = 8;                 // partial rows per lane (G <= 256)
        for (int ch = c0 + warp; ch < c1; ch += kWarps + 1) {
            // all of the lane's loads in flight at once, then added in order
            float4 v[kMaxPer];
#pragma unroll
            for (int i = 0; i < kMaxPer; ++i)
                v[i] = g0 + i < g1 ? __ldcg(reinterpret_cast<const float4 *>(a.partial + static_cast<int64_t>(g0 + i) * d) + ch)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kMaxPer; ++i) {
                acc.x += v[i].x;
                acc.y += v[i].y;
                acc.z += v[i].z;
                acc.w += v[i].w;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
                acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
                acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
                acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
            }
            if (lane == 0) {
                if (a.y_f32) {
                    reinterpret_cast<float4 *>(a.y)[ch] = acc;
                } else {
                    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
                    uint2 pk;
                    pk.x = *reinterpret_cast<uint32_t *>(&lo);
                    pk.y = *reinterpret_cast<uint32_t *>(&hi);
                    reinterpret_cast<uint2 *>(a.y)[ch] = pk;
                }
            }
        }
    }
}

}  // namespace dm

bool decode_m1_eligible(int M, int k, int d, int I, int E)
{
    // (route, neuron) indices times the grid stay within 32 bits; the final
    // reduction takes at most 8 partial rows per lane (grid <= 256)
    return device_sm_count() <= 256 && M == 1 && k >= 1 && k <= dm::kMaxK && (d == 1024 || d == 2048) && I % 32 == 0 && I >= 32 &&
           I <= 65536 && E >= 1;
}

size_t decode_m1_workspace(int d)
{
    return kWsReserved + ws_round(static_cast<size_t>(device_sm_count()) * d * sizeof(float));
}

bool decode_m1_route_eligible(int E, int k)
{
    return E >= k && E <= 512;
}

moe_status_t decode_m1_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                              const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                              const uint8_t *s13, const uint8_t *q2t, const uint8_t *s2t, void *y, bool y_f32,
                              void *ws, int32_t *dev_status, cudaStream_t stream)
{
    using namespace dm;
    const int G = device_sm_count();
    const Geo geo{d};
    const size_t smem = static_cast<size_t>(kStages) * geo.bytes() + 4 * kR * sizeof(float) +
                        2 * kStages * sizeof(uint64_t) + 2 * kMaxK * sizeof(int) + 4 * sizeof(int);
    if (smem > 220 * 1024 || !aligned(y, 16))
        return MOE_ERR_UNSUPPORTED;
    uint8_t *w = static_cast<uint8_t *>(ws);
    Args a{x,  ids, wts, logits, ids_out, wts_out, q13, s13, q2t, s2t, reinterpret_cast<unsigned long long *>(w),
           reinterpret_cast<float *>(w + kWsReserved), y, dev_status, y_f32 ? 1 : 0, k, d, I, E};
    auto go = [&](auto kern) -> moe_status_t {
        if (!smem_attr(reinterpret_cast<const void *>(kern), 220 * 1024))
            return MOE_ERR_CUDA;
        return launch_pdl(kern, dim3(G), dim3(kThreads), smem, stream, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    };
    if (logits) {
        if (!decode_m1_route_eligible(E, k))
            return MOE_ERR_UNSUPPORTED;
        const int pl = (E + 31) / 32;
        if (d == 2048)
            return pl <= 4 ? go(m1_kernel<4, 4>) : pl <= 8 ? go(m1_kernel<4, 8>) : go(m1_kernel<4, 16>);
        if (d == 1024)
            return pl <= 4 ? go(m1_kernel<2, 4>) : pl <= 8 ? go(m1_kernel<2, 8>) : go(m1_kernel<2, 16>);
        return MOE_ERR_UNSUPPORTED;
    }
    if (d == 2048)
        return go(m1_kernel<4, 0>);
    if (d == 1024)
        return go(m1_kernel<2, 0>);
    return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe
