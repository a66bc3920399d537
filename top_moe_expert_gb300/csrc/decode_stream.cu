// decode_stream.cu -- the output-centric decode path for MXFP8 weights,
// restructured for GB300's memory system.
//
// The method is the one of "Warp decode" (cursor.com blog), sections on what
// changed and how the two kernels work: parallelism over outputs, weight rows
// streamed once, MXFP8 converted on the fly, FP32 accumulation with warp
// butterflies, the routing weight folded into the down accumulation, and no
// alignment/padding/scatter/combine buffers (h is the only intermediate).
//
// What is GB300-specific here (the page's kernels were written for B200):
//   * Each kernel runs one CTA per SM over an exactly balanced share of the
//     bytes, so there is no second wave and no tail of idle SMs.
//   * A producer warp streams the weight rows with cp.async.bulk (the TMA
//     engine) into a ring of shared-memory stages guarded by mbarriers, so
//     tens of KB per SM stay in flight without tying up registers.
//   * E4M3 pairs are widened with cvt.rn.f16x2.e4m3x2 and cvt.f32.f16 (both
//     exact) and products accumulate with packed fma.rn.f32x2.
//   * The down kernel is launched with programmatic dependent launch.  Its
//     CTAs become resident while the gate/up kernel is still streaming, build
//     the routing plan and pull their W2 rows into shared memory, and only
//     then wait for h: the W2 stream overlaps the W13 stream.
//   * Every mbarrier wait is bounded; on expiry the kernel records
//     MOE_ERR_TIMEOUT in dev_status[1] and returns.
//
// Summation order per output is fixed by (d, I) and the lane layout only, so
// the result for a token does not depend on M, on the other tokens, or on the
// grid size.
#include "attr.h"
#include "common.cuh"
#include "decode_internal.h"
#include "tc.cuh"

namespace moe {
namespace ds {

constexpr int kWarps = 8;                       // compute warps per CTA
constexpr int kThreads = (kWarps + 1) * 32;     // + one producer warp
constexpr int kRowsA = 4;                       // neurons (gate+up row pairs) per stage
constexpr int kMaxStagesA = 4;
constexpr int kMaxStagesB = 8;
constexpr int kMaxRoutesPerBatch = 64;
constexpr uint64_t kWaitNs = 2000000000ull;     // 2 s

// ---------------------------------------------------------------- plan
// Distinct experts of the batch in ascending order and, per expert, its
// routes ordered by route id (the stable construction of "Route-Block
// Membership Selects Packed-AWQ Arithmetic", without padding).
struct Plan {
    int *cnt;      // [E]  scratch: counts, then running positions
    int *dist;     // [MK] distinct expert ids
    int *rstart;   // [MK + 1] start of each expert's routes in rlist
    int *rlist;    // [MK] routes
    int *n_dist;   // [1]
    int *n_invalid;// [1]
};

__device__ __forceinline__ size_t plan_smem_bytes(int E, int MK)
{
    return (static_cast<size_t>(E) + 3 * MK + 4) * sizeof(int);
}

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

// All threads of the CTA call this; ids are read through L2 (ld.global.cg).
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
                p.cnt[e] = off;                  // running position of e
            run_off += __shfl_sync(0xffffffffu, ic, 31);
            run_slot += __shfl_sync(0xffffffffu, iff, 31);
        }
        if (lane == 0) {
            *p.n_dist = run_slot;
            p.rstart[run_slot] = run_off;
        }
        __syncwarp();
        // stable placement: ascending route id within each expert
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

// ---------------------------------------------------------------- math

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n .reg .b64 A, B, C;\n mov.b64 A, {%2, %3};\n mov.b64 B, {%4, %5};\n"
        " mov.b64 C, {%6, %7};\n fma.rn.f32x2 A, A, B, C;\n mov.b64 {%0, %1}, A;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Two E4M3 codes (bytes 0,1 of `two`) -> (w0, w1) as floats: widened to an
// fp16 pair by the hardware (exact: E4M3 is a subset of fp16), then each
// half to fp32 (exact).
__device__ __forceinline__ float2 w_pair(uint32_t two)
{
    float2 f;
    asm("{\n .reg .b32 r;\n .reg .b16 l, h;\n cvt.rn.f16x2.e4m3x2 r, %2;\n mov.b32 {l, h}, r;\n"
        " cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}"
        : "=f"(f.x), "=f"(f.y) : "h"(static_cast<uint16_t>(two)));
    return f;
}

// sum_{i<16} w_i * x_i for one 16-byte chunk of E4M3 codes; x as 8 float2.
__device__ __forceinline__ float chunk16_dot(uint4 q, const float2 (&x)[8])
{
    float2 acc = make_float2(0.f, 0.f);
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc = fma2(w_pair(qw[i] & 0xFFFFu), x[2 * i], acc);
        acc = fma2(w_pair(qw[i] >> 16), x[2 * i + 1], acc);
    }
    return acc.x + acc.y;
}

// sum_{i<8} w_i * h_i for one 8-byte chunk of E4M3 codes.
__device__ __forceinline__ float chunk8_dot(uint2 q, const float4 ha, const float4 hb)
{
    float2 acc = make_float2(0.f, 0.f);
    acc = fma2(w_pair(q.x & 0xFFFFu), make_float2(ha.x, ha.y), acc);
    acc = fma2(w_pair(q.x >> 16), make_float2(ha.z, ha.w), acc);
    acc = fma2(w_pair(q.y & 0xFFFFu), make_float2(hb.x, hb.y), acc);
    acc = fma2(w_pair(q.y >> 16), make_float2(hb.z, hb.w), acc);
    return acc.x + acc.y;
}

__device__ __forceinline__ void load_x16(const __nv_bfloat16 *xs, float2 (&x)[8])
{
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(xs));
    const uint4 b = __ldg(reinterpret_cast<const uint4 *>(xs) + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        x[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
}

__device__ __forceinline__ float e8m0f(uint32_t s)
{
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

__device__ __forceinline__ void set_timeout(int32_t *dev_status)
{
    if (dev_status)
        atomicCAS(dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
}

// Before the producer leaves: wait (bounded) until every copy it issued has
// landed, so no bulk copy can target shared memory of a finished CTA.
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

// ============================================================ kernel A
// gate/up: h[r][n] = SiLU(W13[e][n] . x[t]) * (W13[e][I+n] . x[t]) for every
// route r = (t, j) of every distinct expert e; CTA c owns row pairs
// [c*P/G, (c+1)*P/G) of the flattened (distinct expert, neuron) space.
struct ArgsA {
    const __nv_bfloat16 *x;
    const int32_t *ids;
    const uint8_t *q13;
    const uint8_t *s13;
    float *h;
    int32_t *dev_status;
    int M, k, d, I, E;
    int stages;         // ring depth
};

template <int NCH>   // NCH = d / 512 when x is held in registers (M == 1), else 0
__global__ void __launch_bounds__(kThreads, 1) gate_up_kernel(const ArgsA a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int MK = a.M * a.k, d = a.d, I = a.I;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row_bytes = d, srow_bytes = d / 32;
    const int stage_bytes = 2 * kRowsA * (row_bytes + srow_bytes);

    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    // shared memory carve-up
    uint8_t *stages = smem;                                               // a.stages stages
    float *res = reinterpret_cast<float *>(smem + a.stages * stage_bytes); // [2][8][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(res + 2 * kWarps * kMaxRoutesPerBatch);
    int *plan_base = reinterpret_cast<int *>(bars + 2 * kMaxStagesA + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * kMaxStagesA);
    const Plan P = plan_carve(plan_base, a.E, MK);
    const uint32_t full0 = tc::smem_u32(bars), empty0 = tc::smem_u32(bars + kMaxStagesA);

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    plan_build(P, a.ids, MK, a.E);
    if (blockIdx.x == 0 && tid == 0 && *P.n_invalid && a.dev_status)
        atomicAdd(a.dev_status, *P.n_invalid);

    const int nd = *P.n_dist;
    const long long Ptot = static_cast<long long>(nd) * I;
    const long long p0 = Ptot * blockIdx.x / gridDim.x, p1 = Ptot * (blockIdx.x + 1) / gridDim.x;

    if (warp == kWarps) {
        // ---------------- producer
        if (lane == 0) {
            int s = 0, issued = 0;
            uint32_t ph = 0;
            for (long long p = p0; p < p1; ++issued) {
                const int u = static_cast<int>(p / I), n = static_cast<int>(p % I);
                const int nr = static_cast<int>(p1 - p < (long long)min(kRowsA, I - n) ? p1 - p : (long long)min(kRowsA, I - n));
                if (!tc::mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, kWaitNs))
                    break;
                const int e = P.dist[u];
                uint8_t *st = stages + s * stage_bytes;
                const uint32_t b = full0 + 8 * s;
                const uint32_t bytes = 2u * nr * (row_bytes + srow_bytes);
                tc::mbar_arrive_expect_tx(b, bytes);
                const int64_t grow = static_cast<int64_t>(e) * 2 * I + n;
                tc::bulk_load(tc::smem_u32(st), a.q13 + grow * row_bytes, nr * row_bytes, b);
                tc::bulk_load(tc::smem_u32(st + kRowsA * row_bytes), a.q13 + (grow + I) * row_bytes,
                              nr * row_bytes, b);
                uint8_t *ss = st + 2 * kRowsA * row_bytes;
                tc::bulk_load(tc::smem_u32(ss), a.s13 + grow * srow_bytes, nr * srow_bytes, b);
                tc::bulk_load(tc::smem_u32(ss + kRowsA * srow_bytes), a.s13 + (grow + I) * srow_bytes,
                              nr * srow_bytes, b);
                p += nr;
                if (++s == a.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            drain_copies(full0, s, ph, issued, a.stages);
        }
        return;
    }

    // ---------------- compute warps: warp w < 4 -> gate row w, else up row w-4
    float2 xr[NCH > 0 ? NCH * 8 : 1];
    if constexpr (NCH > 0) {
        // M == 1: the token's activation slice of this lane, kept in registers
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            float2 t[8];
            load_x16(a.x + (i * 32 + lane) * 16, t);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                xr[i * 8 + q] = t[q];
        }
    }
    const int nch = d / 512;            // 16-byte chunks per lane per row
    int s = 0, rb = 0;
    uint32_t ph = 0;
    for (long long p = p0; p < p1;) {
        const int u = static_cast<int>(p / I), n = static_cast<int>(p % I);
        const int nr = static_cast<int>(p1 - p < (long long)min(kRowsA, I - n) ? p1 - p : (long long)min(kRowsA, I - n));
        // On a timeout every compute warp records it and keeps walking the
        // same loop (later waits return at once), so all warps still meet at
        // every named barrier below; the results are then garbage but the
        // status word says so.
        if (!tc::mbar_wait(full0 + 8 * s, ph, abort_flag, kWaitNs))
            set_timeout(a.dev_status);
        const uint8_t *st = stages + s * stage_bytes;
        const int rs = P.rstart[u], re = P.rstart[u + 1];
        const int wr = warp & 3;
        const bool active = wr < nr;
        const uint8_t *row = st + (warp < 4 ? 0 : kRowsA * row_bytes) + wr * row_bytes;
        const uint8_t *srow = st + 2 * kRowsA * row_bytes + (warp < 4 ? 0 : kRowsA * srow_bytes) + wr * srow_bytes;
        for (int r0 = rs; r0 < re; r0 += kMaxRoutesPerBatch) {
            const int nrt = min(kMaxRoutesPerBatch, re - r0);
            float *rb_res = res + rb * kWarps * kMaxRoutesPerBatch;
            if (active) {
                for (int ri = 0; ri < nrt; ++ri) {
                    const int t = P.rlist[r0 + ri] / a.k;
                    float acc = 0.f;
                    if constexpr (NCH > 0) {
#pragma unroll
                        for (int i = 0; i < NCH; ++i) {
                            const int c = i * 32 + lane;
                            const uint4 q = *reinterpret_cast<const uint4 *>(row + c * 16);
                            const float sc = e8m0f(srow[c >> 1]);
                            float2 xx[8];
#pragma unroll
                            for (int qq = 0; qq < 8; ++qq)
                                xx[qq] = xr[i * 8 + qq];
                            acc = fmaf(chunk16_dot(q, xx), sc, acc);
                        }
                    } else {
                        const __nv_bfloat16 *xt = a.x + static_cast<int64_t>(t) * d;
                        for (int i = 0; i < nch; ++i) {
                            const int c = i * 32 + lane;
                            const uint4 q = *reinterpret_cast<const uint4 *>(row + c * 16);
                            const float sc = e8m0f(srow[c >> 1]);
                            float2 xx[8];
                            load_x16(xt + c * 16, xx);
                            acc = fmaf(chunk16_dot(q, xx), sc, acc);
                        }
                    }
                    acc = warp_sum(acc);
                    if (lane == 0)
                        rb_res[warp * kMaxRoutesPerBatch + ri] = acc;
                }
            }
            tc::named_bar(1, kWarps * 32);
            // the stage's rows are consumed once every warp passed the barrier
            if (r0 + kMaxRoutesPerBatch >= re && tid == 0)
                tc::mbar_arrive(empty0 + 8 * s);
            for (int i = tid; i < nr * nrt; i += kWarps * 32) {
                const int nn = i % nr, ri = i / nr;
                const float g = rb_res[nn * kMaxRoutesPerBatch + ri];
                const float uu = rb_res[(4 + nn) * kMaxRoutesPerBatch + ri];
                a.h[static_cast<int64_t>(P.rlist[r0 + ri]) * I + n + nn] = silu_mul(g, uu);
            }
            rb ^= 1;
        }
        if (rs == re && tid == 0)           // expert without routes cannot occur; keep the ring moving
            tc::mbar_arrive(empty0 + 8 * s);
        p += nr;
        if (++s == a.stages) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ============================================================ kernel B
// down + combine: y[t][o] = sum over routes (t,j) of w[t][j] * W2[e_j][o] . h[t,j],
// accumulated in ascending expert order; CTA c owns rows [o0, o1).
struct ArgsB {
    const float *h;
    const int32_t *ids;
    const float *wts;
    const uint8_t *q2;
    const uint8_t *s2;
    void *y;
    int32_t *dev_status;
    int M, k, d, I, E;
    int gran;           // row granule keeping scale copies 16-byte aligned
    int rows_stage;     // rows per stage
    int stages;         // ring depth
    int y_f32;
};

__global__ void __launch_bounds__(kThreads, 1) down_kernel(const ArgsB a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int MK = a.M * a.k, d = a.d, I = a.I;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int srow_bytes = I / 32;
    const int RS = a.rows_stage;
    const int stage_bytes = RS * I + ((RS * srow_bytes + 127) & ~127);
    const int units = d / a.gran;
    const int o0 = static_cast<int>(static_cast<long long>(units) * blockIdx.x / gridDim.x) * a.gran;
    const int o1 = static_cast<int>(static_cast<long long>(units) * (blockIdx.x + 1) / gridDim.x) * a.gran;
    const int nrows = o1 - o0;
    const int nblk = (nrows + RS - 1) / RS;            // row blocks per expert

    uint8_t *stages = smem;
    float *yacc = reinterpret_cast<float *>(smem + a.stages * stage_bytes);   // [M][nrows_max]
    const int ystride = ((d / a.gran + gridDim.x - 1) / gridDim.x) * a.gran;
    uint64_t *bars = reinterpret_cast<uint64_t *>(yacc + ((a.M * ystride + 3) & ~3));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * kMaxStagesB);
    int *plan_base = reinterpret_cast<int *>(bars + 2 * kMaxStagesB + 2);
    const Plan P = plan_carve(plan_base, a.E, MK);
    const uint32_t full0 = tc::smem_u32(bars), empty0 = tc::smem_u32(bars + kMaxStagesB);

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    for (int i = tid; i < a.M * ystride; i += blockDim.x)
        yacc[i] = 0.f;
    // the routing inputs do not depend on the gate/up kernel: plan now
    plan_build(P, a.ids, MK, a.E);
    const int nd = *P.n_dist;
    const int nwork = nd * nblk;                        // (expert, row block) stages

    if (warp == kWarps) {
        // ---------------- producer: W2 rows do not depend on h either
        if (lane == 0) {
            int s = 0, issued = 0;
            uint32_t ph = 0;
            for (int wi = 0; wi < nwork; ++wi, ++issued) {
                const int u = wi / nblk, blk = wi % nblk;
                const int ra = o0 + blk * RS, nr = min(RS, o1 - ra);
                if (!tc::mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, kWaitNs))
                    break;
                const int e = P.dist[u];
                uint8_t *st = stages + s * stage_bytes;
                const uint32_t b = full0 + 8 * s;
                tc::mbar_arrive_expect_tx(b, nr * (I + srow_bytes));
                const int64_t row = static_cast<int64_t>(e) * d + ra;
                tc::bulk_load(tc::smem_u32(st), a.q2 + row * I, nr * I, b);
                tc::bulk_load(tc::smem_u32(st + RS * I), a.s2 + row * srow_bytes, nr * srow_bytes, b);
                if (++s == a.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            drain_copies(full0, s, ph, issued, a.stages);
        }
        return;
    }

    // h is written by the gate/up kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int nch = I / 256;            // 8-byte chunks per lane per row
    int s = 0;
    uint32_t ph = 0;
    for (int wi = 0; wi < nwork; ++wi) {
        const int u = wi / nblk, blk = wi % nblk;
        const int ra = o0 + blk * RS, nr = min(RS, o1 - ra);
        // On a timeout every compute warp records it and keeps walking the
        // same loop (later waits return at once), so all warps still meet at
        // every named barrier below; the results are then garbage but the
        // status word says so.
        if (!tc::mbar_wait(full0 + 8 * s, ph, abort_flag, kWaitNs))
            set_timeout(a.dev_status);
        const uint8_t *st = stages + s * stage_bytes;
        const int rs = P.rstart[u], re = P.rstart[u + 1];
        for (int i = warp; i < nr; i += kWarps) {
            const uint8_t *row = st + i * I;
            const uint8_t *srow = st + RS * I + i * srow_bytes;
            for (int ri = rs; ri < re; ++ri) {
                const int r = P.rlist[ri];
                const float *hr = a.h + static_cast<int64_t>(r) * I;
                float acc = 0.f;
                for (int j = 0; j < nch; ++j) {
                    const int c = j * 32 + lane;                 // 8-element chunk
                    const uint2 q = *reinterpret_cast<const uint2 *>(row + c * 8);
                    const float4 ha = __ldcg(reinterpret_cast<const float4 *>(hr + c * 8));
                    const float4 hb = __ldcg(reinterpret_cast<const float4 *>(hr + c * 8) + 1);
                    acc = fmaf(chunk8_dot(q, ha, hb), e8m0f(srow[c >> 2]), acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) {
                    const int t = r / a.k;
                    float *ya = yacc + t * ystride + (ra - o0) + i;
                    *ya = fmaf(__ldcg(a.wts + r), acc, *ya);
                }
            }
        }
        tc::named_bar(1, kWarps * 32);
        if (tid == 0)
            tc::mbar_arrive(empty0 + 8 * s);
        if (++s == a.stages) {
            s = 0;
            ph ^= 1u;
        }
    }
    tc::named_bar(1, kWarps * 32);
    for (int i = tid; i < a.M * nrows; i += kWarps * 32) {
        const int t = i / nrows, o = i % nrows;
        const float v = yacc[t * ystride + o];
        const int64_t idx = static_cast<int64_t>(t) * d + o0 + o;
        if (a.y_f32)
            static_cast<float *>(a.y)[idx] = v;
        else
            static_cast<__nv_bfloat16 *>(a.y)[idx] = __float2bfloat16_rn(v);
    }
}

}  // namespace ds

// ---------------------------------------------------------------- host side

bool decode_stream_eligible(int M, int k, int d, int I, int E, const void *q13, const void *s13,
                            const void *q2, const void *s2)
{
    return M >= 1 && M * k <= 512 && E <= 1024 && d % 512 == 0 && I % 256 == 0 &&
           aligned(q13, 16) && aligned(s13, 16) && aligned(q2, 16) && aligned(s2, 16);
}

moe_status_t decode_stream_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                  const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                  const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32, float *h,
                                  int32_t *dev_status, cudaStream_t stream)
{
    using namespace ds;
    const int MK = M * k;
    const int G = device_sm_count();
    // ---- kernel A
    const size_t stage_a = 2 * kRowsA * (d + d / 32);
    int stages_a = static_cast<int>((128 * 1024) / stage_a);
    stages_a = stages_a < 2 ? 2 : (stages_a > kMaxStagesA ? kMaxStagesA : stages_a);
    ArgsA aa{x, ids, q13, s13, h, dev_status, M, k, d, I, E, stages_a};
    const size_t plan_b = (static_cast<size_t>(E) + 3 * MK + 4) * sizeof(int);
    const size_t smem_a = stages_a * stage_a + 2 * kWarps * kMaxRoutesPerBatch * sizeof(float) +
                          (2 * kMaxStagesA + 2) * sizeof(uint64_t) + plan_b;
    // ---- kernel B
    int gran = 1;
    while ((gran * (I / 32)) % 16 != 0)
        gran *= 2;
    int rows_stage = (16384 / I) / gran * gran;
    if (rows_stage < gran)
        rows_stage = gran;
    const int units = d / gran;
    const int GB = units < G ? units : G;
    const int rows_cta = ((units + GB - 1) / GB) * gran;
    if (rows_stage > rows_cta)
        rows_stage = rows_cta;
    const size_t stage_b = static_cast<size_t>(rows_stage) * I + ((rows_stage * (I / 32) + 127) & ~127);
    int stages_b = static_cast<int>((96 * 1024) / stage_b);
    stages_b = stages_b < 2 ? 2 : (stages_b > kMaxStagesB ? kMaxStagesB : stages_b);
    const size_t yacc_b = ((static_cast<size_t>(M) * rows_cta + 3) & ~size_t(3)) * sizeof(float);
    const size_t smem_b = stages_b * stage_b + yacc_b + (2 * kMaxStagesB + 2) * sizeof(uint64_t) + plan_b;
    if (smem_a > 200 * 1024 || smem_b > 200 * 1024)
        return MOE_ERR_UNSUPPORTED;
    ArgsB ab{h, ids, wts, q2, s2, y, dev_status, M, k, d, I, E, gran, rows_stage, stages_b, y_f32 ? 1 : 0};

    auto ka = (M == 1 && d == 2048) ? gate_up_kernel<4>
            : (M == 1 && d == 1024) ? gate_up_kernel<2>
            : (M == 1 && d == 512) ? gate_up_kernel<1> : gate_up_kernel<0>;
    if (!smem_attr(reinterpret_cast<const void *>(ka), 200 * 1024) ||
        !smem_attr(reinterpret_cast<const void *>(down_kernel), 200 * 1024))
        return MOE_ERR_CUDA;
    if (launch_pdl(ka, dim3(G), dim3(kThreads), smem_a, stream, aa) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_pdl(down_kernel, dim3(GB), dim3(kThreads), smem_b, stream, ab) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace moe
