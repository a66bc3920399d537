// host_mx_grouped.cu -- host emulation of the small-batch MXFP8 kernel
// (top_moe_expert_gb300/csrc/grouped_mx_mma.cu) and the grouped combine, for
// the CPU tests.
//
// It runs the kernel's two phases CTA by CTA and warp by warp with the lanes
// looped, through the kernel's own lane functions (grouped_mx_mma.cuh,
// decode_mx_m1.cuh): the unit split over CTAs and warps, the staged operands
// with their row padding and scale exponents, the piece loads and their
// addresses, the block fold, and the per-block completion counts.  mma.sync m16n8k16 is emulated
// from the PTX fragment layouts (products exact, sums in double, rounded to
// float).  Reads of Yr entries that phase 2 never wrote show up as NaN.
#include <cmath>
#include <cstring>
#include <vector>
#include <cuda_bf16.h>
#include "grouped_mx_mma.cuh"

using namespace moe::gmx;

static float bfly_max(float (&v)[32])
{
    for (int o = 16; o > 0; o >>= 1) {
        float t[32];
        for (int l = 0; l < 32; ++l)
            t[l] = fmaxf(v[l], v[l ^ o]);
        memcpy(v, t, sizeof t);
    }
    return v[0];
}

static float h2f(uint16_t b) { return moe::da1::f16bits(b); }
static uint16_t f2h(float v)
{
    __half h = __float2half_rn(v);
    return __half_raw(h).x;
}
static float lo16(uint32_t r) { return h2f(static_cast<uint16_t>(r & 0xFFFFu)); }
static float hi16(uint32_t r) { return h2f(static_cast<uint16_t>(r >> 16)); }

// D += A B for one warp (m16n8k16, f16 inputs, f32 accumulate).
static void mma_warp(float (&D)[32][4], const uint32_t (&A)[32][4], const uint32_t (&B)[32][2])
{
    double a[16][16], bm[16][8], dm[16][8];
    for (int l = 0; l < 32; ++l) {
        const int g = l >> 2, t = l & 3;
        a[g][2 * t] = lo16(A[l][0]);         a[g][2 * t + 1] = hi16(A[l][0]);
        a[g + 8][2 * t] = lo16(A[l][1]);     a[g + 8][2 * t + 1] = hi16(A[l][1]);
        a[g][2 * t + 8] = lo16(A[l][2]);     a[g][2 * t + 9] = hi16(A[l][2]);
        a[g + 8][2 * t + 8] = lo16(A[l][3]); a[g + 8][2 * t + 9] = hi16(A[l][3]);
        bm[2 * t][g] = lo16(B[l][0]);        bm[2 * t + 1][g] = hi16(B[l][0]);
        bm[2 * t + 8][g] = lo16(B[l][1]);    bm[2 * t + 9][g] = hi16(B[l][1]);
        dm[g][2 * t] = D[l][0];     dm[g][2 * t + 1] = D[l][1];
        dm[g + 8][2 * t] = D[l][2]; dm[g + 8][2 * t + 1] = D[l][3];
    }
    for (int l = 0; l < 32; ++l) {
        const int g = l >> 2, t = l & 3;
        const int rows[4] = {g, g, g + 8, g + 8}, cols[4] = {2 * t, 2 * t + 1, 2 * t, 2 * t + 1};
        for (int i = 0; i < 4; ++i) {
            double s = dm[rows[i]][cols[i]];
            for (int kk = 0; kk < 16; ++kk)
                s += a[rows[i]][kk] * bm[kk][cols[i]];
            D[l][i] = static_cast<float>(s);
        }
    }
}

static int f16_sigma_h(float m)
{
    if (!(m > 0.f))
        return 0;
    int ex;
    frexpf(m, &ex);
    return 15 - ex;
}

static float silu_mul_h(float g, float u) { return g / (1.0f + std::exp(-g)) * u; }

// One unit of either phase for one warp (K = Kd, items of 64 values): the
// lanes' accumulators.  alo is the second half of a hi + lo operand (or null).
static void run_unit(const uint8_t *q, const uint8_t *sc, int64_t wrow0, int Kd, const uint8_t *ahi,
                     const uint8_t *alo, int rs, float (&acc)[32][4])
{
    for (int l = 0; l < 32; ++l)
        acc[l][0] = acc[l][1] = acc[l][2] = acc[l][3] = 0.f;
    for (int c = 0; c < Kd / 64; ++c) {
        Ld ld[32];
        for (int l = 0; l < 32; ++l)
            mx_load(q, sc, wrow0, Kd, c, l, ld[l]);
        for (int p = 0; p < 2; ++p) {
            float D[32][4] = {};
            for (int t = 0; t < 2; ++t) {
                uint32_t B[32][2];
                for (int l = 0; l < 32; ++l)
                    mx_b(ld[l], p, t, B[l][0], B[l][1]);
                for (const uint8_t *abase : {ahi, alo}) {
                    if (!abase)
                        continue;
                    uint32_t A[32][4];
                    for (int l = 0; l < 32; ++l) {
                        uint32_t aa[4];
                        a_regs(abase, rs, c * 64, p, t, l, aa);
                        memcpy(A[l], aa, sizeof aa);
                    }
                    mma_warp(D, A, B);
                }
            }
            for (int l = 0; l < 32; ++l) {
                const float dd[4] = {D[l][0], D[l][1], D[l][2], D[l][3]};
                fold4(acc[l], dd, ld[l], p);
            }
        }
    }
}

extern "C" int mx_grouped_emulate(const uint16_t *x, const int32_t *ids, const float *wts, const int32_t *sorted,
                                  const int32_t *expert_ids, int npp, const uint8_t *q13, const uint8_t *s13,
                                  const uint8_t *q2, const uint8_t *s2, float *gu, float *yr, float *y, int M, int k,
                                  int d, int I, int E, int G)
{
    const int b = kRows;
    if (d % 64 || I % 64)
        return -1;
    const int mk = M * k, nblk = npp / b, RB1 = 2 * I / 8, RB2 = d / 8;
    const Smem L{d, I};
    std::vector<uint8_t> sm(L.bytes());
    uint8_t *A = sm.data() + L.a();
    std::vector<int> done(nblk > 0 ? nblk : 1, 0);
    auto xval = [&](int64_t i) -> float {
        __nv_bfloat16_raw r;
        r.x = x[i];
        return __bfloat162float(__nv_bfloat16(r));
    };
    int route[kRows], sig[kRows];
    auto rows_of = [&](int blk) {
        const int e_raw = expert_ids[blk];
        for (int r = 0; r < kRows; ++r) {
            const int rt = r < b ? sorted[static_cast<int64_t>(blk) * b + r] : mk;
            route[r] = rt >= 0 && rt < mk && e_raw >= 0 && e_raw < E ? rt : -1;
        }
        return e_raw >= 0 && e_raw < E ? e_raw : 0;
    };
    // ---- phase 1
    for (int cta = 0; cta < G; ++cta) {
        const int T = nblk * RB1;
        const int c0 = static_cast<int>(static_cast<int64_t>(T) * cta / G);
        const int c1 = static_cast<int>(static_cast<int64_t>(T) * (cta + 1) / G);
        const int rs = L.xrow();
        for (int u = c0; u < c1;) {
            const int blk = u / RB1, seg_end = c1 < (blk + 1) * RB1 ? c1 : (blk + 1) * RB1;
            const int e = rows_of(blk);
            memset(sm.data(), 0xFF, sm.size());            // stale contents must not leak into results
            for (int r = 0; r < kRows; ++r) {
                float v[32];
                for (int l = 0; l < 32; ++l) {
                    v[l] = 0.f;
                    if (route[r] >= 0)
                        for (int i = l; i < d; i += 32)
                            v[l] = fmaxf(v[l], fabsf(xval(static_cast<int64_t>(route[r] / k) * d + i)));
                }
                sig[r] = f16_sigma_h(bfly_max(v));
                uint16_t *row = reinterpret_cast<uint16_t *>(A + r * rs);
                for (int i = 0; i < d; ++i)
                    row[i] = f2h(route[r] >= 0 ? ldexpf(xval(static_cast<int64_t>(route[r] / k) * d + i), sig[r])
                                               : 0.f);
            }
            const int n = seg_end - u;
            for (int wp = 0; wp < kWarps; ++wp) {
                const int v0 = u + n * wp / kWarps, v1 = u + n * (wp + 1) / kWarps;
                for (int v = v0; v < v1; ++v) {
                    float acc[32][4];
                    run_unit(q13, s13, static_cast<int64_t>(e) * 2 * I + (v - blk * RB1) * 8, d, A, nullptr, rs, acc);
                    for (int l = 0; l < 32; ++l) {
                        const int col = (v - blk * RB1) * 8 + 2 * (l & 3);
                        for (int h = 0; h < 2; ++h) {
                            const int r = (l >> 2) + 8 * h;
                            if (r < b && route[r] >= 0) {
                                const float un = ldexpf(1.0f, -sig[r]);
                                gu[static_cast<int64_t>(route[r]) * 2 * I + col] = acc[l][2 * h] * un;
                                gu[static_cast<int64_t>(route[r]) * 2 * I + col + 1] = acc[l][2 * h + 1] * un;
                            }
                        }
                    }
                    ++done[blk];
                }
            }
            u = seg_end;
        }
    }
    for (int blk = 0; blk < nblk; ++blk)
        if (done[blk] != RB1)
            return -2;                                      // a block's gate/up units were not all run once
    // ---- phase 2
    for (int cta = 0; cta < G; ++cta) {
        const int T = nblk * RB2;
        const int c0 = static_cast<int>(static_cast<int64_t>(T) * cta / G);
        const int c1 = static_cast<int>(static_cast<int64_t>(T) * (cta + 1) / G);
        const int rs = L.hrow();
        uint8_t *Ahi = A, *Alo = A + kRows * rs;
        for (int u = c0; u < c1;) {
            const int blk = u / RB2, seg_end = c1 < (blk + 1) * RB2 ? c1 : (blk + 1) * RB2;
            const int e = rows_of(blk);
            memset(sm.data(), 0xFF, sm.size());
            for (int r = 0; r < kRows; ++r) {
                const float w = route[r] >= 0 ? wts[route[r]] : 0.f;
                const float *g_row = gu + static_cast<int64_t>(route[r] >= 0 ? route[r] : 0) * 2 * I;
                float v[32];
                for (int l = 0; l < 32; ++l) {
                    v[l] = 0.f;
                    if (route[r] >= 0)
                        for (int n2 = l; n2 < I; n2 += 32)
                            v[l] = fmaxf(v[l], fabsf(w * silu_mul_h(g_row[n2], g_row[I + n2])));
                }
                sig[r] = f16_sigma_h(bfly_max(v));
                uint16_t *hi = reinterpret_cast<uint16_t *>(Ahi + r * rs);
                uint16_t *lo = reinterpret_cast<uint16_t *>(Alo + r * rs);
                for (int i = 0; i < I; ++i) {
                    float hv = 0.f;
                    if (route[r] >= 0)
                        hv = ldexpf(w * silu_mul_h(g_row[i], g_row[I + i]), sig[r]);
                    hi[i] = f2h(hv);
                    lo[i] = f2h(hv - h2f(hi[i]));
                }
            }
            const int n = seg_end - u;
            for (int wp = 0; wp < kWarps; ++wp) {
                const int v0 = u + n * wp / kWarps, v1 = u + n * (wp + 1) / kWarps;
                for (int v = v0; v < v1; ++v) {
                    float acc[32][4];
                    run_unit(q2, s2, static_cast<int64_t>(e) * d + (v - blk * RB2) * 8, I, Ahi, Alo, rs, acc);
                    for (int l = 0; l < 32; ++l) {
                        const int col = (v - blk * RB2) * 8 + 2 * (l & 3);
                        for (int h = 0; h < 2; ++h) {
                            const int r = (l >> 2) + 8 * h;
                            if (r < b && route[r] >= 0) {
                                const float un = ldexpf(1.0f, -sig[r]);
                                yr[static_cast<int64_t>(route[r]) * d + col] = acc[l][2 * h] * un;
                                yr[static_cast<int64_t>(route[r]) * d + col + 1] = acc[l][2 * h + 1] * un;
                            }
                        }
                    }
                }
            }
            u = seg_end;
        }
    }
    // ---- combine: valid slots in order
    for (int t = 0; t < M; ++t)
        for (int o = 0; o < d; ++o) {
            float s = 0.f;
            for (int j = 0; j < k; ++j) {
                const int e = ids[t * k + j];
                if (e >= 0 && e < E)
                    s += yr[static_cast<int64_t>(t * k + j) * d + o];
            }
            y[static_cast<int64_t>(t) * d + o] = s;
        }
    return L.bytes();
}
