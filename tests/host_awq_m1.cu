// host_awq_m1.cu -- host emulation of the single-token AWQ kernel
// (top_moe_expert_gb300/csrc/decode_awq_m1.cu) for the CPU tests.
//
// It runs the kernel's steps CTA by CTA and warp by warp with the lanes
// looped, through the kernel's own lane functions (decode_awq_m1.cuh): the
// item split, the operand loads and their addresses, the staged orders, the
// piece numbering and the fold.  mma.sync m16n8k16 is emulated from the
// PTX fragment layouts (products exact, sums in double, rounded to float);
// the bulk copies become memcpy after the same alignment checks.  The result
// is compared with the oracle, so an index or layout mistake in the kernel's
// host-visible arithmetic fails on the CPU before the kernel ever runs.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <vector>
#include <cuda_bf16.h>
#include "decode_awq_m1.cuh"

using namespace moe::da1;

static float bfly_sum(float (&v)[32])
{
    for (int o = 16; o > 0; o >>= 1) {
        float t[32];
        for (int l = 0; l < 32; ++l)
            t[l] = v[l] + v[l ^ o];
        memcpy(v, t, sizeof t);
    }
    return v[0];
}

static float h2f(uint16_t b) { return f16bits(b); }
static uint16_t f2h(float v)
{
    __half h = __float2half_rn(v);
    return __half_raw(h).x;
}
static float lo16(uint32_t r) { return h2f(static_cast<uint16_t>(r & 0xFFFFu)); }
static float hi16(uint32_t r) { return h2f(static_cast<uint16_t>(r >> 16)); }

// D (+)= A B for one warp: A 16x16, B 16x8 (f16), D 16x8 (f32).
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
    double out[16][8];
    for (int m = 0; m < 16; ++m)
        for (int n = 0; n < 8; ++n) {
            double s = dm[m][n];
            for (int kk = 0; kk < 16; ++kk)
                s += a[m][kk] * bm[kk][n];
            out[m][n] = s;
        }
    for (int l = 0; l < 32; ++l) {
        const int g = l >> 2, t = l & 3;
        D[l][0] = static_cast<float>(out[g][2 * t]);
        D[l][1] = static_cast<float>(out[g][2 * t + 1]);
        D[l][2] = static_cast<float>(out[g + 8][2 * t]);
        D[l][3] = static_cast<float>(out[g + 8][2 * t + 1]);
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

extern "C" int awq_m1_emulate(const void *x, int x_bf16, const int32_t *ids, const float *wts, const uint32_t *q13,
                           const uint16_t *s13, const int32_t *z13, const uint32_t *q2, const uint16_t *s2,
                           const int32_t *z2, float *gp, float *y, int k, int d, int I, int E, int G, int *status)
{
    Args a{x, ids, wts, q13, s13, z13, q2, s2, z2, nullptr, gp, y, nullptr, x_bf16, 1, k, d, I, E};
    const int NG = d / 128, G2 = I / 128, RB = 2 * I / 8;
    int r_e[kMaxK], nv = 0;
    float r_w[kMaxK];
    for (int j = 0; j < k; ++j)
        if (ids[j] >= 0 && ids[j] < E) {
            r_e[nv] = ids[j];
            r_w[nv] = wts[j];
            ++nv;
        }
    status[0] = k - nv;
    status[1] = 0;
    auto xval = [&](int i) -> float {
        if (x_bf16) {
            __nv_bfloat16_raw r;
            r.x = reinterpret_cast<const uint16_t *>(x)[i];
            return __bfloat162float(__nv_bfloat16(r));
        }
        return h2f(reinterpret_cast<const uint16_t *>(x)[i]);
    };
    float xm = 0.f;
    for (int i = 0; i < d; ++i)
        xm = fmaxf(xm, fabsf(xval(i)));
    const int sigx = f16_sigma_h(xm);
    std::vector<uint16_t> xp(d);
    for (int i = 0; i < d; ++i)
        xp[i] = f2h(ldexpf(xval((i & ~7) + interleave(i & 7)), sigx));
    std::vector<float> xsum(NG);
    for (int g = 0; g < NG; ++g) {
        float v[32];
        for (int l = 0; l < 32; ++l) {
            v[l] = 0.f;
            for (int t = 0; t < 4; ++t)
                v[l] += h2f(xp[g * 128 + t * 32 + l]);
        }
        xsum[g] = bfly_sum(v);
    }
    const int T = nv * RB * NG;
    int maxsmem = 0;
    // ---- phase 1, every CTA
    for (int b = 0; b < G; ++b) {
        const int c0 = split_lo(T, b, G), c1 = split_lo(T, b + 1, G), n = c1 - c0;
        float p1v[kWarps * 4 * 8];
        int p1u[kWarps * 4];
        for (int i = 0; i < kWarps * 4; ++i)
            p1u[i] = -1;
        for (int w = 0; w < kWarps; ++w) {
            const int i0 = c0 + split_lo(n, w, kWarps), i1 = c0 + split_lo(n, w + 1, kWarps);
            float acc[32][2] = {};
            int cur = i0 < i1 ? i0 / NG : -1, slot = 0;
            for (int i = i0; i < i1; ++i) {
                const int u = i / NG, g = i - u * NG;
                if (u != cur) {
                    if (slot >= 4) {
                        status[1] = 7;
                        return -3;
                    }
                    for (int l = 0; l < 4; ++l) {
                        p1v[(w * 4 + slot) * 8 + 2 * l] = acc[l][0];
                        p1v[(w * 4 + slot) * 8 + 2 * l + 1] = acc[l][1];
                    }
                    p1u[w * 4 + slot] = cur;
                    ++slot;
                    cur = u;
                    memset(acc, 0, sizeof acc);
                }
                uint32_t A[32][4], Bm[8][32][2];
                P1Ld ld[32];
                float D[32][4] = {};
                for (int l = 0; l < 32; ++l) {
                    p1_load(a, r_e, i, NG, l, ld[l]);
                    uint32_t bb[8][2];
                    chunk_b(ld[l].c, bb);
                    for (int t = 0; t < 8; ++t) {
                        Bm[t][l][0] = bb[t][0];
                        Bm[t][l][1] = bb[t][1];
                    }
                }
                for (int t = 0; t < 8; ++t) {
                    for (int l = 0; l < 32; ++l) {
                        const uint32_t *h32 = reinterpret_cast<const uint32_t *>(xp.data()) + (g * 128 + 32 * (l & 3)) / 2;
                        uint32_t aa[4];
                        chunk_a(h32, t, aa);
                        memcpy(A[l], aa, sizeof aa);
                    }
                    mma_warp(D, A, Bm[t]);
                }
                for (int l = 0; l < 32; ++l) {
                    float dd[4] = {D[l][0], D[l][1], D[l][2], D[l][3]};
                    const float sv[2] = {ld[l].s[0], ld[l].s[1]};
                    fold(acc[l], dd, sv, ld[l].zw, l, xsum[g]);
                }
            }
            if (cur >= 0) {
                if (slot >= 4) {
                    status[1] = 7;
                    return -3;
                }
                for (int l = 0; l < 4; ++l) {
                    p1v[(w * 4 + slot) * 8 + 2 * l] = acc[l][0];
                    p1v[(w * 4 + slot) * 8 + 2 * l + 1] = acc[l][1];
                }
                p1u[w * 4 + slot] = cur;
            }
        }
        if (c1 > c0) {
            const int u0 = c0 / NG, u1 = (c1 - 1) / NG;
            const float unscale = ldexpf(1.0f, -sigx);
            for (int t = 0; t < (u1 - u0 + 1) * 8; ++t) {
                const int u = u0 + t / 8, r = t % 8;
                float v = 0.f;
                for (int w = 0; w < kWarps * 4; ++w)
                    if (p1u[w] == u)
                        v += p1v[w * 8 + r];
                const int piece = b - owner(u * NG, T, G);
                if (piece < 0 || piece >= kMaxPieces) {
                    status[1] = 8;
                    return -4;
                }
                gp[(static_cast<int64_t>(u) * kMaxPieces + piece) * 8 + r] = v * unscale;
            }
        }
    }
    // ---- phase 2, every CTA
    const int B2 = d / 8;
    for (int b = 0; b < G; ++b) {
        const int blk0 = split_lo(B2, b, G), nb = split_lo(B2, b + 1, G) - blk0;
        const Smem L{d, I, k, nb};
        if (L.bytes() > maxsmem)
            maxsmem = L.bytes();
        std::vector<uint8_t> sm(L.bytes());
        uint32_t *w2s = reinterpret_cast<uint32_t *>(sm.data() + L.w2());
        float *sc2 = reinterpret_cast<float *>(sm.data() + L.sz2());
        float *zz2 = sc2 + k * nb * 8 * G2;
        float *hf = reinterpret_cast<float *>(sm.data() + L.hf());
        uint16_t *hp = reinterpret_cast<uint16_t *>(sm.data() + L.hp());
        float *hsum = reinterpret_cast<float *>(sm.data() + L.hsum());
        float *part2 = reinterpret_cast<float *>(sm.data() + L.part2());
        const int rowb = I / 2;
        for (int r = 0; r < nv * nb * 8; ++r) {
            const int j = r / (nb * 8), o = blk0 * 8 + (r - j * nb * 8);
            const uint8_t *src = reinterpret_cast<const uint8_t *>(q2) + (static_cast<int64_t>(r_e[j]) * d + o) * rowb;
            if ((reinterpret_cast<uintptr_t>(src) & 15) || ((L.w2() + r * rowb) & 15) || (rowb & 15))
                return -5;
            memcpy(reinterpret_cast<uint8_t *>(w2s) + r * rowb, src, rowb);
        }
        for (int i = 0; i < nv * nb * 8 * G2; ++i) {
            const int r = i / G2, g = i - r * G2;
            const int j = r / (nb * 8), o = blk0 * 8 + (r - j * nb * 8);
            const int64_t e = r_e[j];
            sc2[i] = h2f(s2[(e * d + o) * G2 + g]);
            zz2[i] = nib(static_cast<uint32_t>(z2[(e * (d / 8) + o / 8) * G2 + g]), o & 7);
        }
        for (int t = 0; t < nv * I; ++t) {
            const int j = t / I, n = t - j * I;
            const int ug = j * RB + n / 8, uu = j * RB + (I + n) / 8, r = n % 8;
            float gv = 0.f, uv = 0.f;
            const int pg = owner(ug * NG + NG - 1, T, G) - owner(ug * NG, T, G) + 1;
            const int pu = owner(uu * NG + NG - 1, T, G) - owner(uu * NG, T, G) + 1;
            for (int p = 0; p < pg; ++p)
                gv += gp[(static_cast<int64_t>(ug) * kMaxPieces + p) * 8 + r];
            for (int p = 0; p < pu; ++p)
                uv += gp[(static_cast<int64_t>(uu) * kMaxPieces + p) * 8 + r];
            hf[t] = r_w[j] * silu_mul_h(gv, uv);
        }
        int r_sig[kMaxK];
        for (int j = 0; j < nv; ++j) {
            float m = 0.f;
            for (int n = 0; n < I; ++n)
                m = fmaxf(m, fabsf(hf[j * I + n]));
            r_sig[j] = f16_sigma_h(m);
        }
        for (int t = 0; t < nv * I; ++t) {
            const int j = t / I, n = t - j * I;
            const float v = ldexpf(hf[j * I + (n & ~7) + interleave(n & 7)], r_sig[j]);
            const uint16_t hi = f2h(v);
            hp[t] = hi;
            hp[nv * I + t] = f2h(v - h2f(hi));
        }
        for (int t = 0; t < nv * G2; ++t) {
            float v[32];
            for (int l = 0; l < 32; ++l) {
                v[l] = 0.f;
                for (int c = 0; c < 4; ++c) {
                    const int idx = t * 128 + c * 32 + l;
                    v[l] += h2f(hp[idx]) + h2f(hp[nv * I + idx]);
                }
            }
            hsum[t] = bfly_sum(v);
        }
        const uint32_t *h32 = reinterpret_cast<const uint32_t *>(hp);
        const int rw = I / 8;
        for (int v = 0; v < nv * nb; ++v) {
            const int j = v / nb, bl = v - j * nb;
            const int rbase = j * nb * 8 + bl * 8;
            float acc[32][2] = {};
            for (int g = 0; g < G2; ++g) {
                uint32_t Bm[8][32][2];
                for (int l = 0; l < 32; ++l) {
                    const uint4 c = *reinterpret_cast<const uint4 *>(w2s + static_cast<int64_t>(rbase + (l >> 2)) * rw + g * 16 + (l & 3) * 4);
                    uint32_t bb[8][2];
                    chunk_b(c, bb);
                    for (int t = 0; t < 8; ++t) {
                        Bm[t][l][0] = bb[t][0];
                        Bm[t][l][1] = bb[t][1];
                    }
                }
                float D[32][4] = {};
                for (int t = 0; t < 8; ++t) {
                    uint32_t A[32][4];
                    for (int l = 0; l < 32; ++l) {
                        uint32_t aa[4];
                        chunk_a(h32 + (j * I + g * 128 + 32 * (l & 3)) / 2, t, aa);
                        memcpy(A[l], aa, sizeof aa);
                    }
                    mma_warp(D, A, Bm[t]);
                    for (int l = 0; l < 32; ++l) {
                        uint32_t aa[4];
                        chunk_a(h32 + (nv * I + j * I + g * 128 + 32 * (l & 3)) / 2, t, aa);
                        memcpy(A[l], aa, sizeof aa);
                    }
                    mma_warp(D, A, Bm[t]);
                }
                for (int l = 0; l < 32; ++l) {
                    const int r0 = rbase + 2 * (l & 3);
                    const float hs = hsum[j * G2 + g];
                    for (int r = 0; r < 2; ++r)
                        acc[l][r] = fmaf(sc2[(r0 + r) * G2 + g], fmaf(-(1024.0f + zz2[(r0 + r) * G2 + g]), hs, D[l][r]),
                                         acc[l][r]);
                }
            }
            const float un = ldexpf(1.0f, -r_sig[j]);
            for (int l = 0; l < 4; ++l) {
                part2[(j * nb + bl) * 8 + 2 * l] = acc[l][0] * un;
                part2[(j * nb + bl) * 8 + 2 * l + 1] = acc[l][1] * un;
            }
        }
        for (int t = 0; t < nb * 8; ++t) {
            float yo = 0.f;
            for (int j = 0; j < nv; ++j)
                yo += part2[(j * nb + t / 8) * 8 + t % 8];
            y[blk0 * 8 + t] = yo;
        }
    }
    return maxsmem;
}
