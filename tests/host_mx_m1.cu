// host_mx_m1.cu -- host emulation of the single-token MXFP8 kernel
// (top_moe_expert_gb300/csrc/decode_mx_m1.cu) for the CPU tests.
//
// It runs the kernel's steps CTA by CTA and warp by warp with the lanes
// looped, through the kernel's own lane functions (decode_mx_m1.cuh): the
// item split, the piece loads and their addresses (global for W13, the staged
// rows for W2), the block fold, the piece numbering across CTAs, the h split
// and the slot sum.  mma.sync m16n8k16 is emulated from the PTX fragment
// layouts (products exact, sums in double, rounded to float).  The routing
// is given (the kernel's in-kernel top-k is the tested routing kernel's).
#include <cmath>
#include <cstring>
#include <vector>
#include <cuda_bf16.h>
#include "decode_mx_m1.cuh"

using namespace moe::dx1;

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

static float h2f(uint16_t b)
{
    __half_raw r;
    r.x = b;
    return __half2float(__half(r));
}
static uint16_t f2h(float v)
{
    __half h = __float2half_rn(v);
    return __half_raw(h).x;
}
static float lo16(uint32_t r) { return h2f(static_cast<uint16_t>(r & 0xFFFFu)); }
static float hi16(uint32_t r) { return h2f(static_cast<uint16_t>(r >> 16)); }

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

// One item of a warp: acc[lane][2] += the item's block-folded dots.
static void emu_item(float (&acc)[32][2], const Ld (&ld)[32], const uint32_t *a32, int base)
{
    for (int p = 0; p < 2; ++p) {
        float D[32][4] = {};
        for (int t = 0; t < 2; ++t) {
            uint32_t A[32][4], B[32][2];
            for (int l = 0; l < 32; ++l) {
                uint32_t aa[4];
                mx_a(a32, base, p, t, l, aa);
                memcpy(A[l], aa, sizeof aa);
                mx_b(ld[l], p, t, B[l][0], B[l][1]);
            }
            mma_warp(D, A, B);
        }
        for (int l = 0; l < 32; ++l) {
            const float dd[4] = {D[l][0], D[l][1], D[l][2], D[l][3]};
            mx_fold(acc[l], dd, ld[l], p);
        }
    }
}

extern "C" int mx_m1_emulate(const uint16_t *x_bf16, const int32_t *ids, const float *wts, const uint8_t *q13,
                             const uint8_t *s13, const uint8_t *q2, const uint8_t *s2, float *gp, float *y, int k,
                             int d, int I, int E, int G, int stage, int *status)
{
    const int NG = d / 64, NG2 = I / 64, RB = 2 * I / 8;
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
        __nv_bfloat16_raw r;
        r.x = x_bf16[i];
        return __bfloat162float(__nv_bfloat16(r));
    };
    float xm = 0.f;
    for (int i = 0; i < d; ++i)
        xm = fmaxf(xm, fabsf(xval(i)));
    const int sigx = f16_sigma_h(xm);
    std::vector<uint16_t> xp(d);
    for (int i = 0; i < d; ++i)
        xp[i] = f2h(ldexpf(xval(i), sigx));
    const uint32_t *x32 = reinterpret_cast<const uint32_t *>(xp.data());
    const int T = nv * RB * NG;
    int maxsmem = 0;
    // ---- phase 1
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
                const int u = i / NG, c = i - u * NG;
                if (u != cur) {
                    if (slot >= 4)
                        return -3;
                    for (int l = 0; l < 4; ++l) {
                        p1v[(w * 4 + slot) * 8 + 2 * l] = acc[l][0];
                        p1v[(w * 4 + slot) * 8 + 2 * l + 1] = acc[l][1];
                    }
                    p1u[w * 4 + slot] = cur;
                    ++slot;
                    cur = u;
                    memset(acc, 0, sizeof acc);
                }
                const int j = u / RB, rb = u - j * RB;
                Ld ld[32];
                for (int l = 0; l < 32; ++l)
                    mx_load(q13, s13, static_cast<int64_t>(r_e[j]) * 2 * I + rb * 8, d, c, l, ld[l]);
                emu_item(acc, ld, x32, c * 64);
            }
            if (cur >= 0) {
                if (slot >= 4)
                    return -3;
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
                if (piece < 0 || piece >= kMaxPieces)
                    return -4;
                gp[(static_cast<int64_t>(u) * kMaxPieces + piece) * 8 + r] = v * unscale;
            }
        }
    }
    // ---- phase 2
    const int B2 = d / 8;
    for (int b = 0; b < G; ++b) {
        const int blk0 = split_lo(B2, b, G), nb = split_lo(B2, b + 1, G) - blk0;
        const Smem L{d, I, k, nb, stage};
        if (L.bytes() > maxsmem)
            maxsmem = L.bytes();
        std::vector<uint8_t> sm(L.bytes(), 0xFF);
        uint8_t *w2s = sm.data() + L.w2();
        uint8_t *s2s = sm.data() + L.s2();
        float *hf = reinterpret_cast<float *>(sm.data() + L.hf());
        uint16_t *hp = reinterpret_cast<uint16_t *>(sm.data() + L.hp());
        float *part2 = reinterpret_cast<float *>(sm.data() + L.part2());
        for (int r = 0; stage && r < nv * nb * 8; ++r) {
            const int j = r / (nb * 8), o = blk0 * 8 + (r - j * nb * 8);
            const uint8_t *src = q2 + (static_cast<int64_t>(r_e[j]) * d + o) * I;
            if ((reinterpret_cast<uintptr_t>(src) & 15) || ((L.w2() + r * I) & 15) || (I & 15))
                return -5;
            memcpy(w2s + r * I, src, I);
        }
        for (int i = 0; stage && i < nv * nb * 8 * (I / 32); ++i) {
            const int r = i / (I / 32), c = i - r * (I / 32);
            const int j = r / (nb * 8), o = blk0 * 8 + (r - j * nb * 8);
            s2s[i] = s2[(static_cast<int64_t>(r_e[j]) * d + o) * (I / 32) + c];
        }
        for (int t = 0; t < nv * I; ++t) {
            const int j = t / I, n2 = t - j * I;
            const int ug = j * RB + n2 / 8, uu = j * RB + (I + n2) / 8, r = n2 % 8;
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
            for (int n2 = 0; n2 < I; ++n2)
                m = fmaxf(m, fabsf(hf[j * I + n2]));
            r_sig[j] = f16_sigma_h(m);
        }
        for (int t = 0; t < nv * I; ++t) {
            const float v = ldexpf(hf[t], r_sig[t / I]);
            hp[t] = f2h(v);
            hp[nv * I + t] = f2h(v - h2f(hp[t]));
        }
        const uint32_t *h32 = reinterpret_cast<const uint32_t *>(hp);
        for (int v = 0; v < nv * nb; ++v) {
            const int j = v / nb, bl = v - j * nb, rbase = j * nb * 8 + bl * 8;
            float acc[32][2] = {};
            for (int c = 0; c < NG2; ++c) {
                Ld ld[32];
                for (int l = 0; l < 32; ++l)
                    if (stage)
                        mx_load(w2s, s2s, rbase, I, c, l, ld[l]);
                    else
                        mx_load(q2, s2, static_cast<int64_t>(r_e[j]) * d + (blk0 + bl) * 8, I, c, l, ld[l]);
                emu_item(acc, ld, h32 + j * I / 2, c * 64);
                emu_item(acc, ld, h32 + (nv + j) * I / 2, c * 64);
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
