// decode_mx_m1.cuh -- lane-level pieces of the single-token MXFP8 kernel
// (decode_mx_m1.cu), __host__ __device__ so that a host build can run the
// kernel's index arithmetic lane by lane on the CPU.
//
// MXFP8 weights (OCP microscaling): E4M3 codes with one E8M0 scale per 32
// values along K.  Dot products run on mma.sync m16n8k16 (f16 x f16 -> f32):
// the B operand is eight weight rows, each E4M3 pair converted exactly to an
// f16 pair (E4M3 is a subset of f16); A is the activation vector in every
// row (only row 0 of D is read).  An item is 8 rows x 64 K values; lane
// (g = lane/4, q = lane%4) loads two 8-byte pieces of row g -- K values
// [8q, 8q+8) and [32 + 8q, 32 + 8q + 8) of the item -- so that each pair of
// MMAs covers exactly one 32-value scale block.  The block's result is
// D * 2^(s - 127), added in FP32.
#pragma once
#include <cstdint>
#include <cstring>
#include <cuda_fp16.h>

#include "decode_awq_m1.cuh"

namespace moe {
namespace dx1 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxK = 32;
constexpr int kMaxPieces = 4;        // CTAs one unit of phase 1 may span

struct Args {
    const __nv_bfloat16 *x;     // [d]
    const int32_t *ids;         // [k] (given routing) ...
    const float *wts;
    const float *logits;        // ... or [E] router logits (routing in the kernel)
    int32_t *ids_out;           // CTA 0 writes the chosen ids / weights
    float *wts_out;
    const uint8_t *q13;         // [E][2I][d] E4M3
    const uint8_t *s13;         // [E][2I][d/32] E8M0
    const uint8_t *q2;          // [E][d][I]
    const uint8_t *s2;          // [E][d][I/32]
    unsigned long long *bar;    // arrival counter (workspace bytes 0..8)
    float *gp;                  // [k * 2I / 8][kMaxPieces][8] phase-1 partials (workspace from byte 256)
    void *y;                    // [d] bf16 or f32
    int32_t *dev_status;
    int y_f32;
    int k, d, I, E;
};

DA1_HD int split_lo(int T, int b, int G) { return static_cast<int>(static_cast<int64_t>(T) * b / G); }
DA1_HD int owner(int i, int T, int G) { return static_cast<int>((static_cast<int64_t>(i + 1) * G - 1) / T); }

// E4M3 pair (low byte first) -> f16 pair, exact.
DA1_HD uint32_t e4m3x2_f16x2(uint32_t v16)
{
#ifdef __CUDA_ARCH__
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(v16)));
    return r;
#else
    // OCP E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; S.1111.111 is NaN
    auto one = [](uint32_t c) -> uint16_t {
        const uint32_t s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
        float v;
        if (e == 15 && m == 7)
            v = nanf("");
        else if (e == 0)
            v = ldexpf(static_cast<float>(m), -9);
        else
            v = ldexpf(static_cast<float>(8 + m), static_cast<int>(e) - 10);
        __half h = __float2half_rn(s ? -v : v);
        return __half_raw(h).x;
    };
    return static_cast<uint32_t>(one(v16 & 0xFFu)) | (static_cast<uint32_t>(one((v16 >> 8) & 0xFFu)) << 16);
#endif
}

// E8M0 scale byte -> 2^(s - 127) (s = 0 -> 2^-127).
DA1_HD float e8m0(uint32_t s)
{
    const uint32_t bits = s == 0 ? 0x00400000u : (s << 23);
#ifdef __CUDA_ARCH__
    return __uint_as_float(bits);
#else
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
#endif
}

// Operands of one item (unit = 8 rows of a K-contiguous E4M3 matrix starting
// at wrow0, chunk c of 64 K values) for one lane: its two 8-byte pieces of
// row wrow0 + lane/4 and the scale bytes of rows wrow0 + 2(lane%4) + {0, 1}
// for the chunk's two blocks (low byte: first block).
struct Ld {
    uint2 p[2];
    uint32_t s[2];
};

// Plain loads: the same loader reads the weights from global memory (phase
// 1) and the staged down-projection rows from shared memory (phase 2).
#define DX1_LD8(p) (*reinterpret_cast<const uint2 *>(p))
#define DX1_LDU16(p) (*reinterpret_cast<const unsigned short *>(p))

DA1_HD void mx_load(const uint8_t *q, const uint8_t *s, int64_t wrow0, int Kd, int c, int lane, Ld &o)
{
    const int q4 = lane & 3;
    const uint8_t *row = q + (wrow0 + (lane >> 2)) * Kd + c * 64 + 8 * q4;
    o.p[0] = DX1_LD8(row);
    o.p[1] = DX1_LD8(row + 32);
    const int64_t sr = wrow0 + 2 * q4;
    o.s[0] = DX1_LDU16(s + sr * (Kd / 32) + 2 * c);
    o.s[1] = DX1_LDU16(s + (sr + 1) * (Kd / 32) + 2 * c);
}

// B registers of MMA t (0, 1) of piece p: values 4t .. 4t+3 of the piece.
DA1_HD void mx_b(const Ld &o, int p, int t, uint32_t &b0, uint32_t &b1)
{
    const uint32_t w = t == 0 ? o.p[p].x : o.p[p].y;
    b0 = e4m3x2_f16x2(w & 0xFFFFu);
    b1 = e4m3x2_f16x2(w >> 16);
}

// A registers of MMA t of piece p from the staged activation (natural
// order, f16): halves base + 32p + 8q + 4t + {0, 1} and {2, 3}, the same
// vector in every row.
DA1_HD void mx_a(const uint32_t *x32, int base, int p, int t, int lane, uint32_t (&a)[4])
{
    const int h = base + 32 * p + 8 * (lane & 3) + 4 * t;
    a[0] = a[1] = x32[h / 2];
    a[2] = a[3] = x32[h / 2 + 1];
}

// Block fold of the lane's two rows: acc += D * 2^(s - 127).
DA1_HD void mx_fold(float (&acc)[2], const float (&dd)[4], const Ld &o, int p)
{
#pragma unroll
    for (int r = 0; r < 2; ++r)
        acc[r] = fmaf(dd[r], e8m0((o.s[r] >> (8 * p)) & 0xFFu), acc[r]);
}

// Shared-memory plan (bytes from the dynamic base, 16-byte aligned regions).
//   nb: output blocks of 8 of this CTA (phase 2); stage: 1 when the CTA's W2
//   rows and their scales are staged in shared memory, 0 when phase 2 reads
//   them from global memory (shapes whose rows do not fit)
struct Smem {
    int d, I, k, nb, stage;
    DA1_HD static int al(int v) { return (v + 15) & ~15; }
    DA1_HD int xp() const { return 0; }                                   // [d] f16
    DA1_HD int route() const { return al(xp() + 2 * d); }                 // e [32], w [32], sigma [32]
    DA1_HD int mbar() const { return route() + 3 * kMaxK * 4; }           // u64
    DA1_HD int part1() const { return al(mbar() + 8); }                   // [16][4][8] f32 + [16][4] unit ids
    DA1_HD int w2() const { return al(part1() + kWarps * 4 * 8 * 4 + kWarps * 4 * 4); }  // [k][nb*8][I] E4M3
    DA1_HD int s2() const { return al(w2() + stage * k * nb * 8 * I); }  // [k][nb*8][I/32] E8M0
    DA1_HD int hf() const { return al(s2() + stage * k * nb * 8 * (I / 32)); }   // [k][I] f32 (h)
    DA1_HD int hp() const { return al(hf() + 4 * k * I); }               // [2][k][I] f16 hi / lo
    DA1_HD int part2() const { return al(hp() + 2 * 2 * k * I); }        // [k][nb][8] f32
    DA1_HD int bytes() const { return al(part2() + 4 * k * nb * 8); }
};

}  // namespace dx1
}  // namespace moe
