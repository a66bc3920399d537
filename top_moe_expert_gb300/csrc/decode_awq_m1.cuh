// decode_awq_m1.cuh -- lane-level pieces of the single-token 4-bit AWQ
// kernel (decode_awq_m1.cu).  They are __host__ __device__ so that a host
// build can run the kernel's index arithmetic lane by lane on the CPU.
//
// Weights are packed AWQ ("Route-Block Membership Selects Packed-AWQ
// Arithmetic", opening paragraph): 4-bit values q with a 4-bit zero z and an
// fp16 scale s per group of 128 along K, weight = (q - z) s.
//
// Dot products run on mma.sync m16n8k16 (f16 x f16 -> f32) used as a dot
// engine: B = eight weight rows x 16 K values, A = the activation vector in
// every row (only row 0 of D is read).  A packed word w (values v0..v7 of a
// row, value i in bits 4i..4i+3) gives four f16x2 registers with one logic
// operation each and no conversion:
//     ((w >> 4i) & 0x000F000F) | 0x64006400  =  (1024 + v_i, 1024 + v_{i+4})
// (0x6400 is 1024 in f16, whose unit in the last place is 1).  A lane's
// 16-byte chunk (32 values of one row) is thus the B operand of eight MMAs in
// K order 0,4,1,5,2,6,3,7 within each word, and the activation is staged in
// the same order.  Over a group the MMAs form D = sum (1024 + v) a in FP32;
// the group's result is s (D - (1024 + z) sum a), which equals
// s sum (v - z) a: the zero and the offset leave in one FP32 step.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

#define DA1_HD __host__ __device__ __forceinline__

namespace moe {
namespace da1 {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxK = 32;
constexpr int kMaxPieces = 4;        // CTAs one unit of phase 1 may span

struct Args {
    const void *x;              // [d] fp16 (x_bf16 == 0) or bf16
    const int32_t *ids;         // [k]
    const float *wts;           // [k]
    const uint32_t *q13;        // [E][2I][d/8]
    const uint16_t *s13;        // [E][2I][d/128] fp16 bits
    const int32_t *z13;         // [E][2I/8][d/128]
    const uint32_t *q2;         // [E][d][I/8]
    const uint16_t *s2;         // [E][d][I/128]
    const int32_t *z2;          // [E][d/8][I/128]
    unsigned long long *bar;    // arrival counter (workspace bytes 0..8)
    float *gp;                  // [k * 2I / 8][kMaxPieces][8] phase-1 partials (workspace from byte 256)
    void *y;                    // [d] bf16 or f32
    int32_t *dev_status;
    int x_bf16, y_f32;
    int k, d, I, E;
};

// CTA b of G owns items [T b / G, T (b + 1) / G); the owner of item i.
DA1_HD int split_lo(int T, int b, int G) { return static_cast<int>(static_cast<int64_t>(T) * b / G); }
DA1_HD int owner(int i, int T, int G) { return static_cast<int>((static_cast<int64_t>(i + 1) * G - 1) / T); }

// Position p (0..7) of a staged word holds value interleave(p) of the word.
DA1_HD int interleave(int p) { return (p >> 1) + 4 * (p & 1); }

DA1_HD uint32_t nib_pair(uint32_t w, int i) { return ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u; }

// B operand of the eight MMAs of one 16-byte chunk: MMA t uses
// (b[t][0], b[t][1]) = words t/2, nibble pairs 2(t%2) and 2(t%2)+1.
DA1_HD void chunk_b(const uint4 &c, uint32_t (&b)[8][2])
{
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        b[t][0] = nib_pair(w[t >> 1], 2 * (t & 1));
        b[t][1] = nib_pair(w[t >> 1], 2 * (t & 1) + 1);
    }
}

// A operand of MMA t from 32 staged halves (the lane's chunk): registers
// a0 = a1 = halves 4t, 4t+1;  a2 = a3 = halves 4t+2, 4t+3.
DA1_HD void chunk_a(const uint32_t *h32, int t, uint32_t (&a)[4])
{
    a[0] = a[1] = h32[2 * t];
    a[2] = a[3] = h32[2 * t + 1];
}

DA1_HD float f16bits(uint16_t b)
{
    __half_raw r;
    r.x = b;
    return __half2float(__half(r));
}

DA1_HD float nib(uint32_t w, int i) { return static_cast<float>((w >> (4 * i)) & 0xFu); }

// Shared-memory plan (bytes from the dynamic base, 16-byte aligned regions).
//   nb: output blocks of 8 of this CTA (phase 2)
struct Smem {
    int d, I, k, nb;
    DA1_HD static int al(int v) { return (v + 15) & ~15; }
    DA1_HD int xp() const { return 0; }                                   // [d] f16, staged order
    DA1_HD int xsum() const { return al(xp() + 2 * d); }                  // [d/128] f32
    DA1_HD int route() const { return al(xsum() + 4 * (d / 128)); }       // e [32], w [32], sigma [32]
    DA1_HD int mbar() const { return route() + 3 * kMaxK * 4; }           // u64
    DA1_HD int part1() const { return al(mbar() + 8); }                   // [16 warps][4][8] f32 + [16][4] unit ids
    DA1_HD int w2() const { return al(part1() + kWarps * 4 * 8 * 4 + kWarps * 4 * 4); }  // [k][nb*8][I/8] u32
    DA1_HD int sz2() const { return al(w2() + k * nb * 8 * (I / 2)); }    // [k][nb*8][I/128] scale, then zero
    DA1_HD int hf() const { return al(sz2() + 2 * k * nb * 8 * (I / 128) * 4); }   // [k][I] f32 (h)
    DA1_HD int hp() const { return al(hf() + 4 * k * I); }                // [2][k][I] f16 hi / lo, staged order
    DA1_HD int hsum() const { return al(hp() + 2 * 2 * k * I); }          // [k][I/128] f32
    DA1_HD int part2() const { return al(hsum() + 4 * k * (I / 128)); }   // [k][nb][8] f32
    DA1_HD int bytes() const { return al(part2() + 4 * k * nb * 8); }
};


#ifdef __CUDA_ARCH__
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
#define DA1_LD4(p) ld_stream(p)
#define DA1_LDU16(p) __ldg(reinterpret_cast<const unsigned short *>(p))
#define DA1_LDI32(p) __ldg(p)
#else
#define DA1_LD4(p) (*reinterpret_cast<const uint4 *>(p))
#define DA1_LDU16(p) (*reinterpret_cast<const unsigned short *>(p))
#define DA1_LDI32(p) (*(p))
#endif

// Operands of one phase-1 item (unit u = 8 rows of W13 of one slot, group g)
// for one lane: its 16-byte chunk of row rb*8 + lane/4, and the scale and
// zero of rows rb*8 + 2(lane%4) + {0, 1} (the rows its D registers hold).
struct P1Ld {
    uint4 c;
    float s[2];
    uint32_t zw;
};

DA1_HD void p1_load(const Args &a, const int *r_e, int i, int NG, int lane, P1Ld &o)
{
    const int I = a.I, RB = 2 * I / 8;
    const int u = i / NG, g = i - u * NG;
    const int j = u / RB, rb = u - j * RB;
    const int64_t e = r_e[j];
    const int q = lane & 3;
    const int64_t row = e * 2 * I + rb * 8 + (lane >> 2);
    o.c = DA1_LD4(a.q13 + row * (a.d / 8) + g * 16 + q * 4);
    const int64_t srow = e * 2 * I + rb * 8 + 2 * q;
    o.s[0] = f16bits(DA1_LDU16(a.s13 + srow * NG + g));
    o.s[1] = f16bits(DA1_LDU16(a.s13 + (srow + 1) * NG + g));
    o.zw = static_cast<uint32_t>(DA1_LDI32(a.z13 + (e * RB + rb) * NG + g));
}

// Group result of the lane's two rows: s (D - (1024 + z) sum a).
DA1_HD void fold(float (&acc)[2], const float (&dd)[4], const float (&s)[2], uint32_t zw, int lane, float asum)
{
    const int q = lane & 3;
#pragma unroll
    for (int r = 0; r < 2; ++r)
        acc[r] = fmaf(s[r], fmaf(-(1024.0f + nib(zw, 2 * q + r)), asum, dd[r]), acc[r]);
}

}  // namespace da1
}  // namespace moe
