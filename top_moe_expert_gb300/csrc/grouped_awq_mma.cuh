// grouped_awq_mma.cuh -- lane-level pieces of the small-block grouped AWQ
// kernel (grouped_awq_mma.cu), __host__ __device__ so that a host build can
// run the kernel's index arithmetic lane by lane on the CPU.  The operand
// forms are those of decode_awq_m1.cuh.
#pragma once
#include "decode_awq_m1.cuh"

namespace moe {
namespace gsm {

using da1::chunk_b;
using da1::f16bits;
using da1::interleave;
using da1::nib;
#ifdef __CUDA_ARCH__
using da1::ld_stream;
#endif

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 16;                 // rows of an M-tile: b <= 16
constexpr int kPF = 4;                    // items in flight per warp
constexpr uint64_t kWaitNs = 2000000000ull;

struct Args {
    const void *x;                        // [M][d] fp16 or bf16
    const float *wts;                     // [M*k]
    const int32_t *sorted;                // [cap_rows] route ids, sentinel M*k
    const int32_t *expert_ids;            // [cap_rows / b]
    const int32_t *npp;                   // [1] rows after padding
    const uint32_t *q13;                  // [E][2I][d/8]
    const uint16_t *s13;                  // [E][2I][d/128]
    const int32_t *z13;                   // [E][2I/8][d/128]
    const uint32_t *q2;                   // [E][d][I/8]
    const uint16_t *s2;                   // [E][d][I/128]
    const int32_t *z2;                    // [E][d/8][I/128]
    int32_t *done;                        // [cap_rows / b] gate/up units finished per block (zeroed)
    float *gu;                            // [M*k][2I]
    float *yr;                            // [M*k][d]
    int32_t *dev_status;
    int x_bf16;
    int M, k, d, I, E, b, mk;
    int cap_blocks;                       // entries of expert_ids / done: the blocks read are clamped to it
};

// Shared memory: the A operand of one block (rows padded by 16 bytes so
// that the eight rows a warp reads at once fall in different banks), its
// per-row scale exponents and routes, and per-(row, group) sums.  Phase 1
// stages x ([16][d]), phase 2 h hi and lo ([2][16][I]) in the same region.
struct Smem {
    int d, I;
    DA1_HD static int al(int v) { return (v + 15) & ~15; }
    DA1_HD int xrow() const { return 2 * d + 16; }                    // bytes per staged x row
    DA1_HD int hrow() const { return 2 * I + 16; }                    // bytes per staged h row
    DA1_HD int a() const { return 0; }
    DA1_HD int a_bytes() const { return kRows * xrow() > 2 * kRows * hrow() ? kRows * xrow() : 2 * kRows * hrow(); }
    DA1_HD int sums() const { return al(a() + a_bytes()); }            // [16][max(d, I)/128] f32
    DA1_HD int rows() const { return al(sums() + 4 * kRows * ((d > I ? d : I) / 128)); }   // route, sigma [16] each
    DA1_HD int bytes() const { return al(rows() + 2 * 4 * kRows); }
};

// Operands of one item (unit = 8 weight rows starting at wrow0 of a matrix
// with K = Kd, group g) for one lane: its 16-byte chunk of row wrow0 + lane/4,
// the scales of rows wrow0 + 2(lane%4) + {0, 1} and their zero word.
struct Ld {
    uint4 c;
    float s[2];
    uint32_t zw;
};

DA1_HD void load_item(const uint32_t *q, const uint16_t *s, const int32_t *z, int64_t wrow0, int Kd, int g,
                      int lane, Ld &o)
{
    const int NG = Kd / 128, q4 = lane & 3;
    o.c = DA1_LD4(q + (wrow0 + (lane >> 2)) * (Kd / 8) + g * 16 + q4 * 4);
    const int64_t sr = wrow0 + 2 * q4;
    o.s[0] = f16bits(DA1_LDU16(s + sr * NG + g));
    o.s[1] = f16bits(DA1_LDU16(s + (sr + 1) * NG + g));
    o.zw = static_cast<uint32_t>(DA1_LDI32(z + (wrow0 / 8) * NG + g));
}

// A registers of MMA t of an item: rows lane/4 and lane/4 + 8 of the staged
// operand (row stride `rs` bytes), the lane's 32 values starting at half
// `off`: a0 / a1 = halves 4t, 4t+1 of the two rows, a2 / a3 = halves 4t+2, 4t+3.
DA1_HD void a_regs(const uint8_t *abase, int rs, int off, int lane, int t, uint32_t (&aa)[4])
{
    const int gl = lane >> 2;
    const uint32_t *r0 = reinterpret_cast<const uint32_t *>(abase + gl * rs + off * 2);
    const uint32_t *r1 = reinterpret_cast<const uint32_t *>(abase + (gl + 8) * rs + off * 2);
    aa[0] = r0[2 * t];
    aa[1] = r1[2 * t];
    aa[2] = r0[2 * t + 1];
    aa[3] = r1[2 * t + 1];
}

// Fold of one group into the lane's four accumulators: rows lane/4 (D 0, 1)
// and lane/4 + 8 (D 2, 3) of A against weight rows 2(lane%4) + {0, 1}.
DA1_HD void fold4(float (&acc)[4], const float (&dd)[4], const Ld &ld, int lane, float sum0, float sum1)
{
    const int q4 = lane & 3;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float off = -(1024.0f + nib(ld.zw, 2 * q4 + r));
        acc[r] = fmaf(ld.s[r], fmaf(off, sum0, dd[r]), acc[r]);
        acc[2 + r] = fmaf(ld.s[r], fmaf(off, sum1, dd[2 + r]), acc[2 + r]);
    }
}

}  // namespace gsm
}  // namespace moe
