// grouped_mx_mma.cuh -- lane-level pieces of the small-block MXFP8 kernel
// (grouped_mx_mma.cu), __host__ __device__ so that a host build can run the
// kernel's index arithmetic lane by lane on the CPU.  The weight operand is
// that of decode_mx_m1.cuh (E4M3 pairs converted exactly to f16, one E8M0
// scale per 32-value block applied to the block's FP32 sum); the activation
// operand is one MoE block of up to 16 rows, staged in f16 in natural order.
#pragma once
#include "decode_mx_m1.cuh"

namespace moe {
namespace gmx {

using dx1::Ld;
using dx1::e8m0;
using dx1::mx_b;
using dx1::mx_load;

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 16;                 // rows of an M-tile: blocks of 16 rows
constexpr int kPF = 4;                    // items in flight per warp
constexpr uint64_t kWaitNs = 2000000000ull;

struct Args {
    const __nv_bfloat16 *x;               // [M][d]
    const float *wts;                     // [M*k]
    const int32_t *sorted;                // [cap_rows] route ids, sentinel M*k
    const int32_t *expert_ids;            // [cap_blocks]
    const int32_t *npp;                   // [1] rows after padding
    const uint8_t *q13, *s13;             // [E][2I][d], [E][2I][d/32]
    const uint8_t *q2, *s2;               // [E][d][I],  [E][d][I/32]
    int32_t *done;                        // [cap_blocks] gate/up units finished per block (zeroed)
    float *gu;                            // [M*k][2I]
    float *yr;                            // [M*k][d]
    int32_t *dev_status;
    int M, k, d, I, E, mk, cap_blocks;
};

// Shared memory: the A operand of one block (16 rows, each padded by 16
// bytes so that the eight rows a warp reads at once fall in different banks)
// and per-row routes and scale exponents.  Phase 1 stages x ([16][d]),
// phase 2 h hi and lo ([2][16][I]) in the same region.
struct Smem {
    int d, I;
    DA1_HD static int al(int v) { return (v + 15) & ~15; }
    DA1_HD int xrow() const { return 2 * d + 16; }
    DA1_HD int hrow() const { return 2 * I + 16; }
    DA1_HD int a() const { return 0; }
    DA1_HD int a_bytes() const { return kRows * xrow() > 2 * kRows * hrow() ? kRows * xrow() : 2 * kRows * hrow(); }
    DA1_HD int rows() const { return al(a() + a_bytes()); }          // route, sigma [16] each
    DA1_HD int bytes() const { return al(rows() + 2 * 4 * kRows); }
};

// A registers of MMA t of piece p: rows lane/4 and lane/4 + 8 of the staged
// operand (row stride `rs` bytes), halves base + 32p + 8(lane%4) + 4t + {0,1}
// (a0 / a1) and {2, 3} (a2 / a3).
DA1_HD void a_regs(const uint8_t *abase, int rs, int base, int p, int t, int lane, uint32_t (&aa)[4])
{
    const int gl = lane >> 2;
    const int h = base + 32 * p + 8 * (lane & 3) + 4 * t;
    const uint32_t *r0 = reinterpret_cast<const uint32_t *>(abase + gl * rs);
    const uint32_t *r1 = reinterpret_cast<const uint32_t *>(abase + (gl + 8) * rs);
    aa[0] = r0[h / 2];
    aa[1] = r1[h / 2];
    aa[2] = r0[h / 2 + 1];
    aa[3] = r1[h / 2 + 1];
}

// Block fold: rows lane/4 (D 0, 1) and lane/4 + 8 (D 2, 3) against weight rows
// 2(lane%4) + {0, 1}: acc += D * 2^(s - 127) of piece p's block.
DA1_HD void fold4(float (&acc)[4], const float (&dd)[4], const Ld &o, int p)
{
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float sc = e8m0((o.s[r] >> (8 * p)) & 0xFFu);
        acc[r] = fmaf(dd[r], sc, acc[r]);
        acc[2 + r] = fmaf(dd[2 + r], sc, acc[2 + r]);
    }
}

}  // namespace gmx
}  // namespace moe
