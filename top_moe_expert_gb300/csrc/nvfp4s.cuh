// nvfp4s.cuh -- decoding of paired 4:8 sparse NVFP4 weights, usable on the
// device and (for the host emulation test) on the CPU.
//
// "Hardware-Native Joint Sparse-Quantization for Trillion-Scale
// Mixture-of-Experts", App. A: in every group of 8 weights along K two
// adjacent pairs are kept; the 16 kept values of a block of 32 weights are
// E2M1 codes that share one UE4M3 scale; one FP32 constant per matrix.
// Packed layout of one row (K % 64 == 0), as include/moe_ffn.h states it:
//   vals  K/4 bytes:  group g's four kept codes in bytes 2g, 2g+1, low
//                     nibble first (pair p0's two values, then pair p1's)
//   meta  K/16 bytes: group g's pattern nibble p0 | p1 << 2 in byte g/2,
//                     low nibble for even g
//   scale K/32 bytes: UE4M3 codes
// A 64-weight chunk c is 16 bytes of vals, 4 bytes of meta and 2 scale bytes,
// all at naturally aligned offsets (16c, 4c, 2c).
#pragma once

#include <cstdint>
#include <cmath>

#if defined(__CUDACC__)
#define NV4_HD __host__ __device__ __forceinline__
#else
#define NV4_HD inline
#endif

namespace moe {
namespace nv4 {

// E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0
// is subnormal.  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
NV4_HD float e2m1(uint32_t c)
{
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const float mag = e ? static_cast<float>(2u + m) * static_cast<float>(1u << e) * 0.25f : 0.5f * m;
    return (c & 8u) ? -mag : mag;
}

// UE4M3 scale: E4M3 with the sign bit clear (codes 0x00..0x7E), exponent
// bias 7, exponent 0 subnormal.  Exact in binary32.
NV4_HD float ue4m3(uint32_t c)
{
    const int e = static_cast<int>((c >> 3) & 15u), m = static_cast<int>(c & 7u);
    return ldexpf(static_cast<float>(e ? 8 + m : m), (e ? e : 1) - 10);
}

// Sum over the chunk's 64 logical weights of weight * x, without the
// per-matrix constant: per block of 32, UE4M3(scale) * sum of the kept
// E2M1 values times their activations.  v: the 16 value bytes as four
// little-endian words; meta: the 4 pattern bytes; sc2: the 2 scale bytes;
// x: the chunk's 64 activations.  Every x index stays inside its group of 8.
NV4_HD float chunk_dot(const uint32_t (&v)[4], uint32_t meta, uint32_t sc2, const float *x)
{
    float acc = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        float sb = 0.f;
#pragma unroll
        for (int gi = 4 * blk; gi < 4 * blk + 4; ++gi) {
            const uint32_t nib = (meta >> (4 * gi)) & 15u;
            const int o0 = 8 * gi + 2 * static_cast<int>(nib & 3u), o1 = 8 * gi + 2 * static_cast<int>(nib >> 2);
            const uint32_t codes = (v[gi >> 1] >> (16 * (gi & 1))) & 0xFFFFu;
            sb = fmaf(e2m1(codes & 15u), x[o0], sb);
            sb = fmaf(e2m1((codes >> 4) & 15u), x[o0 + 1], sb);
            sb = fmaf(e2m1((codes >> 8) & 15u), x[o1], sb);
            sb = fmaf(e2m1((codes >> 12) & 15u), x[o1 + 1], sb);
        }
        acc = fmaf(ue4m3((sc2 >> (8 * blk)) & 0xFFu), sb, acc);
    }
    return acc;
}

}  // namespace nv4
}  // namespace moe
