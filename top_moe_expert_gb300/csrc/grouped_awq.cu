// grouped_awq.cu -- expert-centric grouped path for 4-bit AWQ weights.
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic" (arXiv 2607.26316),
// opening paragraph: packed-AWQ MoE GEMMs (4-bit values, group 128 along K,
// fp16 scale and 4-bit zero per group) applied to the aligned rows, one MoE
// block of b rows at a time; its schedule paragraphs show that a split-K
// schedule with a global reduction makes a route's bits depend on its block
// membership.  Here every output element accumulates its K-tiles in one
// fixed ascending order in one TMEM accumulator -- no split-K, no atomics --
// so the result depends on neither membership nor grid, and repeats are
// bit-identical.
//
// The tensor cores take fp16 x fp16 (tcgen05 kind::f16, FP32 accumulate):
//   gather_kernel   : Xg[rho] = x[route(rho) / k] as fp16 (zero for padding)
//   gemm_kernel     : both GEMMs in one persistent kernel -- first-GEMM tiles
//                     [g;u] = W13_e Xg^T, epilogue h = SiLU(g) * u -> fp16 Hg;
//                     then second-GEMM tiles W2_e Hg^T, epilogue
//                     Yr[route] = w_route * acc
//   combine         : y[t] = sum over slots j (in order) of Yr[t*k + j]
// The A operand is dequantized on chip into tensor memory: TMA brings each
// k-step's packed tile (256 rows x 128 values = 64 bytes per row) and the
// activation tile into shared memory, bulk copies bring each tile's group
// scales and zeros, and dequantizing warps turn the nibbles into fp16
// w = (q - z) * s -- (q - z) exactly through the 0x6400 exponent trick, one
// rounding in the multiply -- and store them with tcgen05.st as the MMA's A
// operand: row m in TMEM lane m, two values per column.  Four warps (one per
// TMEM lane quadrant) dequantize one half of a k-step (a "unit", 128 rows);
// kDqGroups such groups take the units in turn, so each has several units'
// time for its chain of waits and stores.  Shared memory then holds only the
// packed ring, deep enough to cover DRAM latency.
//
// K order inside the tensor-core operands.  One AND-OR of a packed word with
// 0x000F000F | 0x64006400 yields nibbles i and i + 4 as an fp16 pair, so the
// dequantized row holds each run of 8 values in the order
// 0, 4, 1, 5, 2, 6, 3, 7.  The contraction does not care about the order of
// its terms as long as both operands use the same one: the gather writes Xg
// and the GEMM1 epilogue writes Hg in that order too (interleave_pos).
//
// The same kernel, instantiated for paired 4:8 sparse NVFP4 weights ("Hardware-
// Native Joint Sparse-Quantization for Trillion-Scale Mixture-of-Experts",
// Sec. 3.4 and App. D.1: E2M1 values, pair metadata and one UE4M3 scale per
// 32 weights; activations quantized at run time into 32-element blocks;
// the tensor-wide scales folded into one factor per expert, applied to the
// FP32 accumulator in the epilogue), runs the W4A4 grouped layer:
//   gather_nv4_kernel : Xg[rho] = S * E2M1 of Q_a(x[route(rho) / k]) as fp16,
//                       natural order (the block's alpha_x left out)
//   gemm_kernel<Nv4>  : per k-step TMA brings the kept codes (32 bytes a row)
//                       and a prepared 16-byte side record (8 bytes of pair
//                       patterns, 4 UE4M3 scales); dequantizing warps expand
//                       each group of 8 into fp16 UE4M3 * E2M1 at the kept
//                       pairs and zero elsewhere (exact), into tensor memory;
//                       GEMM1's epilogue scales by alpha_e, forms h and
//                       quantizes it by Q_a into Hg (S * E2M1, fp16); GEMM2's
//                       epilogue scales by w_route * alpha_e.
// The tensor core then multiplies exact products of the quantized operands,
// as the block-scaled MMA does; it runs dense fp16 MMAs over the expanded
// weights (half of them zero) instead of the sparse MMA.
//
// Roles (one CTA per SM, persistent over tiles): warp 0 TMA and bulk copies,
// warps 1 and 2 TMEM and MMA issue (one per 128-row half of a tile), warps
// 3..6 epilogue, warps 7..18 dequantization.
// Every mbarrier wait is bounded; an expired wait records MOE_ERR_TIMEOUT in
// dev_status[1].
#include <cuda.h>

#include <type_traits>

#include "attr.h"
#include "common.cuh"
#include "grouped_internal.h"
#include "tc.cuh"

namespace moe {
namespace ga {

constexpr int kMaxStages = 32;                   // packed ring
constexpr int kDqGroups = 3;                     // groups of 4 dequantizing warps
constexpr int kDqWarps = 4 * kDqGroups;
constexpr int kEpiWarp0 = 3;                     // warps 3..6: epilogue
constexpr int kDqWarp0 = 7;                      // warps 7..18: dequantization
constexpr int kThreads = (kDqWarp0 + kDqWarps) * 32;   // 608
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxASlots = 7;                    // dequantized half-k-steps in TMEM, 64 columns each
constexpr int kHeaderBytes = 1024;
constexpr int kMaxG = 64;                        // K <= 8192
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kAwq = 0;                          // weight formats of the kernel template
constexpr int kNv4 = 1;
constexpr int kNv4SideBytes = 16;                // per weight row and k-step: 8 pattern bytes, 4 scales, 4 unused

// position of value j (0..7) inside its run of 8 in the operand order
__host__ __device__ constexpr int interleave_pos(int j) { return ((j & 3) << 1) | (j >> 2); }

struct Args {
    const uint16_t *s;        // scales [E*N][K/128] fp16 bits
    const int32_t *z;         // zeros  [E][N/8][K/128]
    const int32_t *expert_ids;
    const int32_t *npp;
    const int32_t *sorted;
    const float *wts;
    __half *hg;               // kind 1: [cap_rows][I]
    float *yr;                // kind 2: [MK][d]
    int32_t *dev_status;
    int b, n_mma, n_t, KT, I, d, MK, N, G, stages, aslots, acc_cols, nbuf;
    int E, cap_blocks;        // experts, and the blocks the operands hold (debug bounds checks)
    const float *ce;          // NVFP4S: per-expert factor alpha_w[e] * alpha_in, fp32 [E]
    const float *qa;          // NVFP4S, first GEMM: Q_a constants of h (alpha_h, binary32(1 / (6 alpha_h)))
};

// A tile is 256 weight rows of one expert, in two halves of 128 that two MMA
// issuers (warps 1 and 2) accumulate independently -- one issuing thread
// cannot keep the tensor core busy with N = 16 MMAs.  Kind 1 pairs the gate
// rows of 128 neurons (half 0) with the up rows of the same neurons (half 1),
// so the SwiGLU epilogue finds g and u in the same TMEM lane; kind 2 takes
// 256 consecutive output rows.
//
// A k-step covers 128 values of K -- one quantization group, so one scale
// and zero per weight row.  A stage of the packed ring holds what TMA brings
// for one k-step: the B operand as two 64-wide tiles (fp16 [n_mma][64] each,
// 128-byte swizzled), shared by both halves, and the packed A tile
// ([256][64 bytes]).  It is free again once the dequantizing warps have read
// the packed bytes and both issuers' MMAs that read B have completed.  A
// dequantized half-k-step ("unit") occupies 64 TMEM columns.
//
// NVFP4S: the packed part of a stage is the kept codes ([256][32 bytes],
// half 1 at +4096) and then the side records ([256][16 bytes], half 1 at
// +2048).
struct Geo {
    int n_mma, nv4;
    __host__ __device__ int b_off() const { return 0; }
    __host__ __device__ int raw_off() const { return n_mma * 256; }
    __host__ __device__ int side_off() const { return raw_off() + 8192; }   // NVFP4S
    // multiple of 1024 (n_mma % 8 == 0)
    __host__ __device__ int bytes() const { return n_mma * 256 + (nv4 ? 8192 + 256 * kNv4SideBytes : 16384); }
};

// Packed word -> four fp16 pairs (n0, n4) (n1, n5) (n2, n6) (n3, n7), each
// (n - z) * s with one rounding.  An AND-OR with 0x64006400 turns the nibbles
// at bits 0..3 / 16..19 into 1024 + n (exact in fp16) and those at bits
// 4..7 / 20..23 into 1024 + 16 n; (1024 + n) - (1024 + z) and
// (1024 + 16 n) / 16 - (64 + z) are exact small integers, so the only
// rounding is the multiply by s.  One shift per word reaches nibbles 2, 3,
// 6 and 7; the integer pipe (half the rate of the fp16 pipe) does 5
// operations per word.
//   zb: 1024 + z in both halves; zb16: -(64 + z) in both halves; sc: s in both
template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop_or(uint32_t w)
{
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, 0x64006400, 0xEA;" : "=r"(v) : "r"(w), "n"(MASK));   // (w & MASK) | 0x64006400
    return v;
}

__device__ __forceinline__ void dq_word(uint32_t w, uint32_t zb, uint32_t zb16, uint32_t sc, uint32_t *out)
{
    const __half2 z2 = *reinterpret_cast<const __half2 *>(&zb), z16 = *reinterpret_cast<const __half2 *>(&zb16);
    const __half2 s2 = *reinterpret_cast<const __half2 *>(&sc);
    const __half2 r16 = __float2half2_rn(0.0625f);
    const uint32_t w8 = w >> 8;
    uint32_t t[4] = {lop_or<0x000F000Fu>(w), lop_or<0x00F000F0u>(w), lop_or<0x000F000Fu>(w8), lop_or<0x00F000F0u>(w8)};
    __half2 r[4];
    r[0] = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&t[0]), z2), s2);
    r[1] = __hmul2(__hfma2(*reinterpret_cast<const __half2 *>(&t[1]), r16, z16), s2);
    r[2] = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&t[2]), z2), s2);
    r[3] = __hmul2(__hfma2(*reinterpret_cast<const __half2 *>(&t[3]), r16, z16), s2);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        out[j] = *reinterpret_cast<const uint32_t *>(&r[j]);
}

// 32 packed values (4 words) -> 16 fp16 pairs, each run of 8 in the order
// 0, 4, 1, 5, 2, 6, 3, 7
__device__ __forceinline__ void dq_words(const uint4 &a, const uint4 &b, uint32_t zb2, uint32_t zb16, uint32_t sc2,
                                         uint32_t (&out)[32])
{
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int c = 0; c < 8; ++c)
        dq_word(wd[c], zb2, zb16, sc2, out + 4 * c);
}

// ---------------------------------------------------------------- NVFP4S

// Two E2M1 codes (low nibble first) -> the fp16 pair of their values (exact).
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte)
{
    uint32_t r;
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(r) : "r"(byte));
    return r;
}

// A UE4M3 scale code (sign bit clear) -> the fp16 pair (S, S) (exact).
__device__ __forceinline__ uint32_t ue4m3_f16x2(uint32_t s)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(s | (s << 8))));
    return r;
}

// One group of 8 weights: its four kept codes (pair p0's two values, then
// pair p1's, low nibble first), its pattern nibble p0 | p1 << 2 and its
// block's scale pair -> four fp16 pairs in natural order, UE4M3 * E2M1 at
// the kept pairs (exact: at most 6 significant bits, within fp16's range)
// and 0 at the others.
__device__ __forceinline__ void dq_nv4_group(uint32_t codes16, uint32_t nib, uint32_t s2, uint32_t *out)
{
    const __half2 S = *reinterpret_cast<const __half2 *>(&s2);
    const uint32_t a = e2m1x2_f16x2(codes16 & 0xFFu), b = e2m1x2_f16x2(codes16 >> 8);
    const __half2 ha = __hmul2(*reinterpret_cast<const __half2 *>(&a), S);
    const __half2 hb = __hmul2(*reinterpret_cast<const __half2 *>(&b), S);
    const uint32_t P0 = *reinterpret_cast<const uint32_t *>(&ha), P1 = *reinterpret_cast<const uint32_t *>(&hb);
    // place P0 at pair p0 (0..2) and P1 at pair p1 (1..3), without branches
    asm("{\n .reg .pred a0, a1, a2, b1, b2, b3;\n .reg .b32 p0, p1;\n"
        " and.b32 p0, %4, 3;\n shr.b32 p1, %4, 2;\n"
        " setp.eq.u32 a0, p0, 0;\n setp.eq.u32 a1, p0, 1;\n setp.eq.u32 a2, p0, 2;\n"
        " setp.eq.u32 b1, p1, 1;\n setp.eq.u32 b2, p1, 2;\n setp.eq.u32 b3, p1, 3;\n"
        " selp.b32 %0, %5, 0, a0;\n"
        " selp.b32 %1, %6, 0, b1;\n selp.b32 %1, %5, %1, a1;\n"
        " selp.b32 %2, %6, 0, b2;\n selp.b32 %2, %5, %2, a2;\n"
        " selp.b32 %3, %6, 0, b3;\n}"
        : "=&r"(out[0]), "=&r"(out[1]), "=&r"(out[2]), "=&r"(out[3])
        : "r"(nib), "r"(P0), "r"(P1));
}

// 64 weights of one row: kept codes (16 bytes, group g in bytes 2g, 2g + 1),
// the eight groups' pattern nibbles (group g in bits 4g .. 4g + 3) and the
// two blocks' scale codes (bits 0..7, 8..15) -> 32 fp16 pairs in natural order.
__device__ __forceinline__ void dq_nv4_words(const uint4 &c, uint32_t meta, uint32_t sc, uint32_t (&out)[32])
{
    const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
    const uint32_t s0 = ue4m3_f16x2(sc & 0xFFu), s1 = ue4m3_f16x2((sc >> 8) & 0xFFu);
#pragma unroll
    for (int g = 0; g < 8; ++g)
        dq_nv4_group((wd[g >> 1] >> (16 * (g & 1))) & 0xFFFFu, (meta >> (4 * g)) & 0xFu, g < 4 ? s0 : s1,
                     out + 4 * g);
}

// The run-time activation quantizer Q_a of one 32-element block ("Hardware-
// Native Joint Sparse-Quantization ...", Sec. 3.4 and App. D.1; block scale
// by Eq. 5 with the tensor-wide factor 1 / alpha), every decision in
// binary32: t = amax * r6 (r6 = binary32(1 / (6 alpha))) rounded to nearest
// even onto UE4M3 with saturation at 448 gives the scale S; each value v
// becomes sign(v) | |v * q| rounded to nearest even onto the E2M1
// magnitudes with saturation at 6, q = 1 / binary32(alpha * S) (all codes 0
// when S = 0).  The operand the tensor core takes is S * E2M1 as fp16 (exact);
// alpha goes to the epilogue.
struct QaBlock {
    float q;         // 1 / (alpha S), 0 when S = 0
    uint32_t s16;    // S as fp16 bits
};

__device__ __forceinline__ QaBlock qa_block(float amax, float alpha, float r6)
{
    const float t = __fmul_rn(amax, r6);
    uint16_t code;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(code) : "f"(0.0f), "f"(t));
    const uint32_t s2 = ue4m3_f16x2(code & 0xFFu);
    const float S = __low2float(*reinterpret_cast<const __half2 *>(&s2));
    QaBlock b;
    b.q = S > 0.f ? __frcp_rn(__fmul_rn(alpha, S)) : 0.f;
    b.s16 = s2 & 0xFFFFu;
    return b;
}

// fp16 bits of a (>= 0) rounded to nearest onto {0, .5, 1, 1.5, 2, 3, 4, 6},
// saturating at 6; a midpoint (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) goes to
// the neighbour whose E2M1 mantissa bit is 0.
__device__ __forceinline__ uint32_t e2m1_rne_f16(float a)
{
    uint32_t h = 0u;
    h = a > 0.25f ? 0x3800u : h;
    h = a >= 0.75f ? 0x3C00u : h;
    h = a > 1.25f ? 0x3E00u : h;
    h = a >= 1.75f ? 0x4000u : h;
    h = a > 2.5f ? 0x4200u : h;
    h = a >= 3.5f ? 0x4400u : h;
    h = a > 5.0f ? 0x4600u : h;
    return h;
}

// S * E2M1(code of v) as fp16 bits, the sign bit that of v.
__device__ __forceinline__ uint32_t qa_value_f16(float v, const QaBlock &b)
{
    const uint32_t m = e2m1_rne_f16(fabsf(__fmul_rn(v, b.q)));
    const __half p = __hmul(__ushort_as_half(static_cast<unsigned short>(m)),
                            __ushort_as_half(static_cast<unsigned short>(b.s16)));
    return __half_as_ushort(p) | ((__float_as_uint(v) >> 16) & 0x8000u);
}

// Per-tile group scales and zeros, as copied from global memory: the scale
// rows of the tile's 256 weight rows, [256][G] fp16, then their zero words,
// [32][G] int32 (row r's zero in nibble r % 8 of word [r / 8][g]).
__host__ __device__ inline int sbuf_bytes(int G) { return 640 * G; }

// Both GEMMs in one persistent kernel: the tile list is every first-GEMM
// tile (gate/up, SwiGLU into Hg), block-major, then every second-GEMM tile
// (down, w_route * acc into Yr).  CTA c takes tiles c, c + grid, ..., so it
// finishes its first-GEMM tiles first; a second-GEMM tile of block jb waits
// (bounded) until every first-GEMM tile of jb has published Hg through a
// per-block counter (release add after proxy fences; acquire load and proxy
// fence before the TMA reads).  SMs that run out of first-GEMM tiles start on
// the second GEMM instead of idling at a kernel boundary.  Every CTA must be
// resident: the grid is one CTA per SM.
__device__ __forceinline__ int tile_kind(int t, int total1, int n_t1, int n_t2, int &jb, int &T)
{
    if (t < total1) {
        jb = t / n_t1;
        T = t - jb * n_t1;
        return 1;
    }
    t -= total1;
    jb = t / n_t2;
    T = t - jb * n_t2;
    return 2;
}

// FMT = kAwq: AWQ codes with per-tile scales and zeros (tmS1 / tmS2
// unused); FMT = kNv4: NVFP4S kept codes with per-k-step side records
// (tmS1 / tmS2, no per-tile buffers).
template <int FMT>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmB1,
            const __grid_constant__ CUtensorMap tmQ2, const __grid_constant__ CUtensorMap tmB2,
            const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmS2, const Args a1,
            const Args a2, int32_t *done, int sbuf_g)
{
    constexpr bool kN = FMT == kNv4;
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t raw = tc::smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const Geo geo{a1.n_mma, kN ? 1 : 0};
    // kDqGroups <= AS, ceil(AS / 2) < S
    const int S = a1.stages, SB = geo.bytes(), AS = a1.aslots, NB = a1.nbuf;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * SB);
    const uint32_t rfull0 = tc::smem_u32(bars), rempty0 = rfull0 + 8 * S, afull0 = rempty0 + 8 * S;
    const uint32_t accf0 = afull0 + 8 * AS;      // [half][buf]
    const uint32_t acce0 = accf0 + 32;           // [half][buf]
    const uint32_t sfull0 = acce0 + 32, sempty0 = sfull0 + 16, fin0 = sempty0 + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + AS + 14);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *t_route = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(bars) + kHeaderBytes);   // [256]
    float *t_w = reinterpret_cast<float *>(t_route + 256);                                       // [256]
    uint8_t *sbuf = reinterpret_cast<uint8_t *>(t_w + 256);                                      // [2][sbuf_bytes]
    const int SBUF = sbuf_bytes(sbuf_g);                                                        // both GEMMs' G fit

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            tc::mbar_init(rfull0 + 8 * s, 1);
            tc::mbar_init(rempty0 + 8 * s, 8 + 2);   // the k-step's two units' dequantizing warps + two commits
        }
        for (int s = 0; s < AS; ++s)
            tc::mbar_init(afull0 + 8 * s, 4);
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(accf0 + 8 * i, 1);
            tc::mbar_init(acce0 + 8 * i, 4);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(sfull0 + 8 * i, 1);
            tc::mbar_init(sempty0 + 8 * i, kDqWarps);
            tc::mbar_init(fin0 + 8 * i, 1);
        }
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&tmQ1);
        tc::prefetch_tmap(&tmB1);
        tc::prefetch_tmap(&tmQ2);
        tc::prefetch_tmap(&tmB2);
        if (kN) {
            tc::prefetch_tmap(&tmS1);
            tc::prefetch_tmap(&tmS2);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    const int b = a1.b;
    int n_blocks = *a1.npp / b;
#ifdef MOE_DEBUG_BOUNDS
    {
        // debug build: the block count and every block's expert inside
        // their buffers, or no tile runs at all (every role sees the same)
        bool bad = n_blocks < 0 || n_blocks > a1.cap_blocks;
        for (int j = threadIdx.x; !bad && j < n_blocks; j += blockDim.x)
            bad = a1.expert_ids[j] < 0 || a1.expert_ids[j] >= a1.E;
        if (__syncthreads_or(bad)) {
            MOE_IN_BOUNDS(false, a1.dev_status);
            n_blocks = 0;
        }
    }
#endif
    const int n_t1 = a1.n_t, n_t2 = a2.n_t;
    const int total1 = n_blocks * n_t1, total = total1 + n_blocks * n_t2;
    const uint32_t a_base = static_cast<uint32_t>(2 * NB * a1.acc_cols);   // first A-unit column

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0, issued = 0, ti = 0;
            uint32_t ph = 0;
            const uint32_t tx = static_cast<uint32_t>(SB);
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++ti) {
                int jb, T;
                const int kind = tile_kind(t, total1, n_t1, n_t2, jb, T);
                const int e = a1.expert_ids[jb];
                const int N = kind == 1 ? a1.N : a2.N, G = kind == 1 ? a1.G : a2.G, KT = kind == 1 ? a1.KT : a2.KT;
                const uint16_t *sp = kind == 1 ? a1.s : a2.s;
                const int32_t *zp = kind == 1 ? a1.z : a2.z;
                const CUtensorMap *tQ = kind == 1 ? &tmQ1 : &tmQ2;
                const CUtensorMap *tB = kind == 1 ? &tmB1 : &tmB2;
                const CUtensorMap *tS = kind == 1 ? &tmS1 : &tmS2;
                const int row0 = e * N;
                // first weight row of each half
                const int r0 = kind == 1 ? row0 + 128 * T : row0 + 256 * T;
                const int r1 = kind == 1 ? row0 + a1.I + 128 * T : row0 + 256 * T + 128;
                if (kind == 2) {
                    // block jb's Hg: every first-GEMM tile of jb published
                    const long long t0 = clock64();
                    const long long limit = static_cast<long long>(kWaitNs) * 5 / 2;
                    int v;
                    for (;;) {
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(done + jb) : "memory");
                        if (v >= n_t1)
                            break;
                        if (*abort_flag || clock64() - t0 > limit) {
                            *abort_flag = 1;
                            break;
                        }
                    }
                    if (v < n_t1)
                        break;
                    // the tensor-memory-access proxy reads what generic stores wrote
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                // AWQ: the tile's scales and zeros (buffer ti % 2, freed by
                // the dequantizing warps when they finish tile ti - 2)
                const int sb = ti & 1;
                if (!kN && !tc::mbar_wait(sempty0 + 8 * sb, ((ti >> 1) & 1) ^ 1u, abort_flag, kWaitNs))
                    break;
                if (!kN) {
                    const uint32_t fb = sfull0 + 8 * sb;
                    const uint32_t dst = tc::smem_u32(sbuf + sb * SBUF);
                    const int64_t zr0 = static_cast<int64_t>(e) * (N / 8) + (r0 - row0) / 8;
                    const int64_t zr1 = static_cast<int64_t>(e) * (N / 8) + (r1 - row0) / 8;
                    tc::mbar_arrive_expect_tx(fb, static_cast<uint32_t>(sbuf_bytes(G)));
                    tc::bulk_load(dst, sp + static_cast<int64_t>(r0) * G, 256u * G, fb);
                    tc::bulk_load(dst + 256u * G, sp + static_cast<int64_t>(r1) * G, 256u * G, fb);
                    tc::bulk_load(dst + 512u * G, zp + zr0 * G, 64u * G, fb);
                    tc::bulk_load(dst + 576u * G, zp + zr1 * G, 64u * G, fb);
                }
                for (int kt = 0; kt < KT; ++kt, ++issued) {
                    if (!tc::mbar_wait(rempty0 + 8 * s, ph ^ 1u, abort_flag, kWaitNs))
                        break;
                    uint8_t *st = smem + s * SB;
                    const uint32_t fb = rfull0 + 8 * s;
                    tc::mbar_arrive_expect_tx(fb, tx);
                    if (kN) {
                        // kept codes: 32 bytes (128 weights) of each row; side records: 16 bytes
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off()), tQ, kt * 32, r0, fb);
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off() + 4096), tQ, kt * 32, r1, fb);
                        tc::tma_load_2d(tc::smem_u32(st + geo.side_off()), tS, kt * kNv4SideBytes, r0, fb);
                        tc::tma_load_2d(tc::smem_u32(st + geo.side_off() + 2048), tS, kt * kNv4SideBytes, r1, fb);
                    } else {
                        // packed A rows: 64 bytes (128 values) of each, x in bytes
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off()), tQ, kt * 64, r0, fb);
                        tc::tma_load_2d(tc::smem_u32(st + geo.raw_off() + 8192), tQ, kt * 64, r1, fb);
                    }
                    // B: two tiles of n_mma rows x 64 fp16, x in elements
                    tc::tma_load_2d(tc::smem_u32(st + geo.b_off()), tB, kt * 128, jb * b, fb);
                    tc::tma_load_2d(tc::smem_u32(st + geo.b_off() + geo.n_mma * 128), tB, kt * 128 + 64, jb * b, fb);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // copies still in flight land before the CTA exits
            volatile int never = 0;
            const int n = issued < S ? issued : S;
            for (int i = 1; i <= n; ++i) {
                int st = s - i;
                uint32_t pp = ph;
                if (st < 0) {
                    st += S;
                    pp ^= 1u;
                }
                tc::mbar_wait(rfull0 + 8 * st, pp, &never, kWaitNs);
            }
            for (int i = 1; !kN && i <= 2 && i <= ti; ++i)
                tc::mbar_wait(sfull0 + 8 * ((ti - i) & 1), ((ti - i) >> 1) & 1u, &never, kWaitNs);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------ MMA issuers (warp 1: half 0, warp 2: half 1)
        // The issuing thread's own instructions serialize with the MMA issue,
        // so the loop keeps them few: descriptors advance by constants, one
        // wait and one commit per k-step of 8 MMAs.  afull implies the
        // stage's TMA data landed (the dequantizing warps waited for it
        // before arriving), and the commit to rempty both frees the packed
        // stage (with the other issuer's) and tells the dequantizing warps
        // that the unit's TMEM columns have been read.
        if (lane == 0) {
            const int h = warp - 1;
            int s = 0, ti = 0, sa = h;                // unit 2 i + h of k-step i sits in slot (2 i + h) % AS
            uint32_t pha = 0;
            const uint32_t idesc = tc::idesc_f16(128, geo.n_mma, false);
            const uint64_t bd0 = tc::smem_desc(tc::smem_u32(smem + geo.b_off()), 16, 1024, tc::kLayoutSw128);
            const uint64_t bd_step = static_cast<uint64_t>(SB >> 4);
            const uint64_t bd_half = static_cast<uint64_t>(geo.n_mma * 8);   // second B tile: n_mma * 128 bytes on
            for (int t = blockIdx.x; t < total && !*abort_flag; t += gridDim.x, ++ti) {
                const int KT = t < total1 ? a1.KT : a2.KT;
                const int buf = NB == 2 ? (ti & 1) : 0;
                const uint32_t use = static_cast<uint32_t>(NB == 2 ? (ti >> 1) : ti);
                const int ab = h * 2 + buf;
                if (!tc::mbar_wait(acce0 + 8 * ab, (use & 1u) ^ 1u, abort_flag, kWaitNs))
                    break;
                tc::tc_fence_after();
                const uint32_t acc = tmem + static_cast<uint32_t>((h * NB + buf) * a1.acc_cols);
                uint64_t bd = bd0 + bd_step * static_cast<uint64_t>(s);
                for (int kt = 0; kt < KT; ++kt) {
                    if (!tc::mbar_wait(afull0 + 8 * sa, pha, abort_flag, kWaitNs))
                        break;
                    tc::tc_fence_after();
                    const uint32_t a_t = tmem + a_base + 64 * sa;
                    // 16 values of K per MMA: 8 TMEM columns of A, 32 bytes of B
                    tc::mma_f16_ts(acc, a_t, bd, idesc, kt != 0 ? 1u : 0u);
                    tc::mma_f16_ts(acc, a_t + 8, bd + 2, idesc, 1u);
                    tc::mma_f16_ts(acc, a_t + 16, bd + 4, idesc, 1u);
                    tc::mma_f16_ts(acc, a_t + 24, bd + 6, idesc, 1u);
                    tc::mma_f16_ts(acc, a_t + 32, bd + bd_half, idesc, 1u);
                    tc::mma_f16_ts(acc, a_t + 40, bd + bd_half + 2, idesc, 1u);
                    tc::mma_f16_ts(acc, a_t + 48, bd + bd_half + 4, idesc, 1u);
                    tc::mma_f16_ts(acc, a_t + 56, bd + bd_half + 6, idesc, 1u);
                    tc::tc_commit(rempty0 + 8 * s);
                    if (++s == S) {
                        s = 0;
                        bd = bd0;
                    } else {
                        bd += bd_step;
                    }
                    if ((sa += 2) >= AS) {
                        sa -= AS;
                        pha ^= 1u;
                    }
                }
                tc::tc_commit(accf0 + 8 * ab);
            }
            tc::tc_commit(fin0 + 8 * h);
            volatile int never = 0;
            tc::mbar_wait(fin0 + 8 * h, 0, &never, kWaitNs);
        }
    } else if (warp < kDqWarp0) {
        // ------------------------------------------------ epilogue (warps 3..6)
        const int q = warp & 3;                       // TMEM lane quadrant
        const int etid = threadIdx.x - kEpiWarp0 * 32;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
        // NVFP4S: Q_a constants of h
        const float qa_alpha = kN ? a1.qa[0] : 0.f, qa_r6 = kN ? a1.qa[1] : 0.f;
        int ti = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++ti) {
            int jb, T;
            const int kind = tile_kind(t, total1, n_t1, n_t2, jb, T);
            const int buf = NB == 2 ? (ti & 1) : 0;
            const uint32_t use = static_cast<uint32_t>(NB == 2 ? (ti >> 1) : ti);
            const int rho0 = jb * b;
            // NVFP4S: the expert's factor alpha_w * alpha_in
            const float ce = kN ? (kind == 1 ? a1.ce : a2.ce)[a1.expert_ids[jb]] : 1.f;
            if (kind == 2) {
                for (int c = etid; c < b; c += 128) {
                    int r = a2.sorted[rho0 + c];
                    if (!MOE_IN_BOUNDS(r >= 0 && r <= a2.MK, a2.dev_status))
                        r = a2.MK;                            // read as padding
                    t_route[c] = r;
                    if constexpr (kN)
                        t_w[c] = r < a2.MK ? a2.wts[r] * ce : 0.f;
                    else
                        t_w[c] = r < a2.MK ? a2.wts[r] : 0.f;
                }
            }
            bool ok = tc::mbar_wait(accf0 + 8 * buf, use & 1u, abort_flag, kWaitNs);
            ok = tc::mbar_wait(accf0 + 8 * (2 + buf), use & 1u, abort_flag, kWaitNs) && ok;
            if (!ok && a1.dev_status)
                atomicCAS(a1.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
            tc::tc_fence_after();
            tc::named_bar(1, 128);
            const uint32_t acc0 = tmem + lane_off + static_cast<uint32_t>(buf * a1.acc_cols);
            const uint32_t acc1 = tmem + lane_off + static_cast<uint32_t>((NB + buf) * a1.acc_cols);
            for (int c0 = 0; c0 < b; c0 += 32) {
                const int ncol = min(32, b - c0);
                if (kind == 1) {
                    // gate and up of neuron n share the lane; h -> column n of Hg in the operand order
                    uint32_t g[32], u[32];
                    tc::tmem_ld_32x32b_x32(acc0 + c0, g);
                    tc::tmem_ld_32x32b_x32(acc1 + c0, u);
                    tc::tmem_ld_wait();
                    const int n = 128 * T + 32 * q + lane;
                    if constexpr (kN) {
                        // h -> Q_a: the warp's 32 lanes are the 32 neurons of one block
                        uint16_t *hrow = reinterpret_cast<uint16_t *>(a1.hg) + static_cast<int64_t>(rho0 + c0) * a1.I + n;
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (c < ncol) {
                                const float hv = silu_mul(__fmul_rn(__uint_as_float(g[c]), ce),
                                                          __fmul_rn(__uint_as_float(u[c]), ce));
                                const float amax =
                                    __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv))));
                                hrow[static_cast<int64_t>(c) * a1.I] =
                                    static_cast<uint16_t>(qa_value_f16(hv, qa_block(amax, qa_alpha, qa_r6)));
                            }
                    } else {
                        __half *hrow = a1.hg + static_cast<int64_t>(rho0 + c0) * a1.I + (n & ~7) + interleave_pos(n & 7);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (c < ncol)
                                hrow[static_cast<int64_t>(c) * a1.I] =
                                    __float2half_rn(silu_mul(__uint_as_float(g[c]), __uint_as_float(u[c])));
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t v[32];
                        tc::tmem_ld_32x32b_x32((h ? acc1 : acc0) + c0, v);
                        tc::tmem_ld_wait();
                        float *yo = a2.yr + 256 * T + 128 * h + 32 * q + lane;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int r = t_route[c0 + c];   // same address in every lane: broadcast
                            if (c < ncol && r < a2.MK)
                                yo[static_cast<int64_t>(r) * a2.d] = t_w[c0 + c] * __uint_as_float(v[c]);
                        }
                    }
                }
            }
            if (kind == 1)
                asm volatile("fence.proxy.async.global;" ::: "memory");   // Hg is read by TMA
            tc::tc_fence_before();
            tc::named_bar(1, 128);
            if (lane == 0) {
                tc::mbar_arrive(acce0 + 8 * buf);
                tc::mbar_arrive(acce0 + 8 * (2 + buf));
            }
            if (kind == 1 && etid == 0)                // every epilogue thread's stores are ordered before this
                asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(done + jb) : "memory");
        }
    } else {
        // ------------------------------------------------ dequantization (warps 7..18)
        // Unit v = 2 i + h is half h of the CTA's k-step i (counted over all
        // of its tiles); group g of four warps takes units g, g + kDqGroups,
        // ...  Each thread dequantizes row m = 32 * quadrant + lane of the
        // half into TMEM slot v % AS.
        const int g = (warp - kDqWarp0) >> 2, q = warp & 3;
        const int m = 32 * q + lane;
        const int zsh = 4 * (m & 7);
        const uint32_t a_lane = tmem + (static_cast<uint32_t>(32 * q) << 16) + a_base;
        int v = g, sa = g, ti = 0;
        int s = v >> 1;                               // stage of k-step v / 2 (< S) and its phase
        uint32_t ph = 0;
        int kbase = 0;                                // the CTA's k-steps before this tile
        // after a timeout the waits return at once and the loops run out
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++ti) {
            const int sb = ti & 1;
            const int G = t < total1 ? a1.G : a2.G, KT = t < total1 ? a1.KT : a2.KT;
            if (!kN && !tc::mbar_wait(sfull0 + 8 * sb, (ti >> 1) & 1u, abort_flag, kWaitNs) && a1.dev_status)
                atomicCAS(a1.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
            const uint16_t *sc = reinterpret_cast<const uint16_t *>(sbuf + sb * SBUF);
            const uint32_t *zs = reinterpret_cast<const uint32_t *>(sbuf + sb * SBUF + 512 * G);
            for (; (v >> 1) < kbase + KT;) {
                const int i = v >> 1, h = v & 1;
                const int kt = i - kbase;              // = the quantization group
                const int r = 128 * h + m;             // row of the tile
                uint32_t sc2 = 0, zb2 = 0, zb16 = 0;
                if (!kN) {
                    const uint32_t sv = sc[r * G + kt];
                    const uint32_t zv = (zs[(r >> 3) * G + kt] >> zsh) & 0xFu;
                    sc2 = sv | (sv << 16);
                    zb2 = 0x64006400u | zv | (zv << 16);
                    zb16 = 0xD400D400u | (zv << 4) | (zv << 20);   // -(64 + z): ulp 1/16 in [64, 128)
                }
                if (!tc::mbar_wait(rfull0 + 8 * s, ph, abort_flag, kWaitNs) && a1.dev_status)
                    atomicCAS(a1.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
                // AWQ: 64 packed bytes of row r; NVFP4S: 32 bytes of kept codes and the 16-byte side record
                uint4 w0, w1, w2, w3;
                if (kN) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(smem + s * SB + geo.raw_off() + r * 32);
                    w0 = src[0];
                    w1 = src[1];
                    w2 = *reinterpret_cast<const uint4 *>(smem + s * SB + geo.side_off() + r * kNv4SideBytes);
                    w3 = make_uint4(0, 0, 0, 0);
                } else {
                    const uint4 *src = reinterpret_cast<const uint4 *>(smem + s * SB + geo.raw_off() + r * 64);
                    w0 = src[0];
                    w1 = src[1];
                    w2 = src[2];
                    w3 = src[3];
                }
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(rempty0 + 8 * s);  // packed bytes read
                // slot sa is free once the MMAs of unit v - AS completed: the
                // commits completed phase (i' / S) of k-step i' = (v - AS) / 2's stage
                if (v >= AS) {
                    const int ip = (v - AS) >> 1;
                    if (!tc::mbar_wait(rempty0 + 8 * (ip % S), static_cast<uint32_t>(ip / S) & 1u, abort_flag,
                                       kWaitNs) &&
                        a1.dev_status)
                        atomicCAS(a1.dev_status + 1, 0, static_cast<int>(MOE_ERR_TIMEOUT));
                }
                tc::tc_fence_after();
                if (kN) {
                    uint32_t out[32];
                    dq_nv4_words(w0, w2.x, w2.z & 0xFFFFu, out);   // weights 0..63 -> columns 0..31
                    tc::tmem_st_32x32b_x32(a_lane + 64 * sa, out);
                    dq_nv4_words(w1, w2.y, w2.z >> 16, out);       // weights 64..127 -> columns 32..63
                    tc::tmem_st_32x32b_x32(a_lane + 64 * sa + 32, out);
                } else {
                    {
                        uint32_t out[32];
                        dq_words(w0, w1, zb2, zb16, sc2, out);   // values 0..63 -> columns 0..31
                        tc::tmem_st_32x32b_x32(a_lane + 64 * sa, out);
                    }
                    {
                        uint32_t out[32];
                        dq_words(w2, w3, zb2, zb16, sc2, out);   // values 64..127 -> columns 32..63
                        tc::tmem_st_32x32b_x32(a_lane + 64 * sa + 32, out);
                    }
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    tc::mbar_arrive(afull0 + 8 * sa);
                // next unit: v + kDqGroups
                const int di = ((v + kDqGroups) >> 1) - i;
                v += kDqGroups;
                if ((s += di) >= S) {
                    s -= S;
                    ph ^= 1u;
                }
                if ((sa += kDqGroups) >= AS)
                    sa -= AS;
            }
            __syncwarp();
            if (!kN && lane == 0)
                tc::mbar_arrive(sempty0 + 8 * sb);
            kbase += KT;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// Xg[rho] = x[route / k] as fp16 (zero rows for padding), each run of 8 in
// the operand order 0, 4, 1, 5, 2, 6, 3, 7; 8 values per thread
template <typename XT>
__global__ void gather_kernel(const XT *__restrict__ x, int d, int k, int MK, const int32_t *__restrict__ sorted,
                              const int32_t *__restrict__ npp, __half *__restrict__ xg, int b, int32_t *__restrict__ done,
                              int cap_rows, int32_t *__restrict__ dev_status)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    int rows = *npp;
    if (!MOE_IN_BOUNDS(rows >= 0 && rows <= cap_rows, dev_status))
        rows = 0;
    // the GEMM's per-block counters of finished first-GEMM tiles start at 0
    for (int jb = blockIdx.x * blockDim.x + threadIdx.x; jb < rows / b; jb += gridDim.x * blockDim.x)
        done[jb] = 0;
    const int d8 = d / 8;
    const int64_t total = static_cast<int64_t>(rows) * d8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int rho = static_cast<int>(i / d8), c = static_cast<int>(i - static_cast<int64_t>(rho) * d8);
        int r = sorted[rho];
        if (!MOE_IN_BOUNDS(r >= 0 && r <= MK, dev_status))
            r = MK;                                   // read as padding
        uint4 out = make_uint4(0, 0, 0, 0);
        if (r < MK) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(r / k) * d) + c);
            uint32_t o[4] = {v.x, v.y, v.z, v.w};     // fp16 pairs (0,1) (2,3) (4,5) (6,7)
            if constexpr (!std::is_same<XT, __half>::value) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 h = __floats2half2_rn(__uint_as_float(o[j] << 16), __uint_as_float(o[j] & 0xFFFF0000u));
                    o[j] = *reinterpret_cast<const uint32_t *>(&h);
                }
            }
            out = make_uint4(__byte_perm(o[0], o[2], 0x5410), __byte_perm(o[0], o[2], 0x7632),
                             __byte_perm(o[1], o[3], 0x5410), __byte_perm(o[1], o[3], 0x7632));
        }
        reinterpret_cast<uint4 *>(xg + static_cast<int64_t>(rho) * d)[c] = out;
    }
}

// Xg[rho] = S * E2M1 of Q_a(x[route / k]) as fp16 bits, natural order (the
// block's tensor-wide scale alpha_x left out; padding rows zero).  Each
// thread takes 8 values; 4 neighbouring threads form a block of 32 and share
// its maximum (d % 256 == 0, so a warp's 32 threads lie in one row).
template <typename XT>
__global__ void gather_nv4_kernel(const XT *__restrict__ x, int d, int k, int MK, const int32_t *__restrict__ sorted,
                                  const int32_t *__restrict__ npp, uint16_t *__restrict__ xg, int b,
                                  int32_t *__restrict__ done, int cap_rows, int32_t *__restrict__ dev_status,
                                  const float *__restrict__ qa)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    int rows = *npp;
    if (!MOE_IN_BOUNDS(rows >= 0 && rows <= cap_rows, dev_status))
        rows = 0;
    for (int jb = blockIdx.x * blockDim.x + threadIdx.x; jb < rows / b; jb += gridDim.x * blockDim.x)
        done[jb] = 0;
    const float alpha = qa[0], r6 = qa[1];
    const int d8 = d / 8;
    const int64_t total = static_cast<int64_t>(rows) * d8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int rho = static_cast<int>(i / d8), c = static_cast<int>(i - static_cast<int64_t>(rho) * d8);
        int r = sorted[rho];
        if (!MOE_IN_BOUNDS(r >= 0 && r <= MK, dev_status))
            r = MK;                                   // read as padding
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (r < MK) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(r / k) * d) + c);
            const uint32_t o[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if constexpr (std::is_same<XT, __half>::value) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&o[j]));
                    v[2 * j] = f.x;
                    v[2 * j + 1] = f.y;
                } else {
                    v[2 * j] = __uint_as_float(o[j] << 16);
                    v[2 * j + 1] = __uint_as_float(o[j] & 0xFFFF0000u);
                }
            }
        }
        float am = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            am = fmaxf(am, fabsf(v[j]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const QaBlock qb = qa_block(am, alpha, r6);
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            out[j] = qa_value_f16(v[2 * j], qb) | (qa_value_f16(v[2 * j + 1], qb) << 16);
        reinterpret_cast<uint4 *>(xg + static_cast<int64_t>(rho) * d)[c] = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// Prepared NVFP4S projection (moe_grouped_prepare_nvfp4s): a 256-byte head
// (alpha_in, binary32(1 / (6 alpha_in)) of the activation the projection
// takes), the per-expert factors alpha_w[e] * alpha_in (fp32 [E], rounded up
// to 256 bytes), then one 16-byte side record per weight row and k-step of
// 128: that k-step's 8 pattern bytes, its 4 UE4M3 scale bytes, 4 zero bytes.
struct Nv4Prep {
    size_t head, ce, side, total;
};

static Nv4Prep nv4_prep_layout(int E, int N, int K)
{
    Nv4Prep P;
    P.head = 0;
    P.ce = 256;
    P.side = P.ce + ws_round(static_cast<size_t>(E) * sizeof(float));
    P.total = P.side + static_cast<size_t>(E) * N * (K / 128) * kNv4SideBytes;
    return P;
}

__global__ void prepare_nv4_side_kernel(const uint8_t *__restrict__ meta, const uint8_t *__restrict__ sc, int64_t rows,
                                        int K, uint4 *__restrict__ side)
{
    const int KS = K / 128;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < rows * KS;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t row = i / KS;
        const int kt = static_cast<int>(i - row * KS);
        const uint2 m = *reinterpret_cast<const uint2 *>(meta + row * (K / 16) + 8 * kt);
        const uint32_t s4 = *reinterpret_cast<const uint32_t *>(sc + row * (K / 32) + 4 * kt);
        side[i] = make_uint4(m.x, m.y, s4, 0u);
    }
}

__global__ void prepare_nv4_head_kernel(const float *__restrict__ alpha_w, int E, float alpha_in, float r6,
                                        float *__restrict__ head, float *__restrict__ ce)
{
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        head[0] = alpha_in;
        head[1] = r6;
    }
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
        ce[e] = __fmul_rn(alpha_w[e], alpha_in);
}

struct WsLayout {
    size_t xg, hg, yr, done, total;
};

static WsLayout ws_layout(int M, int k, int d, int I, int b, int cap_rows)
{
    WsLayout L;
    size_t off = 0;
    L.xg = off;
    off += ws_round(static_cast<size_t>(cap_rows) * d * 2);
    L.hg = off;
    off += ws_round(static_cast<size_t>(cap_rows) * I * 2);
    L.yr = off;
    off += ws_round(static_cast<size_t>(M) * k * d * sizeof(float));
    L.done = off;
    off += ws_round(static_cast<size_t>(cap_rows / b) * sizeof(int32_t));
    L.total = off;
    return L;
}

}  // namespace ga

size_t grouped_awq_workspace(int M, int k, int d, int I, int b, int cap_rows)
{
    return ga::ws_layout(M, k, d, I, b, cap_rows).total;
}

moe_status_t grouped_awq_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                const int32_t *sorted, const int32_t *expert_ids, const int32_t *npp, int b,
                                int cap_rows, void *y, bool y_f32, void *ws, int32_t *dev_status, cudaStream_t s)
{
    using namespace ga;
    const int64_t mk = static_cast<int64_t>(M) * k;
    const int n_mma = (b + 15) / 16 * 16;
    const WsLayout L = ws_layout(M, k, d, I, b, cap_rows);
    uint8_t *w = static_cast<uint8_t *>(ws);
    __half *xg = reinterpret_cast<__half *>(w + L.xg);
    __half *hg = reinterpret_cast<__half *>(w + L.hg);
    float *yr = reinterpret_cast<float *>(w + L.yr);
    int32_t *done = reinterpret_cast<int32_t *>(w + L.done);

    // launch configuration first: every check comes before the first launch
    const int G1 = d / 128, G2 = I / 128, Gmax = G1 > G2 ? G1 : G2;
    if (Gmax > kMaxG || n_mma > 128 || d % 256)
        return MOE_ERR_UNSUPPORTED;
    const int stage_bytes = Geo{n_mma}.bytes();
    const size_t fixed = 1024 + kHeaderBytes + 512 * 4 + 2 * static_cast<size_t>(sbuf_bytes(Gmax));
    int stages = static_cast<int>((227 * 1024 - fixed) / stage_bytes);
    stages = stages > kMaxStages ? kMaxStages : stages;
    // TMEM: accumulators [half][buf] of acc_cols columns, then the A units
    const int acc_cols = (n_mma + 31) / 32 * 32;
    const int nbuf = 4 * acc_cols + 64 * kDqGroups <= static_cast<int>(kTmemCols) ? 2 : 1;
    int aslots = (static_cast<int>(kTmemCols) - 2 * nbuf * acc_cols) / 64;
    aslots = aslots > kMaxASlots ? kMaxASlots : aslots;
    aslots = aslots > 2 * stages - 2 ? 2 * stages - 2 : aslots;
    const size_t smem = fixed + static_cast<size_t>(stages) * stage_bytes;
    if (aslots < kDqGroups || smem > 227 * 1024)
        return MOE_ERR_UNSUPPORTED;
    static std::atomic<uint64_t> attr_done{0};
    if (!smem_attr_once(attr_done, reinterpret_cast<const void *>(gemm_kernel<kAwq>), 227 * 1024))
        return MOE_ERR_CUDA;

    // tensor maps: packed weights as bytes [E*N][K/2]; activations fp16 [cap_rows][K]
    CUtensorMap tQ1, tB1, tQ2, tB2;
    if (!grouped_tmap_2d(&tQ1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w13->q, d / 2, static_cast<uint64_t>(E) * 2 * I, 64,
                         128, false) ||
        !grouped_tmap_2d(&tB1, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xg, d, cap_rows, 64, n_mma, true) ||
        !grouped_tmap_2d(&tQ2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w2->q, I / 2, static_cast<uint64_t>(E) * d, 64, 128,
                         false) ||
        !grouped_tmap_2d(&tB2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hg, I, cap_rows, 64, n_mma, true))
        return MOE_ERR_CUDA;

    const int gblocks = grouped_sm_count() * 4;
    const cudaError_t ge =
        x_bf16 ? launch_pdl(gather_kernel<__nv_bfloat16>, dim3(gblocks), dim3(256), 0, s,
                            static_cast<const __nv_bfloat16 *>(x), d, k, static_cast<int>(mk), sorted, npp, xg, b, done,
                            cap_rows, dev_status)
               : launch_pdl(gather_kernel<__half>, dim3(gblocks), dim3(256), 0, s, static_cast<const __half *>(x), d, k,
                            static_cast<int>(mk), sorted, npp, xg, b, done, cap_rows, dev_status);
    if (ge != cudaSuccess)
        return MOE_ERR_CUDA;
    const int grid = grouped_sm_count();
    Args a1{static_cast<const uint16_t *>(w13->scale), static_cast<const int32_t *>(w13->zero), expert_ids, npp, sorted,
            wts, hg, nullptr, dev_status, b, n_mma, I / 128, d / 128, I, d, static_cast<int>(mk), 2 * I, G1, stages,
            aslots, acc_cols, nbuf, E, cap_rows / b};
    Args a2{static_cast<const uint16_t *>(w2->scale), static_cast<const int32_t *>(w2->zero), expert_ids, npp, sorted,
            wts, nullptr, yr, dev_status, b, n_mma, d / 256, I / 128, I, d, static_cast<int>(mk), d, G2, stages,
            aslots, acc_cols, nbuf, E, cap_rows / b};
    if (launch_pdl(gemm_kernel<kAwq>, dim3(grid), dim3(kThreads), smem, s, tQ1, tB1, tQ2, tB2, tQ1, tQ2, a1, a2, done,
                   Gmax) != cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, ids, M, k, d, E, y, y_f32, s);
}

size_t grouped_nv4_prepare_bytes(int E, int N, int K)
{
    return ga::nv4_prep_layout(E, N, K).total;
}

moe_status_t grouped_nv4_prepare(const moe_weights_t *w, float alpha_in, void *out, cudaStream_t s)
{
    using namespace ga;
    const Nv4Prep P = nv4_prep_layout(w->E, w->N, w->K);
    uint8_t *o = static_cast<uint8_t *>(out);
    const float r6 = static_cast<float>(1.0 / (6.0 * static_cast<double>(alpha_in)));
    prepare_nv4_head_kernel<<<1, 256, 0, s>>>(w->alpha, w->E, alpha_in, r6, reinterpret_cast<float *>(o + P.head),
                                              reinterpret_cast<float *>(o + P.ce));
    if (launch_status() != MOE_OK)
        return MOE_ERR_CUDA;
    const int64_t rows = static_cast<int64_t>(w->E) * w->N;
    const int64_t n = rows * (w->K / 128);
    const int blocks = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
    prepare_nv4_side_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint8_t *>(w->zero),
                                                   static_cast<const uint8_t *>(w->scale), rows, w->K,
                                                   reinterpret_cast<uint4 *>(o + P.side));
    return launch_status();
}

moe_status_t grouped_nv4_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                const void *p13, const void *p2, const int32_t *sorted, const int32_t *expert_ids,
                                const int32_t *npp, int b, int cap_rows, void *y, bool y_f32, void *ws,
                                int32_t *dev_status, cudaStream_t s)
{
    using namespace ga;
    const int64_t mk = static_cast<int64_t>(M) * k;
    const int n_mma = (b + 15) / 16 * 16;
    const WsLayout L = ws_layout(M, k, d, I, b, cap_rows);
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint16_t *xg = reinterpret_cast<uint16_t *>(w + L.xg);
    __half *hg = reinterpret_cast<__half *>(w + L.hg);
    float *yr = reinterpret_cast<float *>(w + L.yr);
    int32_t *done = reinterpret_cast<int32_t *>(w + L.done);
    const Nv4Prep P13 = nv4_prep_layout(E, 2 * I, d), P2 = nv4_prep_layout(E, d, I);
    const uint8_t *q13 = static_cast<const uint8_t *>(p13), *q2 = static_cast<const uint8_t *>(p2);

    if (n_mma > 128 || d % 256 || I % 128)
        return MOE_ERR_UNSUPPORTED;
    const int stage_bytes = Geo{n_mma, 1}.bytes();
    const size_t fixed = 1024 + kHeaderBytes + 512 * 4;
    int stages = static_cast<int>((227 * 1024 - fixed) / stage_bytes);
    stages = stages > kMaxStages ? kMaxStages : stages;
    const int acc_cols = (n_mma + 31) / 32 * 32;
    const int nbuf = 4 * acc_cols + 64 * kDqGroups <= static_cast<int>(kTmemCols) ? 2 : 1;
    int aslots = (static_cast<int>(kTmemCols) - 2 * nbuf * acc_cols) / 64;
    aslots = aslots > kMaxASlots ? kMaxASlots : aslots;
    aslots = aslots > 2 * stages - 2 ? 2 * stages - 2 : aslots;
    const size_t smem = fixed + static_cast<size_t>(stages) * stage_bytes;
    if (aslots < kDqGroups || smem > 227 * 1024)
        return MOE_ERR_UNSUPPORTED;
    static std::atomic<uint64_t> attr_done{0};
    if (!smem_attr_once(attr_done, reinterpret_cast<const void *>(gemm_kernel<kNv4>), 227 * 1024))
        return MOE_ERR_CUDA;

    // tensor maps: kept codes as bytes [E*N][K/4]; side records [E*N][K/128 * 16]; activations fp16 [cap_rows][K]
    CUtensorMap tQ1, tB1, tQ2, tB2, tS1, tS2;
    if (!grouped_tmap_2d(&tQ1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w13->q, d / 4, static_cast<uint64_t>(E) * 2 * I, 32,
                         128, false) ||
        !grouped_tmap_2d(&tS1, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q13 + P13.side, (d / 128) * kNv4SideBytes,
                         static_cast<uint64_t>(E) * 2 * I, kNv4SideBytes, 128, false) ||
        !grouped_tmap_2d(&tB1, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, xg, d, cap_rows, 64, n_mma, true) ||
        !grouped_tmap_2d(&tQ2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w2->q, I / 4, static_cast<uint64_t>(E) * d, 32, 128,
                         false) ||
        !grouped_tmap_2d(&tS2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q2 + P2.side, (I / 128) * kNv4SideBytes,
                         static_cast<uint64_t>(E) * d, kNv4SideBytes, 128, false) ||
        !grouped_tmap_2d(&tB2, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, hg, I, cap_rows, 64, n_mma, true))
        return MOE_ERR_CUDA;

    const float *qa_x = reinterpret_cast<const float *>(q13 + P13.head);
    const float *qa_h = reinterpret_cast<const float *>(q2 + P2.head);
    const int gblocks = grouped_sm_count() * 4;
    const cudaError_t ge =
        x_bf16 ? launch_pdl(gather_nv4_kernel<__nv_bfloat16>, dim3(gblocks), dim3(256), 0, s,
                            static_cast<const __nv_bfloat16 *>(x), d, k, static_cast<int>(mk), sorted, npp, xg, b, done,
                            cap_rows, dev_status, qa_x)
               : launch_pdl(gather_nv4_kernel<__half>, dim3(gblocks), dim3(256), 0, s, static_cast<const __half *>(x),
                            d, k, static_cast<int>(mk), sorted, npp, xg, b, done, cap_rows, dev_status, qa_x);
    if (ge != cudaSuccess)
        return MOE_ERR_CUDA;
    const int grid = grouped_sm_count();
    Args a1{nullptr, nullptr, expert_ids, npp, sorted, wts, hg, nullptr, dev_status, b, n_mma, I / 128, d / 128, I, d,
            static_cast<int>(mk), 2 * I, d / 128, stages, aslots, acc_cols, nbuf, E, cap_rows / b,
            reinterpret_cast<const float *>(q13 + P13.ce), qa_h};
    Args a2{nullptr, nullptr, expert_ids, npp, sorted, wts, nullptr, yr, dev_status, b, n_mma, d / 256, I / 128, I, d,
            static_cast<int>(mk), d, I / 128, stages, aslots, acc_cols, nbuf, E, cap_rows / b,
            reinterpret_cast<const float *>(q2 + P2.ce), nullptr};
    if (launch_pdl(gemm_kernel<kNv4>, dim3(grid), dim3(kThreads), smem, s, tQ1, tB1, tQ2, tB2, tS1, tS2, a1, a2, done,
                   0) != cudaSuccess)
        return MOE_ERR_CUDA;
    return grouped_combine_launch(yr, ids, M, k, d, E, y, y_f32, s);
}

}  // namespace moe
