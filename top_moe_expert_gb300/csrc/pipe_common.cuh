// pipe_common.cuh -- helpers shared by the three single-token decode kernels
// (decode_pipe.cu, decode_pipe_awq.cu, decode_pipe_nv4.cu): fp16 dot products
// with FP32 accumulation, the 8-way lane reduction, the exact power-of-two
// rescale into fp16, the relaxed loads and stores of the tagged h exchange,
// and each CTA's split of the layer.
#pragma once

#include <cstdint>

namespace moe {
namespace pipe {

__device__ __forceinline__ void set_err(int32_t *st, int code)
{
    if (st)
        atomicCAS(st + 1, 0, code);
}


// acc + w.lo * a.lo + w.hi * a.hi: fp16 products exact in FP32, one rounding each
__device__ __forceinline__ float fma2(uint32_t w, uint32_t a, float acc)
{
    asm("{\n .reg .f16 w0, w1, a0, a1;\n mov.b32 {w0, w1}, %1;\n mov.b32 {a0, a1}, %2;\n"
        " fma.rn.f32.f16 %0, w0, a0, %0;\n fma.rn.f32.f16 %0, w1, a1, %0;\n}"
        : "+f"(acc) : "r"(w), "r"(a));
    return acc;
}

// Sum over 8 values of 32 lanes at once: lane l ends with the total of value
// v_index(l) = 4 * bit4(l) + 2 * bit3(l) + bit2(l) in every lane of its quad.
__device__ __forceinline__ float reduce8(const float (&v)[8], int lane)
{
    float u[4], t[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? v[i] : v[i + 4];
        u[i] = (b4 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? u[i] : u[i + 2];
        t[i] = (b3 ? u[i + 2] : u[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float r = (b2 ? t[1] : t[0]) + __shfl_xor_sync(0xffffffffu, b2 ? t[0] : t[1], 4);
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    return r;
}

// exponent p with m * 2^p in [2^14, 2^15) for a finite m > 0 (the largest
// magnitude of a vector); 0 for m == 0
__device__ __forceinline__ int f16_shift(float m)
{
    if (!(m > 0.f))
        return 0;
    int ex;
    frexpf(m, &ex);            // m = f * 2^ex, f in [0.5, 1)
    const int p = 15 - ex;
    return p < -100 ? -100 : (p > 100 ? 100 : p);
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_relaxed_add(unsigned long long *p)
{
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(p) : "memory");
}

// one (value, tag) word of the h exchange: 8-byte aligned, so single-copy atomic
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// two consecutive exchange words (16-byte aligned); each word is read
// single-copy atomically on its own
__device__ __forceinline__ void ld_relaxed_u64x2(const unsigned long long *p, unsigned long long &a,
                                                 unsigned long long &b)
{
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// This CTA's share of a single-token layer call: the (route, neuron) pairs
// q = r * I + n in [q_lo, q_lo + P), S gate/up stages of PS neurons, and the
// output rows [o0, o0 + nrows), SW down stages of RPS routes; both spaces
// split evenly over the G CTAs (one per SM).  32-bit arithmetic: the plans
// accept nv * I <= 24576 and d <= 2048, so nv * I * G and d * G stay below
// 2^31 for any G below 87000.
struct Split {
    int q_lo, P, S, o0, nrows, SW;
};

template <int PS>
__host__ __device__ __forceinline__ Split cta_split(int nv, int I, int d, int c, int G, int RPS)
{
    const unsigned g = static_cast<unsigned>(G);
    Split s;
    s.q_lo = static_cast<int>(static_cast<unsigned>(nv * I * c) / g);
    s.P = static_cast<int>(static_cast<unsigned>(nv * I * (c + 1)) / g) - s.q_lo;
    s.S = (s.P + PS - 1) / PS;
    s.o0 = static_cast<int>(static_cast<unsigned>(d * c) / g);
    s.nrows = static_cast<int>(static_cast<unsigned>(d * (c + 1)) / g) - s.o0;
    s.SW = s.nrows > 0 ? (nv + RPS - 1) / RPS : 0;
    return s;
}

}  // namespace pipe
}  // namespace moe
