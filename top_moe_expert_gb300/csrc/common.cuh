// common.cuh -- shared device/host helpers of libmoe_ffn (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_ffn.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

constexpr int kWarp = 32;

// Host: turn the last launch error into a status.
inline moe_status_t launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Round up to a multiple of 256 bytes (workspace carving).
inline size_t ws_round(size_t n) { return (n + 255) & ~size_t(255); }

// ---------------------------------------------------------------- device

// Debug bounds checks.  Built with MOE_DEBUG_BOUNDS, MOE_IN_BOUNDS(cond, st)
// evaluates cond (an index taken from device data against its buffer) and,
// when it fails, writes MOE_ERR_BOUNDS to st[1] (if st is not null); the
// caller skips the access.  In the release build it is the constant true and
// costs nothing.
#ifdef MOE_DEBUG_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, int32_t *st)
{
    if (!ok && st)
        atomicCAS(st + 1, 0, static_cast<int32_t>(MOE_ERR_BOUNDS));
    return ok;
}
#define MOE_IN_BOUNDS(cond, st) ::moe::in_bounds((cond), (st))
#else
#define MOE_IN_BOUNDS(cond, st) true
#endif

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16-byte global load that bypasses L1 allocation: weights are streamed
// once per launch.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_u4(const void *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

// Two E4M3 codes (low and high byte of a 16-bit value) -> two exact fp16.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint16_t v)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return *reinterpret_cast<__half2 *>(&r);
}

// Four E4M3 codes of a 32-bit word -> four exact floats (byte order).
__device__ __forceinline__ void e4m3x4_to_float(uint32_t w, float &f0, float &f1, float &f2, float &f3)
{
    __half2 lo = e4m3x2_to_half2(static_cast<uint16_t>(w & 0xFFFFu));
    __half2 hi = e4m3x2_to_half2(static_cast<uint16_t>(w >> 16));
    float2 a = __half22float2(lo);
    float2 b = __half22float2(hi);
    f0 = a.x; f1 = a.y; f2 = b.x; f3 = b.y;
}

// Two packed bf16 -> two floats (exact).
__device__ __forceinline__ void bf16x2_to_float(uint32_t w, float &lo, float &hi)
{
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

__device__ __forceinline__ void f16x2_to_float(uint32_t w, float &lo, float &hi)
{
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    float2 f = __half22float2(h);
    lo = f.x;
    hi = f.y;
}

// 2^(s-127) of an E8M0 byte as a float (s = 0 gives 2^-127, a subnormal).
__device__ __forceinline__ float e8m0_to_float(uint32_t s)
{
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

// SiLU(g) * u in FP32.
__device__ __forceinline__ float silu_mul(float g, float u)
{
    return g / (1.0f + expf(-g)) * u;
}

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel on the stream is still running; it must execute
// griddepcontrol.wait before touching that kernel's outputs.
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace moe
