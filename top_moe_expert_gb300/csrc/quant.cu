// quant.cu -- MXFP8 quantization (OCP MX rule), one warp per 32-element block.
//
// "Hardware-Native Joint Sparse-Quantization for Trillion-Scale MoE",
// Sec. 3.4 and App. D.1: activations are quantized at run time into
// 32-element scale blocks; the microscaling formats are the OCP MX ones the
// page cites.  Per block: X = floor(log2 amax) - 8 (8 = emax of E4M3),
// clamped to [-127, 127], amax = 0 giving -127; scale byte X + 127; element
// = RNE(v * 2^-X) onto E4M3 with saturation at +-448 (cvt .satfinite).
// v * 2^-X is exact in FP32 for every value that can round to a non-zero
// code, so the element rounding is the single rounding of the definition.
#include "common.cuh"

namespace moe {

// Shared exponent X of a block from the bit pattern of its FP32 amax.
__device__ __forceinline__ int mx_shared_exp(uint32_t amax_bits)
{
    const int ef = static_cast<int>((amax_bits >> 23) & 0xFFu);
    if (ef == 0)
        return -127;                       // zero or subnormal amax: clamped
    int X = ef - 127 - 8;
    return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// 2^-X as an exact float for X in [-127, 127].
__device__ __forceinline__ float mx_inv_scale(int X)
{
    return X <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - X) << 23)
                    : __uint_as_float(0x00400000u);
}

// One value -> E4M3 code, round to nearest even, saturating finite.
__device__ __forceinline__ uint32_t f32_to_e4m3(float u)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(u));
    return r & 0xFFu;
}

template <typename VT>
__device__ __forceinline__ float load_as_float(const VT *p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}

template <typename VT>
__global__ void __launch_bounds__(256)
mxfp8_quantize_kernel(const VT *__restrict__ v, int64_t nblocks, uint8_t *__restrict__ q,
                      uint8_t *__restrict__ s)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t blk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         blk < nblocks; blk += warps) {
        const float val = load_as_float(v + blk * 32 + lane);
        const uint32_t bits = __float_as_uint(fabsf(val));
        const uint32_t amax = __reduce_max_sync(0xffffffffu, bits);
        const int X = mx_shared_exp(amax);
        q[blk * 32 + lane] = static_cast<uint8_t>(f32_to_e4m3(val * mx_inv_scale(X)));
        if (lane == 0)
            s[blk] = static_cast<uint8_t>(X + 127);
    }
}

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_mxfp8_quantize(const void *v, int32_t vdt, int64_t rows, int32_t K,
                                        uint8_t *q, uint8_t *s, void *stream)
{
    if (rows < 0 || K <= 0 || K % 32 != 0)
        return MOE_ERR_INVALID_ARG;
    if (vdt != MOE_FP32 && vdt != MOE_BF16)
        return MOE_ERR_UNSUPPORTED;
    if (rows == 0)
        return MOE_OK;
    if (!v || !q || !s)
        return MOE_ERR_INVALID_ARG;
    const int64_t nblocks = rows * (K / 32);
    int64_t grid64 = (nblocks + 7) / 8;
    const int grid = static_cast<int>(grid64 < 152 * 64 ? grid64 : 152 * 64);
    cudaStream_t st = as_stream(stream);
    if (vdt == MOE_FP32)
        mxfp8_quantize_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float *>(v), nblocks, q, s);
    else
        mxfp8_quantize_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(v), nblocks, q, s);
    return launch_status();
}

