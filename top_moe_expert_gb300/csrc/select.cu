// select.cu -- host-side choice between the two paths of the layer.
//
// "Warp decode" (cursor.com blog, sections on what changed and on hardware
// efficiency) keeps the expert-centric grouped path for large batches and
// uses the output-centric path where few tokens make the grouped path's
// alignment, padding and combine dominant.  Where the two cross is a matter
// of measurement; the rule below follows the crossover measured on GB300 at
// d = 2048, I = 768, E = 128, k = 8 (us per step, routing included, steps
// back to back over copies of the layer's weights larger than the L2):
//
//     M                    1      2      4      8     16     32     64    512
//     MXFP8 decode      15.4      -    179      -    696      -      -      -
//     MXFP8 grouped     27.8   34.0   41.5   57.3   80.5  102.0  113.8  144.6
//
// At M = 1 the decode figure is the single-kernel form, built for a few
// (d, I) pairs; elsewhere the decode path runs its two-kernel form, which
// loses to the grouped path at every M measured (at d = 7168, I = 2048,
// E = 384, M = 1: 250 us against 80.9 us).  For 4-bit AWQ the single-token
// kernel is ahead at one token (14.7 against 34.3 us for the grouped path)
// and the grouped path from two tokens (far ahead at M = 21).  For paired
// 4:8 sparse NVFP4 the single-token kernel takes one token and the W4A4
// grouped path every batch from two tokens (40.9 us at M = 1 against 76 us
// for the two-kernel decode, and faster at every larger M measured).
// Host only: nothing here touches a GPU.
#include "common.cuh"
#include "decode_internal.h"

namespace moe {

static bool decode_shape_ok(int k, int d, int I, int fmt)
{
    if (static_cast<size_t>(k) * I * sizeof(float) > 200 * 1024)
        return false;
    if (fmt == MOE_W_NVFP4S)
        return d % 64 == 0 && I % 64 == 0;
    return fmt == MOE_W_MXFP8 ? (d % 512 == 0 && I % 32 == 0) : (d % 1024 == 0 && I % 128 == 0);
}

static bool grouped_shape_ok(int d, int I, int b, int fmt)
{
    if (d % 128 || I % 128)
        return false;
    if (fmt == MOE_W_AWQ4)
        return d % 256 == 0 && d / 128 <= 64 && I / 128 <= 64 && b <= 128 && (d <= 8064 || b <= 112);
    if (fmt == MOE_W_NVFP4S)
        return d % 256 == 0 && b <= 128;
    return true;
}

// The SM count the single-kernel decode is planned for (GB300); a GPU with
// another count re-checks the plan at dispatch and falls back if it misses.
constexpr int kSelectSMs = 152;

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_ffn_select_path(int32_t M, int32_t k, int32_t E, int32_t d, int32_t I, int32_t fmt,
                                         int32_t *path, int32_t *block)
{
    if (M < 0 || k < 1 || k > 32 || E < 1 || d < 1 || I < 1 || !path || !block)
        return MOE_ERR_INVALID_ARG;
    if (fmt != MOE_W_MXFP8 && fmt != MOE_W_AWQ4 && fmt != MOE_W_NVFP4S)
        return MOE_ERR_UNSUPPORTED;
    // block size: twice the expected rows per expert, a power of two within
    // [16, 128] (MXFP8) or [8, 128] (AWQ, NVFP4S), so most experts fill one block
    const int64_t rows = 2 * static_cast<int64_t>(M) * k / E;
    int b = fmt == MOE_W_MXFP8 ? 16 : 8;
    while (b < rows && b < 128)
        b *= 2;
    if (fmt == MOE_W_AWQ4 && d > 8064 && b > 64)
        b = 64;
    const bool dec = decode_shape_ok(k, d, I, fmt), grp = grouped_shape_ok(d, I, b, fmt);
    // the output-centric path for one token where its single-kernel form is
    // built for the format; the grouped path otherwise
    const bool want_decode =
        M <= 1 && (fmt == MOE_W_MXFP8  ? decode_pipe_shape_fits(k, d, I, kSelectSMs)
                   : fmt == MOE_W_AWQ4 ? decode_pipe_awq_shape_fits(k, d, I, kSelectSMs)
                                       : decode_pipe_nv4_shape_fits(k, d, I, kSelectSMs));
    if (want_decode ? dec : !grp) {
        if (!dec)
            return MOE_ERR_UNSUPPORTED;
        *path = MOE_PATH_DECODE;
        *block = 0;
        return MOE_OK;
    }
    if (!grp)
        return MOE_ERR_UNSUPPORTED;
    *path = MOE_PATH_GROUPED;
    *block = b;
    return MOE_OK;
}
