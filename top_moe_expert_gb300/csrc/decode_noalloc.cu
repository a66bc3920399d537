// decode_noalloc.cu -- moe_ffn_decode_noalloc: the two-kernel MXFP8 decode
// with its scratch in library-owned static device memory.
//
// Some callers cannot allocate device memory when they run the layer: code
// that executes while a CUDA graph is being captured with a strict capture
// mode, inference runtimes whose memory is handed out up front by a planner
// and that refuse any allocation afterwards, and plugins that only receive
// the tensors of one operator.  For them this entry point takes only the
// inputs and the output; the FP32 intermediate h that moe_ffn_decode keeps
// in the caller's workspace lives here in a fixed device array instead.
#include <mutex>

#include "common.cuh"
#include "decode_internal.h"

namespace moe {

// Largest intermediate the array holds: M * k * I floats.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB per device

// Every GPU that loads the library keeps this array until the process
// exits.  It is shared by all calls on a device and keeps the last call's
// contents; nothing in it has to start at zero (each call writes every h
// element it reads).  Calls that overlap on the GPU -- on two streams, or on
// one stream from two host threads without ordering -- race on it.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Host-side address of the array on each device, looked up once per device
// with that device current.  In host code the symbol itself is only a
// stand-in, not a device address.
static constexpr int kMaxDevices = 64;
static std::mutex g_noalloc_mutex;
static float *g_noalloc_ptr[kMaxDevices] = {};

static moe_status_t noalloc_scratch(float **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_ffn_decode_noalloc(const void *x, int32_t xdt, int32_t M, int32_t d,
                                            const int32_t *topk_ids, const float *topk_w, int32_t k,
                                            const moe_weights_t *w13, const moe_weights_t *w2, void *y,
                                            int32_t ydt, int32_t *dev_status, void *stream)
{
    if (M < 0 || d < 1 || k < 1 || k > 32 || !w13 || !w2)
        return MOE_ERR_INVALID_ARG;
    if (w13->fmt != MOE_W_MXFP8 || w2->fmt != MOE_W_MXFP8 || xdt != MOE_BF16)
        return MOE_ERR_UNSUPPORTED;
    const int I = w2->K;
    if (w13->N != 2 * I || w13->K != d || w2->N != d || w13->E != w2->E || w13->E < 1)
        return MOE_ERR_INVALID_ARG;
    if (!w13->q || !w13->scale || !w2->q || !w2->scale)
        return MOE_ERR_INVALID_ARG;
    if (ydt != MOE_BF16 && ydt != MOE_FP32)
        return MOE_ERR_UNSUPPORTED;
    if (M == 0)
        return MOE_OK;
    if (!decode_stream_eligible(M, k, d, I, w13->E, w13->q, w13->scale, w2->q, w2->scale))
        return MOE_ERR_UNSUPPORTED;
    // the intermediate must fit the fixed array
    if (static_cast<size_t>(M) * k * I * sizeof(float) > kNoAllocScratchBytes)
        return MOE_ERR_CAPACITY;
    if (!x || !topk_ids || !topk_w || !y || !aligned(x, 16))
        return MOE_ERR_INVALID_ARG;
    float *h = nullptr;
    const moe_status_t st = noalloc_scratch(&h);
    if (st != MOE_OK)
        return st;
    return decode_stream_launch(static_cast<const __nv_bfloat16 *>(x), M, d, I, w13->E, topk_ids, topk_w, k,
                                static_cast<const uint8_t *>(w13->q), static_cast<const uint8_t *>(w13->scale),
                                static_cast<const uint8_t *>(w2->q), static_cast<const uint8_t *>(w2->scale), y,
                                ydt == MOE_FP32, h, dev_status, as_stream(stream));
}
