// decode_internal.h -- entries of the specialised decode kernels
// (decode_pipe.cu, decode_stream.cu, decode_nvfp4s.cu), called by
// moe_ffn_decode when the shape qualifies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ffn.h"

namespace moe {

// The start of a decode workspace is reserved for the single-token kernel
// (zero before the first use): its CTA count over all launches in
// ws[0..8), then, from kWsCounterBytes, its h exchange words (8 bytes per
// (route, neuron), at most kWsTagBytes).  No other path writes there: the
// other decode paths place their data after kWsReserved.
constexpr size_t kWsCounterBytes = 256;
constexpr size_t kWsTagBytes = 80 * 1024;
constexpr size_t kWsReserved = kWsCounterBytes + kWsTagBytes;

bool decode_stream_eligible(int M, int k, int d, int I, int E, const void *q13, const void *s13,
                            const void *q2, const void *s2);

moe_status_t decode_stream_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                  const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                  const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32, float *h,
                                  int32_t *dev_status, cudaStream_t stream);

// single-token MXFP8 layer in one kernel on the standard layout, optionally
// with the routing (decode_pipe.cu); it uses only the reserved start of ws
bool decode_pipe_eligible(int M, int k, int d, int I, int E);
// the shape check alone, for a grid of G CTAs (host only, no device query)
bool decode_pipe_shape_fits(int k, int d, int I, int G);
bool decode_pipe_route_eligible(int E, int k);
// the failure-detection hook's flag (moe_debug_exchange_stall), read at launch
int decode_exchange_stall();
moe_status_t decode_pipe_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                                const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                                const uint8_t *s13, const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32,
                                void *ws, int32_t *dev_status, cudaStream_t stream);

// single-token 4-bit AWQ layer in one kernel (decode_pipe_awq.cu), the same
// structure and workspace use as decode_pipe.cu; x fp16 or bf16
bool decode_pipe_awq_shape_fits(int k, int d, int I, int G);
bool decode_pipe_awq_eligible(int M, int k, int d, int I, int E);
bool decode_pipe_awq_route_eligible(int E, int k);
moe_status_t decode_pipe_awq_launch(const void *x, bool x_bf16, int d, int I, int E, const int32_t *ids,
                                    const float *wts, const float *logits, int32_t *ids_out, float *wts_out, int k,
                                    const moe_weights_t *w13, const moe_weights_t *w2, void *y, bool y_f32, void *ws,
                                    int32_t *dev_status, cudaStream_t s);

// single-token paired 4:8 sparse NVFP4 layer in one kernel (decode_pipe_nv4.cu),
// the same structure and workspace use as decode_pipe.cu; x fp16 or bf16
bool decode_pipe_nv4_shape_fits(int k, int d, int I, int G);
bool decode_pipe_nv4_eligible(int M, int k, int d, int I, int E);
bool decode_pipe_nv4_route_eligible(int E, int k);
moe_status_t decode_pipe_nv4_launch(const void *x, bool x_bf16, int d, int I, int E, const int32_t *ids,
                                    const float *wts, const float *logits, int32_t *ids_out, float *wts_out, int k,
                                    const moe_weights_t *w13, const moe_weights_t *w2, void *y, bool y_f32, void *ws,
                                    int32_t *dev_status, cudaStream_t s);

// paired 4:8 sparse NVFP4 decode (decode_nvfp4s.cu): a gate/up kernel and a
// down kernel, h [M*k][I] f32 in `h`
bool decode_nvfp4s_eligible(int k, int d, int I);
moe_status_t decode_nvfp4s_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                  const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                  void *y, bool y_f32, float *h, int32_t *dev_status, cudaStream_t s);

}  // namespace moe
