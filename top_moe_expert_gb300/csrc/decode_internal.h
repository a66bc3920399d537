// decode_internal.h -- entries of the specialised decode kernels
// (decode_stream.cu, decode_fused.cu, decode_m1.cu, decode_awq_m1.cu), called
// by moe_ffn_decode when the shape qualifies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ffn.h"

namespace moe {

// Bytes at the start of a decode workspace reserved for the arrival counter
// of the one-kernel single-token paths (ws[0..8), zero before the first use);
// the other decode paths place their data after them.
constexpr size_t kWsReserved = 256;

bool decode_stream_eligible(int M, int k, int d, int I, int E, const void *q13, const void *s13,
                            const void *q2, const void *s2);

moe_status_t decode_stream_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                  const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                  const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32, float *h,
                                  int32_t *dev_status, cudaStream_t stream);

size_t decode_fused_workspace(int M, int d);
bool decode_fused_eligible(int M, int k, int d, int I, int E);
moe_status_t decode_fused_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                 const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                 const uint8_t *q2t, const uint8_t *s2t, void *y, bool y_f32, float *partial,
                                 int32_t *dev_status, cudaStream_t stream);

// single-token MXFP8 layer in one kernel on the standard layout, optionally
// with the routing (decode_pipe.cu); ws holds the arrival counter in its first
// 8 bytes (zero before the first use), then h past kWsReserved
bool decode_pipe_eligible(int M, int k, int d, int I, int E);
bool decode_pipe_route_eligible(int E, int k);
size_t decode_pipe_workspace(int k, int I);
moe_status_t decode_pipe_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                                const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                                const uint8_t *s13, const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32,
                                void *ws, int32_t *dev_status, cudaStream_t stream);

bool decode_m1_eligible(int M, int k, int d, int I, int E);
size_t decode_m1_workspace(int d);
bool decode_m1_route_eligible(int E, int k);
// ids / wts given, or logits given (then ids_out / wts_out receive the routing)
moe_status_t decode_m1_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                              const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                              const uint8_t *s13, const uint8_t *q2t, const uint8_t *s2t, void *y, bool y_f32,
                              void *ws, int32_t *dev_status, cudaStream_t stream);

// single-token MXFP8 layer in one kernel on the standard (K-contiguous) layout
// of both projections, optionally with the routing (decode_mx_m1.cu); ws holds
// the grid-barrier counter in its first 8 bytes (zero before the first use)
bool decode_mx_m1_eligible(int M, int k, int d, int I, int E);
size_t decode_mx_m1_workspace(int k, int I);
moe_status_t decode_mx_m1_launch(const __nv_bfloat16 *x, int d, int I, int E, const int32_t *ids, const float *wts,
                                 const float *logits, int32_t *ids_out, float *wts_out, int k, const uint8_t *q13,
                                 const uint8_t *s13, const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32,
                                 void *ws, int32_t *dev_status, cudaStream_t stream);

// Workspace of the small-batch paths (2 <= M <= 64), each part rounded up to
// 256 bytes: [align ws | sorted route ids | expert ids | rows after padding |
// done | gu | yr], the alignment in blocks of 16 rows
struct SmallWs {
    size_t align_ws, sorted, expert, npp, done, gu, yr, total;
    int cap_rows, cap_blocks;
};
SmallWs small_ws_layout(int M, int k, int d, int I, int E);

// 4-bit AWQ layer for 2 <= M <= 64 through moe_ffn_decode (grouped_awq_mma.cu):
// alignment into blocks of 16 rows, the small-block AWQ kernel, the combine
bool decode_awq_small_eligible(int M, int k, int d, int I, int E);
moe_status_t decode_awq_small_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                     const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                     void *y, bool y_f32, void *ws, size_t ws_bytes, int32_t *dev_status,
                                     cudaStream_t s);

// MXFP8 layer for 2 <= M <= 64 on the standard layout (grouped_mx_mma.cu):
// alignment into blocks of 16 rows, one mma.sync kernel for both GEMMs, then
// the combine; ws as laid out there
bool decode_mx_small_eligible(int M, int k, int d, int I, int E);
size_t decode_mx_small_workspace(int M, int k, int d, int I, int E);
moe_status_t decode_mx_small_launch(const __nv_bfloat16 *x, int M, int d, int I, int E, const int32_t *ids,
                                    const float *wts, int k, const uint8_t *q13, const uint8_t *s13,
                                    const uint8_t *q2, const uint8_t *s2, void *y, bool y_f32, void *ws,
                                    size_t ws_bytes, int32_t *dev_status, cudaStream_t s);

// single-token 4-bit AWQ layer in one kernel (decode_awq_m1.cu); ws holds the
// grid-barrier counter in its first 8 bytes (zero before the first use)
bool decode_awq_m1_eligible(int M, int k, int d, int I, int E);
size_t decode_awq_m1_workspace(int k, int I);
moe_status_t decode_awq_m1_launch(const void *x, bool x_bf16, const int32_t *ids, const float *wts, int k, int d,
                                  int I, int E, const void *q13, const void *s13, const void *z13, const void *q2,
                                  const void *s2, const void *z2, void *y, bool y_f32, void *ws,
                                  int32_t *dev_status, cudaStream_t stream);

// paired 4:8 sparse NVFP4 decode (decode_nvfp4s.cu): a gate/up kernel and a
// down kernel, h [M*k][I] f32 in `h`
bool decode_nvfp4s_eligible(int k, int d, int I);
moe_status_t decode_nvfp4s_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                  const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                  void *y, bool y_f32, float *h, int32_t *dev_status, cudaStream_t s);

}  // namespace moe
