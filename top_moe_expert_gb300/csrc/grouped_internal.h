// grouped_internal.h -- pieces shared by the MXFP8 (grouped.cu) and 4-bit
// AWQ (grouped_awq.cu) expert-centric grouped paths.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ffn.h"

namespace moe {

// 2D tensor map [rows][inner] of `elem_bytes`-byte elements (row stride =
// inner elements), box box_inner x box_rows, optional 128-byte swizzle.
bool grouped_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, int elem_bytes, const void *base, uint64_t inner,
                     uint64_t rows, uint32_t box_inner, uint32_t box_rows, bool sw128);
int grouped_sm_count();
// y[t] = sum over slots j (in order) of Yr[t*k + j] for valid ids
moe_status_t grouped_combine_launch(const float *yr, const int32_t *ids, int M, int k, int d, int E, void *y,
                                    bool y_f32, cudaStream_t s);

// 4-bit AWQ grouped path (kind::f16 on weights dequantized into tensor memory)
size_t grouped_awq_workspace(int M, int k, int d, int I, int b, int cap_rows);
moe_status_t grouped_awq_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                const int32_t *sorted, const int32_t *expert_ids, const int32_t *npp, int b,
                                int cap_rows, void *y, bool y_f32, void *ws, int32_t *dev_status, cudaStream_t s);

// paired 4:8 sparse NVFP4 grouped path (the same kernel, W4A4 with Q_a)
size_t grouped_nv4_prepare_bytes(int E, int N, int K);
moe_status_t grouped_nv4_prepare(const moe_weights_t *w, float alpha_in, void *out, cudaStream_t s);
moe_status_t grouped_nv4_launch(const void *x, bool x_bf16, int M, int d, int I, int E, const int32_t *ids,
                                const float *wts, int k, const moe_weights_t *w13, const moe_weights_t *w2,
                                const void *p13, const void *p2, const int32_t *sorted, const int32_t *expert_ids,
                                const int32_t *npp, int b, int cap_rows, void *y, bool y_f32, void *ws,
                                int32_t *dev_status, cudaStream_t s);

}  // namespace moe
