/*
 * moe_ffn.h -- C ABI of libmoe_ffn.so, the GB300 (sm_103a) routed
 * Mixture-of-Experts expert-FFN layer.
 *
 * The layer (pages cited by title and section):
 *   - "Route-Block Membership Selects Packed-AWQ Arithmetic" (arXiv
 *     2607.26316), opening paragraph: a top-k router produces an M x k array
 *     of expert ids; flattening it row-major gives route ids r = t*k + j;
 *     alignment groups the valid routes by expert, pads each expert to a
 *     multiple of a block size b and emits a parallel expert-block vector.
 *   - "Warp decode" (cursor.com blog), section on how the two kernels work:
 *     per routed expert a gate/up projection, SiLU(gate) x up, a down
 *     projection, and the routing-weighted combine folded into the down
 *     accumulation; MXFP8 weights, BF16 activations, FP32 accumulation.
 *   - "Hardware-Native Joint Sparse-Quantization for Trillion-Scale
 *     Mixture-of-Experts" (arXiv 2610.02241), Sec. 3.4 and App. D.1: the
 *     expert products Y_e = X_e W_e^T of a grouped GEMM, computed with the
 *     weights as the left operand (Y_e^T = W_e X_e^T), activations quantized
 *     at run time into 32-element scale blocks, fused SwiGLU + requantization.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and densely packed, unless a parameter says otherwise.  The library
 *     allocates and frees nothing; scratch memory is the caller's `ws`.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work
 *     is enqueued on it and never synchronised; results are ready when the
 *     stream reaches them.  Calls that share `ws` must not overlap.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-MOE_OK status means nothing was enqueued (MOE_ERR_CUDA: a launch
 *     failed; the stream may hold earlier work of the same call).
 *   - Expert ids outside [0, E) are invalid routes: they are skipped and
 *     contribute nothing.  dev_status is NULL or a device int32[2] that the
 *     caller zeroes: dev_status[0] is INCREASED by the number of invalid
 *     routes seen; dev_status[1] receives the first error a kernel detected
 *     on the device (MOE_ERR_TIMEOUT when a bounded wait on an mbarrier
 *     expired; the outputs of that call are then undefined).
 *   - Debug bounds-check build (libmoe_ffn_debug.so, the same sources built
 *     with MOE_DEBUG_BOUNDS): every global index that a kernel takes from
 *     device data -- expert ids, route ids, block rows and row counts of the
 *     alignment outputs -- is checked against its buffer before use; a
 *     failed check skips the access (and the tile that depends on it) and
 *     writes MOE_ERR_BOUNDS to dev_status[1].  The release build trusts the
 *     contracts below and does not check.
 *   - Shapes are int32; M*k and the padded row counts must fit in int32.
 *
 * Weight formats (one projection of all E experts, [E][N][K], K contracted):
 *   MOE_W_MXFP8: q uint8 [E][N][K] OCP E4M3 codes; scale uint8 [E][N][K/32]
 *                OCP E8M0 bytes (value 2^(s-127)); zero NULL.  K % 32 == 0.
 *   MOE_W_AWQ4:  q int32 [E][N][K/8], element 8c+i of a row in bits
 *                4i..4i+3 of word c; scale fp16 [E][N][K/128];
 *                zero int32 [E][N/8][K/128], the zero of row 8a+i in nibble i
 *                of word a; weight = (q - zero) * scale.  K % 128 == 0,
 *                N % 8 == 0.
 *   MOE_W_NVFP4S: paired 4:8 sparse NVFP4 ("Hardware-Native Joint Sparse-
 *                Quantization ...", App. A, Eq. 6 and 7): in every group of
 *                8 weights along K two adjacent pairs are kept, 2.75 bits
 *                per weight.  q uint8 [E][N][K/4]: group g's four kept E2M1
 *                codes in bytes 2g, 2g+1, low nibble first, the two values
 *                of pair p0 then those of pair p1; zero uint8 [E][N][K/16]:
 *                group g's pattern nibble p0 | p1 << 2 (p0 < p1, the kept
 *                pair indices) in byte g/2, low nibble for even g; scale
 *                uint8 [E][N][K/32] UE4M3 codes (0x00..0x7E); alpha fp32
 *                [E].  weight = alpha[e] * UE4M3(scale) * E2M1(code) at the
 *                kept positions, 0 elsewhere.  K % 64 == 0.  A nibble that
 *                is not one of the six patterns gives undefined values (every
 *                read stays inside its group).
 *   W13 is the fused gate/up projection: N = 2I (rows 0..I-1 gate, rows
 *   I..2I-1 up), K = d.  W2 is the down projection: N = d, K = I.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_FFN_ABI_VERSION 3

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, bad enum       */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (format/size) */
    MOE_ERR_CAPACITY = 3,     /* an output capacity is too small         */
    MOE_ERR_WORKSPACE = 4,    /* ws too small or misaligned (256 B)      */
    MOE_ERR_CUDA = 5,         /* a CUDA launch/attribute call failed      */
    MOE_ERR_TIMEOUT = 6,      /* a bounded device wait expired (dev_status[1]) */
    MOE_ERR_BOUNDS = 7        /* debug build only: an index read from device data was out of its
                                 buffer; the access was skipped (dev_status[1]) */
} moe_status_t;

/* (value 2 is retired: it named an MXFP8 layout stored K-outer) */
typedef enum { MOE_W_MXFP8 = 0, MOE_W_AWQ4 = 1, MOE_W_NVFP4S = 3 } moe_wfmt_t;
typedef enum { MOE_BF16 = 0, MOE_FP16 = 1, MOE_FP32 = 2 } moe_dtype_t;
typedef enum { MOE_PATH_DECODE = 0, MOE_PATH_GROUPED = 1 } moe_path_t;

/* One projection of all experts; see "Weight formats" above. */
typedef struct {
    int32_t fmt;         /* moe_wfmt_t                                   */
    int32_t E, N, K;
    const void *q;       /* codes / packed nibbles                       */
    const void *scale;   /* E8M0 bytes / fp16 group scales               */
    const void *zero;    /* NULL / packed zero nibbles / NVFP4S patterns */
    const float *alpha;  /* MOE_W_NVFP4S: fp32 [E] per-expert constant;
                            read for no other format (may be left unset) */
} moe_weights_t;

/* Human-readable name of a status code (static storage). */
const char *moe_status_string(moe_status_t s);
/* MOE_FFN_ABI_VERSION of the loaded library. */
int32_t moe_abi_version(void);
/* ---------------------------------------------------------------- routing
 * Top-k softmax routing ("Warp decode", section on the conventional MoE
 * path: each token selects k of E experts, e.g. 8 of 128).
 *   logits  fp32 [M][E];  topk_ids int32 [M][k];  topk_w fp32 [M][k].
 * Experts are selected by logit (ties to the lower id), slots in descending
 * order; topk_w = softmax over the E logits renormalised over the k chosen
 * (= softmax over the chosen logits).  Logits must be finite.
 * Limits: 1 <= k <= min(E, 32), E <= 4096. */
moe_status_t moe_topk_softmax(const float *logits, int32_t M, int32_t E, int32_t k,
                              int32_t *topk_ids, float *topk_w, void *stream);

/* --------------------------------------------------------------- alignment
 * Route alignment by stable construction ("Route-Block Membership Selects
 * Packed-AWQ Arithmetic", opening and stable-construction paragraphs).
 * Valid routes (id in [0,E)) are ordered by (expert id, route id); each
 * active expert's run is padded with the sentinel M*k to a multiple of b;
 * experts without routes get no block.
 *   topk_ids          int32 [M*k] (the M x k router output, flattened)
 *   sorted_route_ids  int32 [cap_rows]: aligned rows; rows past the padded
 *                     end also hold the sentinel M*k
 *   expert_ids        int32 [cap_blocks]: expert of aligned block j (rows
 *                     j*b .. j*b+b-1); -1 past the last active block
 *   num_rows_post_pad int32 [1]: b * number of active blocks
 * The result is unique, so it is bit-exact and history-independent.
 * moe_align_capacity gives the worst-case cap_rows / cap_blocks
 * (M*k + min(E, M*k)*(b-1), rounded up to b); smaller capacities are
 * accepted, and MOE_ERR_CAPACITY is returned if they are below that bound.
 * ws: moe_align_workspace_size bytes (may be 0).  Limits: E <= 1024,
 * 1 <= b <= 256. */
moe_status_t moe_align_capacity(int32_t M, int32_t k, int32_t E, int32_t b,
                                int32_t *cap_rows, int32_t *cap_blocks);
moe_status_t moe_align_workspace_size(int32_t M, int32_t k, int32_t E, int32_t b, size_t *bytes);
moe_status_t moe_align_block_size(const int32_t *topk_ids, int32_t M, int32_t k, int32_t E,
                                  int32_t b, int32_t *sorted_route_ids, int32_t *expert_ids,
                                  int32_t *num_rows_post_pad, int32_t cap_rows, int32_t cap_blocks,
                                  void *ws, size_t ws_bytes, int32_t *dev_status, void *stream);

/* Fixed-capacity (batched) layout, the alternative to alignment that
 * "Hardware-Native Joint Sparse-Quantization ...", App. D.1 uses: expert e
 * owns rows e*C .. e*C + C - 1 of the operands at a fixed stride, so no
 * prefix over experts is needed, and only its ceil(N_e / b) active blocks
 * are computed.  Inside an expert the routes keep the stable-construction
 * order (route id ascending).
 *   C        rows per expert, a multiple of b; it must be at least every
 *            expert's route count N_e (the page takes the largest count):
 *            routes past C get no row, are counted in dev_status[0] with the
 *            invalid routes, and their tokens' layer output is then not
 *            defined
 *   sorted_route_ids int32 [E*C]: row e*C + i holds the i-th route of
 *            expert e, rows past N_e the sentinel M*k
 *   expert_ids, block_rows int32 [E*C/b]: the active blocks in expert
 *            order, compacted: block j is expert expert_ids[j]'s rows
 *            block_rows[j] .. block_rows[j] + b - 1; the tail -1 / 0
 *   num_rows_post_pad int32 [1]: b * (number of active blocks)
 * Deterministic (the same bits on every call).  Limits: E <= 1024,
 * 1 <= b <= 256, E*C < 2^31.  No workspace. */
moe_status_t moe_align_fixed_capacity(const int32_t *topk_ids, int32_t M, int32_t k, int32_t E, int32_t b,
                                      int32_t C, int32_t *sorted_route_ids, int32_t *expert_ids,
                                      int32_t *block_rows, int32_t *num_rows_post_pad,
                                      int32_t *dev_status, void *stream);

/* ---------------------------------------------------------- quantization
 * MXFP8 quantization of rows of K values, per 32-element block along K
 * ("Hardware-Native Joint Sparse-Quantization ...", Sec. 3.4 / App. D.1:
 * 32-element scale blocks; OCP MX rule): X = floor(log2 amax) - 8 clamped to
 * [-127,127] (amax = 0 gives -127), s = X + 127, q = RNE(v / 2^X) on the E4M3
 * grid, saturating at +-448, sign kept.  Used to build MXFP8 weights and by
 * the grouped path's activation quantization.
 *   v: [rows][K] of vdt (MOE_FP32 or MOE_BF16); q uint8 [rows][K];
 *   s uint8 [rows][K/32].  Inputs must be finite. */
moe_status_t moe_mxfp8_quantize(const void *v, int32_t vdt, int64_t rows, int32_t K,
                                uint8_t *q, uint8_t *s, void *stream);

/* ------------------------------------------------------------ the layer
 * Output-centric decode path ("Warp decode", sections on what changed and
 * how the two kernels work): parallelism over outputs, weight rows streamed
 * once with on-the-fly dequantisation, FP32 accumulation, warp butterfly
 * reductions, the routing weight folded into the down accumulation; no
 * alignment, padding, scatter or combine buffer.
 *   x        [M][d] of xdt (MOE_BF16; MOE_FP16 or MOE_BF16 for AWQ)
 *   topk_ids int32 [M][k], topk_w fp32 [M][k]
 *   w13      N = 2I, K = d (MOE_W_MXFP8, MOE_W_AWQ4 or MOE_W_NVFP4S)
 *   w2       N = d, K = I, same format as w13
 *   y        [M][d] of ydt (MOE_BF16 or MOE_FP32)
 *   ws       moe_ffn_decode_workspace_size bytes, 256-byte aligned; its
 *            first 82176 bytes (256 + 80 KiB) must be zero before the
 *            first call that uses it (e.g. cudaMemset once) and then left
 *            alone: the single-token kernel keeps there a count of its CTAs
 *            over all calls, which gives each call its own tag, and its
 *            exchange of h, each value written with the tag of its call.
 *            Every other path keeps its data after those bytes, so one
 *            workspace sized for the largest batch serves calls of any
 *            batch size in turn.  A tag repeats only after 2^32 calls.
 * y[t] = sum_j topk_w[t][j] * W2_{e_j} (SiLU(g) * u),  [g; u] = W13_{e_j} x[t].
 * Kernels by case: MOE_W_MXFP8 (standard layout) with M == 1,
 * (d, I) in {(512, 256), (1024, 512), (2048, 512), (2048, 768),
 * (2048, 1024)}, k small enough for the shared-memory plan and for every
 * CTA's gate/up stages to fit one lap of its ring (k <= 8 at d = 2048,
 * I = 768 on 152 SMs) -> one kernel, one CTA per SM (each CTA an
 * even share of the (route, neuron) pairs: gate/up rows streamed by
 * cp.async.bulk, h = SiLU(g)*u published in ws with the call's tag; each
 * CTA reads all of h back once every value carries the tag, then forms its
 * own d / #SM output rows of every route's down projection, from those rows
 * streamed into the same ring and h as fp16 after an exact power-of-two
 * rescale per lane, and the routing-weighted sum over the k slots; with
 * moe_ffn_decode_logits the routing runs in it too);
 * MXFP8 with M*k <= 512 -> a gate/up kernel and a
 * down kernel chained by programmatic dependent launch;
 * MOE_W_AWQ4 or MOE_W_NVFP4S with M == 1 and (d, I) in {(1024, 256),
 * (1024, 512), (2048, 512), (2048, 768)} (k <= 13 at d = 2048, I = 768)
 * -> the same one-kernel structure on the 4-bit
 * weights (AWQ: (q - z) exact in fp16, the group scale per lane; NVFP4S:
 * kept pairs times the activation pairs at their pattern positions, the
 * block scale per lane, alpha per row), code, pattern and scale arrays
 * 16-byte aligned (NVFP4S down scales 8-byte aligned), with the routing
 * inside under moe_ffn_decode_logits;
 * MOE_W_NVFP4S otherwise -> a gate/up kernel and a down kernel, one warp per
 * intermediate / output scalar, 16-byte loads of 64 packed weights, the
 * kept values decoded on the fly, FP32 sums, h in ws past its first 256
 * bytes; d % 64 == 0, I % 64 == 0, x MOE_BF16 or MOE_FP16;
 * otherwise one warp per intermediate / output scalar.  Every output's summation order is fixed
 * by the shapes, the path and (one-kernel path) the grid size,
 * so identical inputs give identical bits; the two-kernel and per-scalar
 * paths are also independent of the other tokens in the batch.
 * Limits: d % 512 == 0 and I % 32 == 0 (MXFP8); d % 1024 == 0 and
 * I % 128 == 0 (AWQ4); k <= 32; M <= 65535. */
moe_status_t moe_ffn_decode_workspace_size(int32_t M, int32_t k, int32_t d, int32_t I, size_t *bytes);
moe_status_t moe_ffn_decode(const void *x, int32_t xdt, int32_t M, int32_t d,
                            const int32_t *topk_ids, const float *topk_w, int32_t k,
                            const moe_weights_t *w13, const moe_weights_t *w2,
                            void *y, int32_t ydt, void *ws, size_t ws_bytes,
                            int32_t *dev_status, void *stream);

/* Routing and the decode layer in one call: the same result, bit for bit, as
 * moe_topk_softmax(logits, M, w13->E, k, topk_ids, topk_w) followed by
 * moe_ffn_decode(x, ..., topk_ids, topk_w, ...).  The whole decode step of
 * "Warp decode" (section on the conventional MoE path: route, then the
 * experts): for a single token (M == 1) with the shapes of moe_ffn_decode's
 * one-kernel case and E <= 768 it is one kernel that routes the token itself
 * in every CTA (each CTA ranks the logits: an expert's slot is the number of
 * experts with a larger logit, or an equal one and a lower id); otherwise it
 * launches the two calls.
 *   logits   fp32 [M][E] router logits, E = w13->E
 *   topk_ids int32 [M][k], topk_w fp32 [M][k]: outputs (the routing used)
 *   other arguments and the workspace contract as moe_ffn_decode. */
moe_status_t moe_ffn_decode_logits(const float *logits, const void *x, int32_t xdt, int32_t M, int32_t d,
                                   int32_t k, const moe_weights_t *w13, const moe_weights_t *w2,
                                   int32_t *topk_ids, float *topk_w, void *y, int32_t ydt, void *ws,
                                   size_t ws_bytes, int32_t *dev_status, void *stream);

/* Failure-detection test hook (no counterpart on the pages).  The one-kernel
 * single-token path waits, in every CTA, until every value of h carries the
 * call's tag -- a wait bounded by a time limit of about 2 s, after which the
 * CTA stops, writes MOE_ERR_TIMEOUT to dev_status[1] and returns, leaving
 * the context usable.  on = 1 makes the launches that follow wait for a tag
 * that no CTA writes, so that a test can make that wait run out without
 * faulting or hanging the GPU; on = 0 (the default) restores normal
 * operation.  The workspace stays valid: the next call takes a new tag.
 * Process-wide; on other than 0 or 1 returns MOE_ERR_INVALID_ARG. */
moe_status_t moe_debug_exchange_stall(int32_t on);

/* ------------------------------------------------- expert-centric path
 * Grouped path for larger batches ("Hardware-Native Joint Sparse-
 * Quantization ...", Sec. 3.4 and App. D.1): the expert products
 * Y_e = X_e W_e^T as a grouped GEMM on the tensor cores (tcgen05
 * kind::mxf8f6f4 with E8M0 block scaling), weights on the left operand;
 * activations quantized to MXFP8 at run time into 32-element blocks; fused
 * SwiGLU + requantization after the first GEMM; the routing weight applied
 * in the second GEMM's epilogue; a fixed-order combine over the k slots.
 * Rows are the aligned routes of moe_align_block_size (same b); one MMA
 * N-tile is one MoE block.  Each output element accumulates its K-tiles in
 * ascending order in one accumulator (no split-K, no atomics), so a route's
 * result does not depend on its block membership or on the grid size.
 *
 * moe_grouped_prepare packs the E8M0 scales of both projections once into
 * the tensor-core scale layout (sizes from moe_grouped_prepare_size):
 *   sfa13: [E][I/64][d/128][512] bytes, sfa2: [E][d/128][I/128][512] bytes.
 * moe_ffn_grouped:
 *   x bf16 [M][d]; topk_ids / topk_w [M][k]; w13, w2 MOE_W_MXFP8;
 *   sorted_route_ids [cap_rows], expert_ids, num_rows_post_pad: the output
 *   of moe_align_block_size for the same ids, E and b (8 <= b <= 256,
 *   b % 8 == 0); y [M][d] bf16 or fp32;
 *   ws: moe_ffn_grouped_workspace_size bytes, 256-aligned, laid out as
 *   [Xq | Xs | Hq | Hs | Yr | D], each part rounded up to 256 bytes:
 *     Xq uint8 [cap_rows][d]    MXFP8 codes of x per aligned row (rows of
 *                               padding sentinels are zero)
 *     Xs uint8 [cap_rows/b][d/128][nsf][512]  their E8M0 scales, in the
 *                               scale layout: byte (m%32)*16 + (m/32)*4 + kb
 *                               of atom m/128 holds block kb of row m
 *     Hq uint8 [cap_rows][I]    MXFP8 codes of SiLU(g)*u per aligned row
 *     Hs uint8 [cap_rows/b][I/128][nsf][512]  their scales (same layout)
 *     Yr f32 [M*k][d]           w_route * (W2 h) per route
 *     D  int32 [cap_rows/b]     per block, how many first-GEMM tiles have
 *                               written Hq/Hs (set by the call itself; both
 *                               GEMMs run in one persistent kernel and a
 *                               block's second-GEMM tiles wait for it)
 *   with nsf = ceil(roundup16(b) / 128).
 * 4-bit AWQ weights ("Route-Block Membership Selects Packed-AWQ
 * Arithmetic", opening paragraph): w13 and w2 both MOE_W_AWQ4, x MOE_FP16
 * or MOE_BF16, sfa13 / sfa2 unused (NULL).  The tensor cores take fp16 x fp16
 * (tcgen05 kind::f16, FP32 accumulate): each weight tile is dequantized on
 * chip to fp16 (q - z) * s (one rounding), x is rounded to fp16 and
 * h = SiLU(g) * u is rounded to fp16 before the second GEMM.  ws is laid out
 * as [Xg | Hg | Yr | D], each part rounded up to 256 bytes:
 *     Xg fp16 [cap_rows][d]     x per aligned row (padding rows zero)
 *     Hg fp16 [cap_rows][I]     h per aligned row
 *     Yr f32 [M*k][d]           w_route * (W2 h) per route
 *     D  int32 [cap_rows/b]     per-block counters of the fused GEMM kernel
 *                               (set by the call itself)
 *   Inside every run of 8 columns Xg and Hg hold the values in the order
 *   0, 4, 1, 5, 2, 6, 3, 7 (the order the on-chip dequantization produces).
 *   Extra limits: b <= 128, d % 256 == 0, d / 128 <= 64, I / 128 <= 64,
 *   and b <= 112 when d > 8064 (MOE_ERR_UNSUPPORTED); scale and zero arrays
 *   16-byte aligned (MOE_ERR_INVALID_ARG).
 * Limits: d % 128 == 0, I % 128 == 0, M * d / 4 <= INT32_MAX
 * (MOE_ERR_UNSUPPORTED otherwise); x and y 16-byte aligned
 * (MOE_ERR_INVALID_ARG otherwise). */
moe_status_t moe_grouped_prepare_size(const moe_weights_t *w13, const moe_weights_t *w2,
                                      size_t *sfa13_bytes, size_t *sfa2_bytes);
moe_status_t moe_grouped_prepare(const moe_weights_t *w13, const moe_weights_t *w2,
                                 void *sfa13, void *sfa2, void *stream);
/* Paired 4:8 sparse NVFP4 weights ("Hardware-Native Joint Sparse-Quantization
 * for Trillion-Scale Mixture-of-Experts", Sec. 3.4 and App. D.1: the W4A4
 * grouped path).  moe_grouped_prepare_nvfp4s prepares both projections once
 * (sizes from moe_grouped_prepare_size with MOE_W_NVFP4S weights; p13 / p2
 * 256-byte aligned device buffers, passed to moe_ffn_grouped as sfa13 /
 * sfa2):
 *   alpha_x, alpha_h  the tensor-wide scales of the layer's activations (the
 *     block input x and h = SiLU(g) * u), finite and > 0, constants of the
 *     layer (e.g. calibrated offline); each expert's factor alpha_e =
 *     alpha_w[e] * alpha_in is formed here;
 *   p = [head 256 B: alpha_in, binary32(1 / (6 alpha_in)) | alpha_e fp32 [E]
 *     rounded up to 256 B | side records [E][N][K/128][16 B]: the k-step's 8
 *     pattern bytes, its 4 UE4M3 scale bytes, 4 zero bytes].
 * Run time: Q_a quantizes x and h into 32-element blocks of E2M1 codes with
 * a UE4M3 scale each, every decision in binary32 -- S = the UE4M3 value
 * nearest (ties to even, saturating at 448) binary32(amax * binary32(1 / (6
 * alpha))), and each value's code the E2M1 magnitude nearest (ties to even,
 * saturating at 6) |binary32(v * binary32(1 / binary32(alpha * S)))|, sign
 * kept (all magnitudes 0 when S = 0).  The tensor cores multiply exact
 * products of the quantized operands (fp16 S * E2M1 on both sides) in FP32;
 * the epilogues apply alpha_e (and w_route) to the FP32 accumulators.
 * moe_ffn_grouped with w13 / w2 MOE_W_NVFP4S (alpha as stated under "Weight
 * formats"), x MOE_BF16 or MOE_FP16, sfa13 = p13, sfa2 = p2: ws as for AWQ,
 * [Xg | Hg | Yr | D], where Xg / Hg hold S * E2M1 of Q_a(x) / Q_a(h) as fp16
 * in natural order (alpha_x / alpha_h left out).  Extra limits: b <= 128,
 * d % 256 == 0 (MOE_ERR_UNSUPPORTED); p13 / p2 256-byte aligned, w13->q and
 * w2->q 16-byte aligned (MOE_ERR_INVALID_ARG).  The fixed-capacity layout
 * (moe_ffn_grouped_batched) returns MOE_ERR_UNSUPPORTED. */
moe_status_t moe_grouped_prepare_nvfp4s(const moe_weights_t *w13, const moe_weights_t *w2, float alpha_x,
                                        float alpha_h, void *p13, void *p2, void *stream);
moe_status_t moe_ffn_grouped_workspace_size(int32_t M, int32_t k, int32_t d, int32_t I, int32_t b,
                                            int32_t cap_rows, size_t *bytes);
moe_status_t moe_ffn_grouped(const void *x, int32_t xdt, int32_t M, int32_t d,
                             const int32_t *topk_ids, const float *topk_w, int32_t k,
                             const moe_weights_t *w13, const moe_weights_t *w2,
                             const void *sfa13, const void *sfa2,
                             const int32_t *sorted_route_ids, const int32_t *expert_ids,
                             const int32_t *num_rows_post_pad, int32_t b, int32_t cap_rows,
                             void *y, int32_t ydt, void *ws, size_t ws_bytes,
                             int32_t *dev_status, void *stream);

/* moe_ffn_grouped on the fixed-capacity layout of moe_align_fixed_capacity
 * (MOE_W_MXFP8 only; AWQ returns MOE_ERR_UNSUPPORTED): the same arguments
 * plus block_rows, with cap_rows = E*C (any multiple of b) and ws sized by
 * moe_ffn_grouped_workspace_size for that cap_rows.  Every route's result
 * is the same, bit for bit, as on the aligned layout: a route's output does
 * not depend on the rows it shares a block with. */
moe_status_t moe_ffn_grouped_batched(const void *x, int32_t xdt, int32_t M, int32_t d,
                                     const int32_t *topk_ids, const float *topk_w, int32_t k,
                                     const moe_weights_t *w13, const moe_weights_t *w2,
                                     const void *sfa13, const void *sfa2,
                                     const int32_t *sorted_route_ids, const int32_t *expert_ids,
                                     const int32_t *block_rows, const int32_t *num_rows_post_pad, int32_t b,
                                     int32_t cap_rows, void *y, int32_t ydt, void *ws, size_t ws_bytes,
                                     int32_t *dev_status, void *stream);

/* ------------------------------------------------------- path selection
 * Which of the two paths to run for a batch ("Warp decode", sections on
 * what changed and on hardware efficiency: the output-centric path for few
 * tokens, the expert-centric grouped path for large batches), at the
 * crossover measured on GB300 at d = 2048, I = 768, E = 128, k = 8:
 *   MOE_W_MXFP8: MOE_PATH_DECODE for M <= 1 where the single-kernel decode
 *                is built for (k, d, I) on GB300's 152 SMs (d = 512,
 *                I = 256; d = 1024, I = 512; d = 2048, I = 512, 768 or
 *                1024; k small enough for its plan, k <= 8 at d = 2048,
 *                I = 768), else MOE_PATH_GROUPED (decode 15.4
 *                against grouped 27.8 us at M = 1; grouped 41.5 against
 *                179 us at M = 4 and faster at every larger M; at d = 7168,
 *                I = 2048, M = 1, grouped 80.9 against 250 us);
 *   MOE_W_AWQ4:  MOE_PATH_DECODE for M <= 1 where the single-kernel AWQ
 *                decode is built for (k, d, I) (d = 1024, I = 256 or 512;
 *                d = 2048, I = 512 or 768), else MOE_PATH_GROUPED (14.7
 *                against 34.3 us at M = 1 on the decode shapes).
 *   MOE_W_NVFP4S: MOE_PATH_DECODE for M <= 1 where the single-kernel NVFP4S
 *                decode is built for (k, d, I) (the same (d, I) pairs),
 *                else MOE_PATH_GROUPED (the W4A4 grouped path, which needs
 *                moe_grouped_prepare_nvfp4s: 21.4 against 40.9 us at M = 1;
 *                the grouped path from M = 2, faster than the two-kernel
 *                decode at every M measured).  Blocks as for AWQ.
 * When the preferred path does not take the shape (the limits of
 * moe_ffn_decode and moe_ffn_grouped on d, I and k), the other one is
 * returned; when neither does, MOE_ERR_UNSUPPORTED.
 *   fmt    MOE_W_MXFP8, MOE_W_AWQ4 or MOE_W_NVFP4S (MOE_ERR_UNSUPPORTED
 *          otherwise)
 *   path   out: a moe_path_t
 *   block  out: the block size b for moe_align_block_size and
 *          moe_ffn_grouped when the path is grouped (twice the expected
 *          rows per expert, 2*M*k/E, rounded up to a power of two within
 *          [16, 128] for MXFP8 and [8, 128] for AWQ, at most 64 for AWQ
 *          with d > 8064), else 0.
 * Host only; launches nothing. */
moe_status_t moe_ffn_select_path(int32_t M, int32_t k, int32_t E, int32_t d, int32_t I, int32_t fmt,
                                 int32_t *path, int32_t *block);

/* ---------------------------------------------- expert-parallel sharding
 * "Hardware-Native Joint Sparse-Quantization ...", App. D.3 (serving with the
 * experts sharded over an expert-parallel group).  The rank that owns experts
 * [e_lo, e_hi) keeps them as its own weights, indexed 0 .. e_hi - e_lo - 1;
 * this maps the routing to those indices: local_ids[i] = topk_ids[i] - e_lo
 * for e_lo <= topk_ids[i] < e_hi, else -1 (an invalid route, which every
 * layer call skips and counts in dev_status[0]).  Running the layer on the
 * rank's weights with the mapped routing gives that rank's experts' share of
 * y; the shares of all ranks sum to the full layer.
 *   topk_ids, local_ids  int32 device arrays of n elements (may be the same)
 * n = 0 is a no-op; n < 0, e_lo < 0, e_hi < e_lo or null arrays return
 * MOE_ERR_INVALID_ARG before anything is launched. */
moe_status_t moe_ep_local_routes(const int32_t *topk_ids, int64_t n, int32_t e_lo, int32_t e_hi,
                                 int32_t *local_ids, void *stream);

/* ------------------------------------------------ allocation-free decode
 * No counterpart on the pages: a convenience for callers that cannot hand
 * the library any device memory of its own -- code running under a strict
 * CUDA-graph capture, serving runtimes that plan all device memory up front
 * and forbid later allocation, operator plugins that only see the tensors
 * of the call.  Same arguments and result as moe_ffn_decode on its
 * two-kernel MXFP8 path, but without ws: the FP32 intermediate h
 * (M*k*I floats) lives in a fixed 4 MiB array inside the library.
 *   - Only MOE_W_MXFP8 weights (standard layout), MOE_BF16 x, and the shapes
 *     of the two-kernel path (M*k <= 512, d % 512 == 0, I % 256 == 0,
 *     E <= 1024); MOE_ERR_UNSUPPORTED otherwise.
 *   - M*k*I*4 bytes above 4 MiB return MOE_ERR_CAPACITY (nothing launched).
 *   - Allocates and frees nothing.  Every GPU that loads the library holds
 *     the array until the process exits.  The first call on each device
 *     looks the array's device address up (with that device current); make
 *     that first call before any stream capture.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (nothing in it needs to start at zero).  Calls that overlap
 *     on the GPU race on it: order them on one stream. */
moe_status_t moe_ffn_decode_noalloc(const void *x, int32_t xdt, int32_t M, int32_t d,
                                    const int32_t *topk_ids, const float *topk_w, int32_t k,
                                    const moe_weights_t *w13, const moe_weights_t *w2,
                                    void *y, int32_t ydt, int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
