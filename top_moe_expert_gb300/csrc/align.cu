// align.cu -- route alignment by stable construction.
//
// "Route-Block Membership Selects Packed-AWQ Arithmetic", opening paragraph:
// alignment groups the valid routes by expert, pads each expert's count to a
// multiple of the block size b and emits a parallel expert-block vector;
// stable-construction paragraph: valid routes are ordered by (expert id,
// flattened route id), which makes the result history-independent.
//
// GPU design: a counting sort whose every step is deterministic.
//   pass 1 (only when M*k > one chunk): each CTA histograms a chunk of
//          kChunk routes into ws[chunk][E];
//   pass 2: each CTA recomputes the per-expert totals, the padded exclusive
//          prefix over experts and its chunk's base, then places its routes:
//          every warp owns a contiguous slice of the chunk and ranks routes
//          of equal expert with __match_any_sync, so the position of route r
//          is off[e] + (#routes of e before r) exactly as the definition.
// No atomics decide a position, so repeated calls give identical bits.

#include "attr.h"
#include "common.cuh"

namespace moe {

constexpr int kAlignThreads = 256;                 // multi-chunk kernels
constexpr int kAlignThreads1 = 1024;               // the single-chunk placement
constexpr int kChunk = 2048;                       // routes per CTA
constexpr int kAlignMaxE = 1024;

__device__ __forceinline__ bool valid_id(int e, int E) { return e >= 0 && e < E; }

// Pass 1: per-chunk histogram.
__global__ void __launch_bounds__(kAlignThreads)
align_hist_kernel(const int32_t *__restrict__ ids, int MK, int E,
                  int32_t *__restrict__ hist, int32_t *__restrict__ dev_status)
{
    extern __shared__ int32_t sm_hist[];
    __shared__ int inval;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int c = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += kAlignThreads)
        sm_hist[e] = 0;
    if (threadIdx.x == 0)
        inval = 0;
    __syncthreads();
    const int r0 = c * kChunk, r1 = min(MK, r0 + kChunk);
    int my_inval = 0;
    for (int r = r0 + threadIdx.x; r < r1; r += kAlignThreads) {
        int e = ids[r];
        if (valid_id(e, E))
            atomicAdd(&sm_hist[e], 1);
        else
            ++my_inval;
    }
    if (my_inval)
        atomicAdd(&inval, my_inval);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kAlignThreads)
        hist[static_cast<int64_t>(c) * E + e] = sm_hist[e];
    if (threadIdx.x == 0 && inval && dev_status)
        atomicAdd(dev_status, inval);
}

// Block-wide exclusive scan of n <= 4*THREADS ints in place; returns the
// total to every thread.
template <int THREADS>
__device__ int block_exclusive_scan(int32_t *a, int n)
{
    constexpr int kAlignWarps = THREADS / 32;
    __shared__ int warp_tot[kAlignWarps];
    const int per = 4;
    const int base = threadIdx.x * per;
    static_assert(THREADS * per >= 1024, "E up to 1024");
    int v[per];
    int s = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        v[i] = (base + i < n) ? a[base + i] : 0;
        s += v[i];
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        warp_tot[w] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int i = 0; i < kAlignWarps; ++i) {
        if (i < w)
            wbase += warp_tot[i];
        total += warp_tot[i];
    }
    int run = wbase + incl - s;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        if (base + i < n)
            a[base + i] = run;
        run += v[i];
    }
    __syncthreads();
    return total;
}

// Largest e in [0, n) with a[e] <= v, for ascending a with a[0] <= v.
__device__ __forceinline__ int last_le(const int32_t *a, int n, int v)
{
    int lo = 0, hi = n;              // a[lo] <= v, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= v)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Pass 2: offsets, padding, tails and stable placement of one chunk.
template <int THREADS>
__global__ void __launch_bounds__(THREADS)
align_place_kernel(const int32_t *__restrict__ ids, int MK, int E, int b, int nchunks,
                   const int32_t *__restrict__ hist,      // [nchunks][E] or null (1 chunk)
                   int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
                   int32_t *__restrict__ num_rows_post_pad, int cap_rows, int cap_blocks,
                   int32_t *__restrict__ dev_status)
{
    constexpr int kAlignThreads = THREADS, kAlignWarps = THREADS / 32;
    extern __shared__ int32_t sm[];
    int32_t *tot = sm;                 // [E] routes of expert e
    int32_t *cbase = sm + E;           // [E] routes of e in earlier chunks
    int32_t *off = sm + 2 * E;         // [E] first aligned row of e
    int32_t *wcnt = sm + 3 * E;        // [kAlignWarps][E]
    int32_t *s_ids = wcnt + kAlignWarps * E;   // [kChunk] this chunk's ids
    __shared__ int inval;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int c = blockIdx.x;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int r0 = c * kChunk, r1 = min(MK, r0 + kChunk);

    for (int r = r0 + threadIdx.x; r < r1; r += kAlignThreads)
        s_ids[r - r0] = __ldg(ids + r);
    for (int i = threadIdx.x; i < (3 + kAlignWarps) * E; i += kAlignThreads)
        sm[i] = 0;
    if (threadIdx.x == 0)
        inval = 0;
    __syncthreads();
    if (hist == nullptr) {
        // single chunk: histogram here
        int my_inval = 0;
        for (int r = r0 + threadIdx.x; r < r1; r += kAlignThreads) {
            int e = s_ids[r - r0];
            if (valid_id(e, E))
                atomicAdd(&tot[e], 1);
            else
                ++my_inval;
        }
        if (my_inval)
            atomicAdd(&inval, my_inval);
    } else {
        for (int e = threadIdx.x; e < E; e += kAlignThreads) {
            int t = 0, cb = 0;
            for (int cc = 0; cc < nchunks; ++cc) {
                int h = hist[static_cast<int64_t>(cc) * E + e];
                t += h;
                if (cc < c)
                    cb += h;
            }
            tot[e] = t;
            cbase[e] = cb;
        }
    }
    __syncthreads();
    if (hist == nullptr && threadIdx.x == 0 && inval && dev_status)
        atomicAdd(dev_status, inval);
    for (int e = threadIdx.x; e < E; e += kAlignThreads)
        off[e] = (tot[e] + b - 1) / b * b;
    __syncthreads();
    const int total_rows = block_exclusive_scan<THREADS>(off, E);

    // bookkeeping, spread over all CTAs' threads: every aligned row that is
    // padding (its expert's rows end before it) and every row past the end
    // gets the sentinel MK; every block gets its expert id, -1 past the end.
    // The expert of row i is the last e with off[e] <= i (experts without
    // rows share their offset with the next one and never match).
    {
        const int stride = nchunks * kAlignThreads;
        for (int i = c * kAlignThreads + threadIdx.x; i < cap_rows; i += stride) {
            if (i >= total_rows) {
                sorted_ids[i] = MK;
            } else {
                const int e = last_le(off, E, i);
                if (i - off[e] >= tot[e])
                    sorted_ids[i] = MK;
            }
        }
        const int nblk = total_rows / b;
        for (int j = c * kAlignThreads + threadIdx.x; j < cap_blocks; j += stride)
            expert_ids[j] = j < nblk ? last_le(off, E, j * b) : -1;
    }
    if (c == 0 && threadIdx.x == 0)
        *num_rows_post_pad = total_rows;

    // stable placement: warp w owns routes [s0, s1) of this chunk (slices
    // of whole 32-route groups, spread over all warps)
    const int slice = ((r1 - r0 + kAlignWarps - 1) / kAlignWarps + 31) / 32 * 32;
    const int s0 = min(r1, r0 + w * slice), s1 = min(r1, s0 + slice);
    int32_t *mycnt = wcnt + w * E;
    for (int r = s0 + lane; r < s1; r += 32) {
        int e = s_ids[r - r0];
        if (valid_id(e, E))
            atomicAdd(&mycnt[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kAlignThreads) {
        int run = 0;
        for (int ww = 0; ww < kAlignWarps; ++ww) {
            int v = wcnt[ww * E + e];
            wcnt[ww * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int base = s0; base < s1; base += 32) {
        const int r = base + lane;
        const bool in = r < s1;
        const int e = in ? s_ids[r - r0] : -1;
        const bool ok = in && valid_id(e, E);
        const unsigned key = ok ? static_cast<unsigned>(e) : 0xffffffffu;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const unsigned lt = (1u << lane) - 1u;
        const int rank = __popc(peers & lt);
        int before = 0;
        if (ok)
            before = mycnt[e];
        __syncwarp();
        if (ok) {
            sorted_ids[off[e] + cbase[e] + before + rank] = r;
            if ((peers & lt) == 0)                 // leader of its group
                mycnt[e] = before + __popc(peers);
        }
        __syncwarp();
    }
}

}  // namespace moe

using namespace moe;

static int64_t align_bound_rows(int64_t M, int64_t k, int64_t E, int64_t b)
{
    int64_t mk = M * k;
    int64_t rows = mk + (E < mk ? E : mk) * (b - 1);
    return (rows + b - 1) / b * b;
}

MOE_API moe_status_t moe_align_capacity(int32_t M, int32_t k, int32_t E, int32_t b,
                                        int32_t *cap_rows, int32_t *cap_blocks)
{
    if (M < 0 || k < 1 || E < 1 || b < 1 || !cap_rows || !cap_blocks)
        return MOE_ERR_INVALID_ARG;
    int64_t rows = align_bound_rows(M, k, E, b);
    if (rows > INT32_MAX)
        return MOE_ERR_UNSUPPORTED;
    *cap_rows = static_cast<int32_t>(rows);
    *cap_blocks = static_cast<int32_t>(rows / b);
    return MOE_OK;
}

MOE_API moe_status_t moe_align_workspace_size(int32_t M, int32_t k, int32_t E, int32_t b, size_t *bytes)
{
    if (M < 0 || k < 1 || E < 1 || b < 1 || !bytes)
        return MOE_ERR_INVALID_ARG;
    int64_t mk = static_cast<int64_t>(M) * k;
    int64_t nchunks = (mk + kChunk - 1) / kChunk;
    *bytes = nchunks > 1 ? ws_round(static_cast<size_t>(nchunks) * E * sizeof(int32_t)) : 0;
    return MOE_OK;
}

MOE_API moe_status_t moe_align_block_size(const int32_t *topk_ids, int32_t M, int32_t k, int32_t E,
                                          int32_t b, int32_t *sorted_route_ids, int32_t *expert_ids,
                                          int32_t *num_rows_post_pad, int32_t cap_rows,
                                          int32_t cap_blocks, void *ws, size_t ws_bytes,
                                          int32_t *dev_status, void *stream)
{
    if (M < 0 || k < 1 || E < 1 || b < 1)
        return MOE_ERR_INVALID_ARG;
    if (E > kAlignMaxE || b > 256)
        return MOE_ERR_UNSUPPORTED;
    const int64_t mk = static_cast<int64_t>(M) * k;
    const int64_t bound = align_bound_rows(M, k, E, b);
    if (bound > INT32_MAX)
        return MOE_ERR_UNSUPPORTED;
    if ((cap_rows > 0 && !sorted_route_ids) || (cap_blocks > 0 && !expert_ids) || !num_rows_post_pad ||
        (mk > 0 && !topk_ids))
        return MOE_ERR_INVALID_ARG;
    if (cap_rows < bound || cap_blocks < bound / b)
        return MOE_ERR_CAPACITY;
    size_t need = 0;
    moe_align_workspace_size(M, k, E, b, &need);
    if (need > 0 && (ws == nullptr || ws_bytes < need || !aligned(ws, 256)))
        return MOE_ERR_WORKSPACE;

    const int nchunks = static_cast<int>(mk > 0 ? (mk + kChunk - 1) / kChunk : 1);
    cudaStream_t s = as_stream(stream);
    int32_t *hist = nullptr;
    if (nchunks > 1) {
        hist = static_cast<int32_t *>(ws);
        if (launch_pdl(align_hist_kernel, dim3(nchunks), dim3(kAlignThreads), E * sizeof(int32_t), s, topk_ids,
                       static_cast<int>(mk), E, hist, dev_status) != cudaSuccess)
            return MOE_ERR_CUDA;
        const size_t smem = (static_cast<size_t>(3 + kAlignThreads / 32) * E + kChunk) * sizeof(int32_t);
        static std::atomic<uint64_t> attr_m{0};
        if (smem > 100 * 1024 ||
            !smem_attr_once(attr_m, reinterpret_cast<const void *>(align_place_kernel<kAlignThreads>), 100 * 1024))
            return MOE_ERR_CUDA;
        return launch_pdl(align_place_kernel<kAlignThreads>, dim3(nchunks), dim3(kAlignThreads), smem, s, topk_ids,
                          static_cast<int>(mk), E, b, nchunks, static_cast<const int32_t *>(hist), sorted_route_ids,
                          expert_ids, num_rows_post_pad, cap_rows, cap_blocks, dev_status) == cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }
    // one chunk: a single CTA of 1024 threads does everything
    const size_t smem = (static_cast<size_t>(3 + kAlignThreads1 / 32) * E + kChunk) * sizeof(int32_t);
    static std::atomic<uint64_t> attr_1{0};
    if (smem > 200 * 1024 ||
        !smem_attr_once(attr_1, reinterpret_cast<const void *>(align_place_kernel<kAlignThreads1>), 200 * 1024))
        return MOE_ERR_CUDA;
    return launch_pdl(align_place_kernel<kAlignThreads1>, dim3(1), dim3(kAlignThreads1), smem, s, topk_ids,
                      static_cast<int>(mk), E, b, 1, static_cast<const int32_t *>(nullptr), sorted_route_ids,
                      expert_ids, num_rows_post_pad, cap_rows, cap_blocks, dev_status) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

namespace moe {

// ---------------------------------------------------------------- fixed capacity
// The batched operand layout of "Hardware-Native Joint Sparse-Quantization
// for Trillion-Scale Mixture-of-Experts", App. D.1: every expert owns C rows
// at a fixed stride (rows e*C .. e*C + C - 1), so its operands need no
// prefix sum; a tile list covers only ceil(N_e / b) blocks of expert e.
// Inside an expert the routes keep the stable-construction order (route id
// ascending), as in moe_align_block_size.

// One CTA per expert: its routes in route-id order into its C rows (routes
// past C are dropped and counted), the rest of its rows the sentinel M*k;
// its route count (capped at C) into cnt[e].
__global__ void __launch_bounds__(1024) align_fixed_place_kernel(const int32_t *__restrict__ ids, int MK, int E,
                                                                 int C, int32_t *__restrict__ sorted,
                                                                 int32_t *__restrict__ cnt,
                                                                 int32_t *__restrict__ dev_status)
{
    __shared__ int warp_tot[32];
    __shared__ int base_s;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    int32_t *rows = sorted + static_cast<int64_t>(e) * C;
    if (tid == 0)
        base_s = 0;
    __syncthreads();
    for (int r0 = 0; r0 < MK; r0 += blockDim.x) {
        const int r = r0 + tid;
        const bool mine = r < MK && ids[r] == e;
        const unsigned m = __ballot_sync(0xffffffffu, mine);
        if (lane == 0)
            warp_tot[wid] = __popc(m);
        __syncthreads();
        int before = base_s;
        for (int w = 0; w < wid; ++w)
            before += warp_tot[w];
        const int pos = before + __popc(m & ((1u << lane) - 1u));
        if (mine && pos < C)
            rows[pos] = r;
        __syncthreads();
        if (tid == 0) {
            int t = 0;
            for (int w = 0; w < nw; ++w)
                t += warp_tot[w];
            base_s += t;
        }
        __syncthreads();
    }
    const int n = base_s;
    for (int i = (n < C ? n : C) + tid; i < C; i += blockDim.x)
        rows[i] = MK;
    if (tid == 0) {
        cnt[e] = n < C ? n : C;
        if (n > C && dev_status)
            atomicAdd(dev_status, n - C);
    }
    if (e == 0 && dev_status) {
        // invalid routes (ids outside [0, E)) are counted once
        int bad = 0;
        for (int r = tid; r < MK; r += blockDim.x)
            bad += !valid_id(ids[r], E);
        bad = __reduce_add_sync(0xffffffffu, bad);
        if (lane == 0 && bad)
            atomicAdd(dev_status, bad);
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

// One CTA: the active blocks of every expert in expert order, compacted:
// expert_ids[j], block_rows[j] (the block's first row); the tail -1 / 0;
// num_rows_post_pad = b * (number of active blocks).
__global__ void __launch_bounds__(1024) align_fixed_blocks_kernel(int E, int C, int b, int cap_blocks,
                                                                  int32_t *__restrict__ expert_ids,
                                                                  int32_t *__restrict__ block_rows,
                                                                  int32_t *__restrict__ npp)
{
    extern __shared__ int32_t sm_nb[];          // [E] blocks per expert, then their exclusive prefix
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int tid = threadIdx.x;
    // the counts were parked in expert_ids[0 .. E); read them all first
    for (int e = tid; e < E; e += blockDim.x)
        sm_nb[e] = (expert_ids[e] + b - 1) / b;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            const int nb = sm_nb[e];
            sm_nb[E + e] = run;
            run += nb;
        }
        sm_nb[2 * E] = run;
    }
    __syncthreads();
    const int total = sm_nb[2 * E];
    for (int e = 0; e < E; ++e) {
        const int nb = sm_nb[e], off = sm_nb[E + e];
        for (int t = tid; t < nb; t += blockDim.x) {
            expert_ids[off + t] = e;
            block_rows[off + t] = e * C + t * b;
        }
    }
    for (int j = total + tid; j < cap_blocks; j += blockDim.x) {
        expert_ids[j] = -1;
        block_rows[j] = 0;
    }
    if (tid == 0)
        *npp = total * b;
}

}  // namespace moe

using namespace moe;

MOE_API moe_status_t moe_align_fixed_capacity(const int32_t *topk_ids, int32_t M, int32_t k, int32_t E, int32_t b,
                                              int32_t C, int32_t *sorted_route_ids, int32_t *expert_ids,
                                              int32_t *block_rows, int32_t *num_rows_post_pad,
                                              int32_t *dev_status, void *stream)
{
    if (M < 0 || k < 1 || E < 1 || b < 1 || C < 1 || C % b)
        return MOE_ERR_INVALID_ARG;
    if (E > kAlignMaxE || b > 256)
        return MOE_ERR_UNSUPPORTED;
    const int64_t mk = static_cast<int64_t>(M) * k, rows = static_cast<int64_t>(E) * C;
    if (rows > INT32_MAX || mk >= INT32_MAX)
        return MOE_ERR_UNSUPPORTED;
    if (!sorted_route_ids || !expert_ids || !block_rows || !num_rows_post_pad || (mk > 0 && !topk_ids))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    // per-expert counts go to expert_ids[0 .. E) (E <= E*C/b entries)
    if (launch_pdl(align_fixed_place_kernel, dim3(E), dim3(1024), 0, s, topk_ids, static_cast<int>(mk), E,
                   static_cast<int>(C), sorted_route_ids, expert_ids, dev_status) != cudaSuccess)
        return MOE_ERR_CUDA;
    const size_t smem = (2 * static_cast<size_t>(E) + 1) * sizeof(int32_t);
    return launch_pdl(align_fixed_blocks_kernel, dim3(1), dim3(1024), smem, s, E, static_cast<int>(C), b,
                      static_cast<int>(rows / b), expert_ids, block_rows, num_rows_post_pad) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}
