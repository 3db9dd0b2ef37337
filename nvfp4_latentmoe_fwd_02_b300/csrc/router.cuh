// router.cuh -- the router: canonical fp32 logits, top-k selection, softmax over the k.
//
// Routing (NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph: 512 experts, top-22
// per token; shengxinai.com Nemotron 3 blog, section 2.2: the routing gate stays at width d).
// Logit order (the library's canonical fp32 order, so expert indices are exact):
//   the d axis is cut into chunks of 64; p_c = fmaf chain over the chunk in ascending index
//   starting from +0; chunks form groups of 16; a group sum is ((0 + p_c0) + p_c0+1) + ...
//   over its chunks; logit = ((0 + G_0) + G_1) + ... over the groups; then + bias.
// Selection: logit descending, lower expert index first on ties.  Weights: softmax (fp32,
// expf) over the k selected logits.  Output slots are in ascending expert id.
// Two paths give exactly the selection of these fp32 operations:
//   small T  (memory bound: the weights are streamed once) router_small_kernel computes the
//            group sums G_g(t, e) into G[t][e][g] from the transposed weights Wt[d][E]
//            (consecutive experts consecutive in memory; a block owns one group of 16 chunks);
//            router_topk_kernel adds them in ascending g, adds the bias and selects;
//   large T  (compute bound) tensor-core logits from bf16 hi/lo planes of the weights bound
//            every canonical logit within a certified margin; router_select_kernel decides
//            what the margin leaves open with canonical logits computed on the spot (below).
#pragma once
#include "common.cuh"

namespace lmoe {

constexpr int kChunk = 64;

// Buffers the first kernel of a forward clears (up to four ranges of 16-byte words), so that
// no separate clearing launch is needed: the expert histogram before the top-k kernel counts
// into it, and the fp32 accumulators before the GEMMs reduce into them.
constexpr int kZeroRanges = 6;
struct ZeroRanges {
    uint4 *p[kZeroRanges];
    int64_t n16[kZeroRanges];
};
__device__ __forceinline__ void zero_ranges(const ZeroRanges &z) {
    const int64_t nthreads = (int64_t)gridDim.x * gridDim.y * blockDim.x;
    const int64_t tid = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll
    for (int r = 0; r < kZeroRanges; ++r)
        for (int64_t i = tid; i < z.n16[r]; i += nthreads) z.p[r][i] = make_uint4(0, 0, 0, 0);
}
__global__ void zero_kernel(ZeroRanges z) {
    pdl_wait();
    pdl_trigger();
    zero_ranges(z);
}

// Small T: group sums G[t][e][g].  Block: 32 experts (lanes) x the 16 chunks of group g
// (warps).  The block's router weights, rows [64 c0, 64 (c0 + 16)) of one 32-expert panel
// (Wp: [ceil(E/32)][d][32], router_panels_kernel), are one contiguous slab of up to 128 KB: a
// single bulk copy brings it into shared memory, issued before the wait on the previous grid
// (the weights are static).  Thread (e, c) runs one fmaf chain over its chunk per token, reading
// the weights from shared memory (lane = expert: conflict free); the block then adds its 16
// chunk partials in order per (token, expert) from shared memory.  Tokens are staged 16 at a time
// in shared memory as fp32 (all lanes of a warp read the same element: a broadcast).
// grid = (ceil(E / 32), ceil(C / 16)); T <= 64.
constexpr int kSmallMaxT = 64;
constexpr int kSmallEG = 32, kSmallCG = 16, kSmallTG = 16;
constexpr int kGroupChunks = 16;
constexpr int kRouterSmallSmem = kSmallCG * kChunk * kSmallEG * 4 + kSmallTG * kSmallCG * kChunk * 4 +
                                 kSmallTG * kSmallCG * kSmallEG * 4 + 16;
__global__ void __launch_bounds__(kSmallEG * kSmallCG) router_small_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wp, int T, int d, int E,
    float *__restrict__ G, ZeroRanges zr, unsigned *err) {
    extern __shared__ __align__(16) float wsm[];        // [kSmallCG * 64][32], then xs, ps, the barrier
    float *xs = wsm + kSmallCG * kChunk * kSmallEG;     // [kSmallTG][kSmallCG][64]
    float *ps = xs + kSmallTG * kSmallCG * kChunk;      // [kSmallTG][kSmallCG][32]
    uint64_t *bar = reinterpret_cast<uint64_t *>(ps + kSmallTG * kSmallCG * kSmallEG);
    const int C = d / kChunk;
    const int ng = (C + kGroupChunks - 1) / kGroupChunks;
    const int lane = threadIdx.x & 31, cl = threadIdx.x >> 5;
    const int e = blockIdx.x * kSmallEG + lane;
    const int c0 = blockIdx.y * kSmallCG;
    const int c = c0 + cl;
    const bool active = e < E && c < C;
    const int ncg = min(kSmallCG, C - c0);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        const uint32_t bytes = static_cast<uint32_t>(ncg * kChunk * kSmallEG * 4);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(wsm, Wp + (static_cast<int64_t>(blockIdx.x) * d + static_cast<int64_t>(c0) * kChunk) * kSmallEG,
                  bytes, bar);
    }
    pdl_wait();
    pdl_trigger();
    zero_ranges(zr);
    const int per_tok = ncg * (kChunk / 8);            // uint4 per token
    bool have_w = false;
    float w[kChunk];
    for (int t0 = 0; t0 < T; t0 += kSmallTG) {
        const int nt = min(kSmallTG, T - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < nt * per_tok; i += blockDim.x) {
            const int t = i / per_tok, r = i - t * per_tok;
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t0 + t) * d + c0 * kChunk) + r);
            float4 *dst = reinterpret_cast<float4 *>(xs + (t * kSmallCG) * kChunk + r * 8);
            dst[0] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                 __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
            dst[1] = make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                                 __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u));
        }
        if (!have_w) {                                  // the weight slab has landed (bounded); the
            if (!mbar_wait(bar, 0)) raise_error(err, kErrTimeout);   // thread's 64 weights to registers
            const float *wr = wsm + cl * kChunk * kSmallEG + lane;
#pragma unroll
            for (int i = 0; i < kChunk; ++i) w[i] = wr[i * kSmallEG];
            have_w = true;
        }
        __syncthreads();
        if (active) {
            for (int t = 0; t < nt; ++t) {
                const float4 *xr = reinterpret_cast<const float4 *>(xs + (t * kSmallCG + cl) * kChunk);
                float p = 0.0f;
#pragma unroll
                for (int i4 = 0; i4 < kChunk / 4; ++i4) {
                    const float4 v = xr[i4];
                    p = fmaf(v.x, w[4 * i4], p);
                    p = fmaf(v.y, w[4 * i4 + 1], p);
                    p = fmaf(v.z, w[4 * i4 + 2], p);
                    p = fmaf(v.w, w[4 * i4 + 3], p);
                }
                ps[(t * kSmallCG + cl) * kSmallEG + lane] = p;
            }
        }
        __syncthreads();
        // thread (t, e): the group sum of its 16 chunk partials, in order
        const int tt = threadIdx.x >> 5;
        if (tt < nt && e < E) {
            float gs = 0.0f;
            for (int q = 0; q < ncg; ++q) gs = __fadd_rn(gs, ps[(tt * kSmallCG + q) * kSmallEG + lane]);
            G[(static_cast<int64_t>(t0 + tt) * E + e) * ng + blockIdx.y] = gs;
        }
    }
    if (!have_w && !mbar_wait(bar, 0)) raise_error(err, kErrTimeout);   // no copy in flight at exit
}

// Top-k by sorting.  A selection key packs (logit, expert) into 64 bits so that a larger key
// means a higher logit, then a lower expert index (-0 is folded onto +0 first): the k largest
// keys are exactly the top-k under (logit desc, index asc), and all keys are distinct.
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
    if (v == 0.0f) v = 0.0f;
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);        // order-preserving on floats
    return (static_cast<uint64_t>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
}
__device__ __forceinline__ float key_value(uint64_t k) {
    uint32_t u = static_cast<uint32_t>(k >> 32);
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}
__device__ __forceinline__ int key_index(uint64_t k) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k));
}
__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Two descending 32-lists (lane i holds element i of each): the top 32 of their union,
// descending, lane i holding element i.
__device__ __forceinline__ uint64_t merge_top32(uint64_t a_i, uint64_t b_rev_i, int lane) {
    uint64_t c = a_i > b_rev_i ? a_i : b_rev_i;             // bitonic, holds the top 32
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const uint64_t o = shfl_xor64(c, m);
        const bool lower = (lane & m) == 0;
        c = lower ? (c > o ? c : o) : (c < o ? c : o);
    }
    return c;
}

// ------------------------------------------------------------------------------------
// Large T: selection certified against the canonical order, with tensor-core logits.
//
// A bf16 tensor-core GEMM gives approximate logits a = x (Whi + Wlo)^T, where Whi = bf16(w)
// and Wlo = bf16(w - Whi) (w - Whi - Wlo is at most 2^-18 |w|), accumulated in fp32 over
// `splits` K-slices and summed with fp32 reductions.  For token t every |a_e + b_e -
// canonical_e| is at most delta_t = |x_t| max_e |w_e| (coef + 2^-16) + 2^-22 max|b|: coef
// bounds the tensor-core accumulation (1024 block steps at d = 8192 split 8 ways, each within
// 2^-23 of the running magnitude, times a margin of 4), 2^-16 the split and the canonical
// order's own rounding (at most 88 roundings of 2^-24), Cauchy-Schwarz bounds sum |x_i w_i|.
// Then, with a_(k) the k-th largest approximate logit:
//   * the true top-k lies inside U = { e : a_e >= a_(k) - 2 delta };
//   * e in U is certainly selected when at most k - 1 others have a_f >= a_e - 2 delta;
//   * the rest of U is decided by exact canonical logits computed here by the token's warp.
// Should U not fit in the sorted top 32, or the counts not add up, the warp computes every
// canonical logit of the token and selects from those.  The routing weights are the softmax
// over the selected logits as known here (canonical where computed, otherwise a + b).
// ------------------------------------------------------------------------------------

// Whi / Wlo planes [E][2d] (row e: Whi then Wlo) and an upper bound of |w_e| per expert.
// One block per expert.
__global__ void router_split_kernel(const float *__restrict__ W, int E, int d,
                                    __nv_bfloat16 *__restrict__ wsplit, float *__restrict__ wnorm) {
    __shared__ double part[8];
    const int e = blockIdx.x;
    const float *w = W + static_cast<int64_t>(e) * d;
    __nv_bfloat16 *o = wsplit + static_cast<int64_t>(e) * 2 * d;
    double ss = 0.0;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const float v = w[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi)));
        o[i] = hi;
        o[d + i] = lo;
        ss += static_cast<double>(v) * static_cast<double>(v);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += part[i];
        wnorm[e] = __fmul_ru(__double2float_ru(sqrt(t)), 1.0f + 0x1p-20f);
    }
}

constexpr int kSelWarps = 8;                 // tokens per block: one warp per token
constexpr int kSelMaxD = 16384;

// The canonical logit (64-element fma chunks, 16-chunk groups, then the bias) of one expert
// for one token, by one warp straight from global memory: lane L takes chunks L, L + 32, ...
// (128-byte rows of bf16 x, 256-byte rows of fp32 w: vector loads), each an fma chain in
// ascending index; a 16-chunk group is the half-warp of one round, summed in order through
// shuffles; the group sums are added in order.  Every lane returns the value.
__device__ __forceinline__ float warp_canonical_logit_g(const __nv_bfloat16 *__restrict__ xt,
                                                        const float *__restrict__ wrow, int C, float bias,
                                                        int lane) {
    float acc = 0.0f;
    for (int r = 0; r * 32 < C; ++r) {
        const int c = r * 32 + lane;
        float p = 0.0f;
        if (c < C) {
            const uint4 *xc = reinterpret_cast<const uint4 *>(xt + c * kChunk);
            const float4 *wc = reinterpret_cast<const float4 *>(wrow + c * kChunk);
#pragma unroll
            for (int q = 0; q < kChunk / 8; ++q) {
                const uint4 u = __ldg(xc + q);
                const float4 w0 = __ldg(wc + 2 * q), w1 = __ldg(wc + 2 * q + 1);
                p = fmaf(__uint_as_float(u.x << 16), w0.x, p);
                p = fmaf(__uint_as_float(u.x & 0xFFFF0000u), w0.y, p);
                p = fmaf(__uint_as_float(u.y << 16), w0.z, p);
                p = fmaf(__uint_as_float(u.y & 0xFFFF0000u), w0.w, p);
                p = fmaf(__uint_as_float(u.z << 16), w1.x, p);
                p = fmaf(__uint_as_float(u.z & 0xFFFF0000u), w1.y, p);
                p = fmaf(__uint_as_float(u.w << 16), w1.z, p);
                p = fmaf(__uint_as_float(u.w & 0xFFFF0000u), w1.w, p);
            }
        }
        // chunks past C contribute +0 at the end of their group (only a zero's sign can change)
        float gs = 0.0f;
        const int base = lane & 16;
#pragma unroll
        for (int q = 0; q < kGroupChunks; ++q) gs = __fadd_rn(gs, __shfl_sync(0xffffffffu, p, base + q));
        const float g0 = __shfl_sync(0xffffffffu, gs, 0), g1 = __shfl_sync(0xffffffffu, gs, 16);
        acc = __fadd_rn(acc, g0);
        if (r * 32 + 16 < C) acc = __fadd_rn(acc, g1);
    }
    return __fadd_rn(acc, bias);
}

// The 32 largest keys of the warp (R keys per lane, distinct except padding 0), sorted
// descending, lane j holding the j-th.  Each lane sorts its own keys (in registers), then
// rounds merge the lanes' r-th largest keys into a running top 32 (a bitonic sort of the 32
// candidates and a bitonic merge with the list): after round r the list is the top 32 of every
// key ranked <= r in its lane, so once no lane's next key beats the list's last the list is
// final (with the top 32 spread over the lanes this takes a few rounds).
template <int R>
__device__ __forceinline__ void sort_desc_local(uint64_t (&a)[R]) {
#pragma unroll
    for (int k = 2; k <= R; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j >= 1; j >>= 1)
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int p = i ^ j;
                if (p > i) {
                    const bool desc = (i & k) == 0;
                    const uint64_t x = a[i], y = a[p];
                    const bool swap = desc ? (x < y) : (x > y);
                    a[i] = swap ? y : x;
                    a[p] = swap ? x : y;
                }
            }
}
__device__ __forceinline__ uint64_t warp_sort32_desc(uint64_t a, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j >= 1; j >>= 1) {
            const uint64_t o = shfl_xor64(a, j);
            const bool lower = (lane & j) == 0;
            const bool desc = (lane & k) == 0;
            a = (lower == desc) ? (a > o ? a : o) : (a < o ? a : o);
        }
    return a;
}
template <int R>
__device__ __forceinline__ uint64_t warp_top32(uint64_t (&key)[R], int lane) {
    sort_desc_local<R>(key);
    uint64_t list = warp_sort32_desc(key[0], lane);
#pragma unroll
    for (int r = 1; r < R; ++r) {
        // stop when no lane's next key beats the 32nd of the list
        uint64_t m = key[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t v = shfl_xor64(m, o);
            m = v > m ? v : m;
        }
        const uint64_t last = (static_cast<uint64_t>(__shfl_sync(0xffffffffu, static_cast<uint32_t>(list >> 32), 31)) << 32) |
                              __shfl_sync(0xffffffffu, static_cast<uint32_t>(list), 31);
        if (m <= last) break;
        const uint64_t cand = warp_sort32_desc(key[r], lane);
        // merge: the top 32 of (list, cand) -- list descending, cand reversed gives a bitonic 64
        const uint64_t crev = (static_cast<uint64_t>(__shfl_sync(0xffffffffu, static_cast<uint32_t>(cand >> 32), 31 - lane)) << 32) |
                              __shfl_sync(0xffffffffu, static_cast<uint32_t>(cand), 31 - lane);
        list = merge_top32(list, crev, lane);
    }
    return list;
}

// Output of one token's selection by its warp: the selected lanes (sel) in ascending expert
// id, the softmax of their values, counts and slot offsets.
__device__ __forceinline__ void emit_selection(int t, int k, bool sel, int e, float v, int lane,
                                               int32_t *idx_out, float *w_out, int32_t *counts,
                                               int32_t *slot_off) {
    const int my_idx = sel ? e : 0x7fffffff;
    const float my_val = sel ? v : -INFINITY;
    int rank = 0;
    for (int r = 0; r < 32; ++r) rank += (__shfl_sync(0xffffffffu, my_idx, r) < my_idx) ? 1 : 0;
    float m = my_val;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float ex = sel ? expf(my_val - m) : 0.0f;
    float ssum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (sel) {
        idx_out[static_cast<int64_t>(t) * k + rank] = my_idx;
        w_out[static_cast<int64_t>(t) * k + rank] = __fdiv_rn(ex, ssum);
        if (counts) {
            const int off = atomicAdd(counts + my_idx, 1);
            if (slot_off) slot_off[static_cast<int64_t>(t) * k + rank] = off;
        }
    }
}

// The expert segments, by the last warp to finish routing (the routing kernels count every
// slot into `counts` first): expert e owns rows [seg_start[e], seg_start[e] + counts[e]) of the
// permuted buffers, its segment padded to a multiple of 128 rows (one tensor-core M tile) so
// that every tile's block scales sit in whole scale atoms; mt_start is the prefix of M tiles.
// Padding rows are never written or read (a tile's valid rows end at its expert's count).
__device__ __forceinline__ void segments_if_last(int units, int *done, const int32_t *counts, int E,
                                                 int32_t *seg_start, int32_t *mt_start, int32_t *nrows,
                                                 int lane) {
    __syncwarp();
    __threadfence();                                       // this warp's counts are visible
    int last = 0;
    if (lane == 0) last = atomicAdd(done, 1) == units - 1;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();
    // every count first (independent loads), then the scan
    int cv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) cv[i] = i * 32 + lane < E ? __ldcg(counts + i * 32 + lane) : 0;
    int run = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (i * 32 >= E) break;
        const int e = i * 32 + lane;
        const int p = (cv[i] + 127) & ~127;
        int incl = p;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (e < E) {
            seg_start[e] = run + incl - p;
            mt_start[e] = (run + incl - p) >> 7;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
        seg_start[E] = run;
        mt_start[E] = run >> 7;
        *nrows = run;
    }
}

// The expert segments laid out by the last of `units` blocks to finish (a whole block: one or
// two experts per thread, E <= 2 blockDim), the same layout as segments_if_last.
__device__ __forceinline__ void segments_block_if_last(int units, int *done, const int32_t *counts, int E,
                                                       int32_t *seg_start, int32_t *mt_start, int32_t *nrows,
                                                       int *s_flag, int32_t *s_wsum) {
    __threadfence();                                       // this block's counts are visible
    __syncthreads();
    if (threadIdx.x == 0) *s_flag = atomicAdd(done, 1) == units - 1;
    __syncthreads();
    if (!*s_flag) return;
    __threadfence();
    const int nthr = blockDim.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = nthr >> 5;
    // expert e = threadIdx.x + j nthr: padded count, block-wide exclusive scan in expert order
    int p[2], incl[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = threadIdx.x + j * nthr;
        p[j] = e < E ? ((__ldcg(counts + e) + 127) & ~127) : 0;
        incl[j] = p[j];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl[j], o);
            if (lane >= o) incl[j] += v;
        }
        if (lane == 31) s_wsum[j * nw + warp] = incl[j];
    }
    __syncthreads();
    if (threadIdx.x == 0) {                                // 2 nw warp totals, in expert order
        int run = 0;
        for (int i = 0; i < 2 * nw; ++i) { const int v = s_wsum[i]; s_wsum[i] = run; run += v; }
        seg_start[E] = run;
        mt_start[E] = run >> 7;
        *nrows = run;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = threadIdx.x + j * nthr;
        if (e < E) {
            const int st = s_wsum[j * nw + warp] + incl[j] - p[j];
            seg_start[e] = st;
            mt_start[e] = st >> 7;
        }
    }
}

// Small T: one block of 512 threads per token, one or two experts per thread (E <= 1024,
// k <= 32).  G: group sums [T][E][NG] (router_small_kernel); a logit is their sum in ascending
// group order plus the bias (the canonical order).  Selection by tournament: each warp sorts its
// keys into a top-32 list in registers (warp_top32), the sixteen lists are merged pairwise to
// the top 32 of the token (merge_top32, four rounds through shared memory), and warp 0 emits the
// first k (emit_selection).  The last block lays out the segments (when `done` is given).
constexpr int kTopkThreads = 512;
__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(
    const float *__restrict__ G, int NG, const float *__restrict__ bias, int T, int E, int k,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts,
    int32_t *__restrict__ slot_off, int *__restrict__ done, int32_t *__restrict__ seg_start,
    int32_t *__restrict__ mt_start, int32_t *__restrict__ nrows) {
    constexpr int nw = kTopkThreads / 32;
    __shared__ uint64_t lists[nw][32];
    __shared__ int32_t wsum[2 * nw];
    __shared__ int s_flag;
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *gt = G + static_cast<int64_t>(t) * E * NG;
    uint64_t key[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = threadIdx.x + j * kTopkThreads;
        float acc = 0.0f;
        if (e < E) {
            if (NG % 4 == 0) {
                for (int g0 = 0; g0 < NG; g0 += 4) {
                    const float4 v = __ldg(reinterpret_cast<const float4 *>(gt + static_cast<int64_t>(e) * NG + g0));
                    acc = __fadd_rn(acc, v.x); acc = __fadd_rn(acc, v.y);
                    acc = __fadd_rn(acc, v.z); acc = __fadd_rn(acc, v.w);
                }
            } else {
                for (int g = 0; g < NG; ++g) acc = __fadd_rn(acc, __ldg(gt + static_cast<int64_t>(e) * NG + g));
            }
            key[j] = topk_key(__fadd_rn(acc, bias ? __ldg(bias + e) : 0.0f), e);
        } else {
            key[j] = 0ull;                                 // below every real key
        }
    }
    lists[warp][lane] = warp_top32<2>(key, lane);
    __syncthreads();
#pragma unroll
    for (int n = nw; n > 1; n >>= 1) {
        uint64_t res = 0;
        if (warp < n / 2) res = merge_top32(lists[2 * warp][lane], lists[2 * warp + 1][31 - lane], lane);
        __syncthreads();
        if (warp < n / 2) lists[warp][lane] = res;
        __syncthreads();
    }
    if (warp == 0) {
        const uint64_t best = lists[0][lane];
        emit_selection(t, k, lane < k, key_index(best), key_value(best), lane, idx_out, w_out, counts, slot_off);
    }
    if (done) segments_block_if_last(T, done, counts, E, seg_start, mt_start, nrows, &s_flag, wsum);
}

// One warp per token (kSelWarps tokens per block).  approx: [T][E] fp32 sums of the tensor-core
// GEMM (no bias); wrows: router weights [E][d] fp32; coef: the accumulation bound described
// above.  R: keys per lane (E <= 32 R).
template <int R>
__global__ void __launch_bounds__(32 * kSelWarps) router_select_kernel(
    const float *__restrict__ approx, const float *__restrict__ bias, const __nv_bfloat16 *__restrict__ x,
    const float *__restrict__ wrows, int T, int d, int E, int k, float coef, float wn_max, float bmax,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts,
    int32_t *__restrict__ slot_off, int *__restrict__ done, int32_t *__restrict__ seg_start,
    int32_t *__restrict__ mt_start, int32_t *__restrict__ nrows) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kSelWarps + warp;
    if (t >= T) return;
    const int C = d / kChunk;
    const __nv_bfloat16 *xt = x + static_cast<int64_t>(t) * d;
    // an upper bound of |x_t| (the fp32 sum of d squares is within d * 2^-24 of exact)
    float ss = 0.0f;
    for (int i = lane * 8; i < d; i += 256) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(xt + i));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(w[j] << 16), b = __uint_as_float(w[j] & 0xFFFF0000u);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float nx = __fmul_ru(sqrtf(ss), 1.0f + 0x1p-10f);
    const float delta = __fadd_ru(__fmul_ru(__fmul_ru(nx, wn_max), __fadd_ru(coef, 0x1p-16f)),
                                  __fmul_ru(bmax, 0x1p-22f));
    const float two_d = __fmul_ru(2.0f, delta);
    // approximate logits + bias -> selection keys
    const float *at = approx + static_cast<int64_t>(t) * E;
    uint64_t key[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int e = i * 32 + lane;
        key[i] = e < E ? topk_key(__fadd_rn(__ldg(at + e), __ldg(bias + e)), e) : 0ull;
    }
    uint64_t top = warp_top32<R>(key, lane);
    float v = key_value(top);                              // NaN for padding (E < 32)
    int e_l = key_index(top);
    const float vk = __shfl_sync(0xffffffffu, v, k - 1);
    const bool in_u = v >= __fsub_rd(vk, two_d);
    const bool overflow = __shfl_sync(0xffffffffu, in_u ? 1 : 0, 31) != 0;
    const float lo = __fsub_rd(v, two_d);
    int cnt = 0;
    for (int j = 0; j < 32; ++j) {
        const float vj = __shfl_sync(0xffffffffu, v, j);
        cnt += (j != lane && vj >= lo) ? 1 : 0;
    }
    const bool certain = in_u && cnt <= k - 1;
    const uint32_t cm = __ballot_sync(0xffffffffu, certain);
    const uint32_t um = __ballot_sync(0xffffffffu, in_u && !certain);
    const int need = k - __popc(cm);
    if (!overflow && need >= 0 && need <= __popc(um)) {
        // canonical logits of the uncertain candidates
        float ve = v;
        for (uint32_t m = um; m; m &= m - 1) {
            const int p = __ffs(m) - 1;
            const int e = __shfl_sync(0xffffffffu, e_l, p);
            const float c = warp_canonical_logit_g(xt, wrows + static_cast<int64_t>(e) * d, C, __ldg(bias + e), lane);
            if (lane == p) ve = c;
        }
        const bool unc = (um >> lane) & 1u;
        const uint64_t kx = unc ? topk_key(ve, e_l) : 0ull;
        int r = 0;
        for (int j = 0; j < 32; ++j) {
            const uint64_t kj = (static_cast<uint64_t>(__shfl_sync(0xffffffffu, static_cast<uint32_t>(kx >> 32), j)) << 32) |
                                __shfl_sync(0xffffffffu, static_cast<uint32_t>(kx), j);
            r += (((um >> j) & 1u) && kj > kx) ? 1 : 0;
        }
        const bool sel = ((cm >> lane) & 1u) || (unc && r < need);
        emit_selection(t, k, sel, e_l, ve, lane, idx_out, w_out, counts, slot_off);
        if (done) segments_if_last(T, done, counts, E, seg_start, mt_start, nrows, lane);
        return;
    }
    // slow path: every canonical logit of the token, then the top k of those
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int e0 = i * 32;
        float mine = 0.0f;
        for (int q = 0; q < 32 && e0 + q < E; ++q) {
            const float c = warp_canonical_logit_g(xt, wrows + static_cast<int64_t>(e0 + q) * d, C, __ldg(bias + e0 + q), lane);
            if (lane == q) mine = c;
        }
        const int e = e0 + lane;
        key[i] = e < E ? topk_key(mine, e) : 0ull;
    }
    top = warp_top32<R>(key, lane);
    emit_selection(t, k, lane < k, key_index(top), key_value(top), lane, idx_out, w_out, counts, slot_off);
    if (done) segments_if_last(T, done, counts, E, seg_start, mt_start, nrows, lane);
}

}  // namespace lmoe
