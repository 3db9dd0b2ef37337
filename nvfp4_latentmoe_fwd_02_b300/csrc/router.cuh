// router.cuh -- the router: canonical fp32 logits, top-k selection, softmax over the k.
//
// Routing (NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph: 512 experts, top-22
// per token; shengxinai.com Nemotron 3 blog, section 2.2: the routing gate stays at width d).
// Logit order (the library's canonical fp32 order, so expert indices are exact):
//   the d axis is cut into chunks of 64; p_c = fmaf chain over the chunk in ascending index
//   starting from +0; chunks form groups of 16; a group sum is ((0 + p_c0) + p_c0+1) + ...
//   over its chunks; logit = ((0 + G_0) + G_1) + ... over the groups; then + bias.
// The router weights are kept transposed, Wt[d][E], so that consecutive experts are
// consecutive in memory (coalesced loads for threads that own one expert each).
// Two paths produce exactly these fp32 operations:
//   small T  router_small_kernel computes the group sums G_g(t, e) into G[t][g][e] (a block
//            owns one group of 16 chunks); the top-k kernel adds them in ascending g and the
//            bias;
//   large T  router_logits_kernel: register-tiled, each thread walks the chunks in order.
// Selection: logit descending, lower expert index first on ties.  Weights: softmax (fp32,
// expf) over the k selected logits.  Output slots are in ascending expert id.
#pragma once
#include "common.cuh"

namespace lmoe {

constexpr int kChunk = 64;

// Buffers the first kernel of a forward clears (up to four ranges of 16-byte words), so that
// no separate clearing launch is needed: the expert histogram before the top-k kernel counts
// into it, and the fp32 accumulators before the GEMMs reduce into them.
struct ZeroRanges {
    uint4 *p[4];
    int64_t n16[4];
};
__device__ __forceinline__ void zero_ranges(const ZeroRanges &z) {
    const int64_t nthreads = (int64_t)gridDim.x * gridDim.y * blockDim.x;
    const int64_t tid = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll
    for (int r = 0; r < 4; ++r)
        for (int64_t i = tid; i < z.n16[r]; i += nthreads) z.p[r][i] = make_uint4(0, 0, 0, 0);
}
__global__ void zero_kernel(ZeroRanges z) {
    pdl_wait();
    pdl_trigger();
    zero_ranges(z);
}

// Small T: group sums G[t][g][e].  Block: 32 experts (lanes) x the 16 chunks of group g
// (warps); thread (e, c) loads its 64 weights once (one coalesced 128-byte load per element
// across the warp) and runs one fmaf chain per token; the block then adds its 16 chunk
// partials in order per (token, expert) from shared memory.  Tokens are staged 16 at a time
// in shared memory as fp32 (all lanes of a warp read the same element: a broadcast).
// grid = (ceil(E / 32), ceil(C / 16)); T <= 64.
constexpr int kSmallMaxT = 64;
constexpr int kSmallEG = 32, kSmallCG = 16, kSmallTG = 16;
constexpr int kGroupChunks = 16;
constexpr int kRouterSmallSmem = kSmallTG * kSmallCG * kChunk * 4 + kSmallTG * kSmallCG * kSmallEG * 4;
__global__ void __launch_bounds__(kSmallEG * kSmallCG) router_small_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wt, int T, int d, int E,
    float *__restrict__ G, ZeroRanges zr) {
    extern __shared__ __align__(16) float xs[];        // [kSmallTG][kSmallCG][64], then ps
    float *ps = xs + kSmallTG * kSmallCG * kChunk;      // [kSmallTG][kSmallCG][32]
    const int C = d / kChunk;
    const int ng = (C + kGroupChunks - 1) / kGroupChunks;
    const int lane = threadIdx.x & 31, cl = threadIdx.x >> 5;
    const int e = blockIdx.x * kSmallEG + lane;
    const int c0 = blockIdx.y * kSmallCG;
    const int c = c0 + cl;
    const bool active = e < E && c < C;
    pdl_wait();
    pdl_trigger();
    zero_ranges(zr);
    float w[kChunk];
    if (active) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) w[i] = __ldg(Wt + static_cast<int64_t>(c * kChunk + i) * E + e);
    }
    const int ncg = min(kSmallCG, C - c0);
    const int per_tok = ncg * (kChunk / 8);            // uint4 per token
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
            G[(static_cast<int64_t>(t0 + tt) * ng + blockIdx.y) * E + e] = gs;
        }
    }
}

// Large T: logits[t][e] (bias added).  Tile 128 tokens x 64 experts per block of 128 threads,
// each thread 8 tokens x 8 experts.  Each 64-element chunk is staged through shared memory in
// two halves of 32 (double-buffered: the next half's global loads are in flight while the
// current half is multiplied); the per-chunk fma chain runs across both halves before it is
// added to acc.  The fmas are issued as fma.rn.f32x2 on expert pairs: two independent IEEE
// fp32 fmas, so every (t, e) chain is exactly the scalar canonical one.  Dynamic smem.
constexpr int kRT = 128, kRE = 64, kHalf = 32;
constexpr int kXsStride = kRT + 4, kWsStride = kRE + 4;
constexpr int kRouterLogitsSmem = 2 * kHalf * (kXsStride + kWsStride) * 4 + 128 * 64 * 4;

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__global__ void __launch_bounds__(128) router_logits_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wt,
    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ logits, ZeroRanges zr) {
    pdl_wait();
    pdl_trigger();
    zero_ranges(zr);
    extern __shared__ __align__(16) float rl_smem[];
    float *xs = rl_smem;                              // [2][kHalf][kXsStride]
    float *ws = rl_smem + 2 * kHalf * kXsStride;      // [2][kHalf][kWsStride]
    float4 *gsum = reinterpret_cast<float4 *>(ws + 2 * kHalf * kWsStride) + threadIdx.x;   // [16][128] float4: this thread's group sums
    const int tid = threadIdx.x;
    const int ty = tid >> 3, tx = tid & 7;
    const int t_base = blockIdx.x * kRT, e_base = blockIdx.y * kRE;
    float acc[8][8];
    uint64_t p[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
#pragma unroll
    for (int m = 0; m < 16; ++m) gsum[m * 128] = make_float4(0.f, 0.f, 0.f, 0.f);
    uint4 xr[4];
    float4 wr[4];
    auto load = [&](int h) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = tid + 128 * j;            // x: 128 tokens x 4 uint4
            const int t = i >> 2, q = i & 3;
            xr[j] = t_base + t < T ? __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t_base + t) * d + h * kHalf + q * 8))
                                   : make_uint4(0, 0, 0, 0);
            const int r = i >> 4, qe = i & 15;      // Wt: 32 rows x 16 float4 of 4 experts
            wr[j] = e_base + qe * 4 < E ? __ldg(reinterpret_cast<const float4 *>(Wt + static_cast<int64_t>(h * kHalf + r) * E + e_base + qe * 4))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto store = [&](int buf) {
        float *X = xs + buf * kHalf * kXsStride;
        float *W = ws + buf * kHalf * kWsStride;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = tid + 128 * j;
            const int t = i >> 2, q = i & 3;
            const uint32_t ww[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                X[(q * 8 + 2 * m) * kXsStride + t] = __uint_as_float(ww[m] << 16);
                X[(q * 8 + 2 * m + 1) * kXsStride + t] = __uint_as_float(ww[m] & 0xFFFF0000u);
            }
            const int r = i >> 4, qe = i & 15;
            *reinterpret_cast<float4 *>(W + r * kWsStride + qe * 4) = wr[j];
        }
    };
    const int H = d / kHalf;
    load(0);
    store(0);
    __syncthreads();
    for (int h = 0; h < H; ++h) {
        const int buf = h & 1;
        if (h + 1 < H) load(h + 1);
        if ((h & 1) == 0) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) p[a][q] = 0ull;
        }
        const float *X = xs + buf * kHalf * kXsStride;
        const float *W = ws + buf * kHalf * kWsStride;
#pragma unroll 4
        for (int i = 0; i < kHalf; ++i) {
            const float4 a0 = *reinterpret_cast<const float4 *>(X + i * kXsStride + ty * 8);
            const float4 a1 = *reinterpret_cast<const float4 *>(X + i * kXsStride + ty * 8 + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(W + i * kWsStride + tx * 8);
            const float4 b1 = *reinterpret_cast<const float4 *>(W + i * kWsStride + tx * 8 + 4);
            const uint64_t bp[4] = {pack2(b0.x, b0.y), pack2(b0.z, b0.w), pack2(b1.x, b1.y), pack2(b1.z, b1.w)};
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const uint64_t aa = pack2(av[a], av[a]);
#pragma unroll
                for (int q = 0; q < 4; ++q) p[a][q] = ffma2(aa, bp[q], p[a][q]);
            }
        }
        if (h & 1) {
            // chunk done: add it to the group sum; at a group's end add that to acc
            const int chunk = h >> 1;
            const bool group_end = ((chunk + 1) % kGroupChunks == 0) || (h + 1 == H);
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                float4 g0 = gsum[(2 * a) * 128], g1 = gsum[(2 * a + 1) * 128];
                float lo, hi;
                unpack2(p[a][0], lo, hi); g0.x = __fadd_rn(g0.x, lo); g0.y = __fadd_rn(g0.y, hi);
                unpack2(p[a][1], lo, hi); g0.z = __fadd_rn(g0.z, lo); g0.w = __fadd_rn(g0.w, hi);
                unpack2(p[a][2], lo, hi); g1.x = __fadd_rn(g1.x, lo); g1.y = __fadd_rn(g1.y, hi);
                unpack2(p[a][3], lo, hi); g1.z = __fadd_rn(g1.z, lo); g1.w = __fadd_rn(g1.w, hi);
                if (group_end) {
                    acc[a][0] = __fadd_rn(acc[a][0], g0.x); acc[a][1] = __fadd_rn(acc[a][1], g0.y);
                    acc[a][2] = __fadd_rn(acc[a][2], g0.z); acc[a][3] = __fadd_rn(acc[a][3], g0.w);
                    acc[a][4] = __fadd_rn(acc[a][4], g1.x); acc[a][5] = __fadd_rn(acc[a][5], g1.y);
                    acc[a][6] = __fadd_rn(acc[a][6], g1.z); acc[a][7] = __fadd_rn(acc[a][7], g1.w);
                    g0 = make_float4(0.f, 0.f, 0.f, 0.f);
                    g1 = g0;
                }
                gsum[(2 * a) * 128] = g0;
                gsum[(2 * a + 1) * 128] = g1;
            }
        }
        if (h + 1 < H) store(buf ^ 1);
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int t = t_base + ty * 8 + a;
        if (t >= T) continue;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int e = e_base + tx * 8 + b;
            if (e < E) logits[static_cast<int64_t>(t) * E + e] = __fadd_rn(acc[a][b], bias ? bias[e] : 0.0f);
        }
    }
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

// Descending bitonic sort of the warp's 128 keys, 4 per lane; key r of lane L sits at position
// 4L + r.
__device__ __forceinline__ void warp_sort128_desc(uint64_t (&a)[4], int lane) {
#pragma unroll
    for (int k = 2; k <= 128; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j >= 1; j >>= 1) {
            if (j >= 4) {
                const int m = j >> 2;                      // partner lane distance
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int i = 4 * lane + r;
                    const uint64_t o = shfl_xor64(a[r], m);
                    const bool lower = (i & j) == 0;       // i < partner
                    const bool desc = (i & k) == 0;        // this run sorts descending
                    const bool keep_max = (lower == desc);
                    a[r] = keep_max ? (a[r] > o ? a[r] : o) : (a[r] < o ? a[r] : o);
                }
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int pr = r ^ j;
                    if (pr > r) {
                        const int i = 4 * lane + r;
                        const bool desc = (i & k) == 0;
                        const uint64_t x = a[r], y = a[pr];
                        const bool swap = desc ? (x < y) : (x > y);
                        a[r] = swap ? y : x;
                        a[pr] = swap ? x : y;
                    }
                }
            }
        }
    }
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

// One block of 256 threads (8 warps) per token: each warp sorts 128 selection keys (E <= 1024),
// the per-warp top-32 lists are merged pairwise (8 -> 4 -> 2 -> 1) through shared memory,
// then warp 0 holds the top-k: softmax over their logits, write idx / w in ascending expert
// id, count tokens per expert and record each slot's offset inside its expert's segment.
constexpr int kTopkThreads = 256;
// src: logits[T][E] (C == 0) or group sums G[T][C][E] (C > 0 groups: summed here in
// ascending group order, then the bias).
__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(
    const float *__restrict__ src, int C, const float *__restrict__ bias, int T, int E, int k,
    int32_t *__restrict__ idx_out, float *__restrict__ w_out, int32_t *__restrict__ counts,
    int32_t *__restrict__ slot_off) {
    __shared__ uint64_t lists[8][32];
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    uint64_t key[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int e = warp * 128 + 4 * lane + r;
        float v = 0.0f;
        if (e < E) {
            if (C == 0) {
                v = __ldg(src + static_cast<int64_t>(t) * E + e);
            } else {
                const float *pt = src + static_cast<int64_t>(t) * C * E + e;
                float acc = 0.0f;
                for (int g = 0; g < C; ++g) acc = __fadd_rn(acc, __ldg(pt + static_cast<int64_t>(g) * E));
                v = __fadd_rn(acc, bias ? bias[e] : 0.0f);
            }
        }
        key[r] = e < E ? topk_key(v, e) : 0ull;             // padding sorts last
    }
    warp_sort128_desc(key, lane);
    // positions 0..31 (lanes 0..7) -> list of this warp
    if (lane < 8) {
#pragma unroll
        for (int r = 0; r < 4; ++r) lists[warp][4 * lane + r] = key[r];
    }
    __syncthreads();
#pragma unroll
    for (int n = 8; n > 1; n >>= 1) {
        uint64_t res = 0;
        if (warp < n / 2) res = merge_top32(lists[2 * warp][lane], lists[2 * warp + 1][31 - lane], lane);
        __syncthreads();
        if (warp < n / 2) lists[warp][lane] = res;
        __syncthreads();
    }
    if (warp != 0) return;
    const uint64_t best = lists[0][lane];
    const int my_idx = lane < k ? key_index(best) : 0x7fffffff;
    const float my_val = lane < k ? key_value(best) : -INFINITY;
    int rank = 0;
    for (int r = 0; r < k; ++r) rank += (__shfl_sync(0xffffffffu, my_idx, r) < my_idx) ? 1 : 0;
    float m = my_val;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float ex = lane < k ? expf(my_val - m) : 0.0f;
    float ssum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
    if (lane < k) {
        idx_out[static_cast<int64_t>(t) * k + rank] = my_idx;
        w_out[static_cast<int64_t>(t) * k + rank] = __fdiv_rn(ex, ssum);
        if (counts) {
            // the histogram's old value is this slot's row inside its expert's segment
            const int off = atomicAdd(counts + my_idx, 1);
            if (slot_off) slot_off[static_cast<int64_t>(t) * k + rank] = off;
        }
    }
}

}  // namespace lmoe
