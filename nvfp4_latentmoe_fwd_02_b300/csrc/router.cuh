// router.cuh -- the router: canonical fp32 logits, top-k selection, softmax over the k.
//
// Routing (NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph: 512 experts, top-22
// per token; shengxinai.com Nemotron 3 blog, section 2.2: the routing gate stays at width d).
// Logit order (the library's canonical fp32 order, so expert indices are exact):
//   the d axis is cut into chunks of 64; p_c = fmaf chain over the chunk in ascending index
//   starting from +0; logit = ((0 + p_0) + p_1) + ... in ascending c; then + bias.
// Two kernels produce exactly these fp32 operations:
//   router_small_kernel      small T: one thread per (expert, chunk) computes p_c for a tile
//                            of tokens; the partials are added in order from shared memory;
//   router_logits_kernel     large T: register-tiled, each thread walks the chunks in order.
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

// Small T: logits[t][e] with the chunk partials reduced through shared memory.  Block: four
// experts x 128 threads; the block stages a tile of 8 tokens of x in shared memory (bf16, chunk
// rows padded by 16 bytes against bank conflicts); thread c computes the partial p_c (one
// 64-element fmaf chain) of chunk c for the tile; then one thread per (expert, token) adds the
// chunk partials left to right and the bias.  d <= 8192 (one chunk per thread);
// grid = ceil(E / 4); dynamic smem router_small_smem(d).
constexpr int kSmallTT = 8;
constexpr int kSmallMaxC = 128;
constexpr int kSmallExperts = 4;
constexpr int kXRow = kChunk + 8;   // bf16 elements per staged chunk row (16-byte pad)
__host__ __device__ constexpr int router_small_smem(int d) {
    return kSmallTT * (d / kChunk) * kXRow * 2 + kSmallExperts * kSmallTT * (kSmallMaxC + 4) * 4;
}
__global__ void __launch_bounds__(512) router_small_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wr,
    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ logits, ZeroRanges zr) {
    zero_ranges(zr);
    extern __shared__ __align__(16) uint8_t rs_smem[];
    const int C = d / kChunk;
    uint16_t *xs = reinterpret_cast<uint16_t *>(rs_smem);                                  // [TT][C][kXRow]
    float *ps = reinterpret_cast<float *>(rs_smem + kSmallTT * C * kXRow * 2);             // [4][TT][kSmallMaxC + 4]
    const int grp = threadIdx.x >> 7, c = threadIdx.x & 127;
    const int e = blockIdx.x * kSmallExperts + grp;
    const bool active = e < E && c < C;
    float w[kChunk];
    if (active) {
        const float4 *src = reinterpret_cast<const float4 *>(Wr + static_cast<int64_t>(e) * d + c * kChunk);
#pragma unroll
        for (int i = 0; i < kChunk / 4; ++i) {
            const float4 f = __ldg(src + i);
            w[4 * i] = f.x; w[4 * i + 1] = f.y; w[4 * i + 2] = f.z; w[4 * i + 3] = f.w;
        }
    }
    for (int t0 = 0; t0 < T; t0 += kSmallTT) {
        const int nt = min(kSmallTT, T - t0);
        __syncthreads();
        {
            // loads in flight in groups of 8 before their stores (at most 16 per thread)
            const int total = nt * C * (kChunk / 8);
#pragma unroll
            for (int g0 = 0; g0 < 16; g0 += 8) {
                uint4 buf[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = threadIdx.x + (g0 + j) * 512;
                    if (i < total) {
                        const int t = i / (C * (kChunk / 8));
                        const int r = i - t * (C * (kChunk / 8));
                        buf[j] = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t0 + t) * d + r * 8));
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i = threadIdx.x + (g0 + j) * 512;
                    if (i < total) {
                        const int t = i / (C * (kChunk / 8));
                        const int r = i - t * (C * (kChunk / 8));
                        const int cc = r >> 3, q = r & 7;
                        *reinterpret_cast<uint4 *>(xs + (t * C + cc) * kXRow + q * 8) = buf[j];
                    }
                }
            }
        }
        __syncthreads();
        if (active) {
            float p[kSmallTT];
#pragma unroll
            for (int t = 0; t < kSmallTT; ++t) p[t] = 0.0f;
#pragma unroll
            for (int q = 0; q < kChunk / 8; ++q) {
#pragma unroll
                for (int t = 0; t < kSmallTT; ++t) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(xs + (t * C + c) * kXRow + q * 8);
                    const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        p[t] = fmaf(__uint_as_float(ww[j] << 16), w[q * 8 + 2 * j], p[t]);
                        p[t] = fmaf(__uint_as_float(ww[j] & 0xFFFF0000u), w[q * 8 + 2 * j + 1], p[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kSmallTT; ++t) ps[(grp * kSmallTT + t) * (kSmallMaxC + 4) + c] = p[t];
        }
        __syncthreads();
        if (e < E && c < nt) {
            const float4 *pp = reinterpret_cast<const float4 *>(ps + (grp * kSmallTT + c) * (kSmallMaxC + 4));
            float acc = 0.0f;
            for (int c4 = 0; c4 < C / 4; ++c4) {
                const float4 v = pp[c4];
                acc = __fadd_rn(acc, v.x);
                acc = __fadd_rn(acc, v.y);
                acc = __fadd_rn(acc, v.z);
                acc = __fadd_rn(acc, v.w);
            }
            for (int cc = (C / 4) * 4; cc < C; ++cc) acc = __fadd_rn(acc, ps[(grp * kSmallTT + c) * (kSmallMaxC + 4) + cc]);
            logits[static_cast<int64_t>(t0 + c) * E + e] = __fadd_rn(acc, bias ? bias[e] : 0.0f);
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
constexpr int kRouterLogitsSmem = 2 * kHalf * (kXsStride + kWsStride) * 4;

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
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wr,
    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ logits, ZeroRanges zr) {
    zero_ranges(zr);
    extern __shared__ __align__(16) float rl_smem[];
    float *xs = rl_smem;                              // [2][kHalf][kXsStride]
    float *ws = rl_smem + 2 * kHalf * kXsStride;      // [2][kHalf][kWsStride]
    const int tid = threadIdx.x;
    const int ty = tid >> 3, tx = tid & 7;
    const int t_base = blockIdx.x * kRT, e_base = blockIdx.y * kRE;
    float acc[8][8];
    uint64_t p[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
    uint4 xr[4];
    float4 wr[4];
    auto load = [&](int h) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = tid + 128 * j;            // x: 128 tokens x 4 uint4
            const int t = i >> 2, q = i & 3;
            xr[j] = t_base + t < T ? __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t_base + t) * d + h * kHalf + q * 8))
                                   : make_uint4(0, 0, 0, 0);
            const int e = i >> 3, qw = i & 7;       // W: 64 experts x 8 float4
            wr[j] = e_base + e < E ? __ldg(reinterpret_cast<const float4 *>(Wr + static_cast<int64_t>(e_base + e) * d + h * kHalf + qw * 4))
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
            const int e = i >> 3, qw = i & 7;
            W[(qw * 4) * kWsStride + e] = wr[j].x;
            W[(qw * 4 + 1) * kWsStride + e] = wr[j].y;
            W[(qw * 4 + 2) * kWsStride + e] = wr[j].z;
            W[(qw * 4 + 3) * kWsStride + e] = wr[j].w;
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
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float lo, hi;
                    unpack2(p[a][q], lo, hi);
                    acc[a][2 * q] = __fadd_rn(acc[a][2 * q], lo);
                    acc[a][2 * q + 1] = __fadd_rn(acc[a][2 * q + 1], hi);
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

// One block of 128 threads per token: select the top-k from logits[T][E] (each thread holds
// E/128 logits; every round is a block-wide argmax by (logit desc, index asc)), softmax over
// the selected logits, write idx / w in ascending expert id, count tokens per expert.
constexpr int kTopkThreads = 128;
constexpr int kMaxEPerThread = 8;   // E <= 1024
__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(
    const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ idx_out,
    float *__restrict__ w_out, int32_t *__restrict__ counts) {
    __shared__ float cand_v[2][kTopkThreads / 32];
    __shared__ int cand_i[2][kTopkThreads / 32];
    __shared__ float sel_v[32];
    __shared__ int sel_i[32];
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float v[kMaxEPerThread];
#pragma unroll
    for (int j = 0; j < kMaxEPerThread; ++j) {
        const int e = tid + kTopkThreads * j;
        v[j] = e < E ? __ldg(logits + static_cast<int64_t>(t) * E + e) : -INFINITY;
    }
    uint32_t taken = 0u;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kMaxEPerThread; ++j) {
            const int e = tid + kTopkThreads * j;
            if (e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < bi))) { bv = v[j]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { cand_v[r & 1][warp] = bv; cand_i[r & 1][warp] = bi; }
        __syncthreads();
        bv = cand_v[r & 1][0];
        bi = cand_i[r & 1][0];
#pragma unroll
        for (int q = 1; q < kTopkThreads / 32; ++q) {
            const float ov = cand_v[r & 1][q];
            const int oi = cand_i[r & 1][q];
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (bi % kTopkThreads == tid) taken |= 1u << (bi / kTopkThreads);
        if (tid == 0) { sel_v[r] = bv; sel_i[r] = bi; }
    }
    __syncthreads();
    if (warp != 0) return;
    const int my_idx = lane < k ? sel_i[lane] : 0x7fffffff;
    const float my_val = lane < k ? sel_v[lane] : -INFINITY;
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
        if (counts) atomicAdd(counts + my_idx, 1);
    }
}

}  // namespace lmoe
