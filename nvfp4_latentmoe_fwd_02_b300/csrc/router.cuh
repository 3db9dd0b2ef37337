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

// Small T: logits[t][e] with the chunk partials reduced through shared memory.  Block: two
// experts x 128 threads; thread c computes the partial p_c (one 64-element fmaf chain) of its
// chunk(s) for a tile of 8 tokens, then one thread per token adds the chunk partials of its
// expert left to right and the bias.  grid = ceil(E / 2).
constexpr int kSmallTT = 8;
constexpr int kSmallMaxC = 256;   // d <= 16384
__global__ void __launch_bounds__(256) router_small_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wr,
    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ logits) {
    __shared__ float ps[2][kSmallTT][kSmallMaxC + 1];
    const int grp = threadIdx.x >> 7, tc = threadIdx.x & 127;
    const int e = blockIdx.x * 2 + grp;
    const int C = d / kChunk;
    for (int t0 = 0; t0 < T; t0 += kSmallTT) {
        const int nt = min(kSmallTT, T - t0);
        if (e < E) {
            for (int c = tc; c < C; c += 128) {
                float w[kChunk];
                const float4 *src = reinterpret_cast<const float4 *>(Wr + static_cast<int64_t>(e) * d + c * kChunk);
#pragma unroll
                for (int i = 0; i < kChunk / 4; ++i) {
                    const float4 f = __ldg(src + i);
                    w[4 * i] = f.x; w[4 * i + 1] = f.y; w[4 * i + 2] = f.z; w[4 * i + 3] = f.w;
                }
                float p[kSmallTT];
#pragma unroll
                for (int t = 0; t < kSmallTT; ++t) p[t] = 0.0f;
#pragma unroll
                for (int q = 0; q < kChunk / 8; ++q) {
#pragma unroll
                    for (int t = 0; t < kSmallTT; ++t) {
                        if (t < nt) {
                            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(
                                x + static_cast<int64_t>(t0 + t) * d + c * kChunk + q * 8));
                            const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                p[t] = fmaf(__uint_as_float(ww[j] << 16), w[q * 8 + 2 * j], p[t]);
                                p[t] = fmaf(__uint_as_float(ww[j] & 0xFFFF0000u), w[q * 8 + 2 * j + 1], p[t]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kSmallTT; ++t) ps[grp][t][c] = p[t];
            }
        }
        __syncthreads();
        if (e < E && tc < nt) {
            float acc = 0.0f;
            for (int c = 0; c < C; ++c) acc = __fadd_rn(acc, ps[grp][tc][c]);
            logits[static_cast<int64_t>(t0 + tc) * E + e] = __fadd_rn(acc, bias ? bias[e] : 0.0f);
        }
        __syncthreads();
    }
}

// logits[t][e] (bias added).  Tile: 128 tokens x 64 experts per block of 128 threads, each
// thread 8 tokens x 8 experts.  Each 64-element chunk is staged through shared memory in two
// halves of 32; the per-chunk fma chain runs across both halves before it is added to acc.
constexpr int kRT = 128, kRE = 64, kHalf = 32;
__global__ void __launch_bounds__(128) router_logits_kernel(
    const __nv_bfloat16 *__restrict__ x, const float *__restrict__ Wr,
    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ logits) {
    __shared__ __align__(16) float xs[kHalf][kRT + 4];
    __shared__ __align__(16) float ws[kHalf][kRE + 4];
    const int tid = threadIdx.x;
    const int ty = tid >> 3, tx = tid & 7;
    const int t_base = blockIdx.x * kRT, e_base = blockIdx.y * kRE;
    float acc[8][8], p[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
    const int H = d / kHalf;   // half-chunks
    for (int h = 0; h < H; ++h) {
        __syncthreads();
        // x tile: 128 tokens x 32 bf16 -> xs[i][t]
        for (int i = tid; i < kRT * (kHalf / 8); i += blockDim.x) {
            const int t = i >> 2, q = i & 3;
            uint4 u = make_uint4(0, 0, 0, 0);
            if (t_base + t < T)
                u = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t_base + t) * d +
                                                          h * kHalf + q * 8));
            const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xs[q * 8 + 2 * j][t] = __uint_as_float(ww[j] << 16);
                xs[q * 8 + 2 * j + 1][t] = __uint_as_float(ww[j] & 0xFFFF0000u);
            }
        }
        // W tile: 64 experts x 32 fp32 -> ws[i][e]
        for (int i = tid; i < kRE * (kHalf / 4); i += blockDim.x) {
            const int e = i >> 3, q = i & 7;
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e_base + e < E)
                f = __ldg(reinterpret_cast<const float4 *>(Wr + static_cast<int64_t>(e_base + e) * d +
                                                           h * kHalf + q * 4));
            ws[q * 4][e] = f.x; ws[q * 4 + 1][e] = f.y; ws[q * 4 + 2][e] = f.z; ws[q * 4 + 3][e] = f.w;
        }
        __syncthreads();
        if ((h & 1) == 0) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) p[a][b] = 0.0f;
        }
#pragma unroll 4
        for (int i = 0; i < kHalf; ++i) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&xs[i][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&xs[i][ty * 8 + 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&ws[i][tx * 8]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&ws[i][tx * 8 + 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) p[a][b] = fmaf(av[a], bv[b], p[a][b]);
        }
        if (h & 1) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = __fadd_rn(acc[a][b], p[a][b]);
        }
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

// One warp per token: select top-k from logits[T][E], softmax, write idx / w in ascending
// expert id, count tokens per expert.
constexpr int kMaxEPerLane = 32;   // E <= 1024
__global__ void __launch_bounds__(256) router_topk_kernel(
    const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ idx_out,
    float *__restrict__ w_out,
    int32_t *__restrict__ counts) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int npl = (E + 31) / 32;
    float v[kMaxEPerLane];
#pragma unroll
    for (int j = 0; j < kMaxEPerLane; ++j) {
        v[j] = -INFINITY;
        const int e = lane + 32 * j;
        if (j < npl && e < E) v[j] = logits[static_cast<int64_t>(t) * E + e];
    }
    uint32_t taken = 0u;
    int my_idx = 0;
    float my_val = 0.0f;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < kMaxEPerLane; ++j) {
            const int e = lane + 32 * j;
            if (j < npl && e < E && !((taken >> j) & 1u)) {
                if (v[j] > bv || (v[j] == bv && e < bi)) { bv = v[j]; bi = e; }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == r) { my_idx = bi; my_val = bv; }
    }
    // rank of each selected expert among the selected (ascending id)
    int rank = 0;
    for (int r = 0; r < k; ++r) {
        const int oi = __shfl_sync(0xffffffffu, my_idx, r);
        rank += (oi < my_idx) ? 1 : 0;
    }
    float m = lane < k ? my_val : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float ex = lane < k ? expf(my_val - m) : 0.0f;
    float s = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane < k) {
        idx_out[static_cast<int64_t>(t) * k + rank] = my_idx;
        w_out[static_cast<int64_t>(t) * k + rank] = __fdiv_rn(ex, s);
        if (counts) atomicAdd(counts + my_idx, 1);
    }
}

}  // namespace lmoe
