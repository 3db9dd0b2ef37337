// moe.cuh -- per-expert segments, gather of the latent tokens, and the small element-wise
// passes around the GEMMs (zeroing, z finalize + quantize, combine finalize, y finalize).
//
// Segments: expert e owns rows [seg_start[e], seg_start[e] + counts[e]) of the permuted
// buffers; each segment is padded to a multiple of 128 rows (one tensor-core M tile) so that
// every tile's block scales sit in whole 128-row scale atoms.  row_slot[row] is the routing
// slot (token * k + j) of a row, -1 for padding.  mt_start[e] is the prefix sum of M tiles.
// Rows inside a segment are in atomic-arrival order (the grouping, not the order, is fixed).
#pragma once
#include "common.cuh"
#include "nvfp4.cuh"

namespace lmoe {

// One block per expert e: its segment start is the sum of the padded counts of experts < e
// (a block reduction over the histogram); the block also marks the segment's padding rows.
// Block E - 1 writes the totals.  grid = E, block = 128.
__global__ void __launch_bounds__(128) segments_kernel(
    const int32_t *__restrict__ counts, int E, int32_t *__restrict__ seg_start,
    int32_t *__restrict__ mt_start, int32_t *__restrict__ fill, int32_t *__restrict__ row_slot,
    int32_t *__restrict__ nrows) {
    __shared__ int part[4];
    const int e = blockIdx.x;
    int sum = 0;
    for (int i = threadIdx.x; i < e; i += blockDim.x) sum += (__ldg(counts + i) + 127) & ~127;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sum;
    __syncthreads();
    const int start = part[0] + part[1] + part[2] + part[3];
    const int cnt = __ldg(counts + e);
    const int padded = (cnt + 127) & ~127;
    if (threadIdx.x == 0) {
        seg_start[e] = start;
        mt_start[e] = start >> 7;
        fill[e] = 0;
        if (e == E - 1) {
            seg_start[E] = start + padded;
            mt_start[E] = (start + padded) >> 7;
            *nrows = start + padded;
        }
    }
    for (int r = start + cnt + threadIdx.x; r < start + padded; r += blockDim.x) row_slot[r] = -1;
}

// One warp per routing slot: claim a row of the expert's segment and copy the token's
// quantized latent vector (codes and scales) into it.  l: latent width.
__global__ void __launch_bounds__(256) scatter_kernel(
    const int32_t *__restrict__ idx, int64_t nslots, const int32_t *__restrict__ seg_start,
    int32_t *__restrict__ fill, int32_t *__restrict__ row_slot, int k, int l,
    const uint8_t *__restrict__ zq_codes, const uint8_t *__restrict__ zq_sf,
    uint8_t *__restrict__ a_codes, uint8_t *__restrict__ a_sf) {
    const int lane = threadIdx.x & 31;
    const int64_t s = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    if (s >= nslots) return;
    int pos = 0;
    if (lane == 0) {
        const int e = idx[s];
        pos = seg_start[e] + atomicAdd(fill + e, 1);
        row_slot[pos] = static_cast<int32_t>(s);
    }
    pos = __shfl_sync(0xffffffffu, pos, 0);
    const int64_t t = s / k;
    const int row_bytes = l / 2;
    const uint4 *src = reinterpret_cast<const uint4 *>(zq_codes + t * row_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(a_codes + static_cast<int64_t>(pos) * row_bytes);
    for (int i = lane; i < row_bytes / 16; i += 32) dst[i] = __ldg(src + i);
    const int K64 = l / 64;
    const uint32_t *ssrc = reinterpret_cast<const uint32_t *>(zq_sf + t * (l / 16));
    for (int kb = lane; kb < K64; kb += 32)
        *reinterpret_cast<uint32_t *>(a_sf + sf_atom_offset(pos, 4 * kb, K64)) = __ldg(ssrc + kb);
}

// zacc [T][l] fp32 -> z = bf16(zacc) -> zq (row-major codes and scales); z kept if z_out.
__global__ void z_finalize_kernel(const float *__restrict__ zacc, int64_t T, int l, QScale q,
                                  uint8_t *__restrict__ codes, uint8_t *__restrict__ sf,
                                  __nv_bfloat16 *__restrict__ z_out) {
    const int64_t total = T * (l / 16);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float x[16];
        load16<float>(zacc + i * 16, x);
        uint32_t zb[8];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = bf16_bits_to_f32(f32_to_bf16_bits(x[j]));
#pragma unroll
        for (int j = 0; j < 8; ++j) zb[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
        if (z_out) {
            uint4 *zo = reinterpret_cast<uint4 *>(z_out + i * 16);
            zo[0] = make_uint4(zb[0], zb[1], zb[2], zb[3]);
            zo[1] = make_uint4(zb[4], zb[5], zb[6], zb[7]);
        }
        uint32_t lo, hi;
        const uint32_t s = quant_block16(x, q, lo, hi);
        reinterpret_cast<uint2 *>(codes)[i] = make_uint2(lo, hi);
        sf[i] = static_cast<uint8_t>(s);
    }
}

// acc [n] fp32 -> out [n] bf16 (n % 8 == 0).
__global__ void f32_to_bf16_kernel(const float *__restrict__ acc, int64_t n,
                                   __nv_bfloat16 *__restrict__ out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n / 8;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i + 1);
        reinterpret_cast<uint4 *>(out)[i] =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                       pack_bf16x2(b.z, b.w));
    }
}

}  // namespace lmoe
