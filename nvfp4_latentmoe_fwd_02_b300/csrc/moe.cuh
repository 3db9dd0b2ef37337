// moe.cuh -- per-expert segments, gather of the latent tokens, and the small element-wise
// passes around the GEMMs (zeroing, z finalize + quantize, combine finalize, y finalize).
//
// Segments (laid out by the routing kernels' last warp, router.cuh): expert e owns rows
// [seg_start[e], seg_start[e] + counts[e]) of the permuted buffers, padded to a multiple of
// 128 rows.  row_slot[row] is the routing slot (token * k + j) of a real row; padding rows are
// never written or read.  A slot's row inside its segment is the histogram's old value when
// the routing kernel counted it (atomic-arrival order: the grouping, not the order inside a
// segment, is fixed).
#pragma once
#include "common.cuh"
#include "nvfp4.cuh"

namespace lmoe {

// Where the k copies of token t's quantized latent vector go: segment row of each slot.
__device__ __forceinline__ int slot_row(const int32_t *idx, const int32_t *slot_off,
                                        const int32_t *seg_start, int64_t slot) {
    return __ldg(seg_start + __ldg(idx + slot)) + __ldg(slot_off + slot);
}

// Split-K finalize of the down-projection, one thread per (token, 16-block): z = bf16(zacc),
// zq = NVFP4(z) into the row-major buffers and into the token's k segment rows (codes and
// scale atoms; or, for W4A16, the bf16 z itself); row_slot records the slot of each row.  A block covers whole tokens
// (blockDim / (l/16) of them) and one group of their slots (blockIdx.y of gridDim.y groups: at
// small T the copies are spread over more SMs, so the stores drain sooner); the group's segment
// rows are looked up once into shared memory.  The row-major zq is written by group 0.
__global__ void __launch_bounds__(256) z_finalize_kernel(
    const float *__restrict__ zacc, int64_t T, int l, QScale q, uint8_t *__restrict__ codes,
    uint8_t *__restrict__ sf, __nv_bfloat16 *__restrict__ z_out, const int32_t *__restrict__ idx,
    const int32_t *__restrict__ slot_off, const int32_t *__restrict__ seg_start, int k,
    int32_t *__restrict__ row_slot, uint8_t *__restrict__ a_codes, uint8_t *__restrict__ a_sf,
    __nv_bfloat16 *__restrict__ a_bf16) {
    __shared__ int rows_s[256];   // [tokens per block][slots of the group]
    pdl_wait();
    pdl_trigger();
    const int nb = l / 16, K64 = l / 64;
    const int tpb = blockDim.x / nb;                   // tokens per block (>= 1)
    const int64_t t_first = static_cast<int64_t>(blockIdx.x) * tpb;
    const int spg = (k + gridDim.y - 1) / gridDim.y;   // slots per group
    const int j0 = blockIdx.y * spg, nj = max(0, min(k, j0 + spg) - j0);
    for (int i = threadIdx.x; i < tpb * nj; i += blockDim.x) {
        const int64_t slot = (t_first + i / nj) * k + j0 + i % nj;
        if (t_first + i / nj < T) {
            const int row = slot_row(idx, slot_off, seg_start, slot);
            rows_s[i] = row;
            row_slot[row] = static_cast<int32_t>(slot);
        }
    }
    __syncthreads();
    const int tl = threadIdx.x / nb, b = threadIdx.x - tl * nb;
    const int64_t t = t_first + tl;
    if (tl >= tpb || t >= T) return;
    const int64_t i = t * nb + b;
    float x[16];
    load16<float>(zacc + i * 16, x);
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = bf16_bits_to_f32(f32_to_bf16_bits(x[j]));
    uint32_t zb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) zb[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
    if (z_out && blockIdx.y == 0) {
        uint4 *zo = reinterpret_cast<uint4 *>(z_out + i * 16);
        zo[0] = make_uint4(zb[0], zb[1], zb[2], zb[3]);
        zo[1] = make_uint4(zb[4], zb[5], zb[6], zb[7]);
    }
    uint32_t lo, hi;
    const uint32_t s = quant_block16(x, q, lo, hi);
    if (blockIdx.y == 0) {
        reinterpret_cast<uint2 *>(codes)[i] = make_uint2(lo, hi);
        sf[i] = static_cast<uint8_t>(s);
    }
    for (int j = 0; j < nj; ++j) {
        const int row = rows_s[tl * nj + j];
        if (a_bf16) {       // W4A16: the bf16 z itself goes to the expert segments
            uint4 *o = reinterpret_cast<uint4 *>(a_bf16 + static_cast<int64_t>(row) * l + b * 16);
            o[0] = make_uint4(zb[0], zb[1], zb[2], zb[3]);
            o[1] = make_uint4(zb[4], zb[5], zb[6], zb[7]);
        } else {
            reinterpret_cast<uint2 *>(a_codes + static_cast<int64_t>(row) * (l / 2))[b] = make_uint2(lo, hi);
            a_sf[sf_atom_offset(row, b, K64)] = static_cast<uint8_t>(s);
        }
    }
}

// Copies of each token's quantized latent row into its k expert-segment rows (large T: the
// down-projection epilogue then only writes the row-major zq), one warp per token: the row is
// read once into registers (codes as 16-byte pieces, scales as 4-byte groups), then written to
// each of the token's k rows (codes as 16-byte stores, the scales into the scale atoms) with
// the slot into row_slot.  W4A16: the bf16 z row instead (a_bf16 set).  l <= 4096.
__global__ void __launch_bounds__(256) scatter_rows_kernel(
    const uint8_t *__restrict__ zq_codes, const uint8_t *__restrict__ zq_sf,
    const __nv_bfloat16 *__restrict__ z, const int32_t *__restrict__ idx,
    const int32_t *__restrict__ slot_off, const int32_t *__restrict__ seg_start, int64_t T, int k,
    int l, uint8_t *__restrict__ a_codes, uint8_t *__restrict__ a_sf, __nv_bfloat16 *__restrict__ a_bf16,
    int32_t *__restrict__ row_slot) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    // the token's k rows (k <= 32): lane j looks up slot j
    const int my_row = lane < k ? slot_row(idx, slot_off, seg_start, t * k + lane) : 0;
    if (lane < k) row_slot[my_row] = static_cast<int32_t>(t * k + lane);
    if (a_bf16) {
        const int n16 = l / 8;                             // uint4 per row
        uint4 v[16];
        const uint4 *src = reinterpret_cast<const uint4 *>(z + t * l);
#pragma unroll
        for (int q = 0; q < 16; ++q)
            if (q * 32 + lane < n16) v[q] = __ldg(src + q * 32 + lane);
        for (int j = 0; j < k; ++j) {
            const int row = __shfl_sync(0xffffffffu, my_row, j);
            uint4 *dst = reinterpret_cast<uint4 *>(a_bf16 + static_cast<int64_t>(row) * l);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                if (q * 32 + lane < n16) dst[q * 32 + lane] = v[q];
        }
        return;
    }
    const int n16 = l / 32;                                // uint4 of codes per row
    const int K64 = l / 64;                                // 4-byte scale groups per row
    uint4 cv[4];
    uint32_t sv[2];
    const uint4 *src = reinterpret_cast<const uint4 *>(zq_codes + t * (l / 2));
    const uint32_t *sf4 = reinterpret_cast<const uint32_t *>(zq_sf + t * (l / 16));
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q * 32 + lane < n16) cv[q] = __ldg(src + q * 32 + lane);
#pragma unroll
    for (int q = 0; q < 2; ++q)
        if (q * 32 + lane < K64) sv[q] = __ldg(sf4 + q * 32 + lane);
    for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xffffffffu, my_row, j);
        uint4 *dst = reinterpret_cast<uint4 *>(a_codes + static_cast<int64_t>(row) * (l / 2));
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q * 32 + lane < n16) dst[q * 32 + lane] = cv[q];
#pragma unroll
        for (int q = 0; q < 2; ++q)                        // scales of 16-blocks 4g..4g+3: atom g
            if (q * 32 + lane < K64)
                *reinterpret_cast<uint32_t *>(a_sf + sf_atom_offset(row, 4 * (q * 32 + lane), K64)) = sv[q];
    }
}

// Router weights [E][d] -> 32-expert panels [ceil(E/32)][d][32] (expert e of panel e / 32 at
// lane e % 32; the panels' unused lanes are left as they are, zero after the allocation's clear):
// one block of the small-T router reads a contiguous slab of one panel.
__global__ void router_panels_kernel(const float *__restrict__ in, int64_t E, int64_t d, float *__restrict__ out) {
    __shared__ float tile[32][33];
    const int64_t c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;   // d columns, expert rows (one panel)
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
        const int64_t r = r0 + j, c = c0 + threadIdx.x;
        if (r < E && c < d) tile[j][threadIdx.x] = in[r * d + c];
    }
    __syncthreads();
    for (int j = threadIdx.y; j < 32; j += blockDim.y) {
        const int64_t c = c0 + j, r = r0 + threadIdx.x;
        if (r < E && c < d) out[((r0 / 32) * d + c) * 32 + threadIdx.x] = tile[threadIdx.x][j];
    }
}

// out [n] bf16 = bf16(acc [n] fp32 (+ add [n] bf16, if given)) (n % 8 == 0).
__global__ void f32_to_bf16_kernel(const float *__restrict__ acc, int64_t n,
                                   __nv_bfloat16 *__restrict__ out,
                                   const __nv_bfloat16 *__restrict__ add) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n / 8;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i);
        float4 b = __ldg(reinterpret_cast<const float4 *>(acc) + 2 * i + 1);
        if (add) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(add) + i);
            a.x = __fadd_rn(a.x, __uint_as_float(u.x << 16)); a.y = __fadd_rn(a.y, __uint_as_float(u.x & 0xFFFF0000u));
            a.z = __fadd_rn(a.z, __uint_as_float(u.y << 16)); a.w = __fadd_rn(a.w, __uint_as_float(u.y & 0xFFFF0000u));
            b.x = __fadd_rn(b.x, __uint_as_float(u.z << 16)); b.y = __fadd_rn(b.y, __uint_as_float(u.z & 0xFFFF0000u));
            b.z = __fadd_rn(b.z, __uint_as_float(u.w << 16)); b.w = __fadd_rn(b.w, __uint_as_float(u.w & 0xFFFF0000u));
        }
        reinterpret_cast<uint4 *>(out)[i] =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                       pack_bf16x2(b.z, b.w));
    }
}

}  // namespace lmoe
