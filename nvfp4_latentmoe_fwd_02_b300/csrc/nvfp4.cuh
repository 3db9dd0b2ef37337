// nvfp4.cuh -- NVFP4 quantization on the device.
//
// Format (shengxinai.com Nemotron 3 blog, section 3.1.1 "NVFP4 格式解析"): E2M1 elements,
// one E4M3 block scale per 16 contiguous contraction-axis elements, plus one FP32 tensor
// scale.  The arithmetic (IEEE fp32, round-to-nearest-even, every product written as an
// explicit __fmul_rn so nothing is contracted):
//   amax_t == 0 -> codes 0, scales 0, tensor scale 1
//   s_enc = 2688 / amax_t, s_dec = amax_t / 2688, s_enc6 = s_enc / 6
//   per block:  sf  = e4m3_satfinite(amax_b * s_enc6)
//               bd  = value(sf) * s_dec;  rcp = bd > 0 ? 1/bd : 0
//               q_i = e2m1_satfinite(x_i * rcp)        (sign kept, so a flushed block is +-0)
// The conversions are the hardware cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32 instructions.
#pragma once
#include "common.cuh"

namespace lmoe {

constexpr float kNvfp4S = 2688.0f;   // 448 (E4M3 max) * 6 (E2M1 max)

struct QScale {
    float s_enc6;   // block-scale encode factor (s_enc / 6)
    float s_dec;    // FP32 tensor (decode) scale
    int zero;       // amax_t == 0: everything quantizes to 0
};

__host__ __device__ inline QScale qscale_from_amax(float amax) {
    QScale q;
    if (amax == 0.0f) {
        q.s_enc6 = 0.0f; q.s_dec = 1.0f; q.zero = 1;
        return q;
    }
#ifdef __CUDA_ARCH__
    float s_enc = __fdiv_rn(kNvfp4S, amax);
    q.s_dec = __fdiv_rn(amax, kNvfp4S);
    q.s_enc6 = __fdiv_rn(s_enc, 6.0f);
#else
    volatile float s_enc = kNvfp4S / amax;   // host: IEEE fp32 division
    q.s_dec = amax / kNvfp4S;
    q.s_enc6 = s_enc / 6.0f;
#endif
    q.zero = 0;
    return q;
}

__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(code)));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}
// Two fp32 values -> one byte of E2M1 codes, `lo` in the low nibble.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t; }"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}

// Quantize one 16-element block held in registers.  Returns the E4M3 scale byte; the 16
// codes are returned packed little-endian in two 32-bit words (element 0 = lowest nibble).
__device__ __forceinline__ uint32_t quant_block16(const float (&x)[16], const QScale &q,
                                                  uint32_t &lo, uint32_t &hi) {
    if (q.zero) { lo = hi = 0u; return 0u; }
    float amax_b = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(x[i]));
    const uint32_t sf = f32_to_e4m3_satfinite(__fmul_rn(amax_b, q.s_enc6));
    const float bd = __fmul_rn(e4m3_to_f32(sf), q.s_dec);
    const float rcp = bd > 0.0f ? __frcp_rn(bd) : 0.0f;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = f32x2_to_e2m1x2(__fmul_rn(x[2 * i], rcp), __fmul_rn(x[2 * i + 1], rcp));
        w[i >> 2] |= b << (8 * (i & 3));
    }
    lo = w[0]; hi = w[1];
    return sf;
}

// quant_block16 with the reciprocal looked up: rcp_of[sf] holds the rcp that quant_block16
// derives from the scale byte sf (the same fp32 operations, done once per byte value), so the
// codes are identical.  The block maximum is taken as a tree (max is exact in any order).
__device__ __forceinline__ uint32_t quant_block16_lut(const float (&x)[16], const QScale &q,
                                                      const float *rcp_of, uint32_t &lo, uint32_t &hi) {
    if (q.zero) { lo = hi = 0u; return 0u; }
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(x[2 * i]), fabsf(x[2 * i + 1]));
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], m[i + 4]);
    const float amax_b = fmaxf(fmaxf(m[0], m[2]), fmaxf(m[1], m[3]));
    const uint32_t sf = f32_to_e4m3_satfinite(__fmul_rn(amax_b, q.s_enc6));
    const float rcp = rcp_of[sf];
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = f32x2_to_e2m1x2(__fmul_rn(x[2 * i], rcp), __fmul_rn(x[2 * i + 1], rcp));
    lo = (b[0] | (b[1] << 8)) | ((b[2] << 16) | (b[3] << 24));
    hi = (b[4] | (b[5] << 8)) | ((b[6] << 16) | (b[7] << 24));
    return sf;
}
// The table of quant_block16_lut for quantizer q (rcp_of[0..255]; all zero when q.zero).
__device__ __forceinline__ float quant_rcp_entry(const QScale &q, uint32_t sf) {
    if (q.zero) return 0.0f;
    const float bd = __fmul_rn(e4m3_to_f32(sf), q.s_dec);
    return bd > 0.0f ? __frcp_rn(bd) : 0.0f;
}

// 16 codes of a block whose scale is already decided (rcp = 1 / (value(sf) * s_dec), or 0).
__device__ __forceinline__ void block_codes16(const float (&x)[16], float rcp, uint32_t &lo, uint32_t &hi) {
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = f32x2_to_e2m1x2(__fmul_rn(x[2 * i], rcp), __fmul_rn(x[2 * i + 1], rcp));
        w[i >> 2] |= b << (8 * (i & 3));
    }
    lo = w[0]; hi = w[1];
}

// Byte offset of the scale of (row r, 16-block b) in the tensor-core scale-factor layout:
// atoms of 128 rows x 4 blocks (512 B), ordered [r / 128][b / 4]; inside an atom row r
// sits at (r % 32) * 16 + ((r / 32) % 4) * 4 and block b at + (b % 4).
__host__ __device__ __forceinline__ size_t sf_atom_offset(int64_t r, int64_t b, int64_t K64) {
    return (static_cast<size_t>(r >> 7) * K64 + (b >> 2)) * 512 + (r & 31) * 16 +
           ((r >> 5) & 3) * 4 + (b & 3);
}

// ------------------------------------------------------------------------------------
// kernels
// ------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void load16(const T *p, float (&x)[16]);
template <>
__device__ __forceinline__ void load16<float>(const float *p, float (&x)[16]) {
    const float4 *v = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 f = __ldg(v + i);
        x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
    }
}
template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16 *p, float (&x)[16]) {
    const uint4 *v = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint4 u = __ldg(v + i);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
            x[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}

// max |x| over n elements -> atomicMax on the fp32 bit pattern (order-preserving for >= 0).
template <typename T>
__global__ void amax_kernel(const T *__restrict__ src, int64_t n, unsigned *__restrict__ out) {
    float m = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float v;
        if constexpr (sizeof(T) == 4) v = src[i];
        else v = __bfloat162float(src[i]);
        m = fmaxf(m, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));
}

// Per-segment amax: segment s = [s * seg_len, (s+1) * seg_len), grid.y = segment.
__global__ void amax_segments_kernel(const __nv_bfloat16 *__restrict__ src, int64_t seg_len,
                                     unsigned *__restrict__ out) {
    const __nv_bfloat16 *p = src + blockIdx.y * seg_len;
    float m = 0.0f;
    for (int64_t i = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 8; i < seg_len;
         i += (int64_t)gridDim.x * blockDim.x * 8) {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(p + i));
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(out + blockIdx.y, __float_as_uint(m));
}

// Row-major quantization: one thread per 16-block.  The tensor amax is either the value
// `amax` (>= 0) or, if amax < 0, the bit pattern at amax_bits (written by amax_kernel).
template <typename T>
__global__ void quantize_rows_kernel(const T *__restrict__ src, int64_t rows, int64_t K,
                                     float amax, const unsigned *__restrict__ amax_bits,
                                     uint8_t *__restrict__ codes, uint8_t *__restrict__ sf) {
    const float a = amax >= 0.0f ? amax : __uint_as_float(*amax_bits);
    const QScale q = qscale_from_amax(a);
    const int64_t nb = K / 16;
    const int64_t total = rows * nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float x[16];
        load16<T>(src + i * 16, x);
        uint32_t lo, hi;
        const uint32_t s = quant_block16(x, q, lo, hi);
        reinterpret_cast<uint2 *>(codes)[i] = make_uint2(lo, hi);
        sf[i] = static_cast<uint8_t>(s);
    }
}

// tensor_scale = amax / 2688 (1 when amax == 0), amax read from its bit pattern.
__global__ void tensor_scale_kernel(const unsigned *__restrict__ amax_bits, int n,
                                    float *__restrict__ out) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = qscale_from_amax(__uint_as_float(amax_bits[i])).s_dec;
}

// Expert weights: src [E][N][K] bf16 -> codes [E][N][K/2] and scales in the tensor-core
// atom layout [E][ceil(N/128)][K/64][512], one FP32 tensor scale per expert (amax_bits[e]).
__global__ void quantize_experts_kernel(const __nv_bfloat16 *__restrict__ src, int E, int N,
                                        int K, const unsigned *__restrict__ amax_bits,
                                        uint8_t *__restrict__ codes,
                                        uint8_t *__restrict__ sf_atoms) {
    const int64_t nb = K / 16;
    const int64_t per_e = static_cast<int64_t>(N) * nb;
    const int64_t total = per_e * E;
    const int64_t K64 = K / 64;
    const int64_t NB = (N + 127) / 128;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = i / per_e;
        const int64_t rem = i - e * per_e;
        const int64_t r = rem / nb, b = rem - r * nb;
        const QScale q = qscale_from_amax(__uint_as_float(amax_bits[e]));
        float x[16];
        load16<__nv_bfloat16>(src + i * 16, x);
        uint32_t lo, hi;
        const uint32_t s = quant_block16(x, q, lo, hi);
        reinterpret_cast<uint2 *>(codes)[i] = make_uint2(lo, hi);
        sf_atoms[static_cast<size_t>(e) * NB * K64 * 512 + sf_atom_offset(r, b, K64)] =
            static_cast<uint8_t>(s);
    }
}

// 2-D weight blocks (NVIDIA AI releases Nemotron 3 Ultra, architecture paragraph: weights
// quantized in two-dimensional blocks; 16 x 16 here): one E4M3 scale per 16 rows x 16
// contraction elements from the block's amax, the 1-D arithmetic otherwise.  One thread per
// block; it writes the scale for each of the 16 rows, so the GEMMs read the usual per-row
// layout.  quantize_block2d: rows [r0, r0 + 16) x elements [16 b, 16 b + 16) of src [.][K].
template <typename T, typename SfAt>
__device__ __forceinline__ void quantize_block2d(const T *src, int64_t K, int64_t r0, int64_t b,
                                                 const QScale &q, uint8_t *codes, SfAt sf_at) {
    float amax_b = 0.0f;
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
        float x[16];
        load16<T>(src + (r0 + r) * K + 16 * b, x);
#pragma unroll
        for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(x[i]));
    }
    uint32_t s = 0u;
    float rcp = 0.0f;
    if (!q.zero) {
        s = f32_to_e4m3_satfinite(__fmul_rn(amax_b, q.s_enc6));
        const float bd = __fmul_rn(e4m3_to_f32(s), q.s_dec);
        rcp = bd > 0.0f ? __frcp_rn(bd) : 0.0f;
    }
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
        float x[16];
        load16<T>(src + (r0 + r) * K + 16 * b, x);
        uint32_t lo = 0u, hi = 0u;
        if (!q.zero) block_codes16(x, rcp, lo, hi);
        reinterpret_cast<uint2 *>(codes + (r0 + r) * (K / 2))[b] = make_uint2(lo, hi);
        *sf_at(r0 + r, b) = static_cast<uint8_t>(s);
    }
}

// Row-major 2-D quantization of src [rows][K] (rows % 16 == 0); sf [rows][K/16] per row.
template <typename T>
__global__ void quantize_rows_2d_kernel(const T *__restrict__ src, int64_t rows, int64_t K, float amax,
                                        const unsigned *__restrict__ amax_bits, uint8_t *__restrict__ codes,
                                        uint8_t *__restrict__ sf) {
    const float a = amax >= 0.0f ? amax : __uint_as_float(*amax_bits);
    const QScale q = qscale_from_amax(a);
    const int64_t nb = K / 16;
    const int64_t total = (rows / 16) * nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = i / nb, b = i - g * nb;
        quantize_block2d<T>(src, K, g * 16, b, q, codes,
                            [&](int64_t r, int64_t bb) { return sf + r * nb + bb; });
    }
}

// Expert weights with 2-D blocks: src [E][N][K] bf16 -> codes [E][N][K/2] and the scale atoms
// [E][ceil(N/128)][K/64][512] (N % 16 == 0), one FP32 tensor scale per expert.
__global__ void quantize_experts_2d_kernel(const __nv_bfloat16 *__restrict__ src, int E, int N, int K,
                                           const unsigned *__restrict__ amax_bits,
                                           uint8_t *__restrict__ codes, uint8_t *__restrict__ sf_atoms) {
    const int64_t nb = K / 16;
    const int64_t per_e = static_cast<int64_t>(N / 16) * nb;
    const int64_t total = per_e * E;
    const int64_t K64 = K / 64;
    const int64_t NB = (N + 127) / 128;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = i / per_e;
        const int64_t rem = i - e * per_e;
        const int64_t g = rem / nb, b = rem - g * nb;
        const QScale q = qscale_from_amax(__uint_as_float(amax_bits[e]));
        uint8_t *atoms = sf_atoms + static_cast<size_t>(e) * NB * K64 * 512;
        quantize_block2d<__nv_bfloat16>(src + static_cast<int64_t>(e) * N * K, K, g * 16, b, q,
                                        codes + static_cast<int64_t>(e) * N * (K / 2),
                                        [&](int64_t r, int64_t bb) { return atoms + sf_atom_offset(r, bb, K64); });
    }
}

// Expert weight codes in tile order: for expert e, 128-row block nb and 128-byte column block
// kt, the 128 x 128-byte box that one TMA copy of the GEMMs moves is contiguous (16 KB), so
// the weight stream reads whole 16 KB runs of HBM instead of 128-byte pieces 1 KB apart.
// Byte (e, r, c) of the row-major [E][N][K/2] codes sits at
//   (((e * NB + r / 128) * KT + c / 128) * 128 + r % 128) * 128 + c % 128,
// NB = ceil(N / 128), KT = ceil(K / 256); bytes past N rows or K/2 columns stay 0.
__host__ __device__ __forceinline__ int64_t tiled_code_offset(int64_t e, int64_t r, int64_t c, int64_t NB,
                                                              int64_t KT) {
    return (((e * NB + (r >> 7)) * KT + (c >> 7)) * 128 + (r & 127)) * 128 + (c & 127);
}
__host__ __device__ __forceinline__ size_t tiled_codes_bytes(int64_t E, int64_t N, int64_t K) {
    return static_cast<size_t>(E * ((N + 127) / 128) * ((K + 255) / 256)) * 16384;
}
// row-major codes [E][N][K/2] -> tile order (8-byte pieces: one 16-element block each)
__global__ void tile_codes_kernel(const uint8_t *__restrict__ src, int E, int N, int K,
                                  uint8_t *__restrict__ dst) {
    const int64_t NB = (N + 127) / 128, KT = (K + 255) / 256;
    const int64_t pr = K / 16;                                   // 8-byte pieces per row
    const int64_t total = static_cast<int64_t>(E) * N * pr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / pr, p = i - row * pr;           // row over E * N
        const int64_t e = row / N, r = row - e * N;
        *reinterpret_cast<uint2 *>(dst + tiled_code_offset(e, r, 8 * p, NB, KT)) =
            reinterpret_cast<const uint2 *>(src)[i];
    }
}
// One expert's codes from tile order back to row-major [N][K/2].
__global__ void untile_codes_kernel(const uint8_t *__restrict__ tiled, int e, int N, int K,
                                    uint8_t *__restrict__ out) {
    const int64_t NB = (N + 127) / 128, KT = (K + 255) / 256;
    const int64_t pr = K / 16;
    const int64_t total = static_cast<int64_t>(N) * pr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / pr, p = i - r * pr;
        reinterpret_cast<uint2 *>(out)[i] =
            *reinterpret_cast<const uint2 *>(tiled + tiled_code_offset(e, r, 8 * p, NB, KT));
    }
}

// Atom layout -> row-major [N][K/16] for one matrix (used to hand scales back to callers).
__global__ void sf_atoms_to_rows_kernel(const uint8_t *__restrict__ atoms, int N, int K,
                                        uint8_t *__restrict__ out) {
    const int64_t nb = K / 16;
    const int64_t total = static_cast<int64_t>(N) * nb;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / nb, b = i - r * nb;
        out[i] = atoms[sf_atom_offset(r, b, K / 64)];
    }
}

}  // namespace lmoe
