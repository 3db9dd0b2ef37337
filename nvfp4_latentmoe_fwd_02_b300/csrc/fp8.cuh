// fp8.cuh -- FP8 E4M3 with one FP32 per-tensor scale: the shared expert's format (NVIDIA AI
// releases Nemotron 3 Ultra, quantization paragraph: NVFP4 routed experts beside an FP8
// shared expert).
//
//   s_enc = 448 / amax, s_dec = amax / 448           (IEEE fp32 divisions)
//   code  = e4m3_satfinite(x * s_enc)                 (round to nearest even, +-448 at most)
//   amax == 0: every code is 0 and s_dec = 1
// The conversion is the hardware cvt.rn.satfinite.e4m3x2.f32 instruction.
#pragma once
#include "common.cuh"
#include "nvfp4.cuh"

namespace lmoe {

struct Fp8Scale {
    float s_enc, s_dec;
    bool zero;
};

__host__ __device__ __forceinline__ Fp8Scale fp8scale_from_amax(float amax) {
    Fp8Scale q;
    q.zero = !(amax > 0.0f);
    q.s_enc = q.zero ? 0.0f : 448.0f / amax;
    q.s_dec = q.zero ? 1.0f : amax / 448.0f;
    return q;
}

// Two values -> two E4M3 codes in one 16-bit word (a in the low byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// 16 values (already multiplied by s_enc) -> 16 codes packed little-endian in a uint4.
__device__ __forceinline__ uint4 e4m3x16(const float (&v)[16]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = f32x2_to_e4m3x2(v[4 * i], v[4 * i + 1]) | (f32x2_to_e4m3x2(v[4 * i + 2], v[4 * i + 3]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Per-tensor quantization of n elements (n % 16 == 0), one thread per 16 elements.  The
// tensor amax is the value `amax` (>= 0) or, if amax < 0, the fp32 bit pattern at amax_bits.
template <typename T>
__global__ void quantize_fp8_kernel(const T *__restrict__ src, int64_t n, float amax,
                                    const unsigned *__restrict__ amax_bits,
                                    uint8_t *__restrict__ codes) {
    pdl_wait();
    pdl_trigger();
    const float a = amax >= 0.0f ? amax : __uint_as_float(*amax_bits);
    const Fp8Scale q = fp8scale_from_amax(a);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n / 16;
         i += (int64_t)gridDim.x * blockDim.x) {
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (!q.zero) {
            float x[16];
            load16<T>(src + i * 16, x);
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = __fmul_rn(x[j], q.s_enc);
            out = e4m3x16(x);
        }
        reinterpret_cast<uint4 *>(codes)[i] = out;
    }
}

// tensor_scale = amax / 448 (1 when amax == 0), amax read from its bit pattern.
__global__ void fp8_tensor_scale_kernel(const unsigned *__restrict__ amax_bits, float *__restrict__ out) {
    if (threadIdx.x == 0 && blockIdx.x == 0) out[0] = fp8scale_from_amax(__uint_as_float(*amax_bits)).s_dec;
}

}  // namespace lmoe
