/*
 * lmoe_oracle.h -- plain, slow CPU oracle for the LatentMoE expert layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load or call this library.  It shares no code, header,
 * table or helper with the CUDA library under nvfp4_latentmoe_fwd_02_b300/csrc.
 *
 * Every function states the passage it follows.  Page names used below:
 *   [BLOG]  shengxinai.com blog on Nemotron 3 ("Nemotron 3 不止是模型 ... 可复现的工业级蓝图"),
 *           section 2.2 "LatentMoE：在潜空间中重构专家网络" and section 3.1.1 "NVFP4 格式解析",
 *           section 3.1.3 mixed-precision table (latent projections kept in BF16).
 *   [NEWS]  "NVIDIA AI釋出Nemotron 3 Ultra：一個開放的550B混合專家混合Mamba-Transformer..."
 *           (architecture paragraph: d = 8192, 512 experts, top-22; quantization paragraph:
 *           native FP4 math on Blackwell).
 *   [CARD]  "nvidia/NVIDIA-Nemotron-3-Ultra-550B-A55B-NVFP4 · Hugging Face", Description.
 *   [SUPER] "Nemotron 3 Super：面向智能体推理的混合Mamba-Transformer MoE模型", section "潜在MoE".
 *   [HEIDI] "Heidi 在 Fireworks 上训练并部署 NVIDIA Nemotron 3 Ultra", NVFP4 quantization paragraph
 *           (post-training quantization calibrated on synthetic prompts).
 *
 * Parity status: every function here is pinned by a CPU test (see tests/test_oracle_*.py)
 * except the composition of the whole quantized layer, which is pinned only through its
 * parts and through the special cases (l = d identity projections -> standard MoE;
 * E = k = 1 -> plain squared-ReLU FFN) in unquantized mode: "parity unpinned" for the
 * end-to-end quantized composition beyond those pins; the pages print no worked example.
 */
#ifndef LMOE_ORACLE_H
#define LMOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ([BLOG] 3.1.1: E2M1 elements, E4M3 block scale) ---- */
double  oracle_e2m1_value(uint8_t code);       /* low 4 bits used; bit 3 = sign            */
double  oracle_e4m3_value(uint8_t code);       /* NaN for 0x7F / 0xFF                      */
uint8_t oracle_f32_to_e2m1(float v);           /* round-to-nearest-even, saturate to +-6   */
uint8_t oracle_f32_to_e4m3(float v);           /* round-to-nearest-even, saturate to +-448 */
double  oracle_round_bf16(double v);           /* round-to-nearest-even to bfloat16        */
void    oracle_f32_to_e2m1_array(const float *v, int64_t n, uint8_t *out, int nthreads);
void    oracle_f32_to_e4m3_array(const float *v, int64_t n, uint8_t *out, int nthreads);

/* FP8 E4M3 with one FP32 per-tensor scale (the shared expert: [NEWS] quantization paragraph,
 * NVFP4 routed experts mixed with an FP8 shared expert).  s_enc = 448/amax, s_dec = amax/448 (fp32); code = e4m3_satfinite(x * s_enc).
 * amax < 0: computed from src; amax == 0: all codes 0 and s_dec = 1.  n elements. */
void oracle_quantize_fp8(const float *src, int64_t n, float amax, uint8_t *codes,
                         float *s_dec, int nthreads);

/* Exact E4M3 x E4M3 dot product over K elements (tensor scales NOT applied): every E4M3
 * value is an integer multiple of 2^-9, so the sum is an exact integer count of 2^-18;
 * it is returned as a double (exact for K <= 2^17). */
double oracle_fp8_dot(const uint8_t *a, const uint8_t *b, int64_t K);

/* NVFP4 quantization of a row-major [R][K] fp32 array along K (16-element blocks).
 * amax < 0: the tensor amax is computed from src.  codes: [R][K/2] (even element in
 * the low nibble), sf: [R][K/16] E4M3 bytes, *s_dec: the FP32 tensor (decode) scale.
 * nthreads <= 0: all host cores. */
void oracle_quantize_nvfp4(const float *src, int64_t R, int64_t K, float amax,
                           uint8_t *codes, uint8_t *sf, float *s_dec, int nthreads);

/* The 2-D weight-block variant: one E4M3 scale per 16 rows x 16 contraction elements (same
 * arithmetic, block amax over the 16 x 16 block), written for every row of the block so sf
 * keeps the [R][K/16] layout.  R % 16 == 0. */
void oracle_quantize_nvfp4_2d(const float *src, int64_t R, int64_t K, float amax,
                              uint8_t *codes, uint8_t *sf, float *s_dec, int nthreads);

/* Exact NVFP4 x NVFP4 dot product over K elements (K % 16 == 0), block scales applied,
 * tensor scales NOT applied. */
double oracle_nvfp4_dot(const uint8_t *qa, const uint8_t *sfa,
                        const uint8_t *qb, const uint8_t *sfb, int64_t K);

/* Dense x NVFP4 dot over K elements (W4A16): a holds the dense operand (bf16 values), block
 * scales applied, tensor scale NOT applied; fp64. */
double oracle_nvfp4_dense_dot(const float *a, const uint8_t *qb, const uint8_t *sfb, int64_t K);

/* Router: canonical fp32 logits (64-element fmaf chunks; chunk partials summed left to right
 * in groups of 16 chunks; group sums summed left to right; then the bias), top-k by
 * (logit desc, index asc), softmax over the
 * k selected logits (fp64, rounded to float).  x: [T][d] values, Wr: [E][d], b: [E] or NULL.
 * idx/w: [T][k] in ascending expert id; logits [T][E] and counts [E] optional. */
void oracle_router(const float *x, int64_t T, int d, const float *Wr, const float *b,
                   int E, int k, float *logits, int32_t *idx, float *w, int32_t *counts,
                   int nthreads);

/* The layer. Weight layouts follow y = x * W^T (rows = output features). */
typedef struct {
    int d, l, E, k, ffn;
    const float *w_down;    /* [l][d]  bf16 values                                  */
    const float *w_up;      /* [d][l]  bf16 values                                  */
    const float *w_router;  /* [E][d]  fp32                                         */
    const float *b_router;  /* [E] or NULL                                          */
    /* quantized experts (quant mode); per-expert pointers, NULL = not available     */
    const uint8_t *const *w1_codes; /* [E] -> [ffn][l/2]   */
    const uint8_t *const *w1_sf;    /* [E] -> [ffn][l/16]  */
    const float *w1_sdec;           /* [E]                  */
    const uint8_t *const *w2_codes; /* [E] -> [l][ffn/2]   */
    const uint8_t *const *w2_sf;    /* [E] -> [l][ffn/16]  */
    const float *w2_sdec;           /* [E]                  */
    /* master experts (unquantized mode); per-expert pointers                         */
    const float *const *w1;         /* [E] -> [ffn][l]     */
    const float *const *w2;         /* [E] -> [l][ffn]     */
    float amax_z, amax_h;           /* static activation amax (calibration)          */
    /* optional shared expert, kept at the width d ([BLOG] 2.2, closing remark) and in FP8
     * ([NEWS] quantization paragraph), E4M3 with per-tensor scales:
     *   s = bf16( s_h s_w2 (q8(h) . Ws2q) ),  h = bf16( max(s_x s_w1 (q8(x) . Ws1q), 0)^2 )
     * and y = bf16( c Wu^T + s ).  shared_ffn == 0: no shared expert.                   */
    int shared_ffn;
    const uint8_t *ws1_codes;       /* [shared_ffn][d]  E4M3 (quant mode)             */
    float ws1_sdec;
    const uint8_t *ws2_codes;       /* [d][shared_ffn]  E4M3 (quant mode)             */
    float ws2_sdec;
    const float *ws1;               /* [shared_ffn][d]  bf16 values (unquant mode)    */
    const float *ws2;               /* [d][shared_ffn]  bf16 values (unquant mode)    */
    float amax_xs, amax_hs;         /* static amax of x and of the shared h           */
} oracle_layer;

typedef struct {               /* every pointer optional (NULL = not wanted)          */
    float   *z;        /* [T][l]            bf16 values (quant) / fp64 rounded to float (unquant) */
    uint8_t *zq_codes; /* [T][l/2]          */
    uint8_t *zq_sf;    /* [T][l/16]         */
    float   *logits;   /* [T][E]            */
    int32_t *idx;      /* [T][k]            */
    float   *w;        /* [T][k]            */
    int32_t *counts;   /* [E]               */
    float   *h;        /* [T][k][ffn]       bf16 values, slots in ascending expert id */
    uint8_t *hq_codes; /* [T][k][ffn/2]     */
    uint8_t *hq_sf;    /* [T][k][ffn/16]    */
    double  *c64;      /* [T][l]            combine before rounding */
    float   *c;        /* [T][l]            bf16 values              */
    double  *y64;      /* [T][d]            before the final rounding */
    float   *y;        /* [T][d]            bf16 values              */
    uint8_t *xs_q;     /* [T][d]            shared expert: E4M3 codes of x */
    float   *hs;       /* [T][shared_ffn]   shared expert: h (bf16 values)  */
    uint8_t *hs_q;     /* [T][shared_ffn]   shared expert: E4M3 codes of h */
    float   *s;        /* [T][d]            shared expert output (bf16 values) */
} oracle_out;

/* quant = 1: the NVFP4 layer.  quant = 2: W4A16 (NVFP4 weights, bf16 activations, no activation
 * quantization).  quant = 0: the same layer in plain fp64 with the master weights and no
 * rounding of any intermediate (used by the structural pins).
 * Returns 0, or -1 if an expert that a token selects has no weights. */
int oracle_layer_forward(const oracle_layer *L, const float *x, int64_t T, int quant,
                         oracle_out *out, int nthreads);

/* The NVFP4 layer (quant = 1) with each token's quantized z given (zq_codes [T][l/2],
 * zq_sf [T][l/16]) instead of the quantization of the oracle's own z: routing, experts,
 * combine, up-projection and shared expert are the steps above, applied to that zq.  For a z
 * whose fp32 accumulation order differs (one bf16 ulp away), whose quantization is as correct.
 * Returns 0, or -1 (missing expert weights / NULL zq). */
int oracle_layer_forward_zq(const oracle_layer *L, const float *x, const uint8_t *zq_codes,
                            const uint8_t *zq_sf, int64_t T, oracle_out *out, int nthreads);

/* The shared expert alone on token rows x [T][d] (outputs as in oracle_out; each optional).
 * quant = 0: fp64 with the master weights, no quantization and no rounding. */
int oracle_shared_forward(const oracle_layer *L, const float *x, int64_t T, int quant,
                          uint8_t *xs_q, float *hs, uint8_t *hs_q, float *s, int nthreads);

/* Static activation calibration ([HEIDI]): amax of z and of h over a calibration batch. */
int oracle_calibrate(const oracle_layer *L, const float *x, int64_t T,
                     float *amax_z, float *amax_h, int nthreads);
/* The shared expert's static amax: of x, then of h with x quantized by that amax. */
int oracle_calibrate_shared(const oracle_layer *L, const float *x, int64_t T,
                            float *amax_xs, float *amax_hs, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
