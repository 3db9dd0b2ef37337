/*
 * lmoe_oracle.c -- plain, slow CPU oracle for the LatentMoE expert layer forward.
 *
 * TEST INFRASTRUCTURE ONLY (see lmoe_oracle.h for the page names and the parity status).
 * Built with  gcc -O2 -ffp-contract=off  and no fast-math, so every float operation
 * written here is the IEEE operation it reads as.  Floating-point steps whose result
 * is a float output use fp64 and round once; steps that decide an integer (a code,
 * a block scale, an expert index) use exactly the fp32 operations their definition
 * states.
 */
#include "lmoe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------------------ */
/* threads: a plain parallel-for over [0, n)                                             */
/* ------------------------------------------------------------------------------------ */
typedef void (*range_fn)(int64_t begin, int64_t end, void *arg);
typedef struct { range_fn fn; void *arg; int64_t b, e; } range_job;

static void *range_thread(void *p) {
    range_job *j = (range_job *)p;
    j->fn(j->b, j->e, j->arg);
    return NULL;
}

static int host_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *arg) {
    int nt = host_threads(nthreads);
    if (nt > n) nt = (int)(n > 0 ? n : 1);
    if (nt <= 1) { fn(0, n, arg); return; }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    range_job *jobs = (range_job *)malloc(sizeof(range_job) * nt);
    for (int i = 0; i < nt; ++i) {
        jobs[i].fn = fn; jobs[i].arg = arg;
        jobs[i].b = n * i / nt; jobs[i].e = n * (i + 1) / nt;
        pthread_create(&th[i], NULL, range_thread, &jobs[i]);
    }
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th); free(jobs);
}

/* ------------------------------------------------------------------------------------ */
/* Number formats.  [BLOG] 3.1.1: an NVFP4 element is E2M1 (2 exponent bits, 1 mantissa  */
/* bit); each 16-element micro-block carries one E4M3 scale.  The decoders below are the  */
/* closed forms of those binary formats (E2M1: bias 1; E4M3: bias 7, no infinities,       */
/* S.1111.111 is NaN, largest finite 448).                                               */
/* ------------------------------------------------------------------------------------ */
double oracle_e2m1_value(uint8_t code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

double oracle_e4m3_value(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round |v| to the binary grid with `q` = spacing of the binade, ties to even (the      */
/* default rounding mode of nearbyint), then encode.  E2M1 grid: 0, .5, 1, 1.5, 2, 3, 4, */
/* 6 (codes 0..7); anything at or beyond 6 saturates to 6 (satfinite).                   */
uint8_t oracle_f32_to_e2m1(float v) {
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (!(a < 6.0)) return sign | 7;
    double q = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double r = nearbyint(a / q) * q;
    if (r > 6.0) r = 6.0;
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    for (uint8_t c = 0; c < 8; ++c)
        if (grid[c] == r) return sign | c;
    return sign | 7; /* unreachable */
}

/* E4M3: normal binades [2^E, 2^(E+1)) for E >= -6 have spacing 2^(E-3); below 2^-6 the */
/* subnormal spacing is 2^-9.  Values at or beyond 448 saturate to 448 (satfinite).     */
uint8_t oracle_f32_to_e4m3(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    if (!(a < 448.0)) return sign | 0x7E;
    const double min_normal = ldexp(1.0, -6);
    double q;
    if (a < min_normal) {
        q = ldexp(1.0, -9);
    } else {
        int e; frexp(a, &e);       /* a = f * 2^e, f in [0.5, 1)  =>  floor(log2 a) = e - 1 */
        q = ldexp(1.0, (e - 1) - 3);
    }
    double r = nearbyint(a / q) * q;
    if (r == 0.0) return sign;
    if (r < min_normal) return sign | (uint8_t)(r / ldexp(1.0, -9));
    int e; frexp(r, &e);
    int E = e - 1;
    int m = (int)(r / ldexp(1.0, E - 3)) - 8;
    return sign | (uint8_t)(((E + 7) << 3) | m);
}

/* bfloat16: 8 significant bits, exponent range of fp32 (subnormal spacing 2^-133).      */
double oracle_round_bf16(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    double a = fabs(v);
    int e; frexp(a, &e);
    int qe = (e - 1) - 7;
    if (qe < -133) qe = -133;
    double r = nearbyint(a / ldexp(1.0, qe)) * ldexp(1.0, qe);
    const double bf16_max = ldexp(255.0 / 128.0, 127);
    if (r > bf16_max) r = INFINITY;
    return v < 0 ? -r : r;
}

/* decode tables filled from the closed forms above */
static double g_e4m3[256];
static int g_e2m1x2[16];           /* 2 * value: an integer in {0, 1, 2, 3, 4, 6, 8, 12} */
static int64_t g_e4m3x512[256];    /* 512 * value: an integer (E4M3 values are multiples of 2^-9) */
static pthread_once_t g_once = PTHREAD_ONCE_INIT;
static void init_tables(void) {
    for (int c = 0; c < 256; ++c) {
        g_e4m3[c] = oracle_e4m3_value((uint8_t)c);
        g_e4m3x512[c] = isnan(g_e4m3[c]) ? 0 : (int64_t)(g_e4m3[c] * 512.0);
    }
    for (int c = 0; c < 16; ++c) g_e2m1x2[c] = (int)(2.0 * oracle_e2m1_value((uint8_t)c));
}

/* ------------------------------------------------------------------------------------ */
/* NVFP4 quantization ([BLOG] 3.1.1 gives the format only; the arithmetic below is the   */
/* reading this project takes, all in IEEE fp32 with round-to-nearest-even):             */
/*   amax_t == 0       -> all codes and scales 0, tensor scale 1                         */
/*   s_enc = 2688/amax_t, s_dec = amax_t/2688 (2688 = 448 * 6), s_enc6 = s_enc/6          */
/*   per 16-block:  sf = e4m3(amax_b * s_enc6);  bd = value(sf) * s_dec;                  */
/*                  rcp = bd > 0 ? 1/bd : 0;     q_i = e2m1(x_i * rcp)                     */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    const float *src; int64_t K; float s_enc6, s_dec;
    uint8_t *codes, *sf;
} quant_job;

static void quantize_row(const float *x, int64_t K, float s_enc6, float s_dec,
                         uint8_t *codes, uint8_t *sf) {
    for (int64_t b = 0; b < K / 16; ++b) {
        const float *xb = x + 16 * b;
        float amax_b = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(xb[i]);
            if (a > amax_b) amax_b = a;
        }
        float sc = amax_b * s_enc6;
        uint8_t s = oracle_f32_to_e4m3(sc);
        float bd = (float)g_e4m3[s] * s_dec;
        float rcp = (bd > 0.0f) ? 1.0f / bd : 0.0f;
        sf[b] = s;
        for (int i = 0; i < 16; i += 2) {
            uint8_t q0 = oracle_f32_to_e2m1(xb[i] * rcp);
            uint8_t q1 = oracle_f32_to_e2m1(xb[i + 1] * rcp);
            codes[8 * b + i / 2] = (uint8_t)(q0 | (q1 << 4));
        }
    }
}

static void quant_rows(int64_t b, int64_t e, void *arg) {
    quant_job *j = (quant_job *)arg;
    for (int64_t r = b; r < e; ++r)
        quantize_row(j->src + r * j->K, j->K, j->s_enc6, j->s_dec,
                     j->codes + r * (j->K / 2), j->sf + r * (j->K / 16));
}

void oracle_quantize_nvfp4(const float *src, int64_t R, int64_t K, float amax,
                           uint8_t *codes, uint8_t *sf, float *s_dec_out, int nthreads) {
    pthread_once(&g_once, init_tables);
    if (amax < 0.0f) {
        amax = 0.0f;
        for (int64_t i = 0; i < R * K; ++i) {
            float a = fabsf(src[i]);
            if (a > amax) amax = a;
        }
    }
    if (amax == 0.0f) {
        memset(codes, 0, (size_t)(R * K / 2));
        memset(sf, 0, (size_t)(R * K / 16));
        if (s_dec_out) *s_dec_out = 1.0f;
        return;
    }
    const float S = 2688.0f;
    float s_enc = S / amax;
    float s_dec = amax / S;
    quant_job j = {src, K, s_enc / 6.0f, s_dec, codes, sf};
    parallel_for(R, nthreads, quant_rows, &j);
    if (s_dec_out) *s_dec_out = s_dec;
}

/* 2-D variant ([NEWS] architecture paragraph: NVFP4 pretraining with weights quantized in */
/* two-dimensional blocks; 16 x 16 is this project's reading, matching the 16-element      */
/* contraction blocks).  One E4M3 scale per 16 rows x 16 contraction elements, from the     */
/* block's amax; the same fp32 steps as the 1-D quantizer otherwise.  The scale is written  */
/* for every row of the block, so sf keeps the 1-D layout [R][K/16] (R % 16 == 0).          */
typedef struct { const float *src; int64_t K; float s_enc6, s_dec; uint8_t *codes, *sf; } quant2d_job;

static void quant2d_groups(int64_t gb, int64_t ge, void *arg) {
    quant2d_job *j = (quant2d_job *)arg;
    const int64_t K = j->K;
    for (int64_t g = gb; g < ge; ++g) {               /* 16-row group */
        for (int64_t b = 0; b < K / 16; ++b) {
            float amax_b = 0.0f;
            for (int r = 0; r < 16; ++r)
                for (int i = 0; i < 16; ++i) {
                    float a = fabsf(j->src[(g * 16 + r) * K + 16 * b + i]);
                    if (a > amax_b) amax_b = a;
                }
            uint8_t s = oracle_f32_to_e4m3(amax_b * j->s_enc6);
            float bd = (float)g_e4m3[s] * j->s_dec;
            float rcp = (bd > 0.0f) ? 1.0f / bd : 0.0f;
            for (int r = 0; r < 16; ++r) {
                const float *xb = j->src + (g * 16 + r) * K + 16 * b;
                uint8_t *cb = j->codes + (g * 16 + r) * (K / 2) + 8 * b;
                for (int i = 0; i < 16; i += 2) {
                    uint8_t q0 = oracle_f32_to_e2m1(xb[i] * rcp);
                    uint8_t q1 = oracle_f32_to_e2m1(xb[i + 1] * rcp);
                    cb[i / 2] = (uint8_t)(q0 | (q1 << 4));
                }
                j->sf[(g * 16 + r) * (K / 16) + b] = s;
            }
        }
    }
}

void oracle_quantize_nvfp4_2d(const float *src, int64_t R, int64_t K, float amax,
                              uint8_t *codes, uint8_t *sf, float *s_dec_out, int nthreads) {
    pthread_once(&g_once, init_tables);
    if (amax < 0.0f) {
        amax = 0.0f;
        for (int64_t i = 0; i < R * K; ++i) {
            float a = fabsf(src[i]);
            if (a > amax) amax = a;
        }
    }
    if (amax == 0.0f) {
        memset(codes, 0, (size_t)(R * K / 2));
        memset(sf, 0, (size_t)(R * K / 16));
        if (s_dec_out) *s_dec_out = 1.0f;
        return;
    }
    const float S = 2688.0f;
    float s_enc = S / amax;
    float s_dec = amax / S;
    quant2d_job j = {src, K, s_enc / 6.0f, s_dec, codes, sf};
    parallel_for(R / 16, nthreads, quant2d_groups, &j);
    if (s_dec_out) *s_dec_out = s_dec;
}

/* Exact block-scaled dot: inside a block, 2*e2m1 values are small integers, so the     */
/* 16-term dot is an exact integer; it is scaled by 1/4 and the two E4M3 block scales    */
/* (all exact in fp64).  Blocks are summed in fp64.                                      */
double oracle_nvfp4_dot(const uint8_t *qa, const uint8_t *sfa,
                        const uint8_t *qb, const uint8_t *sfb, int64_t K) {
    pthread_once(&g_once, init_tables);
    double acc = 0.0;
    for (int64_t b = 0; b < K / 16; ++b) {
        int dot = 0;
        for (int i = 0; i < 8; ++i) {
            uint8_t a = qa[8 * b + i], c = qb[8 * b + i];
            dot += g_e2m1x2[a & 15] * g_e2m1x2[c & 15] + g_e2m1x2[a >> 4] * g_e2m1x2[c >> 4];
        }
        acc += (double)dot * 0.25 * g_e4m3[sfa[b]] * g_e4m3[sfb[b]];
    }
    return acc;
}

/* Dense x NVFP4 dot (the W4A16 form): sum over blocks of value(sfb) * sum_i a_i * e2m1(q_i),  */
/* in fp64; every product of a bf16 activation with an E2M1 value is exact in fp64.          */
double oracle_nvfp4_dense_dot(const float *a, const uint8_t *qb, const uint8_t *sfb, int64_t K) {
    pthread_once(&g_once, init_tables);
    double acc = 0.0;
    for (int64_t b = 0; b < K / 16; ++b) {
        double blk = 0.0;
        for (int i = 0; i < 8; ++i) {
            uint8_t c = qb[8 * b + i];
            blk += (double)a[16 * b + 2 * i] * (0.5 * g_e2m1x2[c & 15]) +
                   (double)a[16 * b + 2 * i + 1] * (0.5 * g_e2m1x2[c >> 4]);
        }
        acc += blk * g_e4m3[sfb[b]];
    }
    return acc;
}

/* ------------------------------------------------------------------------------------ */
/* FP8 E4M3 with one per-tensor scale ([NEWS] quantization paragraph: the shared expert is */
/* FP8).  The scale arithmetic is this project's reading, in IEEE fp32: s_enc = 448/amax,  */
/* s_dec = amax/448, code = e4m3_satfinite(x * s_enc); amax == 0 -> codes 0, s_dec = 1.    */
/* ------------------------------------------------------------------------------------ */
typedef struct { const float *src; float s_enc; uint8_t *codes; } fp8_job;
static void fp8_rows(int64_t b, int64_t e, void *arg) {
    fp8_job *j = (fp8_job *)arg;
    for (int64_t i = b; i < e; ++i) j->codes[i] = oracle_f32_to_e4m3(j->src[i] * j->s_enc);
}

void oracle_quantize_fp8(const float *src, int64_t n, float amax, uint8_t *codes,
                         float *s_dec_out, int nthreads) {
    pthread_once(&g_once, init_tables);
    if (amax < 0.0f) {
        amax = 0.0f;
        for (int64_t i = 0; i < n; ++i) {
            float a = fabsf(src[i]);
            if (a > amax) amax = a;
        }
    }
    if (amax == 0.0f) {
        memset(codes, 0, (size_t)n);
        if (s_dec_out) *s_dec_out = 1.0f;
        return;
    }
    fp8_job j = {src, 448.0f / amax, codes};
    parallel_for(n, nthreads, fp8_rows, &j);
    if (s_dec_out) *s_dec_out = amax / 448.0f;
}

/* Exact E4M3 dot: with every value scaled by 512 the products are integers below 2^36, so */
/* an int64 sum is exact; the result counts units of 2^-18.                                */
double oracle_fp8_dot(const uint8_t *a, const uint8_t *b, int64_t K) {
    pthread_once(&g_once, init_tables);
    int64_t acc = 0;
    for (int64_t i = 0; i < K; ++i) acc += g_e4m3x512[a[i]] * g_e4m3x512[b[i]];
    return ldexp((double)acc, -18);
}

/* ------------------------------------------------------------------------------------ */
/* Router.  [NEWS] architecture paragraph: each MoE layer has 512 experts and activates   */
/* the top 22 per token; [BLOG] 2.2 keeps the routing gate at width d.  The logit order   */
/* is this project's canonical fp32 order (the pages are silent): the d axis is cut into */
/* chunks of 64; inside a chunk an fmaf chain in ascending index starting from 0; chunks  */
/* are grouped 16 at a time (1024 elements); a group's chunk partials are added left to   */
/* right starting from 0; the group sums are added left to right starting from 0; then    */
/* the bias.  Selection: logit descending, lower expert index first on ties.  Weights:    */
/* softmax over the k selected logits (fp64).                                             */
/* ------------------------------------------------------------------------------------ */
/* The same source is compiled twice: for CPUs with the FMA instruction set fmaf becomes one  */
/* inline fused multiply-add instead of a libm call (the operation is exactly specified, so  */
/* both clones return the same bits; the loader picks the clone the host supports).          */
__attribute__((target_clones("fma", "default")))
static float canonical_logit(const float *x, const float *w, int d) {
    float acc = 0.0f;
    for (int g = 0; g < d; g += 16 * 64) {
        float gs = 0.0f;
        for (int c = g; c < g + 16 * 64 && c < d; c += 64) {
            float p = 0.0f;
            for (int i = c; i < c + 64; ++i) p = fmaf(x[i], w[i], p);
            gs = gs + p;
        }
        acc = acc + gs;
    }
    return acc;
}

static void topk_softmax(const float *lg, int E, int k, int32_t *idx, float *w, double *w64) {
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * k);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || lg[e] > lg[best]) best = e;  /* strict '>' keeps the lower index */
        }
        taken[best] = 1;
        sel[j] = best;
    }
    /* slot order: ascending expert id */
    int n = 0;
    for (int e = 0; e < E; ++e)
        if (taken[e]) idx[n++] = e;
    double m = -INFINITY;
    for (int j = 0; j < k; ++j) if ((double)lg[idx[j]] > m) m = lg[idx[j]];
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += exp((double)lg[idx[j]] - m);
    for (int j = 0; j < k; ++j) {
        double v = exp((double)lg[idx[j]] - m) / s;
        if (w64) w64[j] = v;
        if (w) w[j] = (float)v;
    }
    free(taken); free(sel);
}

typedef struct {
    const float *x; int d; const float *Wr, *b; int E, k;
    float *logits; int32_t *idx; float *w;
} router_job;

static void router_rows(int64_t tb, int64_t te, void *arg) {
    router_job *j = (router_job *)arg;
    float *lg = (float *)malloc(sizeof(float) * j->E);
    for (int64_t t = tb; t < te; ++t) {
        const float *xt = j->x + t * j->d;
        for (int e = 0; e < j->E; ++e)
            lg[e] = canonical_logit(xt, j->Wr + (int64_t)e * j->d, j->d) + (j->b ? j->b[e] : 0.0f);
        if (j->logits) memcpy(j->logits + t * j->E, lg, sizeof(float) * j->E);
        topk_softmax(lg, j->E, j->k, j->idx + t * j->k, j->w ? j->w + t * j->k : NULL, NULL);
    }
    free(lg);
}

void oracle_router(const float *x, int64_t T, int d, const float *Wr, const float *b,
                   int E, int k, float *logits, int32_t *idx, float *w, int32_t *counts,
                   int nthreads) {
    router_job j = {x, d, Wr, b, E, k, logits, idx, w};
    parallel_for(T, nthreads, router_rows, &j);
    if (counts) {
        memset(counts, 0, sizeof(int32_t) * E);
        for (int64_t i = 0; i < T * k; ++i) counts[idx[i]]++;
    }
}

/* ------------------------------------------------------------------------------------ */
/* The shared expert of one token: it runs at the full width d ([BLOG] 2.2, closing       */
/* remark: the shared expert is not moved into the latent space) in FP8 ([NEWS]            */
/* quantization paragraph), with the routed experts' squared ReLU (the pages name no other */
/* activation for it):                                                                    */
/*   xq = q8(x; amax_xs)                                                                  */
/*   h  = bf16( max(s_x s_w1 (xq . Ws1q_f), 0)^2 )       (exact E4M3 dots, fp64 scaling)  */
/*   hq = q8(h; amax_hs)                                                                  */
/*   s  = bf16( s_h s_w2 (hq . Ws2q_j) )                                                  */
/* Unquantized mode: the same steps in fp64 on the masters with no quantization and no    */
/* rounding.  s64 receives s; hmax (optional) the largest h.                              */
/* ------------------------------------------------------------------------------------ */
static void shared_token(const oracle_layer *L, const float *xt, int quant, float amax_xs,
                         float amax_hs, uint8_t *xq, float *hf, uint8_t *hq, double *h64,
                         double *s64, float *hmax) {
    const int d = L->d, F = L->shared_ffn;
    float mh = 0.0f;
    if (quant) {
        float sdx, sdh;
        oracle_quantize_fp8(xt, d, amax_xs, xq, &sdx, 1);
        double a1 = (double)sdx * (double)L->ws1_sdec;
        for (int f = 0; f < F; ++f) {
            double u = a1 * oracle_fp8_dot(xq, L->ws1_codes + (int64_t)f * d, d);
            double r = u > 0.0 ? u : 0.0;
            hf[f] = (float)oracle_round_bf16(r * r);
            if (hf[f] > mh) mh = hf[f];
        }
        oracle_quantize_fp8(hf, F, amax_hs, hq, &sdh, 1);
        double a2 = (double)sdh * (double)L->ws2_sdec;
        for (int j = 0; j < d; ++j)
            s64[j] = oracle_round_bf16(a2 * oracle_fp8_dot(hq, L->ws2_codes + (int64_t)j * F, F));
    } else {
        for (int f = 0; f < F; ++f) {
            const float *wr = L->ws1 + (int64_t)f * d;
            double u = 0.0;
            for (int i = 0; i < d; ++i) u += (double)xt[i] * (double)wr[i];
            double r = u > 0.0 ? u : 0.0;
            h64[f] = r * r;
            hf[f] = (float)h64[f];
            if (hf[f] > mh) mh = hf[f];
        }
        for (int j = 0; j < d; ++j) {
            const float *wr = L->ws2 + (int64_t)j * F;
            double o = 0.0;
            for (int f = 0; f < F; ++f) o += h64[f] * (double)wr[f];
            s64[j] = o;
        }
    }
    if (hmax) *hmax = mh;
}

static int shared_ready(const oracle_layer *L, int quant) {
    return quant ? (L->ws1_codes && L->ws2_codes) : (L->ws1 && L->ws2);
}

typedef struct {
    const oracle_layer *L; const float *x; int quant;
    uint8_t *xs_q; float *hs; uint8_t *hs_q; float *s; float *hmax_seen; float amax_hs;
} shared_job;

static void shared_rows(int64_t tb, int64_t te, void *arg) {
    shared_job *J = (shared_job *)arg;
    const oracle_layer *L = J->L;
    const int d = L->d, F = L->shared_ffn;
    uint8_t *xq = (uint8_t *)malloc((size_t)d), *hq = (uint8_t *)malloc((size_t)F);
    float *hf = (float *)malloc(sizeof(float) * F);
    double *h64 = (double *)malloc(sizeof(double) * F), *s64 = (double *)malloc(sizeof(double) * d);
    for (int64_t t = tb; t < te; ++t) {
        float mh;
        shared_token(L, J->x + t * d, J->quant, L->amax_xs, J->amax_hs, xq, hf, hq, h64, s64, &mh);
        if (J->hmax_seen) J->hmax_seen[t] = mh;
        if (J->xs_q) memcpy(J->xs_q + t * d, xq, (size_t)d);
        if (J->hs) memcpy(J->hs + t * F, hf, sizeof(float) * F);
        if (J->hs_q) memcpy(J->hs_q + t * F, hq, (size_t)F);
        if (J->s) for (int j = 0; j < d; ++j) J->s[t * d + j] = (float)s64[j];
    }
    free(xq); free(hq); free(hf); free(h64); free(s64);
}

int oracle_shared_forward(const oracle_layer *L, const float *x, int64_t T, int quant,
                          uint8_t *xs_q, float *hs, uint8_t *hs_q, float *s, int nthreads) {
    pthread_once(&g_once, init_tables);
    if (L->shared_ffn <= 0 || !shared_ready(L, quant)) return -1;
    shared_job J = {L, x, quant, quant ? xs_q : NULL, hs, quant ? hs_q : NULL, s, NULL, L->amax_hs};
    parallel_for(T, nthreads, shared_rows, &J);
    return 0;
}

int oracle_calibrate_shared(const oracle_layer *L, const float *x, int64_t T,
                            float *amax_xs, float *amax_hs, int nthreads) {
    pthread_once(&g_once, init_tables);
    if (L->shared_ffn <= 0 || !shared_ready(L, 1)) return -1;
    float mx = 0.0f;
    for (int64_t i = 0; i < T * L->d; ++i) {
        float a = fabsf(x[i]);
        if (a > mx) mx = a;
    }
    oracle_layer Lc = *L;
    Lc.amax_xs = mx;
    float *seen = (float *)calloc((size_t)(T > 0 ? T : 1), sizeof(float));
    shared_job J = {&Lc, x, 1, NULL, NULL, NULL, NULL, seen, 1.0f};
    parallel_for(T, nthreads, shared_rows, &J);
    float mh = 0.0f;
    for (int64_t t = 0; t < T; ++t) if (seen[t] > mh) mh = seen[t];
    free(seen);
    *amax_xs = mx; *amax_hs = mh;
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* The layer ([BLOG] 2.2, steps 1-3; [SUPER] "潜在MoE"):                                  */
/*   z  = bf16( x Wd^T )                      down-projection d -> l, BF16 ([BLOG] 3.1.3) */
/*   zq = NVFP4(z) with the static amax_z                                                */
/*   route x (router above)                                                              */
/*   per selected expert e:  u = s_z s_w1e (zq . W1q_e)    (exact block dots)             */
/*                           h = bf16(max(u,0)^2)          (squared ReLU)                 */
/*                           hq = NVFP4(h) with the static amax_h                         */
/*                           o = s_h s_w2e (hq . W2q_e)                                   */
/*   c  = bf16( sum_j w_j o_j )               routing-weighted combine in l space        */
/*   y  = bf16( c Wu^T )                      up-projection l -> d, BF16                 */
/*        (+ s, the shared expert above, before the rounding, when the layer has one)    */
/* In unquantized mode (quant = 0) the same steps run in fp64 on the master weights with  */
/* no quantization and no rounding.  W4A16 mode (quant = 2; [NEWS] quantization paragraph: */
/* the NVFP4 checkpoint runs as W4A16 on Hopper): NVFP4 weights, bf16 z and h unquantized: */
/*   u = s_w1e (z . dq(W1q_e)), h = bf16(max(u,0)^2), o = s_w2e (h . dq(W2q_e)).           */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    const oracle_layer *L; const float *x; int quant; oracle_out *out;
    float amax_z, amax_h;       /* used by the quantizers */
    float *amax_h_seen;         /* per-token max |h| (calibration), may be NULL */
    /* optional (quant = 1): each token's zq ([T][l/2] codes, [T][l/16] scales) given instead */
    /* of the quantization of this oracle's own z                                          */
    const uint8_t *zq_codes_in, *zq_sf_in;
    volatile int error;
} layer_job;

static void layer_rows(int64_t tb, int64_t te, void *arg) {
    layer_job *J = (layer_job *)arg;
    const oracle_layer *L = J->L;
    const int d = L->d, l = L->l, E = L->E, k = L->k, F = L->ffn;
    oracle_out *O = J->out;
    double *z64 = (double *)malloc(sizeof(double) * l);
    float *zf = (float *)malloc(sizeof(float) * l);
    uint8_t *zc = (uint8_t *)malloc((size_t)l / 2), *zs = (uint8_t *)malloc((size_t)l / 16);
    float *lg = (float *)malloc(sizeof(float) * E);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * k);
    double *w64 = (double *)malloc(sizeof(double) * k);
    float *wf = (float *)malloc(sizeof(float) * k);
    double *u64 = (double *)malloc(sizeof(double) * F);
    float *hf = (float *)malloc(sizeof(float) * F);
    uint8_t *hc = (uint8_t *)malloc((size_t)F / 2), *hs = (uint8_t *)malloc((size_t)F / 16);
    double *c64 = (double *)malloc(sizeof(double) * l);
    double *cin = (double *)malloc(sizeof(double) * l);
    const int FS = L->shared_ffn > 0 ? L->shared_ffn : 1;
    const int has_shared = L->shared_ffn > 0;
    if (has_shared && !shared_ready(L, J->quant)) J->error = 1;
    uint8_t *sxq = (uint8_t *)malloc((size_t)d), *shq = (uint8_t *)malloc((size_t)FS);
    float *shf = (float *)malloc(sizeof(float) * FS);
    double *sh64 = (double *)malloc(sizeof(double) * FS), *ss64 = (double *)malloc(sizeof(double) * d);

    for (int64_t t = tb; t < te; ++t) {
        const float *xt = J->x + t * d;
        /* step 1: down-projection */
        for (int j = 0; j < l; ++j) {
            const float *wr = L->w_down + (int64_t)j * d;
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += (double)xt[i] * (double)wr[i];
            z64[j] = J->quant ? oracle_round_bf16(s) : s;
            zf[j] = (float)z64[j];
        }
        if (O->z) memcpy(O->z + t * l, zf, sizeof(float) * l);
        if (J->quant == 1 && J->zq_codes_in) {
            memcpy(zc, J->zq_codes_in + t * (l / 2), (size_t)l / 2);
            memcpy(zs, J->zq_sf_in + t * (l / 16), (size_t)l / 16);
            if (O->zq_codes) memcpy(O->zq_codes + t * (l / 2), zc, (size_t)l / 2);
            if (O->zq_sf) memcpy(O->zq_sf + t * (l / 16), zs, (size_t)l / 16);
        } else if (J->quant == 1) {
            float sd;
            oracle_quantize_nvfp4(zf, 1, l, J->amax_z, zc, zs, &sd, 1);
            if (O->zq_codes) memcpy(O->zq_codes + t * (l / 2), zc, (size_t)l / 2);
            if (O->zq_sf) memcpy(O->zq_sf + t * (l / 16), zs, (size_t)l / 16);
        }
        /* step 2: routing on x */
        for (int e = 0; e < E; ++e)
            lg[e] = canonical_logit(xt, L->w_router + (int64_t)e * d, d) +
                    (L->b_router ? L->b_router[e] : 0.0f);
        if (O->logits) memcpy(O->logits + t * E, lg, sizeof(float) * E);
        topk_softmax(lg, E, k, idx, wf, w64);
        if (O->idx) memcpy(O->idx + t * k, idx, sizeof(int32_t) * k);
        if (O->w) memcpy(O->w + t * k, wf, sizeof(float) * k);

        /* step 2b: latent experts and the weighted combine */
        for (int j = 0; j < l; ++j) c64[j] = 0.0;
        float hmax = 0.0f;
        float s_dec_z = (J->amax_z == 0.0f) ? 1.0f : J->amax_z / 2688.0f;
        float s_dec_h = (J->amax_h == 0.0f) ? 1.0f : J->amax_h / 2688.0f;
        for (int jj = 0; jj < k; ++jj) {
            int e = idx[jj];
            if (J->quant == 2) {
                /* W4A16: NVFP4 weights, bf16 activations (no activation quantization) */
                if (!L->w1_codes[e] || !L->w1_sf[e] || !L->w2_codes[e] || !L->w2_sf[e]) {
                    J->error = 1; continue;
                }
                for (int f = 0; f < F; ++f) {
                    double u = (double)L->w1_sdec[e] *
                               oracle_nvfp4_dense_dot(zf, L->w1_codes[e] + (int64_t)f * (l / 2),
                                                      L->w1_sf[e] + (int64_t)f * (l / 16), l);
                    double r = u > 0.0 ? u : 0.0;
                    hf[f] = (float)oracle_round_bf16(r * r);
                }
                for (int j = 0; j < l; ++j) {
                    double o = (double)L->w2_sdec[e] *
                               oracle_nvfp4_dense_dot(hf, L->w2_codes[e] + (int64_t)j * (F / 2),
                                                      L->w2_sf[e] + (int64_t)j * (F / 16), F);
                    c64[j] += w64[jj] * o;
                }
            } else if (J->quant) {
                if (!L->w1_codes[e] || !L->w1_sf[e] || !L->w2_codes[e] || !L->w2_sf[e]) {
                    J->error = 1; continue;
                }
                double a1 = (double)s_dec_z * (double)L->w1_sdec[e];
                for (int f = 0; f < F; ++f) {
                    double u = a1 * oracle_nvfp4_dot(zc, zs, L->w1_codes[e] + (int64_t)f * (l / 2),
                                                     L->w1_sf[e] + (int64_t)f * (l / 16), l);
                    double r = u > 0.0 ? u : 0.0;
                    hf[f] = (float)oracle_round_bf16(r * r);
                    if (hf[f] > hmax) hmax = hf[f];
                }
                oracle_quantize_nvfp4(hf, 1, F, J->amax_h, hc, hs, NULL, 1);
                double a2 = (double)s_dec_h * (double)L->w2_sdec[e];
                for (int j = 0; j < l; ++j) {
                    double o = a2 * oracle_nvfp4_dot(hc, hs, L->w2_codes[e] + (int64_t)j * (F / 2),
                                                     L->w2_sf[e] + (int64_t)j * (F / 16), F);
                    c64[j] += w64[jj] * o;
                }
                if (O->hq_codes) memcpy(O->hq_codes + (t * k + jj) * (F / 2), hc, (size_t)F / 2);
                if (O->hq_sf) memcpy(O->hq_sf + (t * k + jj) * (F / 16), hs, (size_t)F / 16);
            } else {
                if (!L->w1[e] || !L->w2[e]) { J->error = 1; continue; }
                for (int f = 0; f < F; ++f) {
                    const float *wr = L->w1[e] + (int64_t)f * l;
                    double u = 0.0;
                    for (int i = 0; i < l; ++i) u += z64[i] * (double)wr[i];
                    double r = u > 0.0 ? u : 0.0;
                    u64[f] = r * r;
                    hf[f] = (float)u64[f];
                }
                for (int j = 0; j < l; ++j) {
                    const float *wr = L->w2[e] + (int64_t)j * F;
                    double o = 0.0;
                    for (int f = 0; f < F; ++f) o += u64[f] * (double)wr[f];
                    c64[j] += w64[jj] * o;
                }
            }
            if (O->h) memcpy(O->h + (t * k + jj) * F, hf, sizeof(float) * F);
        }
        if (J->amax_h_seen) J->amax_h_seen[t] = hmax;
        if (O->c64) memcpy(O->c64 + t * l, c64, sizeof(double) * l);
        for (int j = 0; j < l; ++j) {
            cin[j] = J->quant ? oracle_round_bf16(c64[j]) : c64[j];
            if (O->c) O->c[t * l + j] = (float)cin[j];
        }
        /* shared expert (at width d, on x) */
        if (has_shared && shared_ready(L, J->quant)) {
            shared_token(L, xt, J->quant, L->amax_xs, L->amax_hs, sxq, shf, shq, sh64, ss64, NULL);
            if (O->xs_q && J->quant) memcpy(O->xs_q + t * d, sxq, (size_t)d);
            if (O->hs) memcpy(O->hs + t * L->shared_ffn, shf, sizeof(float) * L->shared_ffn);
            if (O->hs_q && J->quant) memcpy(O->hs_q + t * L->shared_ffn, shq, (size_t)L->shared_ffn);
            if (O->s) for (int j = 0; j < d; ++j) O->s[t * d + j] = (float)ss64[j];
        } else {
            for (int j = 0; j < d; ++j) ss64[j] = 0.0;
        }
        /* step 3: up-projection (plus the shared expert's output) */
        for (int j = 0; j < d; ++j) {
            const float *wr = L->w_up + (int64_t)j * l;
            double s = 0.0;
            for (int i = 0; i < l; ++i) s += cin[i] * (double)wr[i];
            s += ss64[j];
            if (O->y64) O->y64[t * d + j] = s;
            if (O->y) O->y[t * d + j] = (float)(J->quant ? oracle_round_bf16(s) : s);
        }
    }
    free(z64); free(zf); free(zc); free(zs); free(lg); free(idx); free(w64); free(wf);
    free(u64); free(hf); free(hc); free(hs); free(c64); free(cin);
    free(sxq); free(shq); free(shf); free(sh64); free(ss64);
}

int oracle_layer_forward(const oracle_layer *L, const float *x, int64_t T, int quant,
                         oracle_out *out, int nthreads) {
    pthread_once(&g_once, init_tables);
    layer_job J;
    memset(&J, 0, sizeof(J));
    J.L = L; J.x = x; J.quant = quant; J.out = out;
    J.amax_z = L->amax_z; J.amax_h = L->amax_h;
    parallel_for(T, nthreads, layer_rows, &J);
    if (out->counts) {
        /* counts need idx; recompute from the router when idx was not requested */
        memset(out->counts, 0, sizeof(int32_t) * L->E);
        if (out->idx) {
            for (int64_t i = 0; i < T * L->k; ++i) out->counts[out->idx[i]]++;
        } else {
            int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * T * L->k);
            oracle_router(x, T, L->d, L->w_router, L->b_router, L->E, L->k, NULL, idx, NULL,
                          out->counts, nthreads);
            free(idx);
        }
    }
    return J.error ? -1 : 0;
}

/* The NVFP4 layer (quant = 1) with each token's zq given: the steps after the quantization */
/* of z (routing on x, the latent experts, the combine, the up-projection, the shared       */
/* expert) applied to zq_codes [T][l/2] / zq_sf [T][l/16].  z = bf16(x Wd^T) is the bf16     */
/* rounding of a sum whose fp32 accumulation order the method leaves open, so a z one bf16   */
/* ulp away from this oracle's (its sum is exact) is as correct, and so is its              */
/* quantization; this entry point gives the layer's output for such a zq.                    */
int oracle_layer_forward_zq(const oracle_layer *L, const float *x, const uint8_t *zq_codes,
                            const uint8_t *zq_sf, int64_t T, oracle_out *out, int nthreads) {
    pthread_once(&g_once, init_tables);
    if (!zq_codes || !zq_sf) return -1;
    layer_job J;
    memset(&J, 0, sizeof(J));
    J.L = L; J.x = x; J.quant = 1; J.out = out;
    J.amax_z = L->amax_z; J.amax_h = L->amax_h;
    J.zq_codes_in = zq_codes; J.zq_sf_in = zq_sf;
    parallel_for(T, nthreads, layer_rows, &J);
    if (out->counts && out->idx) {
        memset(out->counts, 0, sizeof(int32_t) * L->E);
        for (int64_t i = 0; i < T * L->k; ++i) out->counts[out->idx[i]]++;
    }
    return J.error ? -1 : 0;
}

/* Calibration ([HEIDI]: static scales from a calibration pass on synthetic prompts):     */
/* amax_z = max |z| over the batch; then with zq quantized by that amax, amax_h = max |h|.*/
int oracle_calibrate(const oracle_layer *L, const float *x, int64_t T,
                     float *amax_z, float *amax_h, int nthreads) {
    pthread_once(&g_once, init_tables);
    /* amax_z: the down-projection alone */
    float mz = 0.0f;
    for (int64_t t = 0; t < T; ++t) {
        const float *xt = x + t * L->d;
        for (int j = 0; j < L->l; ++j) {
            const float *wr = L->w_down + (int64_t)j * L->d;
            double s = 0.0;
            for (int i = 0; i < L->d; ++i) s += (double)xt[i] * (double)wr[i];
            float v = (float)fabs(oracle_round_bf16(s));
            if (v > mz) mz = v;
        }
    }
    /* amax_h: the quantized layer with amax_z fixed, recording max |h| per token */
    float *seen_h = (float *)calloc((size_t)T, sizeof(float));
    oracle_out none;
    memset(&none, 0, sizeof(none));
    oracle_layer Lc = *L;
    Lc.shared_ffn = 0;          /* the shared expert does not feed z or h */
    layer_job J;
    memset(&J, 0, sizeof(J));
    J.L = &Lc; J.x = x; J.quant = 1; J.out = &none;
    J.amax_z = mz; J.amax_h = 1.0f; J.amax_h_seen = seen_h;
    parallel_for(T, nthreads, layer_rows, &J);
    float mh = 0.0f;
    for (int64_t t = 0; t < T; ++t) if (seen_h[t] > mh) mh = seen_h[t];
    *amax_z = mz; *amax_h = mh;
    free(seen_h);
    return J.error ? -1 : 0;
}

/* Element-wise conversions over arrays (used by the exhaustive conversion checks). */
typedef struct { const float *v; uint8_t *out; int fmt; } conv_job;
static void conv_rows(int64_t b, int64_t e, void *arg) {
    conv_job *j = (conv_job *)arg;
    if (j->fmt == 0) for (int64_t i = b; i < e; ++i) j->out[i] = oracle_f32_to_e2m1(j->v[i]);
    else             for (int64_t i = b; i < e; ++i) j->out[i] = oracle_f32_to_e4m3(j->v[i]);
}
void oracle_f32_to_e2m1_array(const float *v, int64_t n, uint8_t *out, int nthreads) {
    conv_job j = {v, out, 0};
    parallel_for(n, nthreads, conv_rows, &j);
}
void oracle_f32_to_e4m3_array(const float *v, int64_t n, uint8_t *out, int nthreads) {
    conv_job j = {v, out, 1};
    parallel_for(n, nthreads, conv_rows, &j);
}
