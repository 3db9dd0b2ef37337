/*
 * lmoe.h -- C ABI of liblmoe.so: the LatentMoE expert layer forward on one B300 (sm_103a).
 *
 * The layer (shengxinai.com Nemotron 3 blog, section 2.2 "LatentMoE：在潜空间中重构专家网络",
 * steps 1-3; "Nemotron 3 Super" page, section "潜在MoE"):
 *     z  = bf16(x Wd^T)                       down-projection d -> l (l = d/4), BF16
 *     route x to the top-k of E experts       (NVIDIA AI releases Nemotron 3 Ultra: 512 / top-22)
 *     per selected expert, in latent space:   u = zq W1q_e^T, h = bf16(relu(u)^2), o = hq W2q_e^T
 *                                             (NVFP4 weights and activations)
 *     c  = bf16(sum_j w_j o_j)                routing-weighted combine
 *     y  = bf16(c Wu^T [+ s])                 up-projection l -> d, BF16
 * and, optionally, a shared expert on x at the full width d (same blog, section 2.2, closing
 * remark) in FP8 E4M3 with per-tensor scales (NVIDIA AI releases Nemotron 3 Ultra,
 * quantization paragraph: FP8 shared expert):
 *     s  = bf16(s_h s_w2 (q8(h) Ws2q^T)),  h = bf16(relu(s_x s_w1 (q8(x) Ws1q^T))^2)
 * NVFP4 (same blog, section 3.1.1): E2M1 elements, one E4M3 scale per 16 contiguous
 * contraction-axis elements, one FP32 tensor scale.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers unless the argument says "host".
 *  - Matrices are row-major; weights follow y = x W^T (rows = output features), so every
 *    operand is contiguous along its contraction axis.
 *  - NVFP4 codes are packed two per byte, the even element in the low nibble; block scales
 *    are E4M3 bytes, one per 16 elements along the contraction axis.
 *  - Calls return a status and never abort, exit or throw.  Argument errors are detected on
 *    the host before anything is launched.  Launched work is asynchronous on `stream`;
 *    device-side errors (a bounded wait that ran out) latch into the context's error word and
 *    are reported (and cleared) by the calls that synchronize: lmoe_check() and
 *    lmoe_forward_host().  The asynchronous calls (lmoe_route, lmoe_route_static,
 *    lmoe_forward) never read device memory, so they cannot report them.
 *  - Every wait inside a kernel is bounded.  The GEMM pipeline waits give up after the
 *    context's wait limit (lmoe_set_wait_limit; default about 1 s of SM clock), record
 *    LMOE_ETIMEOUT, drain the kernel's outstanding copies and tensor-core work (with the
 *    default bound) and return; the forward's outputs are then undefined, the context stays
 *    usable and the next forward is unaffected.
 *  - Fault injection for tests of the error paths (read from the environment by each call):
 *    LMOE_FAULT=alloc:N makes the call's N-th device allocation fail (LMOE_ENOMEM, nothing
 *    leaked); LMOE_FAULT=launch:N makes the call's N-th kernel launch fail before it launches
 *    (LMOE_ECUDA); LMOE_FAULT=wait makes lmoe_forward's latent-up GEMM wait on a barrier that
 *    nothing arrives at, so the wait runs out and lmoe_check() returns LMOE_ETIMEOUT.
 *    LMOE_WAIT_LIMIT_CYCLES=n (read by lmoe_create) sets the new context's wait limit.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - The caller owns every buffer it passes; the context owns the quantized weights.
 *  - A context must not run two forwards at once on overlapping workspaces.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *lmoe_stream;   /* == cudaStream_t */

typedef enum {
    LMOE_OK = 0,
    LMOE_EINVAL = 1,        /* bad argument (detected on the host, nothing launched)      */
    LMOE_ENOMEM = 2,        /* device allocation failed, or workspace too small           */
    LMOE_ECUDA = 3,         /* a CUDA runtime/driver call failed                          */
    LMOE_EUNSUPPORTED = 4,  /* device is not sm_103a / sm_100-family, or shape unsupported */
    LMOE_ETIMEOUT = 5,      /* a bounded device-side wait ran out (kernel returned early) */
    LMOE_EDEVICE = 6        /* a device-side check failed (error word set)                */
} lmoe_status;

typedef enum { LMOE_BF16 = 0, LMOE_FP32 = 1 } lmoe_dtype;

typedef struct lmoe_ctx lmoe_ctx;   /* opaque, owned by the library */

/* Weights handed to lmoe_create.  All DEVICE pointers, caller-owned, read only during
 * lmoe_create (the context keeps its own quantized / copied versions). */
typedef struct {
    const void  *w_down;    /* bf16 [l][d]        z = x w_down^T            (BF16, kept)      */
    const void  *w_up;      /* bf16 [d][l]        y = c w_up^T              (BF16, kept)      */
    const float *w_router;  /* fp32 [E][d]        logits = x w_router^T + b                   */
    const float *b_router;  /* fp32 [E] or NULL   router bias (used for selection and weights)*/
    const void  *w1;        /* bf16 [E][ffn][l]   latent-up expert masters, quantized at create */
    const void  *w2;        /* bf16 [E][l][ffn]   latent-down expert masters, quantized at create */
    float amax_z;           /* static amax of z (calibration); > 0                           */
    float amax_h;           /* static amax of h (calibration); > 0                           */
    /* Optional shared expert (ws1 == NULL: none).  Quantized to FP8 E4M3 at create, one FP32
     * tensor scale per matrix from its amax (s_dec = amax / 448).                            */
    const void  *ws1;       /* bf16 [shared_ffn][d]  h = relu(x ws1^T)^2                        */
    const void  *ws2;       /* bf16 [d][shared_ffn]  s = h ws2^T                                */
    int shared_ffn;         /* multiple of 64 when ws1 != NULL                                */
    float amax_xs;          /* static amax of x for its FP8 quantization (calibration); > 0    */
    float amax_hs;          /* static amax of the shared h (calibration); > 0                 */
    /* Expert weight blocks: 0 = one E4M3 scale per 1 x 16 contraction elements; 1 = one scale
     * per 16 output rows x 16 contraction elements (two-dimensional weight blocks, NVIDIA AI
     * releases Nemotron 3 Ultra, architecture paragraph).  The GEMMs are the same: a 2-D
     * block's scale is stored for each of its 16 rows. */
    int weight_blocks_2d;
    /* Expert arithmetic: 0 = W4A4 (z and h quantized to NVFP4, native FP4 MMAs); 1 = W4A16
     * (NVIDIA AI releases Nemotron 3 Ultra, quantization paragraph: the Hopper form of the
     * checkpoint): NVFP4 weights decoded to bf16 on chip (in tensor memory at T <= 32, in
     * shared memory above) and bf16 z and h, with
     * u = s_w1 (z . dq(W1q)), h = bf16(relu(u)^2), o = s_w2 (h . dq(W2q)). */
    int expert_w4a16;
} lmoe_weights;

/* Create a layer context: validates the dims, allocates the context buffers, quantizes every
 * expert matrix to NVFP4 (one FP32 tensor scale per expert per matrix, computed from its amax)
 * and lays the block scales out for the tensor cores; synchronizes `stream` once at the end.
 * Dims: d, l and ffn multiples of 64; d <= 16384; l <= 4096; 1 <= k <= 32; k <= E <= 1024; E % 4 == 0;
 * with a shared expert, shared_ffn a multiple of 64 and amax_xs, amax_hs > 0.
 * (The Ultra layer: d = 8192, l = 2048, E = 512, k = 22; ffn is not given by the pages.)
 * Errors: LMOE_EINVAL (dims / NULL pointers / amax <= 0), LMOE_ENOMEM, LMOE_ECUDA,
 * LMOE_EUNSUPPORTED (device is not compute capability 10.3). */
lmoe_status lmoe_create(int d, int l, int E, int k, int ffn, const lmoe_weights *w,
                        lmoe_stream stream, lmoe_ctx **out);

/* NVFP4 quantization (blog section 3.1.1) of a row-major [rows][K] tensor along K.
 *   src          device, bf16 or fp32 per `dt`
 *   amax         tensor amax; < 0: computed on the device from src
 *   codes        device uint8 [rows][K/2]    (even element in the low nibble)
 *   sf           device uint8 [rows][K/16]   E4M3 block scales, row-major
 *   tensor_scale device float [1]            the FP32 decode scale amax/2688 (1 if amax == 0)
 * Arithmetic (fp32, round-to-nearest-even): s_enc = 2688/amax, s_dec = amax/2688;
 * sf = e4m3_satfinite(amax_block * (s_enc/6)); q = e2m1_satfinite(x * (1/(value(sf)*s_dec))),
 * q = +-0 where value(sf)*s_dec == 0.  K % 16 == 0, rows >= 0 (0 is a no-op). */
lmoe_status lmoe_quantize_nvfp4(const void *src, lmoe_dtype dt, int64_t rows, int64_t K,
                                float amax, uint8_t *codes, uint8_t *sf, float *tensor_scale,
                                lmoe_stream stream);

/* The same with two-dimensional blocks: one E4M3 scale per 16 rows x 16 elements of K, from
 * the block's amax, written to each of the block's 16 rows of sf (so sf has the layout above).
 * rows % 16 == 0, K % 16 == 0. */
lmoe_status lmoe_quantize_nvfp4_2d(const void *src, lmoe_dtype dt, int64_t rows, int64_t K,
                                   float amax, uint8_t *codes, uint8_t *sf, float *tensor_scale,
                                   lmoe_stream stream);

/* FP8 E4M3 quantization with one FP32 per-tensor scale (the shared expert's format):
 *   src          device, bf16 or fp32 per `dt`, n elements (n % 16 == 0, n >= 0; 0 is a no-op)
 *   amax         tensor amax; < 0: computed on the device from src
 *   codes        device uint8 [n]
 *   tensor_scale device float [1]   the FP32 decode scale amax/448 (1 if amax == 0)
 * Arithmetic (fp32, round-to-nearest-even): s_enc = 448/amax; code = e4m3_satfinite(x * s_enc);
 * every code is 0 when amax == 0. */
lmoe_status lmoe_quantize_fp8(const void *src, lmoe_dtype dt, int64_t n, float amax,
                              uint8_t *codes, float *tensor_scale, lmoe_stream stream);

/* Routing alone (top-k of E per token, NVIDIA AI releases Nemotron 3 Ultra, architecture):
 *   x       device bf16 [T][d]
 *   idx     device int32 [T][k]  selected experts, ascending expert id per token
 *   w       device float [T][k]  softmax over the k selected logits, same order as idx
 *   counts  device int32 [E]     tokens per expert (may be NULL)
 * The selection is the one the canonical fp32 logits make (64-element fma chunks; chunk
 * partials added left to right in groups of 16; group sums added left to right; then the
 * bias), so idx and counts are exact.  T <= 64: every canonical logit is computed.  T > 64:
 * tensor-core logits (bf16 hi/lo split of the weights, fp32 accumulation) bound every canonical
 * logit within a certified margin, and the canonical logits of the candidates the margin
 * leaves undecided are computed exactly; w is then the softmax of the selected logits as known
 * (canonical where computed, tensor-core otherwise: within about 1e-5 relative).  Uses context-owned scratch
 * (grown with cudaMallocAsync on first use for a larger T).  T >= 0; x and counts 16-byte
 * aligned (LMOE_EINVAL otherwise, before anything is launched). */
lmoe_status lmoe_route(lmoe_ctx *ctx, const void *x, int64_t T, int32_t *idx, float *w,
                       int32_t *counts, lmoe_stream stream);

/* Allocation-free routing.  The paper has no counterpart: this is a deployment convenience.
 * Some callers cannot allocate device memory at the moment they route: code running inside an
 * allocator or memory-pool callback (where re-entering the allocator can deadlock), serving
 * loops whose device memory is fixed at start-up, and hosts that embed the library without
 * handing it any allocator.  lmoe_route may grow a context-owned scratch with cudaMallocAsync;
 * lmoe_route_static never allocates or frees.  It has lmoe_route's arguments and results, but
 * keeps the router's scratch (fp32 group sums, T x E x ceil(d/1024), when T <= 64; fp32
 * logits, T x E, above) in one fixed array of LMOE_ROUTE_STATIC_SCRATCH_BYTES compiled into
 * liblmoe.so, which every GPU that loads the library holds until the process exits.
 *   - That scratch must fit in LMOE_ROUTE_STATIC_SCRATCH_BYTES (at d = 8192, E = 512: every
 *     T <= 8192); a larger T returns LMOE_EINVAL before anything is launched.
 *   - The first call on a device looks up the array's device address (once per device, with
 *     that device current; the context's device must be current).  Make that first call before
 *     any CUDA stream capture.  The address is cached with the device's current CUDA context;
 *     after a device reset (or a released and re-created primary context) the first call in
 *     the new context looks it up again, so that call too must come before any capture.
 *   - x and counts must be 16-byte aligned (LMOE_EINVAL otherwise, before anything launches).
 *   - Every call on a device shares the one array, and it keeps the last call's contents.  The
 *     scratch is fully written before it is read, and `counts` is zeroed by the call, so no
 *     earlier contents leak into a result; but two calls whose kernels overlap on the GPU (on
 *     different streams, or from different contexts of one device) race on the array: order
 *     such calls on one stream or with events. */
#define LMOE_ROUTE_STATIC_SCRATCH_BYTES (16u << 20)
lmoe_status lmoe_route_static(lmoe_ctx *ctx, const void *x, int64_t T, int32_t *idx, float *w,
                              int32_t *counts, lmoe_stream stream);

/* Bytes of device workspace lmoe_forward needs for T tokens (256-byte aligned pointer). */
size_t lmoe_workspace_size(const lmoe_ctx *ctx, int64_t T);

/* The layer forward: x device bf16 [T][d] -> y device bf16 [T][d].  No host synchronization
 * and no host read of device data.  Work is launched on `stream` and, for small T, partly on a
 * context-owned second stream that forks from `stream` and joins back into it with events, so
 * the whole call is ordered after earlier work on `stream`, later work on `stream` is ordered
 * after it, and it can be captured in a CUDA graph.
 * ws: device workspace of at least lmoe_workspace_size(ctx, T) bytes.
 * Errors: LMOE_EINVAL (NULL / T < 0), LMOE_ENOMEM (ws_bytes too small), LMOE_ECUDA. */
lmoe_status lmoe_forward(lmoe_ctx *ctx, const void *x, int64_t T, void *y, void *ws,
                         size_t ws_bytes, lmoe_stream stream);

/* Bytes of device workspace lmoe_forward_host needs (lmoe_workspace_size + x and y staging). */
size_t lmoe_host_workspace_size(const lmoe_ctx *ctx, int64_t T);

/* The forward from and to HOST memory: copies x_host (bf16 [T][d], pinned for best speed) to
 * the device, runs lmoe_forward, copies y back to y_host and synchronizes `stream`.  On a
 * created (non-default) stream the three steps, and a copy of the context's error word to
 * pinned host memory (read after the synchronization), are captured as one CUDA graph, kept in the
 * context and replayed by later calls with the same T, x_host, y_host, ws, ws_bytes, stream,
 * debug flag and wait limit (the host buffers' contents are read and written at each
 * replay); any other call captures anew.  A call with LMOE_FAULT set runs the steps directly
 * and keeps the cached graph.  If the capture is refused (e.g. pageable host memory) the steps run
 * directly.  The legacy and per-thread default streams, and profiling mode, run directly.
 * The call synchronizes `stream`, so a stream that is being captured is refused with
 * LMOE_EINVAL before anything is enqueued.  After the synchronize it reads the context's
 * error word: a device-side error of this forward returns LMOE_ETIMEOUT / LMOE_EDEVICE. */
lmoe_status lmoe_forward_host(lmoe_ctx *ctx, const void *x_host, int64_t T, void *y_host,
                              void *ws, size_t ws_bytes, lmoe_stream stream);

/* Intermediates of the last lmoe_forward, as byte ranges of its workspace (for parity checks).
 * Stage ids: see lmoe_stage.  Returns LMOE_EINVAL for an unknown stage. */
typedef enum {
    LMOE_STAGE_IDX = 0,      /* int32 [T][k]                                           */
    LMOE_STAGE_W = 1,        /* float [T][k]                                           */
    LMOE_STAGE_COUNTS = 2,   /* int32 [E]                                              */
    LMOE_STAGE_ZQ_CODES = 3, /* uint8 [T][l/2]                                         */
    LMOE_STAGE_ZQ_SF = 4,    /* uint8 [T][l/16]   row-major E4M3                       */
    LMOE_STAGE_C = 5,        /* bf16  [T][l]      combine output                       */
    LMOE_STAGE_Z = 6,        /* bf16  [T][l]      debug mode only                       */
    LMOE_STAGE_ROWS = 7,     /* int32 [R] slot (token*k + j) of each permuted row, -1 = pad */
    LMOE_STAGE_H = 8,        /* bf16  [R][ffn]    permuted rows; W4A4: debug mode only  */
    LMOE_STAGE_HQ_CODES = 9, /* uint8 [R][ffn/2]  permuted rows (W4A4 only)             */
    LMOE_STAGE_HQ_SF = 10,   /* uint8 [R/128][ffn/64][512] tensor-core scale atoms (W4A4) */
    LMOE_STAGE_NROWS = 11,   /* int32 [1]         R actually used                       */
    LMOE_STAGE_XS_Q = 12,    /* uint8 [T][d]      shared expert: E4M3 codes of x        */
    LMOE_STAGE_HS = 13,      /* bf16  [T][shared_ffn] shared expert h, debug mode only   */
    LMOE_STAGE_HS_Q = 14,    /* uint8 [T][shared_ffn] shared expert: E4M3 codes of h     */
    LMOE_STAGE_S = 15,       /* bf16  [T][d]      shared expert output s                */
    LMOE_STAGE_ROUTER = 16   /* fp32  router scratch: T > 64: tensor-core logits [T][E]
                                without the bias; T <= 64: group sums [T][E][d/1024]   */
} lmoe_stage;
lmoe_status lmoe_workspace_range(const lmoe_ctx *ctx, int64_t T, int stage, size_t *offset,
                                 size_t *bytes);

/* Debug mode (0/1): when on, lmoe_forward also writes z and h (bf16) into its workspace,
 * which then needs lmoe_workspace_size() bytes computed after this call. */
lmoe_status lmoe_set_debug(lmoe_ctx *ctx, int on);

/* Wait limit of the GEMM pipeline waits, in SM clock cycles (cycles <= 0: the default, about
 * 1 s at the maximum SM clock).  A wait that runs out makes its kernel record LMOE_ETIMEOUT in
 * the context's error word and return early (see the conventions at the top).  The waits that
 * drain a kernel's in-flight copies and tensor-core work before it exits keep the default
 * bound.  Applies to the forwards launched after the call. */
lmoe_status lmoe_set_wait_limit(lmoe_ctx *ctx, long long cycles);

/* Copy expert e's quantized matrix (which = 1: W1 [ffn][l], which = 2: W2 [l][ffn]) out of the
 * context in the canonical layout: codes device uint8 [N][K/2], sf device uint8 [N][K/16]
 * row-major, *s_dec (host) its FP32 tensor scale.  Synchronizes `stream`. */
lmoe_status lmoe_get_expert_nvfp4(const lmoe_ctx *ctx, int which, int e, uint8_t *codes,
                                  uint8_t *sf, float *s_dec, lmoe_stream stream);

/* Copy the shared expert's quantized matrix (which = 1: Ws1 [shared_ffn][d], which = 2: Ws2
 * [d][shared_ffn]) out of the context: codes device uint8, *s_dec (host) its FP32 tensor
 * scale.  LMOE_EINVAL if the context has no shared expert.  Synchronizes `stream`. */
lmoe_status lmoe_get_shared_fp8(const lmoe_ctx *ctx, int which, uint8_t *codes, float *s_dec,
                                lmoe_stream stream);

/* Number of kernels one lmoe_forward(ctx, ..., T, ...) launches (it depends on T only through
 * the split-K plan of the two projections; a shared expert adds three). */
int lmoe_forward_kernel_count(const lmoe_ctx *ctx, int64_t T);

/* Per-kernel timing of lmoe_forward.  When on, lmoe_forward records a CUDA event on its stream
 * before its first kernel and after every kernel it launches (do not capture a forward into a
 * CUDA graph while this is on).  lmoe_profile_read synchronizes on the last event and writes,
 * for the last forward, each kernel's name (static strings) and duration in milliseconds, in
 * launch order; it returns the number written (<= max), or -1 if nothing was recorded. */
lmoe_status lmoe_set_profile(lmoe_ctx *ctx, int on);
int lmoe_profile_read(lmoe_ctx *ctx, const char **names, float *ms, int max);

/* Synchronize `stream` and report (and clear) the context's device error word. */
lmoe_status lmoe_check(lmoe_ctx *ctx, lmoe_stream stream);

/* Static description of a status code. */
const char *lmoe_status_string(lmoe_status s);

/* Free the context (synchronizes the device once).  NULL is a no-op. */
void lmoe_destroy(lmoe_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif
