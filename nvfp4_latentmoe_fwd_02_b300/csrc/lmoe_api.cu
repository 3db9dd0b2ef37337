// lmoe_api.cu -- host side of liblmoe.so: the C ABI declared in include/lmoe.h.
//
// The LatentMoE expert layer forward (shengxinai.com Nemotron 3 blog, section 2.2, steps 1-3):
// down-projection d -> l, routing on x, NVFP4 latent experts, weighted combine, up-projection,
// plus the optional FP8 shared expert at width d whose output joins the up-projection.
// The host code validates arguments, lays out the workspace, encodes TMA descriptors and
// launches the kernels of this directory on the caller's stream; it never synchronizes or
// reads device memory inside lmoe_forward.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>

#include "lmoe.h"   // include/ (on the include path)
#include "common.cuh"
#include "fp8.cuh"
#include "gemm.cuh"
#include "moe.cuh"
#include "nvfp4.cuh"
#include "router.cuh"
#include "w4dec.cuh"

using namespace lmoe;

namespace {

// NVFP4 prefill, latent-up: 128 x 256 tiles, one N = 256 MMA per K step (each tcgen05.mma
// costs its issuing thread ~85 cycles whatever its N, so wider MMAs feed the tensor core
// faster); one accumulator, one 128-byte column block (54 KB with the scale atoms) per stage,
// four stages.
constexpr int kKbF4Up = 1;
constexpr int kStagesF4 = 4;
constexpr int kBNF4Up = 256;
// NVFP4 prefill, latent-down: 128 x 256 tiles like the latent-up, three 54 KB stages + 32 KB
// of combine staging (8 epilogue warps x 4 KB)
constexpr int kKbF4Dn = 1;
constexpr int kStagesF4Stg = 3;
constexpr bool kStgF4Dn = true;
constexpr int kBNF4Dn = 256;
constexpr int kStagesBF16 = 6;
constexpr int kStagesF4Small = 4;     // decode (T <= 32): 4 KB A boxes, 2 column blocks per stage
constexpr int kStagesBF16Small = 5;
constexpr int kStagesF8 = 6;          // FP8 stages have the BF16 byte layout
constexpr int kStagesF8Small = 5;
constexpr int kStagesWide = 4;        // bf16 / fp8 with 256-column tiles: 48 KB per stage
constexpr int kBNWide = 256;
constexpr int kBNNarrow = 64;         // bf16 GEMMs at decode whose 128-column tiles leave SMs idle
constexpr int kStagesW4 = 5;          // W4A16 above decode: bf16 A + decoded bf16 B + raw E2M1 block per stage
constexpr int kSmallAMaxT = 32;
// up-projection at T <= 8 reading the fp32 combine accumulator (A staged as fp32, 4 KB more per
// stage): 64-column tiles 6 stages, 128-column tiles 4
constexpr int kStagesUpF32N = 6, kStagesUpF32W = 4;
constexpr int kUpF32MaxT = 8;
constexpr int64_t kSharedFirstMaxT = 1;   // forking forwards up to this T put the shared expert first

inline int kb_for(bool small_a) { return small_a ? 2 : 1; }   // column blocks per stage
// tile width of the dense (bf16 / fp8) GEMMs: 256 outside decode (fewer operand bytes per output)
inline int bn_for(bool small_a) { return small_a ? 128 : 256; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D K-major operand: `inner` elements per row (contiguous), `rows` rows, row pitch in bytes.
// Box: one 128-byte swizzle row by `box_rows` rows (128 for weights, 32 for activations).
bool make_map(CUtensorMap *m, bool bf16, const void *ptr, uint64_t inner, uint64_t rows,
              uint64_t pitch_bytes, uint32_t box_rows = 128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {bf16 ? 64u : 128u, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                    const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// fp32 [rows][inner] map, unswizzled, box of 64 elements (256 bytes) x box_rows.
bool make_map_f32(CUtensorMap *m, const float *ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Raw (unswizzled) byte map of E2M1 weight codes [rows][K/2] for the W4A16 decoders: a box
// of 32 bytes (64 elements) by 128 rows lands in smem as [128][32].
bool make_map_raw(CUtensorMap *m, const void *ptr, uint64_t inner_bytes, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner_bytes, rows};
    cuuint64_t strides[1] = {inner_bytes};
    cuuint32_t box[2] = {32u, 128u};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ---------------------------------------------------------------------------------------
// Host-side fault injection (for tests of the error paths; nothing here touches the GPU):
// the environment variable LMOE_FAULT, read at the start of each create / route / forward
// call, selects one failure for that call:
//   alloc:N   the call's N-th device allocation fails as if the device were out of memory
//   launch:N  the call's N-th kernel launch fails before anything is launched
//   wait      the forward's latent-up GEMM makes one pipeline wait on a barrier nothing
//             arrives at, so that wait runs out after the context's wait limit and the
//             kernel takes its timeout path (LMOE_ETIMEOUT from lmoe_check)
// ---------------------------------------------------------------------------------------
enum FaultKind { kFaultNone = 0, kFaultAlloc = 1, kFaultLaunch = 2, kFaultWait = 3 };
struct Fault {
    int kind = kFaultNone;
    int n = 0;
};
Fault read_fault() {
    Fault f;
    const char *e = std::getenv("LMOE_FAULT");
    if (!e) return f;
    if (std::strncmp(e, "alloc:", 6) == 0) { f.kind = kFaultAlloc; f.n = std::atoi(e + 6); }
    else if (std::strncmp(e, "launch:", 7) == 0) { f.kind = kFaultLaunch; f.n = std::atoi(e + 7); }
    else if (std::strcmp(e, "wait") == 0) f.kind = kFaultWait;
    if ((f.kind == kFaultAlloc || f.kind == kFaultLaunch) && f.n <= 0) f.kind = kFaultNone;
    return f;
}
// Launches left before the injected launch failure in this thread's current call (0: none).
thread_local int t_launch_fault = 0;
// Allocations left before the injected allocation failure in this thread's current call.
thread_local int t_alloc_fault = 0;
inline bool injected_launch_failure() { return t_launch_fault > 0 && --t_launch_fault == 0; }
// Arms the call's injected failures from LMOE_FAULT and disarms them when the call returns.
struct FaultScope {
    Fault f;
    FaultScope() : f(read_fault()) {
        t_launch_fault = f.kind == kFaultLaunch ? f.n : 0;
        t_alloc_fault = f.kind == kFaultAlloc ? f.n : 0;
    }
    ~FaultScope() { t_launch_fault = 0; t_alloc_fault = 0; }
};
// cudaMalloc / cudaMallocAsync with the injected allocation failure.
template <typename T>
cudaError_t dev_malloc(T **p, size_t bytes) {
    if (t_alloc_fault > 0 && --t_alloc_fault == 0) return cudaErrorMemoryAllocation;
    return cudaMalloc(reinterpret_cast<void **>(p), bytes);
}
cudaError_t dev_malloc_async(void **p, size_t bytes, cudaStream_t s) {
    if (t_alloc_fault > 0 && --t_alloc_fault == 0) return cudaErrorMemoryAllocation;
    return cudaMallocAsync(p, bytes, s);
}

// Launch with programmatic stream serialization: the kernel's CTAs may be scheduled while the
// previous kernel on the stream drains; each kernel of this library calls pdl_wait() before
// its first global access (see common.cuh), so results are the same as a plain launch.
// prio != 0: the launch's scheduling priority (a stream priority value; lower = more urgent),
// which graph capture keeps with the kernel node.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_prio(int prio, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args &&...args) {
    if (injected_launch_failure()) return cudaErrorLaunchFailure;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributePriority;
    attr[1].val.priority = prio;
    cfg.attrs = attr;
    cfg.numAttrs = prio != 0 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// The priority launch_pdl gives its kernels on this thread (0: the stream's own), set for a
// stretch of launches by PrioScope.
thread_local int t_launch_prio = 0;
struct PrioScope {
    int saved;
    explicit PrioScope(int prio) : saved(t_launch_prio) { t_launch_prio = prio; }
    ~PrioScope() { t_launch_prio = saved; }
};
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    return launch_pdl_prio(t_launch_prio, kernel, grid, block, smem, s, std::forward<Args>(args)...);
}
// The most urgent launch priority of this device (0 if it has a single priority level).
int urgent_priority() {
    static int p = [] {
        int least = 0, greatest = 0;
        return cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess ? greatest : 0;
    }();
    return p;
}
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// One NVTX range around the host side of a forward (its launches), for timeline tools.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

struct WsLayout {
    size_t idx, w, counts, seg, mt, slot_off, nrows, row_slot, router, zacc, zq_codes, zq_sf, z_dbg,
        a_codes, a_sf, h_codes, h_sf, h_dbg, c_acc, c, yacc, xs_q, hs_q, hs_dbg, s_out, a_bf16, h_bf16, total;
    int64_t R;   // row capacity of the permuted buffers (multiple of 128)
    bool small_router, split_down, split_up;
    int down_splits, up_splits;
    int up_bn;                         // tile width of the up-projection
};

}  // namespace

struct lmoe_ctx {
    int d, l, E, k, ffn;
    int dev, num_sms;
    __nv_bfloat16 *w_down, *w_up;
    float *w_router, *b_router;   // w_router in 32-expert panels [ceil(E/32)][d][32] (small-T router)
    // large-T router: bf16 planes [E][2d] (hi | lo) for the tensor-core logits, fp32 rows [E][d]
    // for the canonical recompute, per-expert norm bounds; host copies of max norm and max |b|
    __nv_bfloat16 *w_split;
    float *w_rows, *wnorm;
    float wn_max, bmax;
    CUtensorMap tm_wsplit;
    uint8_t *w1_codes, *w1_sf, *w2_codes, *w2_sf;
    float *w1_sdec, *w2_sdec, *alpha1, *alpha2;
    unsigned *amax_bits;   // [2E]
    float amax_z, amax_h;
    QScale qz, qh;
    CUtensorMap tm_wd, tm_wu, tm_w1, tm_w2;
    CUtensorMap tm_wd_w, tm_wu_w;     // 256-row boxes for the wide (256-column) tiles
    CUtensorMap tm_wu_n;              // 64-row boxes: the up-projection's narrow tiles at decode
    int w4a16;                        // experts in W4A16 form (bf16 z, h; weights decoded in smem)
    CUtensorMap tm_w1raw, tm_w2raw;   // unswizzled code maps for the W4A16 decoders
    // shared expert (FP8 E4M3, per-tensor scales); shared_ffn == 0: none
    int shared_ffn;
    uint8_t *ws1_codes, *ws2_codes;
    float ws1_sdec, ws2_sdec, amax_xs, amax_hs;
    float alpha_s1, alpha_s2, s_enc_hs;
    CUtensorMap tm_ws1, tm_ws2, tm_ws1_w, tm_ws2_w;
    unsigned *err;
    unsigned *err_host;               // pinned: the error word as lmoe_forward_host's graph copied it
    long long wait_limit;             // SM cycles a GEMM pipeline wait may take (<= 0: default)
    int debug;
    void *route_ws;
    size_t route_ws_bytes;
    // second stream: the split-K down-projection runs beside the router (fork / join events)
    cudaStream_t aux;
    cudaEvent_t ev_fork, ev_join, ev_join_s;   // ev_join_s: the shared expert, run on the second stream
    // lmoe_forward_host: its copy-in, forward and copy-out as one CUDA graph, replayed while a
    // call's arguments (and the debug flag) equal those it was captured with
    cudaGraphExec_t host_exec;
    int64_t host_T;
    const void *host_x;
    void *host_y, *host_ws;
    size_t host_ws_bytes;
    cudaStream_t host_stream;
    int host_debug;
    long long host_wait_limit;
    // per-kernel timing (lmoe_set_profile)
    int profile;
    int nprof;
    cudaEvent_t ev[33];
    const char *prof_name[32];
};

namespace {

lmoe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LMOE_OK;
    if (e == cudaErrorMemoryAllocation) return LMOE_ENOMEM;
    return LMOE_ECUDA;
}
#define LMOE_CUDA(call)                                         \
    do {                                                        \
        cudaError_t e_ = (call);                                \
        if (e_ != cudaSuccess) return cuda_status(e_);          \
    } while (0)
#define LMOE_LAUNCH()                                           \
    do {                                                        \
        cudaError_t e_ = cudaGetLastError();                    \
        if (e_ != cudaSuccess) return cuda_status(e_);          \
    } while (0)

// Split-K plan for a dense projection: spread small-M problems over the SMs.
// fill: split only while tiles * fill <= SMs (a split costs a finalize kernel and fp32
// reduction traffic; with N = d the up-projection already has enough tiles unsplit).
int plan_splits(int m_tiles, int n_tiles, int k_tiles, int num_sms, int fill = 2) {
    const int tiles = m_tiles * n_tiles;
    if (tiles * fill > num_sms) return 1;
    int s = std::max(1, num_sms / tiles);
    s = std::min(s, k_tiles);
    const int per = static_cast<int>(cdiv(k_tiles, s));
    return static_cast<int>(cdiv(k_tiles, per));
}

// Tile width of the up-projection: 64 at decode when 128-column tiles would leave more than a
// quarter of the SMs idle and 64-column ones still fit in one wave; else the dense default.
int up_bn(int64_t T, int64_t d, int num_sms) {
    if (T > kSmallAMaxT) return bn_for(false);
    const int64_t t128 = cdiv(d, kBN), t64 = cdiv(d, kBNNarrow);
    return (4 * t128 < 3 * num_sms && t64 <= num_sms) ? kBNNarrow : kBN;
}

WsLayout layout(const lmoe_ctx *c, int64_t T) {
    WsLayout L;
    std::memset(&L, 0, sizeof(L));
    const int64_t d = c->d, l = c->l, E = c->E, k = c->k, F = c->ffn;
    L.R = cdiv(T * k + E * 127, 128) * 128;
    if (L.R == 0) L.R = 128;
    L.small_router = T <= kSmallMaxT;
    const int mt = static_cast<int>(cdiv(T, 128));
    const int kb = kb_for(T <= kSmallAMaxT);
    const int bn = bn_for(T <= kSmallAMaxT);
    L.down_splits = plan_splits(mt, static_cast<int>(cdiv(l, bn)), static_cast<int>(cdiv(d / 64, kb)), c->num_sms);
    L.up_bn = up_bn(T, d, c->num_sms);
    L.up_splits = plan_splits(mt, static_cast<int>(cdiv(d, L.up_bn)), static_cast<int>(cdiv(l / 64, kb)), c->num_sms, 4);
    L.split_down = L.down_splits > 1;
    L.split_up = L.up_splits > 1;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
    L.idx = take(T * k * 4);
    L.w = take(T * k * 4);
    L.counts = take(E * 4 + 16);   // + the routing kernels' done counter (cleared with the counts)
    L.seg = take((E + 1) * 4);
    L.mt = take((E + 1) * 4);
    L.slot_off = take(T * k * 4);
    L.nrows = take(4);
    L.row_slot = take(L.R * 4);
    L.router = take(T <= kSmallMaxT ? T * cdiv(d / kChunk, kGroupChunks) * E * 4 : T * E * 4);
    L.zacc = take(L.split_down ? T * l * 4 : 0);
    L.zq_codes = take(T * l / 2);
    L.zq_sf = take(T * l / 16);
    L.z_dbg = take(c->debug || c->w4a16 ? T * l * 2 : 0);   // W4A16: the scatter copies z rows
    const bool w4 = c->w4a16 != 0;
    L.a_codes = take(w4 ? 0 : L.R * l / 2);
    L.a_sf = take(w4 ? 0 : L.R * l / 16);
    L.h_codes = take(w4 ? 0 : L.R * F / 2);
    L.h_sf = take(w4 ? 0 : L.R * F / 16);
    L.h_dbg = take(c->debug && !w4 ? L.R * F * 2 : 0);
    L.a_bf16 = take(w4 ? L.R * l * 2 : 0);
    L.h_bf16 = take(w4 ? L.R * F * 2 : 0);
    L.c_acc = take(T * l * 4);
    L.c = take(T * l * 2);
    L.yacc = take(L.split_up ? T * d * 4 : 0);
    const int64_t FS = c->shared_ffn;
    L.xs_q = take(FS ? T * d : 0);
    L.hs_q = take(T * FS);
    L.hs_dbg = take(c->debug ? T * FS * 2 : 0);
    L.s_out = take(FS ? T * d * 2 : 0);
    L.total = off;
    return L;
}

template <int KIND, bool SMALLA, int KB, int STAGES, int BN = kBN, bool STG = false>
cudaError_t set_smem_attr() {
    static_assert(gemm_smem_bytes<KIND, SMALLA, KB, BN, STG>(STAGES) <= 232448, "shared memory budget");
    return cudaFuncSetAttribute(gemm_kernel<KIND, SMALLA, KB, STAGES, BN, STG>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                gemm_smem_bytes<KIND, SMALLA, KB, BN, STG>(STAGES));
}

template <int KIND, bool SMALLA, int KB, int STAGES, int BN = kBN, bool STG = false>
cudaError_t launch_gemm_cfg(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &g, int grid,
                            cudaStream_t s) {
    return launch_pdl(gemm_kernel<KIND, SMALLA, KB, STAGES, BN, STG>, dim3(grid),
                      dim3(GemmCfg<KIND, SMALLA, KB, BN, STG>::kThreads),
                      gemm_smem_bytes<KIND, SMALLA, KB, BN, STG>(STAGES), s, ta, tb, g);
}

// small_a: every tile has at most 32 valid A rows (T <= 32); such launches use two column
// blocks per stage, and g.k_tiles must count stages of kb_for(true) blocks.
template <int KIND>
cudaError_t launch_gemm(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &g_in, int grid,
                        bool small_a, cudaStream_t s) {
    // decode launches issue their first weight stages before waiting on the previous kernel:
    // the weights are static and every grouped launch's segment tables come from the router,
    // which completed before the previous kernel of the forward began
    GemmArgs g = g_in;
    g.preload = small_a && KIND != kKindW4A16 ? 1 : 0;
    if (KIND == kKindNvf4)
        return small_a ? launch_gemm_cfg<kKindNvf4, true, 2, kStagesF4Small>(ta, tb, g, grid, s)
               : g.epi == EPI_COMBINE ? launch_gemm_cfg<kKindNvf4, false, kKbF4Dn, kStagesF4Stg, kBNF4Dn, kStgF4Dn>(ta, tb, g, grid, s)
                                      : launch_gemm_cfg<kKindNvf4, false, kKbF4Up, kStagesF4, kBNF4Up>(ta, tb, g, grid, s);
    if (KIND == kKindFp8)
        return small_a ? launch_gemm_cfg<kKindFp8, true, 2, kStagesF8Small>(ta, tb, g, grid, s)
                       : launch_gemm_cfg<kKindFp8, false, 1, kStagesWide, kBNWide>(ta, tb, g, grid, s);
    if (KIND == kKindW4A16)   // (decode: launch_w4dec)
        return small_a ? cudaErrorInvalidValue : launch_gemm_cfg<kKindW4A16, false, 1, kStagesW4>(ta, tb, g, grid, s);
    if (small_a && g.bn == kBNNarrow)
        return launch_gemm_cfg<kKindBf16, true, 2, kStagesBF16Small, kBNNarrow>(ta, tb, g, grid, s);
    return small_a ? launch_gemm_cfg<kKindBf16, true, 2, kStagesBF16Small>(ta, tb, g, grid, s)
                   : launch_gemm_cfg<kKindBf16, false, 1, kStagesWide, kBNWide>(ta, tb, g, grid, s);
}

// W4A16 expert GEMM at decode (every expert segment has at most nt <= 32 rows): tx is the bf16
// activation map with nt-row boxes, tw the expert codes' tile-order map (128-byte swizzle).
cudaError_t launch_w4dec(const CUtensorMap &tx, const CUtensorMap &tw, const GemmArgs &g_in, int grid, int nt,
                         cudaStream_t s) {
    static_assert(w4dec_smem_bytes<16>() <= 232448 && w4dec_smem_bytes<32>() <= 232448, "shared memory budget");
    GemmArgs g = g_in;
    g.preload = 1;
    g.k_tiles = static_cast<int>(cdiv(g.K, 256));   // 256-element chunks per tile
    return nt <= 16 ? launch_pdl(w4_decode_kernel<16>, dim3(grid), dim3(W4Cfg<16>::kThreads), w4dec_smem_bytes<16>(), s,
                                 tx, tw, g)
                    : launch_pdl(w4_decode_kernel<32>, dim3(grid), dim3(W4Cfg<32>::kThreads), w4dec_smem_bytes<32>(), s,
                                 tx, tw, g);
}

// K elements per 128-byte column block: 64 (bf16) or 128 (fp8).
GemmArgs dense_args(int M, int N, int K, int splits, int epi, const lmoe_ctx *c, int kb, int k_block = 64,
                    int bn = kBN) {
    GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.M = M; g.N = N; g.K = K;
    g.bn = bn;
    g.m_tiles = static_cast<int>(cdiv(M, kBM));
    g.n_tiles = static_cast<int>(cdiv(N, bn));
    g.k_tiles = static_cast<int>(cdiv(cdiv(K, k_block), kb));
    g.kt_per_split = static_cast<int>(cdiv(g.k_tiles, splits));
    g.k_splits = static_cast<int>(cdiv(g.k_tiles, g.kt_per_split));
    g.epi = epi;
    g.err = c->err;
    g.wait_limit = c->wait_limit;
    return g;
}

int grid_for(int64_t tiles, int num_sms) {
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles, num_sms)));
}

// Record the end of the kernel just launched (profiling mode only).
// Also an NVTX mark with the kernel's name (free unless a tracing tool is attached), so a
// timeline shows which stage each launch of the forward belongs to.
inline void prof_mark(lmoe_ctx *c, const char *name, cudaStream_t s) {
    nvtxMarkA(name);
    if (!c->profile || c->nprof >= 32) return;
    c->prof_name[c->nprof] = name;
    cudaEventRecord(c->ev[c->nprof + 1], s);
    ++c->nprof;
}

lmoe_status check_error_word(lmoe_ctx *c) {
    unsigned v = 0;
    if (cudaMemcpy(&v, c->err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return LMOE_ECUDA;
    if (v) cudaMemset(c->err, 0, sizeof(unsigned));
    if (v & kErrTimeout) return LMOE_ETIMEOUT;
    if (v) return LMOE_EDEVICE;
    return LMOE_OK;
}
// After a replay of lmoe_forward_host's graph has completed: its last node copied the error
// word to pinned host memory, so a clear word needs no further device round trip.
lmoe_status host_error_word(lmoe_ctx *c) {
    if (*static_cast<volatile unsigned *>(c->err_host) == 0) return LMOE_OK;
    *c->err_host = 0;
    return check_error_word(c);
}

// The router on x.  Small T: canonical chunk-group sums into `scratch`, then top-k, softmax and
// counts; the first kernel also clears the ranges in `zr`.  Large T: a clearing kernel (zr and
// the logits), tensor-core logits into `scratch` (bf16 hi/lo planes of the weights, K split
// over the SMs, fp32 reductions), then the certified selection against the canonical order.
// seg (optional, with done / mt / nrows): the routing kernel's last warp lays out the expert
// segments (done: a zeroed counter).
struct SegOut {
    int *done;
    int32_t *seg, *mt, *nrows;
};
lmoe_status launch_router(lmoe_ctx *c, const __nv_bfloat16 *x, int64_t T, float *scratch,
                          int32_t *idx, float *w, int32_t *counts, int32_t *slot_off,
                          const ZeroRanges &zr, cudaStream_t s, SegOut so = {nullptr, nullptr, nullptr, nullptr},
                          cudaEvent_t after_logits = nullptr) {
    const bool small = T <= kSmallMaxT;
    const int C = c->d / kChunk;
    const int NG = static_cast<int>(cdiv(C, kGroupChunks));
    if (small) {
        // the router and the split-K down-projection (forked stream) each want about 128 SMs
        // at the start of a forward; the router's chain (top-k, segments) is the longer one,
        // so its kernels are scheduled first
        LMOE_CUDA(launch_pdl_prio(urgent_priority(), router_small_kernel,
                             dim3(static_cast<unsigned>(cdiv(c->E, kSmallEG)), static_cast<unsigned>(cdiv(C, kSmallCG))),
                             dim3(kSmallEG * kSmallCG), kRouterSmallSmem, s, x,
                             static_cast<const float *>(c->w_router), static_cast<int>(T), c->d, c->E, scratch, zr,
                             c->err));
        prof_mark(c, "router_small", s);
        if (after_logits) LMOE_CUDA(cudaEventRecord(after_logits, s));
        LMOE_CUDA(launch_pdl_prio(urgent_priority(), router_topk_kernel, dim3(static_cast<unsigned>(T)), dim3(kTopkThreads), 0, s,
                             static_cast<const float *>(scratch), NG, static_cast<const float *>(c->b_router),
                             static_cast<int>(T), c->E, c->k, idx, w, counts, slot_off, so.done, so.seg, so.mt,
                             so.nrows));
        prof_mark(c, "router_topk", s);
        return LMOE_OK;
    }
    ZeroRanges z = zr;
    int free_slot = -1;
    for (int i = 0; i < kZeroRanges; ++i)
        if (!z.p[i] && free_slot < 0) free_slot = i;
    if (free_slot < 0) return LMOE_EINVAL;
    z.p[free_slot] = reinterpret_cast<uint4 *>(scratch);
    z.n16[free_slot] = T * c->E * 4 / 16;
    LMOE_CUDA(launch_pdl(zero_kernel, dim3(c->num_sms * 2), dim3(256), 0, s, z));
    prof_mark(c, "router_zero", s);
    const int d = c->d, E = c->E;
    CUtensorMap tx;
    if (!make_map(&tx, true, x, d, T, static_cast<uint64_t>(d) * 2, kBM)) return LMOE_ECUDA;
    const int m_tiles = static_cast<int>(cdiv(T, kBM)), n_tiles = static_cast<int>(cdiv(E, kBNWide));
    const int k_tiles = 2 * d / 64;
    const int splits = std::min<int>(k_tiles, std::max<int>(8, static_cast<int>(cdiv(2 * c->num_sms, int64_t(m_tiles) * n_tiles))));
    GemmArgs g = dense_args(static_cast<int>(T), E, 2 * d, splits, EPI_RED_F32, c, 1, 64, kBNWide);
    g.out = scratch;
    g.ld_out = E;
    g.a_kwrap = d;
    LMOE_CUDA((launch_gemm<kKindBf16>(tx, c->tm_wsplit, g, grid_for(int64_t(g.m_tiles) * g.n_tiles * g.k_splits, c->num_sms),
                                      false, s)));
    prof_mark(c, "router_approx", s);
    // accumulation bound: per K-slice 4 block steps per k-tile (+2), plus the fp32 sum of the
    // slices, each within 2^-23 of the running magnitude; times a margin of 4
    const float coef = 4.0f * static_cast<float>(4 * g.kt_per_split + 2 + g.k_splits) * 0x1p-23f;
    const dim3 sgrid(static_cast<unsigned>(cdiv(T, kSelWarps))), sblock(32 * kSelWarps);
    const float *ap = scratch;
    const float *wr = c->w_rows;
    const float *bp = c->b_router;
    if (E <= 128)
        LMOE_CUDA(launch_pdl(router_select_kernel<4>, sgrid, sblock, 0, s, ap, bp, x, wr, static_cast<int>(T), d, E,
                             c->k, coef, c->wn_max, c->bmax, idx, w, counts, slot_off, so.done, so.seg, so.mt,
                             so.nrows));
    else if (E <= 512)
        LMOE_CUDA(launch_pdl(router_select_kernel<16>, sgrid, sblock, 0, s, ap, bp, x, wr, static_cast<int>(T), d, E,
                             c->k, coef, c->wn_max, c->bmax, idx, w, counts, slot_off, so.done, so.seg, so.mt,
                             so.nrows));
    else
        LMOE_CUDA(launch_pdl(router_select_kernel<32>, sgrid, sblock, 0, s, ap, bp, x, wr, static_cast<int>(T), d, E,
                             c->k, coef, c->wn_max, c->bmax, idx, w, counts, slot_off, so.done, so.seg, so.mt,
                             so.nrows));
    prof_mark(c, "router_select", s);
    return LMOE_OK;
}

ZeroRanges zero_counts(int32_t *counts, int E) {
    ZeroRanges z;
    std::memset(&z, 0, sizeof(z));
    if (counts) { z.p[0] = reinterpret_cast<uint4 *>(counts); z.n16[0] = cdiv(E * 4, 16); }
    return z;
}

// Scratch bytes the router needs for T tokens: fp32 group sums (T <= 64) or logits.
size_t route_scratch_bytes(const lmoe_ctx *c, int64_t T) {
    return T <= kSmallMaxT ? static_cast<size_t>(T) * cdiv(c->d / kChunk, kGroupChunks) * c->E * 4
                           : static_cast<size_t>(T) * c->E * 4;
}

// ---------------------------------------------------------------------------------------
// Fixed router scratch for callers that cannot allocate (lmoe_route_static).  In host code
// `g_route_static_scratch` names a host-side stand-in, not device memory: its device address
// is looked up once per device with cudaGetSymbolAddress and that address is what the
// kernels receive.
// ---------------------------------------------------------------------------------------
__device__ __align__(256) unsigned char g_route_static_scratch[LMOE_ROUTE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
CUcontext g_static_ctx[kMaxDevices] = {};   // the context each cached address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// The device address of the fixed scratch on device `dev` (current).  Looked up once per device
// and context: a device reset (or a released and re-created primary context) reloads the
// library's module at a possibly different address, so a cached address is only reused while
// the current context is the one it was looked up in.
lmoe_status route_static_scratch(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return LMOE_EUNSUPPORTED;
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (!get) return LMOE_ECUDA;
    CUcontext cur = nullptr;
    if (get(&cur) != CUDA_SUCCESS || !cur) return LMOE_ECUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev] || g_static_ctx[dev] != cur) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_route_static_scratch);
        if (e != cudaSuccess || !p) return e != cudaSuccess ? cuda_status(e) : LMOE_ECUDA;
        g_static_ptr[dev] = p;
        g_static_ctx[dev] = cur;
    }
    *out = g_static_ptr[dev];
    return LMOE_OK;
}

}  // namespace

extern "C" {

const char *lmoe_status_string(lmoe_status s) {
    switch (s) {
    case LMOE_OK: return "ok";
    case LMOE_EINVAL: return "invalid argument";
    case LMOE_ENOMEM: return "out of device memory or workspace too small";
    case LMOE_ECUDA: return "CUDA error";
    case LMOE_EUNSUPPORTED: return "unsupported device or shape";
    case LMOE_ETIMEOUT: return "a bounded device-side wait timed out";
    case LMOE_EDEVICE: return "device-side check failed";
    }
    return "unknown status";
}

static lmoe_status quantize_nvfp4_impl(const void *src, lmoe_dtype dt, int64_t rows, int64_t K, float amax,
                                       uint8_t *codes, uint8_t *sf, float *tensor_scale, lmoe_stream stream,
                                       bool two_d) {
    if (rows < 0 || K <= 0 || K % 16 != 0 || (dt != LMOE_BF16 && dt != LMOE_FP32)) return LMOE_EINVAL;
    if (two_d && rows % 16 != 0) return LMOE_EINVAL;
    if (rows == 0) return LMOE_OK;
    if (!src || !codes || !sf || !tensor_scale) return LMOE_EINVAL;
    if (amax != amax) return LMOE_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t n = rows * K;
    const int64_t blocks = rows * (K / 16);
    const int qgrid = static_cast<int>(std::min<int64_t>(cdiv(blocks, 256), 148 * 16));
    unsigned *bits = reinterpret_cast<unsigned *>(tensor_scale);   // holds amax bits until the end
    if (amax < 0.0f) {
        LMOE_CUDA(cudaMemsetAsync(bits, 0, sizeof(unsigned), s));
        const int agrid = static_cast<int>(std::min<int64_t>(cdiv(n, 256), 148 * 8));
        if (dt == LMOE_BF16)
            amax_kernel<__nv_bfloat16><<<agrid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), n, bits);
        else
            amax_kernel<float><<<agrid, 256, 0, s>>>(static_cast<const float *>(src), n, bits);
        LMOE_LAUNCH();
    } else {
        unsigned ab;
        std::memcpy(&ab, &amax, sizeof(ab));
        LMOE_CUDA(cudaMemcpyAsync(bits, &ab, sizeof(ab), cudaMemcpyHostToDevice, s));
    }
    if (two_d) {
        const int g2 = static_cast<int>(std::min<int64_t>(cdiv(blocks / 16, 256), 148 * 16));
        if (dt == LMOE_BF16)
            quantize_rows_2d_kernel<__nv_bfloat16><<<g2, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src),
                                                                     rows, K, -1.0f, bits, codes, sf);
        else
            quantize_rows_2d_kernel<float><<<g2, 256, 0, s>>>(static_cast<const float *>(src), rows, K, -1.0f,
                                                             bits, codes, sf);
    } else if (dt == LMOE_BF16) {
        quantize_rows_kernel<__nv_bfloat16><<<qgrid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src),
                                                                 rows, K, -1.0f, bits, codes, sf);
    } else {
        quantize_rows_kernel<float><<<qgrid, 256, 0, s>>>(static_cast<const float *>(src), rows, K, -1.0f,
                                                         bits, codes, sf);
    }
    LMOE_LAUNCH();
    tensor_scale_kernel<<<1, 32, 0, s>>>(bits, 1, tensor_scale);
    LMOE_LAUNCH();
    return LMOE_OK;
}

lmoe_status lmoe_quantize_nvfp4(const void *src, lmoe_dtype dt, int64_t rows, int64_t K, float amax,
                                uint8_t *codes, uint8_t *sf, float *tensor_scale, lmoe_stream stream) {
    return quantize_nvfp4_impl(src, dt, rows, K, amax, codes, sf, tensor_scale, stream, false);
}

lmoe_status lmoe_quantize_nvfp4_2d(const void *src, lmoe_dtype dt, int64_t rows, int64_t K, float amax,
                                   uint8_t *codes, uint8_t *sf, float *tensor_scale, lmoe_stream stream) {
    return quantize_nvfp4_impl(src, dt, rows, K, amax, codes, sf, tensor_scale, stream, true);
}

lmoe_status lmoe_quantize_fp8(const void *src, lmoe_dtype dt, int64_t n, float amax, uint8_t *codes,
                              float *tensor_scale, lmoe_stream stream) {
    if (n < 0 || n % 16 != 0 || (dt != LMOE_BF16 && dt != LMOE_FP32)) return LMOE_EINVAL;
    if (n == 0) return LMOE_OK;
    if (!src || !codes || !tensor_scale) return LMOE_EINVAL;
    if (amax != amax) return LMOE_EINVAL;
    if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(codes) % 16) return LMOE_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *bits = reinterpret_cast<unsigned *>(tensor_scale);   // holds amax bits until the end
    if (amax < 0.0f) {
        LMOE_CUDA(cudaMemsetAsync(bits, 0, sizeof(unsigned), s));
        const int agrid = static_cast<int>(std::min<int64_t>(cdiv(n, 256), 148 * 8));
        if (dt == LMOE_BF16)
            amax_kernel<__nv_bfloat16><<<agrid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), n, bits);
        else
            amax_kernel<float><<<agrid, 256, 0, s>>>(static_cast<const float *>(src), n, bits);
        LMOE_LAUNCH();
    } else {
        unsigned ab;
        std::memcpy(&ab, &amax, sizeof(ab));
        LMOE_CUDA(cudaMemcpyAsync(bits, &ab, sizeof(ab), cudaMemcpyHostToDevice, s));
    }
    const int qgrid = static_cast<int>(std::min<int64_t>(cdiv(n / 16, 256), 148 * 16));
    if (dt == LMOE_BF16)
        quantize_fp8_kernel<__nv_bfloat16><<<qgrid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), n,
                                                                -1.0f, bits, codes);
    else
        quantize_fp8_kernel<float><<<qgrid, 256, 0, s>>>(static_cast<const float *>(src), n, -1.0f, bits, codes);
    LMOE_LAUNCH();
    fp8_tensor_scale_kernel<<<1, 32, 0, s>>>(bits, tensor_scale);
    LMOE_LAUNCH();
    return LMOE_OK;
}

lmoe_status lmoe_create(int d, int l, int E, int k, int ffn, const lmoe_weights *w,
                        lmoe_stream stream, lmoe_ctx **out) {
    if (!out) return LMOE_EINVAL;
    *out = nullptr;
    if (!w || !w->w_down || !w->w_up || !w->w_router || !w->w1 || !w->w2) return LMOE_EINVAL;
    if (d <= 0 || l <= 0 || ffn <= 0 || d % 64 || l % 64 || ffn % 64) return LMOE_EINVAL;
    if (l > 4096 || d > kSelMaxD) return LMOE_EINVAL;
    if (k < 1 || k > 32 || E < k || E > 1024 || E % 4) return LMOE_EINVAL;
    if (!(w->amax_z > 0.0f) || !(w->amax_h > 0.0f)) return LMOE_EINVAL;
    if (w->weight_blocks_2d != 0 && w->weight_blocks_2d != 1) return LMOE_EINVAL;
    if (w->expert_w4a16 != 0 && w->expert_w4a16 != 1) return LMOE_EINVAL;
    const bool has_shared = w->ws1 != nullptr;
    if (has_shared && (!w->ws2 || w->shared_ffn <= 0 || w->shared_ffn % 64 || !(w->amax_xs > 0.0f) ||
                       !(w->amax_hs > 0.0f)))
        return LMOE_EINVAL;
    int dev = 0;
    LMOE_CUDA(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    LMOE_CUDA(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || prop.minor != 3) return LMOE_EUNSUPPORTED;
    if (!encode_fn()) return LMOE_ECUDA;
    {
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        std::call_once(once, [] {
            cudaError_t a = set_smem_attr<kKindNvf4, false, kKbF4Up, kStagesF4, kBNF4Up>();
            if (a == cudaSuccess) a = set_smem_attr<kKindNvf4, false, kKbF4Dn, kStagesF4Stg, kBNF4Dn, kStgF4Dn>();
            cudaError_t b = set_smem_attr<kKindBf16, false, 1, kStagesBF16>();
            if (a == cudaSuccess) a = set_smem_attr<kKindNvf4, true, 2, kStagesF4Small>();
            if (b == cudaSuccess) b = set_smem_attr<kKindBf16, true, 2, kStagesBF16Small>();
            if (a == cudaSuccess) a = set_smem_attr<kKindFp8, false, 1, kStagesF8>();
            if (a == cudaSuccess) a = set_smem_attr<kKindW4A16, false, 1, kStagesW4>();
            if (a == cudaSuccess) a = set_smem_attr<kKindBf16, false, 1, kStagesWide, kBNWide>();
            if (a == cudaSuccess) a = set_smem_attr<kKindBf16, true, 2, kStagesBF16Small, kBNNarrow>();
            if (a == cudaSuccess) a = set_smem_attr<kKindFp8, false, 1, kStagesWide, kBNWide>();
            if (a == cudaSuccess) a = set_smem_attr<kKindFp8, true, 2, kStagesF8Small>();
            if (a == cudaSuccess) a = set_smem_attr<kKindBf16, true, 2, kStagesUpF32N, kBNNarrow, true>();
            if (a == cudaSuccess) a = set_smem_attr<kKindBf16, true, 2, kStagesUpF32W, kBN, true>();
            if (a == cudaSuccess)
                a = cudaFuncSetAttribute(w4_decode_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         w4dec_smem_bytes<16>());
            if (a == cudaSuccess)
                a = cudaFuncSetAttribute(w4_decode_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         w4dec_smem_bytes<32>());
            cudaError_t r = cudaFuncSetAttribute(router_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kRouterSmallSmem);
            attr_err = a != cudaSuccess ? a : (b != cudaSuccess ? b : r);
        });
        if (attr_err != cudaSuccess) return cuda_status(attr_err);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    FaultScope fault_scope;
    lmoe_ctx *c = new (std::nothrow) lmoe_ctx;
    if (!c) return LMOE_ENOMEM;
    std::memset(c, 0, sizeof(*c));
    if (const char *wl = std::getenv("LMOE_WAIT_LIMIT_CYCLES")) c->wait_limit = std::atoll(wl);
    c->d = d; c->l = l; c->E = E; c->k = k; c->ffn = ffn;
    c->dev = dev;
    c->num_sms = prop.multiProcessorCount;
    c->amax_z = w->amax_z;
    c->amax_h = w->amax_h;
    c->qz = qscale_from_amax(w->amax_z);
    c->qh = qscale_from_amax(w->amax_h);
    c->w4a16 = w->expert_w4a16;
    auto fail = [&](lmoe_status st) { lmoe_destroy(c); return st; };
#define CREATE_CUDA(call)                                   \
    do {                                                    \
        cudaError_t e_ = (call);                            \
        if (e_ != cudaSuccess) return fail(cuda_status(e_)); \
    } while (0)
    const size_t NB1 = cdiv(ffn, 128), NB2 = cdiv(l, 128);
    const size_t w1_sf_bytes = static_cast<size_t>(E) * NB1 * (l / 64) * 512;
    const size_t w2_sf_bytes = static_cast<size_t>(E) * NB2 * (ffn / 64) * 512;
    CREATE_CUDA(dev_malloc(&c->w_down, static_cast<size_t>(l) * d * 2));
    CREATE_CUDA(dev_malloc(&c->w_up, static_cast<size_t>(d) * l * 2));
    CREATE_CUDA(dev_malloc(&c->w_router, static_cast<size_t>(cdiv(E, 32)) * 32 * d * 4));
    CREATE_CUDA(dev_malloc(&c->b_router, static_cast<size_t>(E) * 4));
    CREATE_CUDA(dev_malloc(&c->w_split, static_cast<size_t>(E) * 2 * d * 2));
    CREATE_CUDA(dev_malloc(&c->w_rows, static_cast<size_t>(E) * d * 4));
    CREATE_CUDA(dev_malloc(&c->wnorm, static_cast<size_t>(E) * 4));
    const size_t w1_bytes = tiled_codes_bytes(E, ffn, l), w2_bytes = tiled_codes_bytes(E, l, ffn);
    CREATE_CUDA(dev_malloc(&c->w1_codes, w1_bytes));
    CREATE_CUDA(dev_malloc(&c->w2_codes, w2_bytes));
    CREATE_CUDA(dev_malloc(&c->w1_sf, w1_sf_bytes));
    CREATE_CUDA(dev_malloc(&c->w2_sf, w2_sf_bytes));
    CREATE_CUDA(dev_malloc(&c->w1_sdec, E * 4));
    CREATE_CUDA(dev_malloc(&c->w2_sdec, E * 4));
    CREATE_CUDA(dev_malloc(&c->alpha1, E * 4));
    CREATE_CUDA(dev_malloc(&c->alpha2, E * 4));
    CREATE_CUDA(dev_malloc(&c->amax_bits, 2 * E * 4));
    CREATE_CUDA(dev_malloc(&c->err, sizeof(unsigned)));
    CREATE_CUDA(cudaMallocHost(reinterpret_cast<void **>(&c->err_host), sizeof(unsigned)));
    *c->err_host = 0;
    CREATE_CUDA(cudaStreamCreateWithFlags(&c->aux, cudaStreamNonBlocking));
    CREATE_CUDA(cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming));
    CREATE_CUDA(cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming));
    CREATE_CUDA(cudaEventCreateWithFlags(&c->ev_join_s, cudaEventDisableTiming));
    CREATE_CUDA(cudaMemsetAsync(c->err, 0, sizeof(unsigned), s));
    CREATE_CUDA(cudaMemcpyAsync(c->w_down, w->w_down, static_cast<size_t>(l) * d * 2, cudaMemcpyDeviceToDevice, s));
    CREATE_CUDA(cudaMemcpyAsync(c->w_up, w->w_up, static_cast<size_t>(d) * l * 2, cudaMemcpyDeviceToDevice, s));
    CREATE_CUDA(cudaMemsetAsync(c->w_router, 0, static_cast<size_t>(cdiv(E, 32)) * 32 * d * 4, s));
    router_panels_kernel<<<dim3(static_cast<unsigned>(cdiv(d, 32)), static_cast<unsigned>(cdiv(E, 32))),
                           dim3(32, 8), 0, s>>>(w->w_router, E, d, c->w_router);
    CREATE_CUDA(cudaGetLastError());
    if (w->b_router)
        CREATE_CUDA(cudaMemcpyAsync(c->b_router, w->b_router, E * 4, cudaMemcpyDeviceToDevice, s));
    else
        CREATE_CUDA(cudaMemsetAsync(c->b_router, 0, E * 4, s));
    CREATE_CUDA(cudaMemcpyAsync(c->w_rows, w->w_router, static_cast<size_t>(E) * d * 4, cudaMemcpyDeviceToDevice, s));
    router_split_kernel<<<E, 256, 0, s>>>(c->w_rows, E, d, c->w_split, c->wnorm);
    CREATE_CUDA(cudaGetLastError());
    CREATE_CUDA(cudaMemsetAsync(c->w1_sf, 0, w1_sf_bytes, s));
    CREATE_CUDA(cudaMemsetAsync(c->w2_sf, 0, w2_sf_bytes, s));
    CREATE_CUDA(cudaMemsetAsync(c->amax_bits, 0, 2 * E * 4, s));
    // expert weights: per-expert amax, then quantization into codes + scale atoms
    const int64_t seg1 = static_cast<int64_t>(ffn) * l, seg2 = static_cast<int64_t>(l) * ffn;
    amax_segments_kernel<<<dim3(16, E), 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w->w1), seg1, c->amax_bits);
    amax_segments_kernel<<<dim3(16, E), 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w->w2), seg2, c->amax_bits + E);
    CREATE_CUDA(cudaGetLastError());
    const int qgrid = c->num_sms * 16;
    {
        // quantize row-major into a scratch buffer, then lay the codes out in tile order
        uint8_t *rowmajor = nullptr;
        CREATE_CUDA(dev_malloc(&rowmajor, static_cast<size_t>(E) * ffn * l / 2));
        cudaError_t qe = cudaMemsetAsync(c->w1_codes, 0, w1_bytes, s);
        if (qe == cudaSuccess) qe = cudaMemsetAsync(c->w2_codes, 0, w2_bytes, s);
        for (int m = 0; m < 2 && qe == cudaSuccess; ++m) {
            const int N = m == 0 ? ffn : l, K = m == 0 ? l : ffn;
            const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(m == 0 ? w->w1 : w->w2);
            unsigned *amax = c->amax_bits + m * E;
            uint8_t *sf = m == 0 ? c->w1_sf : c->w2_sf;
            if (w->weight_blocks_2d)
                quantize_experts_2d_kernel<<<qgrid, 256, 0, s>>>(src, E, N, K, amax, rowmajor, sf);
            else
                quantize_experts_kernel<<<qgrid, 256, 0, s>>>(src, E, N, K, amax, rowmajor, sf);
            tile_codes_kernel<<<qgrid, 256, 0, s>>>(rowmajor, E, N, K, m == 0 ? c->w1_codes : c->w2_codes);
            qe = cudaGetLastError();
        }
        if (qe == cudaSuccess) qe = cudaStreamSynchronize(s);
        const cudaError_t fe = cudaFree(rowmajor);
        CREATE_CUDA(qe);
        CREATE_CUDA(fe);
    }
    tensor_scale_kernel<<<cdiv(E, 256), 256, 0, s>>>(c->amax_bits, E, c->w1_sdec);
    tensor_scale_kernel<<<cdiv(E, 256), 256, 0, s>>>(c->amax_bits + E, E, c->w2_sdec);
    CREATE_CUDA(cudaGetLastError());
    CREATE_CUDA(cudaStreamSynchronize(s));
    // alpha_e = s_dec(activation) * s_dec(weight_e), in fp32
    {
        float *sd1 = new float[E], *sd2 = new float[E], *a1 = new float[E], *a2 = new float[E];
        cudaError_t e1 = cudaMemcpy(sd1, c->w1_sdec, E * 4, cudaMemcpyDeviceToHost);
        cudaError_t e2 = cudaMemcpy(sd2, c->w2_sdec, E * 4, cudaMemcpyDeviceToHost);
        for (int e = 0; e < E; ++e) {
            volatile float p1 = c->qz.s_dec * sd1[e];
            volatile float p2 = c->qh.s_dec * sd2[e];
            a1[e] = p1; a2[e] = p2;
        }
        cudaError_t e3 = cudaMemcpy(c->alpha1, a1, E * 4, cudaMemcpyHostToDevice);
        cudaError_t e4 = cudaMemcpy(c->alpha2, a2, E * 4, cudaMemcpyHostToDevice);
        delete[] sd1; delete[] sd2; delete[] a1; delete[] a2;
        for (cudaError_t e : {e1, e2, e3, e4})
            if (e != cudaSuccess) return fail(cuda_status(e));
    }
    // large-T router: the largest expert norm bound and the largest |bias|
    {
        float *wn = new float[E], *bb = new float[E];
        cudaError_t e1 = cudaMemcpy(wn, c->wnorm, E * 4, cudaMemcpyDeviceToHost);
        cudaError_t e2 = cudaMemcpy(bb, c->b_router, E * 4, cudaMemcpyDeviceToHost);
        c->wn_max = 0.0f;
        c->bmax = 0.0f;
        for (int e = 0; e < E; ++e) {
            c->wn_max = std::max(c->wn_max, wn[e]);
            c->bmax = std::max(c->bmax, std::fabs(bb[e]));
        }
        delete[] wn; delete[] bb;
        for (cudaError_t e : {e1, e2})
            if (e != cudaSuccess) return fail(cuda_status(e));
    }
    // shared expert: per-matrix amax, FP8 E4M3 codes, and the fp32 scale products
    if (has_shared) {
        const int FS = w->shared_ffn;
        const int64_t n = static_cast<int64_t>(FS) * d;
        c->shared_ffn = FS;
        c->amax_xs = w->amax_xs;
        c->amax_hs = w->amax_hs;
        CREATE_CUDA(dev_malloc(&c->ws1_codes, n));
        CREATE_CUDA(dev_malloc(&c->ws2_codes, n));
        unsigned *bits = c->amax_bits;   // reused: [0] ws1, [1] ws2 (the expert amax is done)
        CREATE_CUDA(cudaMemsetAsync(bits, 0, 2 * sizeof(unsigned), s));
        amax_segments_kernel<<<dim3(c->num_sms * 4, 1), 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w->ws1), n, bits);
        amax_segments_kernel<<<dim3(c->num_sms * 4, 1), 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w->ws2), n, bits + 1);
        CREATE_CUDA(cudaGetLastError());
        const int qg = static_cast<int>(std::min<int64_t>(cdiv(n / 16, 256), c->num_sms * 16));
        quantize_fp8_kernel<__nv_bfloat16><<<qg, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w->ws1), n, -1.0f,
                                                             bits, c->ws1_codes);
        quantize_fp8_kernel<__nv_bfloat16><<<qg, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(w->ws2), n, -1.0f,
                                                             bits + 1, c->ws2_codes);
        CREATE_CUDA(cudaGetLastError());
        unsigned hb[2];
        CREATE_CUDA(cudaMemcpyAsync(hb, bits, sizeof(hb), cudaMemcpyDeviceToHost, s));
        CREATE_CUDA(cudaStreamSynchronize(s));
        float a1, a2;
        std::memcpy(&a1, &hb[0], 4);
        std::memcpy(&a2, &hb[1], 4);
        c->ws1_sdec = fp8scale_from_amax(a1).s_dec;
        c->ws2_sdec = fp8scale_from_amax(a2).s_dec;
        volatile float p1 = fp8scale_from_amax(c->amax_xs).s_dec * c->ws1_sdec;
        volatile float p2 = fp8scale_from_amax(c->amax_hs).s_dec * c->ws2_sdec;
        c->alpha_s1 = p1;
        c->alpha_s2 = p2;
        c->s_enc_hs = fp8scale_from_amax(c->amax_hs).s_enc;
        if (!make_map(&c->tm_ws1, false, c->ws1_codes, d, FS, d) ||
            !make_map(&c->tm_ws2, false, c->ws2_codes, FS, d, FS) ||
            !make_map(&c->tm_ws1_w, false, c->ws1_codes, d, FS, d, kBNWide) ||
            !make_map(&c->tm_ws2_w, false, c->ws2_codes, FS, d, FS, kBNWide))
            return fail(LMOE_ECUDA);
    }
    // expert codes in tile order: rows of 128 bytes, one 128-row box per (expert, row block, column block)
    const uint64_t w1_rows = w1_bytes / 128, w2_rows = w2_bytes / 128;
    bool ok = make_map_raw(&c->tm_w1raw, c->w1_codes, 128, w1_rows) &&
              make_map_raw(&c->tm_w2raw, c->w2_codes, 128, w2_rows) &&
              make_map(&c->tm_wsplit, true, c->w_split, 2 * d, E, static_cast<uint64_t>(2 * d) * 2, kBNWide) &&
              make_map(&c->tm_wd_w, true, c->w_down, d, l, static_cast<uint64_t>(d) * 2, kBNWide) &&
              make_map(&c->tm_wu_w, true, c->w_up, l, d, static_cast<uint64_t>(l) * 2, kBNWide) &&
              make_map(&c->tm_wd, true, c->w_down, d, l, static_cast<uint64_t>(d) * 2) &&
              make_map(&c->tm_wu, true, c->w_up, l, d, static_cast<uint64_t>(l) * 2) &&
              make_map(&c->tm_wu_n, true, c->w_up, l, d, static_cast<uint64_t>(l) * 2, kBNNarrow) &&
              make_map(&c->tm_w1, false, c->w1_codes, 128, w1_rows, 128) &&
              make_map(&c->tm_w2, false, c->w2_codes, 128, w2_rows, 128);
    if (!ok) return fail(LMOE_ECUDA);
#undef CREATE_CUDA
    *out = c;
    return LMOE_OK;
}

void lmoe_destroy(lmoe_ctx *c) {
    if (!c) return;
    cudaDeviceSynchronize();
    void *ptrs[] = {c->w_down, c->w_up, c->w_router, c->b_router, c->w1_codes, c->w1_sf,
                    c->w2_codes, c->w2_sf, c->w1_sdec, c->w2_sdec, c->alpha1, c->alpha2,
                    c->amax_bits, c->err, c->route_ws, c->ws1_codes, c->ws2_codes, c->w_split,
                    c->w_rows, c->wnorm};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    for (cudaEvent_t e : c->ev)
        if (e) cudaEventDestroy(e);
    if (c->ev_fork) cudaEventDestroy(c->ev_fork);
    if (c->ev_join) cudaEventDestroy(c->ev_join);
    if (c->ev_join_s) cudaEventDestroy(c->ev_join_s);
    if (c->aux) cudaStreamDestroy(c->aux);
    if (c->host_exec) cudaGraphExecDestroy(c->host_exec);
    if (c->err_host) cudaFreeHost(c->err_host);
    delete c;
}

lmoe_status lmoe_route_static(lmoe_ctx *c, const void *x, int64_t T, int32_t *idx, float *w,
                              int32_t *counts, lmoe_stream stream) {
    if (!c || T < 0) return LMOE_EINVAL;
    if (T == 0) return LMOE_OK;
    if (!x || !idx || !w) return LMOE_EINVAL;
    if (reinterpret_cast<uintptr_t>(x) % 16 || (counts && reinterpret_cast<uintptr_t>(counts) % 16))
        return LMOE_EINVAL;
    if (route_scratch_bytes(c, T) > LMOE_ROUTE_STATIC_SCRATCH_BYTES) return LMOE_EINVAL;
    FaultScope fault_scope;
    int dev = -1;
    LMOE_CUDA(cudaGetDevice(&dev));
    if (dev != c->dev) return LMOE_EINVAL;
    void *scratch = nullptr;
    const lmoe_status st = route_static_scratch(dev, &scratch);
    if (st != LMOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return launch_router(c, static_cast<const __nv_bfloat16 *>(x), T, static_cast<float *>(scratch),
                         idx, w, counts, nullptr, zero_counts(counts, c->E), s);
}

size_t lmoe_workspace_size(const lmoe_ctx *c, int64_t T) {
    if (!c || T < 0) return 0;
    return layout(c, T).total;
}

size_t lmoe_host_workspace_size(const lmoe_ctx *c, int64_t T) {
    if (!c || T < 0) return 0;
    return align256(layout(c, T).total) + 2 * align256(static_cast<size_t>(T) * c->d * 2);
}

lmoe_status lmoe_workspace_range(const lmoe_ctx *c, int64_t T, int stage, size_t *offset,
                                 size_t *bytes) {
    if (!c || T < 0 || !offset || !bytes) return LMOE_EINVAL;
    const WsLayout L = layout(c, T);
    const int64_t k = c->k, l = c->l, F = c->ffn;
    switch (stage) {
    case LMOE_STAGE_IDX: *offset = L.idx; *bytes = T * k * 4; break;
    case LMOE_STAGE_W: *offset = L.w; *bytes = T * k * 4; break;
    case LMOE_STAGE_COUNTS: *offset = L.counts; *bytes = c->E * 4; break;
    case LMOE_STAGE_ZQ_CODES: *offset = L.zq_codes; *bytes = T * l / 2; break;
    case LMOE_STAGE_ZQ_SF: *offset = L.zq_sf; *bytes = T * l / 16; break;
    case LMOE_STAGE_C: *offset = L.c; *bytes = T * l * 2; break;
    case LMOE_STAGE_Z: *offset = L.z_dbg; *bytes = c->debug ? T * l * 2 : 0; break;
    case LMOE_STAGE_ROWS: *offset = L.row_slot; *bytes = L.R * 4; break;
    case LMOE_STAGE_H:
        if (c->w4a16) { *offset = L.h_bf16; *bytes = L.R * F * 2; }
        else { *offset = L.h_dbg; *bytes = c->debug ? L.R * F * 2 : 0; }
        break;
    case LMOE_STAGE_HQ_CODES: *offset = L.h_codes; *bytes = c->w4a16 ? 0 : L.R * F / 2; break;
    case LMOE_STAGE_HQ_SF: *offset = L.h_sf; *bytes = c->w4a16 ? 0 : L.R * F / 16; break;
    case LMOE_STAGE_NROWS: *offset = L.nrows; *bytes = 4; break;
    case LMOE_STAGE_XS_Q: *offset = L.xs_q; *bytes = c->shared_ffn ? T * c->d : 0; break;
    case LMOE_STAGE_HS: *offset = L.hs_dbg; *bytes = c->debug ? T * c->shared_ffn * 2 : 0; break;
    case LMOE_STAGE_HS_Q: *offset = L.hs_q; *bytes = T * c->shared_ffn; break;
    case LMOE_STAGE_S: *offset = L.s_out; *bytes = c->shared_ffn ? T * c->d * 2 : 0; break;
    case LMOE_STAGE_ROUTER: *offset = L.router; *bytes = route_scratch_bytes(c, T); break;
    default: return LMOE_EINVAL;
    }
    return LMOE_OK;
}

lmoe_status lmoe_set_debug(lmoe_ctx *c, int on) {
    if (!c) return LMOE_EINVAL;
    c->debug = on ? 1 : 0;
    return LMOE_OK;
}

lmoe_status lmoe_set_wait_limit(lmoe_ctx *c, long long cycles) {
    if (!c) return LMOE_EINVAL;
    c->wait_limit = cycles > 0 ? cycles : 0;
    return LMOE_OK;
}

lmoe_status lmoe_route(lmoe_ctx *c, const void *x, int64_t T, int32_t *idx, float *w,
                       int32_t *counts, lmoe_stream stream) {
    if (!c || T < 0) return LMOE_EINVAL;
    if (T == 0) return LMOE_OK;
    if (!x || !idx || !w) return LMOE_EINVAL;
    if (reinterpret_cast<uintptr_t>(x) % 16 || (counts && reinterpret_cast<uintptr_t>(counts) % 16))
        return LMOE_EINVAL;
    FaultScope fault_scope;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = route_scratch_bytes(c, T);
    if (need > c->route_ws_bytes) {
        if (c->route_ws) LMOE_CUDA(cudaFreeAsync(c->route_ws, s));
        c->route_ws = nullptr;
        c->route_ws_bytes = 0;
        LMOE_CUDA(dev_malloc_async(&c->route_ws, need, s));
        c->route_ws_bytes = need;
    }
    return launch_router(c, static_cast<const __nv_bfloat16 *>(x), T,
                         static_cast<float *>(c->route_ws), idx, w, counts, nullptr,
                         zero_counts(counts, c->E), s);
}

lmoe_status lmoe_forward(lmoe_ctx *c, const void *x, int64_t T, void *y, void *ws, size_t ws_bytes,
                         lmoe_stream stream) {
    if (!c || T < 0) return LMOE_EINVAL;
    if (T == 0) return LMOE_OK;
    if (!x || !y || !ws) return LMOE_EINVAL;
    if (T > (int64_t(1) << 24)) return LMOE_EINVAL;
    const WsLayout L = layout(c, T);
    if (ws_bytes < L.total) return LMOE_ENOMEM;
    if (reinterpret_cast<uintptr_t>(ws) % 256 || reinterpret_cast<uintptr_t>(x) % 16 ||
        reinterpret_cast<uintptr_t>(y) % 16)
        return LMOE_EINVAL;
    FaultScope fault_scope;
    const Fault &fault = fault_scope.f;
    NvtxRange nvtx_range("lmoe_forward");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *W = static_cast<uint8_t *>(ws);
    auto at = [&](size_t off) { return static_cast<void *>(W + off); };
    int32_t *idx = static_cast<int32_t *>(at(L.idx));
    float *rw = static_cast<float *>(at(L.w));
    int32_t *counts = static_cast<int32_t *>(at(L.counts));
    int32_t *seg = static_cast<int32_t *>(at(L.seg));
    int32_t *mt = static_cast<int32_t *>(at(L.mt));
    int32_t *slot_off = static_cast<int32_t *>(at(L.slot_off));
    int32_t *nrows = static_cast<int32_t *>(at(L.nrows));
    int32_t *row_slot = static_cast<int32_t *>(at(L.row_slot));
    float *zacc = static_cast<float *>(at(L.zacc));
    uint8_t *zq_codes = static_cast<uint8_t *>(at(L.zq_codes));
    uint8_t *zq_sf = static_cast<uint8_t *>(at(L.zq_sf));
    __nv_bfloat16 *z_dbg = c->debug || c->w4a16 ? static_cast<__nv_bfloat16 *>(at(L.z_dbg)) : nullptr;
    uint8_t *a_codes = static_cast<uint8_t *>(at(L.a_codes));
    uint8_t *a_sf = static_cast<uint8_t *>(at(L.a_sf));
    uint8_t *h_codes = static_cast<uint8_t *>(at(L.h_codes));
    uint8_t *h_sf = static_cast<uint8_t *>(at(L.h_sf));
    __nv_bfloat16 *h_dbg = c->debug ? static_cast<__nv_bfloat16 *>(at(L.h_dbg)) : nullptr;
    float *c_acc = static_cast<float *>(at(L.c_acc));
    __nv_bfloat16 *cb = static_cast<__nv_bfloat16 *>(at(L.c));
    float *yacc = static_cast<float *>(at(L.yacc));
    __nv_bfloat16 *a_bf16 = c->w4a16 ? static_cast<__nv_bfloat16 *>(at(L.a_bf16)) : nullptr;
    __nv_bfloat16 *h_bf16 = c->w4a16 ? static_cast<__nv_bfloat16 *>(at(L.h_bf16)) : nullptr;
    uint8_t *xs_q = static_cast<uint8_t *>(at(L.xs_q));
    uint8_t *hs_q = static_cast<uint8_t *>(at(L.hs_q));
    __nv_bfloat16 *hs_dbg = c->debug ? static_cast<__nv_bfloat16 *>(at(L.hs_dbg)) : nullptr;
    __nv_bfloat16 *s_out = static_cast<__nv_bfloat16 *>(at(L.s_out));
    const int d = c->d, l = c->l, E = c->E, k = c->k, F = c->ffn;
    const bool small_a = T <= kSmallAMaxT;   // no GEMM tile then has more than 32 valid rows
    const uint32_t a_box = small_a ? kABoxRows : kBM;   // rows of the activation TMA box
    // W4A16 expert GEMMs: at decode the token rows are the MMA's N (16 or 32; an expert segment
    // has at most T rows, since a token's k experts are distinct)
    const uint32_t w4_box = small_a ? (T <= 16 ? 16u : 32u) : kBM;
    if (c->profile) {
        c->nprof = 0;
        cudaEventRecord(c->ev[0], s);
    }

    // The split-K down-projection does not depend on routing: it runs on the context's second
    // stream, beside the router, and joins before its finalize (which needs the segments).
    const bool fork = L.split_down && !c->profile;
    auto down_proj = [&](cudaStream_t ds) -> lmoe_status {
        CUtensorMap tx;
        if (!make_map(&tx, true, x, d, T, static_cast<uint64_t>(d) * 2, a_box)) return LMOE_ECUDA;
        GemmArgs g = dense_args(static_cast<int>(T), l, d, L.down_splits,
                                L.split_down ? EPI_RED_F32 : EPI_Z_QUANT, c, kb_for(small_a), 64, bn_for(small_a));
        if (L.split_down) {
            g.out = zacc; g.ld_out = l;
        } else {
            // row-major zq (and, W4A16, z) only; scatter_rows_kernel copies the rows into the
            // expert segments (a copy kernel with all SMs beats k scattered stores per row in
            // the GEMM epilogue)
            g.q = c->qz; g.q_codes = zq_codes; g.q_sf = zq_sf; g.dbg = z_dbg;
            g.topk = 0;
        }
        LMOE_CUDA((launch_gemm<kKindBf16>(tx, small_a ? c->tm_wd : c->tm_wd_w, g,
                                      grid_for(int64_t(g.m_tiles) * g.n_tiles * g.k_splits, c->num_sms), small_a, ds)));
        prof_mark(c, "down_proj", ds);
        return LMOE_OK;
    };
    // The split-K down-projection runs on the second stream beside the router.  At small T it
    // forks after the router's logit kernel: both want about 128 SMs, and the router's chain
    // (logits, top-k, segments) is the longer one, so it streams its weights first on an idle
    // GPU; that kernel also clears the down-projection's accumulator.
    const bool fork_late = fork && T <= kSmallMaxT;
    if (fork && !fork_late) LMOE_CUDA(cudaEventRecord(c->ev_fork, s));

    // 1. router (its first kernel also clears the histogram and the fp32 accumulators)
    {
        ZeroRanges z;
        std::memset(&z, 0, sizeof(z));
        z.p[0] = reinterpret_cast<uint4 *>(counts); z.n16[0] = cdiv(E * 4 + 16, 16);   // counts + done
        z.p[1] = reinterpret_cast<uint4 *>(c_acc); z.n16[1] = T * l * 4 / 16;
        if (L.split_down && (!fork || fork_late)) { z.p[2] = reinterpret_cast<uint4 *>(zacc); z.n16[2] = T * l * 4 / 16; }
        if (L.split_up) { z.p[3] = reinterpret_cast<uint4 *>(yacc); z.n16[3] = T * d * 4 / 16; }
        SegOut so = {counts + E, seg, mt, nrows};
        lmoe_status st = launch_router(c, static_cast<const __nv_bfloat16 *>(x), T,
                                       static_cast<float *>(at(L.router)), idx, rw, counts, slot_off, z, s, so,
                                       fork_late ? c->ev_fork : nullptr);
        if (st != LMOE_OK) return st;
    }
    if (fork) {
        LMOE_CUDA(cudaStreamWaitEvent(c->aux, c->ev_fork, 0));
        if (!fork_late) {
            ZeroRanges zz;
            std::memset(&zz, 0, sizeof(zz));
            zz.p[0] = reinterpret_cast<uint4 *>(zacc); zz.n16[0] = T * l * 4 / 16;
            LMOE_CUDA(launch_pdl(zero_kernel, dim3(c->num_sms), dim3(256), 0, c->aux, zz));
        }
        lmoe_status st = down_proj(c->aux);
        if (st != LMOE_OK) return st;
        LMOE_CUDA(cudaEventRecord(c->ev_join, c->aux));
    }
    // 3. down-projection z = x Wd^T, quantized to NVFP4
    {
        if (fork) {
            LMOE_CUDA(cudaStreamWaitEvent(s, c->ev_join, 0));
        } else {
            lmoe_status st = down_proj(s);
            if (st != LMOE_OK) return st;
        }
        if (!L.split_down) {
            LMOE_CUDA(launch_pdl(scatter_rows_kernel, dim3(static_cast<unsigned>(cdiv(T * 32, 256))), dim3(256), 0, s,
                                 static_cast<const uint8_t *>(zq_codes), static_cast<const uint8_t *>(zq_sf),
                                 static_cast<const __nv_bfloat16 *>(z_dbg), static_cast<const int32_t *>(idx),
                                 static_cast<const int32_t *>(slot_off), static_cast<const int32_t *>(seg), T, k, l,
                                 a_codes, a_sf, a_bf16, row_slot));
            prof_mark(c, "scatter", s);
        }
        if (L.split_down) {
            // whole tokens per block: 256 threads cover 256 / (l/16) tokens (l <= 4096, k * tokens <= 256);
            // at T <= 16 one token per block and its k copies in four groups of blocks
            const int nb = l / 16;
            const int tpb = T <= 16 ? 1 : std::max(1, std::min(256 / nb, 256 / k));
            const unsigned groups = T <= 16 ? 4u : 1u;
            LMOE_CUDA(launch_pdl(z_finalize_kernel, dim3(static_cast<unsigned>(cdiv(T, tpb)), groups), dim3(tpb * nb), 0, s,
                                 static_cast<const float *>(zacc), T, l, c->qz, zq_codes, zq_sf, z_dbg,
                                 static_cast<const int32_t *>(idx), static_cast<const int32_t *>(slot_off),
                                 static_cast<const int32_t *>(seg), k, row_slot, a_codes, a_sf, a_bf16));
            prof_mark(c, "z_finalize", s);
        }
    }
    // 5. latent-up grouped GEMM + relu^2 (+ requantize to NVFP4; W4A16: bf16 h)
    {
        CUtensorMap ta;
        const bool ok = c->w4a16 ? make_map(&ta, true, a_bf16, l, L.R, static_cast<uint64_t>(l) * 2, w4_box)
                                 : make_map(&ta, false, a_codes, l / 2, L.R, l / 2, a_box);
        if (!ok) return LMOE_ECUDA;
        GemmArgs g;
        std::memset(&g, 0, sizeof(g));
        g.M = static_cast<int>(L.R); g.N = F; g.K = l;
        g.bn = (c->w4a16 || small_a) ? kBN : kBNF4Up;   // the launch_gemm configuration's tile width
        g.n_tiles = static_cast<int>(cdiv(F, g.bn));
        g.grouped = 1; g.E = E; g.mt_start = mt; g.seg_start = seg; g.counts = counts;
        g.sfb = c->w1_sf; g.NB = static_cast<int>(cdiv(F, 128));
        g.b_kt = static_cast<int>(cdiv(l, 256));
        g.err = c->err;
        g.wait_limit = c->wait_limit;
        g.inject_wait = fault.kind == kFaultWait ? 1 : 0;
        if (c->w4a16) {
            g.k_tiles = static_cast<int>(cdiv(l / 64, kb_for(small_a)));
            g.epi = EPI_H_BF16; g.out = h_bf16; g.alpha = c->w1_sdec;
            if (small_a)
                LMOE_CUDA(launch_w4dec(ta, c->tm_w1, g, c->num_sms, static_cast<int>(w4_box), s));
            else
                LMOE_CUDA((launch_gemm<kKindW4A16>(ta, c->tm_w1raw, g, c->num_sms, small_a, s)));
        } else {
            g.k_tiles = static_cast<int>(cdiv(l, 256 * (small_a ? kb_for(true) : kKbF4Up)));
            g.sfa = a_sf;
            g.epi = EPI_H_QUANT; g.q = c->qh; g.q_codes = h_codes; g.q_sf = h_sf; g.dbg = h_dbg;
            g.alpha = c->alpha1;
            LMOE_CUDA((launch_gemm<kKindNvf4>(ta, c->tm_w1, g, c->num_sms, small_a, s)));
        }
        prof_mark(c, "expert_up", s);
    }
    // 6. latent-down grouped GEMM, routing weight, combine into c_acc
    {
        CUtensorMap ta;
        const bool ok = c->w4a16 ? make_map(&ta, true, h_bf16, F, L.R, static_cast<uint64_t>(F) * 2, w4_box)
                                 : make_map(&ta, false, h_codes, F / 2, L.R, F / 2, a_box);
        if (!ok) return LMOE_ECUDA;
        GemmArgs g;
        std::memset(&g, 0, sizeof(g));
        g.M = static_cast<int>(L.R); g.N = l; g.K = F;
        g.bn = (c->w4a16 || small_a) ? kBN : kBNF4Dn;   // the launch_gemm configuration's tile width
        g.n_tiles = static_cast<int>(cdiv(l, g.bn));
        g.grouped = 1; g.E = E; g.mt_start = mt; g.seg_start = seg; g.counts = counts;
        g.sfb = c->w2_sf; g.NB = static_cast<int>(cdiv(l, 128));
        g.b_kt = static_cast<int>(cdiv(F, 256));
        g.epi = EPI_COMBINE; g.out = c_acc; g.ld_out = l;
        g.row_slot = row_slot; g.route_w = rw; g.topk = k; g.err = c->err;
        g.wait_limit = c->wait_limit;
        if (c->w4a16) {
            g.k_tiles = static_cast<int>(cdiv(F / 64, kb_for(small_a)));
            g.alpha = c->w2_sdec;
            if (small_a)
                LMOE_CUDA(launch_w4dec(ta, c->tm_w2, g, c->num_sms, static_cast<int>(w4_box), s));
            else
                LMOE_CUDA((launch_gemm<kKindW4A16>(ta, c->tm_w2raw, g, c->num_sms, small_a, s)));
        } else {
            g.k_tiles = static_cast<int>(cdiv(F, 256 * (small_a ? kb_for(true) : kKbF4Dn)));
            g.sfa = h_sf;
            g.alpha = c->alpha2;
            LMOE_CUDA((launch_gemm<kKindNvf4>(ta, c->tm_w2, g, c->num_sms, small_a, s)));
        }
        prof_mark(c, "expert_down", s);
    }
    // 7. c = bf16(c_acc) (at T <= 8 the up-projection rounds c_acc itself, below)
    const bool up_f32 = T <= kUpF32MaxT;
    if (!up_f32) {
        const int grid = static_cast<int>(std::min<int64_t>(cdiv(T * l / 8, 256), c->num_sms * 8));
        LMOE_CUDA(launch_pdl(f32_to_bf16_kernel, dim3(grid), dim3(256), 0, s, static_cast<const float *>(c_acc),
                             T * l, cb, static_cast<const __nv_bfloat16 *>(nullptr)));
        prof_mark(c, "combine_cast", s);
    }
    // 7b. shared expert at width d (FP8): xs = q8(x); hs = q8(bf16(relu(alpha_s1 xs Ws1q^T)^2));
    //     s = bf16(alpha_s2 hs Ws2q^T), added to the up-projection before its rounding.  It needs
    //     only x: when the forward forks, it runs on the second stream after the down-projection,
    //     beside the routed experts, and joins before the up-projection.
    const bool shared_aux = c->shared_ffn && fork;
    if (c->shared_ffn) {
        // at T = 1 its 134 MB of FP8 weights outweigh the routed experts' 104 MB: its kernels
        // are scheduled first (at T = 8 and 64 that ordering was slower)
        PrioScope shared_prio(shared_aux && T <= kSharedFirstMaxT ? urgent_priority() : 0);
        const cudaStream_t ss = shared_aux ? c->aux : s;
        const int FS = c->shared_ffn;
        const int qg = static_cast<int>(std::min<int64_t>(cdiv(T * d / 16, 256), c->num_sms * 16));
        LMOE_CUDA(launch_pdl(quantize_fp8_kernel<__nv_bfloat16>, dim3(qg), dim3(256), 0, ss,
                             static_cast<const __nv_bfloat16 *>(x), T * d, c->amax_xs,
                             static_cast<const unsigned *>(nullptr), xs_q));
        prof_mark(c, "shared_quant_x", ss);
        CUtensorMap txs, ths;
        if (!make_map(&txs, false, xs_q, d, T, d, a_box) || !make_map(&ths, false, hs_q, FS, T, FS, a_box))
            return LMOE_ECUDA;
        GemmArgs g1 = dense_args(static_cast<int>(T), FS, d, 1, EPI_FP8_SQRELU, c, kb_for(small_a), 128,
                                 bn_for(small_a));
        g1.alpha_s = c->alpha_s1; g1.s_enc8 = c->s_enc_hs; g1.q_codes = hs_q; g1.dbg = hs_dbg;
        LMOE_CUDA((launch_gemm<kKindFp8>(txs, small_a ? c->tm_ws1 : c->tm_ws1_w, g1, grid_for(int64_t(g1.m_tiles) * g1.n_tiles, c->num_sms),
                                         small_a, ss)));
        prof_mark(c, "shared_up", ss);
        GemmArgs g2 = dense_args(static_cast<int>(T), d, FS, 1, EPI_STORE_SCALED, c, kb_for(small_a), 128,
                                 bn_for(small_a));
        g2.alpha_s = c->alpha_s2; g2.out = s_out; g2.ld_out = d;
        LMOE_CUDA((launch_gemm<kKindFp8>(ths, small_a ? c->tm_ws2 : c->tm_ws2_w, g2, grid_for(int64_t(g2.m_tiles) * g2.n_tiles, c->num_sms),
                                         small_a, ss)));
        prof_mark(c, "shared_down", ss);
        if (shared_aux) {
            LMOE_CUDA(cudaEventRecord(c->ev_join_s, c->aux));
            LMOE_CUDA(cudaStreamWaitEvent(s, c->ev_join_s, 0));
        }
    }
    const __nv_bfloat16 *y_add = c->shared_ffn ? s_out : nullptr;
    // 8. up-projection y = c Wu^T (+ s)
    {
        CUtensorMap tc;
        // T <= 8: A is the fp32 combine accumulator, rounded to bf16 inside the GEMM (which also
        // writes the bf16 c); otherwise the bf16 c of step 7
        const bool ok = up_f32 ? make_map_f32(&tc, static_cast<const float *>(c_acc), l, T, kAF32Rows)
                               : make_map(&tc, true, cb, l, T, static_cast<uint64_t>(l) * 2, a_box);
        if (!ok) return LMOE_ECUDA;
        GemmArgs g = dense_args(static_cast<int>(T), d, l, L.up_splits,
                                L.split_up ? EPI_RED_F32 : EPI_STORE_BF16, c, kb_for(small_a), 64, L.up_bn);
        g.out = L.split_up ? static_cast<void *>(yacc) : y;
        g.ld_out = d;
        if (!L.split_up) g.addend = y_add;
        const CUtensorMap &twu = !small_a ? c->tm_wu_w : (L.up_bn == kBNNarrow ? c->tm_wu_n : c->tm_wu);
        const int grid = grid_for(int64_t(g.m_tiles) * g.n_tiles * g.k_splits, c->num_sms);
        if (up_f32) {
            g.a_copy = cb;
            g.a_rows = static_cast<int>(T);
            g.preload = 1;
            LMOE_CUDA((L.up_bn == kBNNarrow
                           ? launch_gemm_cfg<kKindBf16, true, 2, kStagesUpF32N, kBNNarrow, true>(tc, twu, g, grid, s)
                           : launch_gemm_cfg<kKindBf16, true, 2, kStagesUpF32W, kBN, true>(tc, twu, g, grid, s)));
        } else {
            LMOE_CUDA((launch_gemm<kKindBf16>(tc, twu, g, grid, small_a, s)));
        }
        prof_mark(c, "up_proj", s);
        if (L.split_up) {
            const int grid = static_cast<int>(std::min<int64_t>(cdiv(T * d / 8, 256), c->num_sms * 8));
            LMOE_CUDA(launch_pdl(f32_to_bf16_kernel, dim3(grid), dim3(256), 0, s, static_cast<const float *>(yacc),
                                 T * d, static_cast<__nv_bfloat16 *>(y), y_add));
            prof_mark(c, "y_cast", s);
        }
    }
    return LMOE_OK;
}

lmoe_status lmoe_forward_host(lmoe_ctx *c, const void *x_host, int64_t T, void *y_host, void *ws,
                              size_t ws_bytes, lmoe_stream stream) {
    if (!c || T < 0) return LMOE_EINVAL;
    if (T == 0) return LMOE_OK;
    if (!x_host || !y_host || !ws) return LMOE_EINVAL;
    const size_t main = align256(layout(c, T).total);
    const size_t io = align256(static_cast<size_t>(T) * c->d * 2);
    if (ws_bytes < main + 2 * io) return LMOE_ENOMEM;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *W = static_cast<uint8_t *>(ws);
    void *xd = W + main, *yd = W + main + io;
    const size_t bytes = static_cast<size_t>(T) * c->d * 2;
    // The call synchronizes `stream`, which is not allowed while the stream is being captured.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    LMOE_CUDA(cudaStreamIsCapturing(s, &cap));
    if (cap != cudaStreamCaptureStatusNone) return LMOE_EINVAL;
    auto direct = [&]() -> lmoe_status {
        LMOE_CUDA(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s));
        lmoe_status st = lmoe_forward(c, xd, T, yd, ws, main, stream);
        if (st != LMOE_OK) return st;
        LMOE_CUDA(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s));
        LMOE_CUDA(cudaStreamSynchronize(s));
        return check_error_word(c);
    };
    // the legacy / per-thread default streams cannot be captured; profiling times each kernel;
    // a call with an injected fault runs directly and leaves the cached graph alone
    const bool graphable = s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread && !c->profile &&
                           read_fault().kind == kFaultNone;
    if (!graphable) return direct();
    if (c->host_exec && c->host_T == T && c->host_x == x_host && c->host_y == y_host && c->host_ws == ws &&
        c->host_ws_bytes == ws_bytes && c->host_stream == s && c->host_debug == c->debug &&
        c->host_wait_limit == c->wait_limit) {
        LMOE_CUDA(cudaGraphLaunch(c->host_exec, s));
        LMOE_CUDA(cudaStreamSynchronize(s));
        return host_error_word(c);
    }
    // capture copy-in + forward + copy-out (and the error word); if the capture cannot be made (e.g. pageable host
    // memory), run the same work directly
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        return direct();
    }
    cudaError_t e = cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s);
    lmoe_status st = e == cudaSuccess ? lmoe_forward(c, xd, T, yd, ws, main, stream) : LMOE_ECUDA;
    if (st == LMOE_OK) e = cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s);
    if (st == LMOE_OK && e == cudaSuccess)
        e = cudaMemcpyAsync(c->err_host, c->err, sizeof(unsigned), cudaMemcpyDeviceToHost, s);
    const cudaError_t ec = cudaStreamEndCapture(s, &graph);
    if (st == LMOE_EINVAL || st == LMOE_ENOMEM) {        // argument errors: nothing ran
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    cudaGraphExec_t exec = nullptr;
    if (st == LMOE_OK && e == cudaSuccess && ec == cudaSuccess && graph &&
        cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess) {
        cudaGraphDestroy(graph);
        if (c->host_exec) cudaGraphExecDestroy(c->host_exec);
        c->host_exec = exec;
        c->host_T = T; c->host_x = x_host; c->host_y = y_host; c->host_ws = ws;
        c->host_ws_bytes = ws_bytes; c->host_stream = s; c->host_debug = c->debug;
        c->host_wait_limit = c->wait_limit;
        LMOE_CUDA(cudaGraphLaunch(c->host_exec, s));
        LMOE_CUDA(cudaStreamSynchronize(s));
        return host_error_word(c);
    }
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();                                    // the failed capture's error
    return direct();
}

lmoe_status lmoe_get_expert_nvfp4(const lmoe_ctx *c, int which, int e, uint8_t *codes, uint8_t *sf,
                                  float *s_dec, lmoe_stream stream) {
    if (!c || (which != 1 && which != 2) || e < 0 || e >= c->E || !codes || !sf || !s_dec)
        return LMOE_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int N = which == 1 ? c->ffn : c->l;
    const int K = which == 1 ? c->l : c->ffn;
    const size_t NB = cdiv(N, 128);
    const uint8_t *atoms = (which == 1 ? c->w1_sf : c->w2_sf) + static_cast<size_t>(e) * NB * (K / 64) * 512;
    untile_codes_kernel<<<static_cast<unsigned>(cdiv(static_cast<int64_t>(N) * K / 16, 256)), 256, 0, s>>>(
        which == 1 ? c->w1_codes : c->w2_codes, e, N, K, codes);
    LMOE_LAUNCH();
    sf_atoms_to_rows_kernel<<<static_cast<unsigned>(cdiv(static_cast<int64_t>(N) * K / 16, 256)), 256, 0, s>>>(atoms, N, K, sf);
    LMOE_LAUNCH();
    LMOE_CUDA(cudaMemcpyAsync(s_dec, (which == 1 ? c->w1_sdec : c->w2_sdec) + e, 4, cudaMemcpyDeviceToHost, s));
    LMOE_CUDA(cudaStreamSynchronize(s));
    return LMOE_OK;
}

lmoe_status lmoe_get_shared_fp8(const lmoe_ctx *c, int which, uint8_t *codes, float *s_dec,
                                lmoe_stream stream) {
    if (!c || !c->shared_ffn || (which != 1 && which != 2) || !codes || !s_dec) return LMOE_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t n = static_cast<size_t>(c->shared_ffn) * c->d;
    LMOE_CUDA(cudaMemcpyAsync(codes, which == 1 ? c->ws1_codes : c->ws2_codes, n, cudaMemcpyDeviceToDevice, s));
    LMOE_CUDA(cudaStreamSynchronize(s));
    *s_dec = which == 1 ? c->ws1_sdec : c->ws2_sdec;
    return LMOE_OK;
}

int lmoe_forward_kernel_count(const lmoe_ctx *c, int64_t T) {
    if (!c || T <= 0) return 0;
    const WsLayout L = layout(c, T);
    // router (small T: chunk sums, top-k; large T: clearing, tensor-core logits, selection;
    // its last warp lays out the segments), down-proj, expert-up, expert-down, combine cast,
    // up-proj, plus one finalize per split projection or the row scatter (and, for a split
    // down-projection forked before a large-T router, the clearing of its accumulator), plus
    // the shared expert's quantization of x and its two GEMMs
    const int down_extra = L.split_down && T > kSmallMaxT && !c->profile ? 1 : 0;
    const int cast = T > kUpF32MaxT ? 1 : 0;       // at T <= 8 the up-projection rounds c itself
    return 6 + cast + (T > kSmallMaxT ? 1 : 0) + 1 + down_extra + (L.split_up ? 1 : 0) + (c->shared_ffn ? 3 : 0);
}

lmoe_status lmoe_set_profile(lmoe_ctx *c, int on) {
    if (!c) return LMOE_EINVAL;
    if (on && !c->ev[0]) {
        for (cudaEvent_t &e : c->ev) LMOE_CUDA(cudaEventCreate(&e));
    }
    c->profile = on ? 1 : 0;
    c->nprof = 0;
    return LMOE_OK;
}

int lmoe_profile_read(lmoe_ctx *c, const char **names, float *ms, int max) {
    if (!c || !c->profile || c->nprof == 0 || max < 0) return -1;
    if (cudaEventSynchronize(c->ev[c->nprof]) != cudaSuccess) return -1;
    const int n = std::min(c->nprof, max);
    for (int i = 0; i < n; ++i) {
        float t = 0.0f;
        cudaEventElapsedTime(&t, c->ev[i], c->ev[i + 1]);
        if (names) names[i] = c->prof_name[i];
        if (ms) ms[i] = t;
    }
    return n;
}

lmoe_status lmoe_check(lmoe_ctx *c, lmoe_stream stream) {
    if (!c) return LMOE_EINVAL;
    LMOE_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    return check_error_word(c);
}

}  // extern "C"
