// gemm.cuh -- the tensor-core GEMMs of the layer (tcgen05, TMEM accumulators, TMA operands).
//
// One persistent, warp-specialized kernel template serves
//   * the BF16 latent projections d -> l and l -> d (kind::f16, fp32 accumulate) -- the
//     projections stay in BF16 (shengxinai.com Nemotron 3 blog, section 3.1.3 table), and
//   * the NVFP4 expert GEMMs latent-up and latent-down (kind::mxf4nvf4.block_scale with
//     UE4M3 scales, one per 16 K, E2M1 operands; blog section 3.1.1), grouped per expert, and
//   * the FP8 E4M3 shared-expert GEMMs (kind::f8f6f4, per-tensor scales applied in the
//     epilogue; NVIDIA AI releases Nemotron 3 Ultra, quantization paragraph).
// D[m][n] = sum_k A[m][k] * B[n][k]: A = activations (rows = tokens), B = weights (rows = output
// features); both K-major.  Tile 128 x 128, one SW128 row of 128 bytes per operand per stage
// (64 bf16, 128 e4m3 or 256 e2m1 elements of K).  A is fetched as one box per column block:
// 32 rows at decode (a tile of one token moves 4 KB of A per stage, not 16 KB; rows past the
// box hold stale data whose accumulator rows the epilogue never reads), 128 rows otherwise
// (one TMA request instead of four: the request count, not the bytes, limited the loads).
//
// Warp roles (one CTA per SM; 384 threads; 256 for the grouped NVFP4 GEMMs at prefill, 512 for
// W4A16, whose warps 2..7 decode the weight tiles):
//   warp 0      TMA producer (one elected lane): operand tiles + scale atoms -> smem ring
//   warp 1      TMEM allocator and MMA issuer (one lane): tcgen05.mma into one of two
//               128-column accumulators
//   warps 2, 3  scale-factor copiers (NVFP4 only, one lane each): the A and the B scale atoms
//               of a stage (loaded first, on their own barrier, so they land ahead of the
//               operand tiles), smem -> TMEM with tcgen05.cp, then a commit on the stage's
//               "scales ready" barrier.  Issuing a tensor-core op costs a single thread tens of
//               cycles, so copies and MMAs are issued from three threads in parallel.
//   warps 4..   epilogue: tcgen05.ld of the accumulator (warp w reads lane quadrant w % 4;
//               eight warps: two per quadrant, each taking half of the tile's columns; four
//               warps: one per quadrant), fused output transform, global stores / reductions.
//               A warp loads two 32-column chunks before one wait; the next tile's per-row
//               scalars (expert scale, routing weight, output token) are fetched while the
//               current tile is processed.
// Barriers: full/empty per smem stage, tmem_full/tmem_empty per accumulator.  Every wait is
// bounded (common.cuh); on a timeout the CTA records LMOE_ETIMEOUT, the roles leave their
// loops, outstanding tensor-core work is drained with a bounded wait and TMEM is freed.
#pragma once
#include "common.cuh"
#include "nvfp4.cuh"
#include "fp8.cuh"

namespace lmoe {

// Operand kinds (template argument KIND).
// kKindW4A16 (above decode size; decode has its own kernel, w4dec.cuh): bf16 activations times
// NVFP4 weights that converter warps decode into bf16 tiles in shared memory (E2M1 x E4M3 is
// exact in bf16), then kind::f16 MMAs.
constexpr int kKindBf16 = 0, kKindNvf4 = 1, kKindFp8 = 2, kKindW4A16 = 3;

enum EpiMode : int {
    EPI_STORE_BF16 = 0,   // out bf16 [M][ld] = acc (+ addend bf16 [M][ld], if given)
    EPI_RED_F32 = 1,      // out fp32 [M][ld] += acc (split-K partial)
    EPI_Z_QUANT = 2,      // z = bf16(acc); zq = NVFP4(z) row-major; dbg = z
    EPI_H_QUANT = 3,      // h = bf16(relu(alpha_e acc)^2); hq = NVFP4(h) (scale atoms); dbg = h
    EPI_COMBINE = 4,      // c_acc[token] += w_slot * alpha_e * acc
    EPI_FP8_SQRELU = 5,   // h = bf16(relu(alpha_s acc)^2); q_codes [M][N] = e4m3(h * s_enc8); dbg = h
    EPI_STORE_SCALED = 6, // out bf16 [M][ld] = alpha_s * acc
    EPI_H_BF16 = 7        // W4A16 latent-up: out bf16 [M][N] = bf16(relu(alpha_e acc)^2)
};

constexpr int kBM = 128, kBN = 128;
constexpr int kTileBytes = kBM * 128;     // 16 KB per operand per stage
constexpr int kABoxRows = 32;             // decode: A is loaded as one 32-row box per column block
constexpr int kABoxBytes = kABoxRows * 128;
constexpr int kAF32Rows = 8;              // decode, A staged as fp32: one 8-row box per column block
constexpr int kSfStageBytes = 4 * 512;    // 4 scale atoms (4 x K64) per operand per stage

struct GemmArgs {
    int M, N, K;                 // dense: rows of A, rows of B (= output cols), depth (elements)
    int m_tiles, n_tiles, k_tiles, k_splits, kt_per_split;
    int grouped, E;              // grouped: per-expert segments from the device tables
    const int32_t *mt_start;     // [E+1] prefix of M tiles
    const int32_t *seg_start;    // [E+1] first row of each expert's segment (multiple of 128)
    const int32_t *counts;       // [E]
    const uint8_t *sfa;          // activation scale atoms [rows/128][K/64][512]
    const uint8_t *sfb;          // weight scale atoms [E][NB][K/64][512]
    int NB;                      // ceil(N / 128)
    int b_kt;                    // > 0: B (expert weight codes) in tile order with b_kt 128-byte
                                 // column blocks per 128-row block (tiled_code_offset)
    int epi;
    void *out;                   // see EpiMode
    int64_t ld_out;
    QScale q;                    // quantizer of z or h
    uint8_t *q_codes;            // [rows][N/2]
    uint8_t *q_sf;               // z: [rows][N/16] row-major; h: atoms [rows/128][N/64][512]
    __nv_bfloat16 *dbg;          // optional bf16 copy of z or h, [rows][N]
    const float *alpha;          // [E] per-expert tensor-scale product
    const int32_t *row_slot;     // [rows] routing slot of a permuted row (combine)
    const float *route_w;        // [T*k]
    int topk;
    // z epilogue: copies of each token's zq row into its k expert-segment rows
    const int32_t *idx;          // [T*k] selected experts
    const int32_t *slot_off;     // [T*k] row of each slot inside its expert's segment
    uint8_t *a_codes;            // [R][N/2]
    uint8_t *a_sf;               // scale atoms [R/128][N/64][512]
    int32_t *row_slot_out;       // [R]
    // shared expert (FP8): per-tensor scale product and the h encode scale; up-projection addend
    float alpha_s;
    float s_enc8;
    const __nv_bfloat16 *addend; // EPI_STORE_BF16: bf16 [M][ld_out] added before the rounding
    int a_kwrap;                 // > 0: A's K coordinate wraps at this many elements (B is K-concatenated)
    int bn;                      // tile width (output columns): the kernel's BN
    __nv_bfloat16 *a_bf16;       // W4A16 z epilogue: bf16 z rows copied into the expert segments [R][N]
    unsigned *err;
    long long wait_limit;        // SM cycles a pipeline wait may take before the CTA gives up
    int inject_wait;             // fault injection: the MMA role first waits on a barrier that
                                 // nothing arrives at, so the wait runs out (LMOE_FAULT=wait)
    __nv_bfloat16 *a_copy;       // A staged as fp32 (bf16 GEMM at decode, STG): the bf16 rounding
                                 // of A's first a_rows rows, [a_rows][K], written by the CTAs of n-tile 0
    int a_rows;
    int preload;                 // decode launches: issue the weight (B) loads of the first
                                 // ring pass before waiting on the previous grid (the weights,
                                 // and for grouped launches the segment tables, are complete
                                 // before that grid began)
};

struct Tile {
    int e, a_row0, rows, b_row0, n0, cols, kt0, kt1;
};

// Per-expert tables copied to shared memory at kernel start (grouped GEMMs): every role
// decodes every tile, so the binary search must not walk global memory.
struct SmemTables {
    int32_t mt[1025];    // mt_start[0..E]
    int32_t cnt[1024];   // counts[e]
    float rcp_h[256];    // h quantizer: reciprocal of each block-scale byte (quant_block16_lut)
};

__device__ __forceinline__ Tile decode_tile(const GemmArgs &g, const SmemTables *tb, int t) {
    Tile tl;
    if (g.grouped) {
        const int key = t / g.n_tiles;
        int lo = 0, hi = g.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tb->mt[mid] <= key) lo = mid; else hi = mid - 1;
        }
        const int e = lo;
        const int mt0 = tb->mt[e];
        const int mt_e = tb->mt[e + 1] - mt0;
        const int local = t - mt0 * g.n_tiles;
        const int m = local % mt_e, n = local / mt_e;
        tl.e = e;
        tl.a_row0 = (mt0 + m) * kBM;          // segments are whole 128-row tiles: seg_start = 128 mt_start
        tl.rows = min(kBM, tb->cnt[e] - m * kBM);
        tl.n0 = n * g.bn;
        tl.b_row0 = e * g.N + n * g.bn;
        tl.cols = min(g.bn, g.N - n * g.bn);
        tl.kt0 = 0;
        tl.kt1 = g.k_tiles;
    } else {
        const int m = t % g.m_tiles;
        const int r = t / g.m_tiles;
        const int n = r % g.n_tiles, s = r / g.n_tiles;
        tl.e = 0;
        tl.a_row0 = m * kBM;
        tl.rows = min(kBM, g.M - m * kBM);
        tl.n0 = n * g.bn;
        tl.b_row0 = n * g.bn;
        tl.cols = min(g.bn, g.N - n * g.bn);
        tl.kt0 = s * g.kt_per_split;
        tl.kt1 = min(g.k_tiles, tl.kt0 + g.kt_per_split);
    }
    return tl;
}

// Pipeline wait: gives up after `limit` SM cycles (recording LMOE_ETIMEOUT and telling the
// other roles to stop), or as soon as another role of the CTA has given up.  sleep_ns > 0: the
// waiting thread is suspended between polls (mbar_try_wait_sleep).
__device__ __forceinline__ bool role_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          unsigned *err, long long limit, uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    if (limit <= 0) limit = kWaitLimitCycles;       // unset: the library's default bound
    const long long t0 = clock64();
    while (true) {
        if (sleep_ns ? mbar_try_wait_sleep(bar, parity, sleep_ns) : mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            raise_error(err, kErrTimeout);
            return false;
        }
    }
}

// ------------------------------------------------------------------------------------
// epilogue: one thread owns one accumulator row; 32 columns per call
// ------------------------------------------------------------------------------------
// Per-tile, per-row scalars, loaded before the accumulator is ready so their latency hides
// behind the tile's MMAs.
struct EpiRow {
    float alpha;     // per-expert tensor-scale product (grouped GEMMs)
    float wslot;     // routing weight of the row's slot (combine)
    int64_t orow;    // output row: the token (combine)
    bool valid;
};

__device__ __forceinline__ EpiRow epilogue_row(const GemmArgs &g, const Tile &tl, int row) {
    EpiRow er;
    er.alpha = 1.0f; er.wslot = 0.0f; er.orow = 0;
    er.valid = row < tl.rows;
    if (g.epi == EPI_H_QUANT || g.epi == EPI_COMBINE || g.epi == EPI_H_BF16) er.alpha = __ldg(g.alpha + tl.e);
    if (g.epi == EPI_COMBINE && er.valid) {
        const int slot = __ldg(g.row_slot + tl.a_row0 + row);
        if (slot < 0) {
            er.valid = false;
        } else {
            er.orow = slot / g.topk;
            er.wslot = __ldg(g.route_w + slot);
        }
    }
    return er;
}

// rcp_of: the h quantizer's reciprocal table in shared memory (grouped NVFP4 GEMMs), or null.
__device__ __forceinline__ void epilogue_chunk(const GemmArgs &g, const Tile &tl, const EpiRow &er,
                                               int row, int c0, const uint32_t (&r)[32],
                                               const float *rcp_of) {
    if (!er.valid) return;
    const int64_t grow = static_cast<int64_t>(tl.a_row0) + row;   // global row of A / output
    const int col = tl.n0 + c0;                                    // output column
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    switch (g.epi) {
    case EPI_STORE_BF16:
    case EPI_STORE_SCALED: {
        if (g.epi == EPI_STORE_SCALED) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(g.alpha_s, v[i]);
        } else if (g.addend) {
            const uint4 *a = reinterpret_cast<const uint4 *>(g.addend + grow * g.ld_out + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 u = __ldg(a + i);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * i + 2 * j] = __fadd_rn(v[8 * i + 2 * j], __uint_as_float(w[j] << 16));
                    v[8 * i + 2 * j + 1] = __fadd_rn(v[8 * i + 2 * j + 1], __uint_as_float(w[j] & 0xFFFF0000u));
                }
            }
        }
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(g.out) + grow * g.ld_out + col);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                              pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
        break;
    }
    case EPI_FP8_SQRELU: {
        const float a = g.alpha_s;
        uint32_t hb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float u0 = fmaxf(__fmul_rn(a, v[2 * i]), 0.0f);
            const float u1 = fmaxf(__fmul_rn(a, v[2 * i + 1]), 0.0f);
            hb[i] = pack_bf16x2(__fmul_rn(u0, u0), __fmul_rn(u1, u1));
            v[2 * i] = __fmul_rn(__uint_as_float(hb[i] << 16), g.s_enc8);
            v[2 * i + 1] = __fmul_rn(__uint_as_float(hb[i] & 0xFFFF0000u), g.s_enc8);
        }
        if (g.dbg) {
            uint4 *o = reinterpret_cast<uint4 *>(g.dbg + grow * g.N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
        }
        uint4 *q = reinterpret_cast<uint4 *>(g.q_codes + grow * g.N + col);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = f32x2_to_e4m3x2(v[16 * b + 4 * i], v[16 * b + 4 * i + 1]) |
                       (f32x2_to_e4m3x2(v[16 * b + 4 * i + 2], v[16 * b + 4 * i + 3]) << 16);
            q[b] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        break;
    }
    case EPI_RED_F32: {
        // columns past the tile's valid ones (N % 32 != 0, e.g. N = E experts) are skipped
        float *o = static_cast<float *>(g.out) + grow * g.ld_out + col;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (c0 + 4 * i < tl.cols) red_add_v4_f32(o + 4 * i, v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        break;
    }
    case EPI_Z_QUANT:
    case EPI_H_QUANT: {
        if (g.epi == EPI_H_QUANT) {
            const float a = er.alpha;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float u = fmaxf(__fmul_rn(a, v[i]), 0.0f);
                v[i] = __fmul_rn(u, u);
            }
        }
        uint32_t hb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            hb[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            v[2 * i] = __uint_as_float(hb[i] << 16);
            v[2 * i + 1] = __uint_as_float(hb[i] & 0xFFFF0000u);
        }
        if (g.dbg) {
            uint4 *o = reinterpret_cast<uint4 *>(g.dbg + grow * g.N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
        }
        uint32_t w[4], s[2];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = v[16 * b + i];
            s[b] = rcp_of ? quant_block16_lut(x, g.q, rcp_of, w[2 * b], w[2 * b + 1])
                          : quant_block16(x, g.q, w[2 * b], w[2 * b + 1]);
        }
        *reinterpret_cast<uint4 *>(g.q_codes + grow * (g.N / 2) + col / 2) = make_uint4(w[0], w[1], w[2], w[3]);
        const uint16_t s2 = static_cast<uint16_t>(s[0] | (s[1] << 8));
        if (g.epi == EPI_Z_QUANT) {
            *reinterpret_cast<uint16_t *>(g.q_sf + grow * (g.N / 16) + col / 16) = s2;
            // the token's k expert-segment rows get the same codes and scales (W4A16: bf16 z)
            for (int j = 0; j < g.topk; ++j) {
                const int64_t slot = grow * g.topk + j;
                const int row = __ldg(g.seg_start + __ldg(g.idx + slot)) + __ldg(g.slot_off + slot);
                if (g.a_bf16) {
                    uint4 *o = reinterpret_cast<uint4 *>(g.a_bf16 + static_cast<int64_t>(row) * g.N + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
                } else {
                    *reinterpret_cast<uint4 *>(g.a_codes + static_cast<int64_t>(row) * (g.N / 2) + col / 2) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint16_t *>(g.a_sf + sf_atom_offset(row, col / 16, g.N / 64)) = s2;
                }
                if (col == 0) g.row_slot_out[row] = static_cast<int32_t>(slot);
            }
        } else {
            *reinterpret_cast<uint16_t *>(g.q_sf + sf_atom_offset(grow, col / 16, g.N / 64)) = s2;
        }
        break;
    }
    case EPI_H_BF16: {
        const float a = er.alpha;
        uint32_t hb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float u0 = fmaxf(__fmul_rn(a, v[2 * i]), 0.0f);
            const float u1 = fmaxf(__fmul_rn(a, v[2 * i + 1]), 0.0f);
            hb[i] = pack_bf16x2(__fmul_rn(u0, u0), __fmul_rn(u1, u1));
        }
        uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(g.out) + grow * g.N + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
        break;
    }
    case EPI_COMBINE: {
        const float ws = er.wslot;
        const float a = er.alpha;
        float *o = static_cast<float *>(g.out) + er.orow * g.ld_out + col;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            red_add_v4_f32(o + 4 * i, __fmul_rn(ws, __fmul_rn(a, v[4 * i])),
                           __fmul_rn(ws, __fmul_rn(a, v[4 * i + 1])),
                           __fmul_rn(ws, __fmul_rn(a, v[4 * i + 2])),
                           __fmul_rn(ws, __fmul_rn(a, v[4 * i + 3])));
        break;
    }
    default: break;
    }
}

// EPI_H_QUANT over two adjacent 32-column chunks (columns c0 .. c0 + 63, c0 a multiple of 64)
// in one straight-line block, so the four 16-element blocks' dependency chains interleave.
// Same arithmetic as epilogue_chunk's EPI_H_QUANT.
__device__ __forceinline__ void hquant_pair(const GemmArgs &g, const Tile &tl, const EpiRow &er, int row,
                                            int c0, const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                            const float *rcp_of) {
    if (!er.valid) return;
    const int64_t grow = static_cast<int64_t>(tl.a_row0) + row;
    const int col = tl.n0 + c0;
    const float a = er.alpha;
    float v[64];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float u0 = fmaxf(__fmul_rn(a, __uint_as_float(r0[i])), 0.0f);
        const float u1 = fmaxf(__fmul_rn(a, __uint_as_float(r1[i])), 0.0f);
        v[i] = __fmul_rn(u0, u0);
        v[32 + i] = __fmul_rn(u1, u1);
    }
    uint32_t hb[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        hb[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        v[2 * i] = __uint_as_float(hb[i] << 16);
        v[2 * i + 1] = __uint_as_float(hb[i] & 0xFFFF0000u);
    }
    if (g.dbg) {
        uint4 *o = reinterpret_cast<uint4 *>(g.dbg + grow * g.N + col);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
    }
    uint32_t w[8], s[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = v[16 * b + i];
        s[b] = quant_block16_lut(x, g.q, rcp_of, w[2 * b], w[2 * b + 1]);
    }
    uint4 *q = reinterpret_cast<uint4 *>(g.q_codes + grow * (g.N / 2) + col / 2);
    q[0] = make_uint4(w[0], w[1], w[2], w[3]);
    q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    // blocks col/16 .. col/16 + 3 are the four bytes of one word of the row's scale atom
    *reinterpret_cast<uint32_t *>(g.q_sf + sf_atom_offset(grow, col / 16, g.N / 64)) =
        s[0] | (s[1] << 8) | (s[2] << 16) | (s[3] << 24);
}

// The h quantization of hquant_pair from 64 accumulator values (two 32-column chunks), one
// 16-element block at a time (only one block's temporaries live), with the same results:
// u = alpha acc and h = u^2 as packed fp32 pairs (each lane the __fmul_rn product), h rounded
// to bf16; h >= 0, so the block amax is the maximum of the bf16 values (max.bf16x2, exact);
// then the block scale, its reciprocal from the table, and the E2M1 codes of h * rcp.
__device__ __forceinline__ void hquant_from_acc(const GemmArgs &g, const Tile &tl, int row, int c0, float a,
                                                const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                                const float *rcp_of) {
    const int64_t grow = static_cast<int64_t>(tl.a_row0) + row;
    const int col = tl.n0 + c0;
    const uint64_t a2 = f2_pack(a, a);
    uint32_t w[8], s[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t *rb = (b < 2 ? r0 : r1) + 16 * (b & 1);
        uint32_t hb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float u0, u1, h0, h1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1])), a2), u0, u1);
            const uint64_t q = f2_pack(fmaxf(u0, 0.0f), fmaxf(u1, 0.0f));
            f2_unpack(f2_mul(q, q), h0, h1);
            hb[i] = cvt_bf16x2(h0, h1);
        }
        if (g.dbg) {
            uint4 *o = reinterpret_cast<uint4 *>(g.dbg + grow * g.N + col + 16 * b);
            o[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
            o[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
        }
        if (g.q.zero) { w[2 * b] = w[2 * b + 1] = 0u; s[b] = 0u; continue; }
        const uint32_t m = max_bf16x2(max_bf16x2(max_bf16x2(hb[0], hb[1]), max_bf16x2(hb[2], hb[3])),
                                      max_bf16x2(max_bf16x2(hb[4], hb[5]), max_bf16x2(hb[6], hb[7])));
        const float amax_b = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
        const uint32_t sf = f32_to_e4m3_satfinite(__fmul_rn(amax_b, g.q.s_enc6));
        const float rcp = rcp_of[sf];
        const uint64_t r2 = f2_pack(rcp, rcp);
        uint32_t by[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float y0, y1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(hb[i] << 16), __uint_as_float(hb[i] & 0xFFFF0000u)), r2), y0, y1);
            by[i] = f32x2_to_e2m1x2(y0, y1);
        }
        w[2 * b] = (by[0] | (by[1] << 8)) | ((by[2] << 16) | (by[3] << 24));
        w[2 * b + 1] = (by[4] | (by[5] << 8)) | ((by[6] << 16) | (by[7] << 24));
        s[b] = sf;
    }
    uint4 *qc = reinterpret_cast<uint4 *>(g.q_codes + grow * (g.N / 2) + col / 2);
    qc[0] = make_uint4(w[0], w[1], w[2], w[3]);
    qc[1] = make_uint4(w[4], w[5], w[6], w[7]);
    *reinterpret_cast<uint32_t *>(g.q_sf + sf_atom_offset(grow, col / 16, g.N / 64)) =
        s[0] | (s[1] << 8) | (s[2] << 16) | (s[3] << 24);
}

// The output row of each of the eight rows this lane reduces (rows it * 4 + lane / 8), or -1
// for padding: exchanged once per tile and shared by the tile's chunks.
__device__ __forceinline__ void combine_rows(const EpiRow &er, int lane, int32_t (&orow)[8]) {
    const int32_t mine = er.valid ? static_cast<int32_t>(er.orow) : -1;
#pragma unroll
    for (int it = 0; it < 8; ++it) orow[it] = __shfl_sync(0xffffffffu, mine, it * 4 + (lane >> 3));
}

// Combine through shared memory (prefill tiles): the warp parks its 32 rows x 32 scaled values
// in a 4 KB staging buffer (16-byte chunk c of row r at chunk slot c ^ (r % 8): conflict-free
// both ways), then reads them back four rows per instruction, so each red.add.v4 instruction
// covers four whole 128-byte lines of c_acc instead of 32 scattered 16-byte pieces.  Rows of
// padding (invalid) take part in the exchange but issue no reduction.  Warp-synchronous.
__device__ __forceinline__ void combine_staged(const GemmArgs &g, const Tile &tl, const EpiRow &er,
                                               int c0, const uint32_t (&r)[32], float4 *stg,
                                               int lane, const int32_t (&orow)[8]) {
    const float ws = er.wslot, a = er.alpha;
    float4 *mine = stg + lane * 8;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        mine[c ^ (lane & 7)] = make_float4(__fmul_rn(ws, __fmul_rn(a, __uint_as_float(r[4 * c]))),
                                           __fmul_rn(ws, __fmul_rn(a, __uint_as_float(r[4 * c + 1]))),
                                           __fmul_rn(ws, __fmul_rn(a, __uint_as_float(r[4 * c + 2]))),
                                           __fmul_rn(ws, __fmul_rn(a, __uint_as_float(r[4 * c + 3]))));
    __syncwarp();
    const int col = tl.n0 + c0;
    const int cc = lane & 7;
    const uint64_t pol = policy_evict_last();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = it * 4 + (lane >> 3);
        const float4 v = stg[rr * 8 + (cc ^ (rr & 7))];
        if (orow[it] >= 0)
            red_add_v4_f32_hint(static_cast<float *>(g.out) + static_cast<int64_t>(orow[it]) * g.ld_out + col + 4 * cc,
                                v.x, v.y, v.z, v.w, pol);
    }
    __syncwarp();
}

// KIND: kKindBf16, kKindNvf4 or kKindFp8.  SMALLA (decode): every tile has at most 32 valid A rows, so each column block of a stage
// keeps only one 4 KB A box; the MMA still reads 128 rows from the block's A base, and rows
// 32..127 fall on the following boxes (or on the slack after the last one): they only feed
// accumulator rows the epilogue never reads.  KB: 128-byte column blocks (256 e2m1 or 64 bf16
// elements of K each; 128 e4m3) per pipeline stage; KB = 2 halves the per-stage barrier handshakes and
// copies when each stage carries little MMA work (decode).
template <int KIND, bool SMALLA, int KB, int BN = kBN, bool STG = false>
struct GemmCfg {
    static constexpr bool NVF4 = KIND == kKindNvf4;
    static constexpr bool W4 = KIND == kKindW4A16;
    static constexpr bool kTables = NVF4 || W4;                       // grouped launches: tables in smem
    // bf16 at decode with STG (T <= 8): A arrives as fp32 (the combine accumulator) in 8-row x
    // 64-element boxes, and warps 2-3 round it to bf16 into the SW128 A slot (no cast kernel)
    static constexpr bool kAF32 = KIND == kKindBf16 && SMALLA && STG;
    static constexpr int kRawBlock = W4 ? 128 * 32 + 512                // E2M1 codes + one scale atom per block
                                        : (kAF32 ? kAF32Rows * 64 * 4 : 0);   // or the fp32 A box
    static constexpr int kRawStage = KB * kRawBlock;
    static constexpr int kEpi0 = W4 ? 8 : 4;                          // first epilogue warp
    // epilogue warps: 4 for the grouped NVFP4 GEMMs at prefill with 128-column tiles (one per
    // TMEM lane quadrant, four 32-column chunks each: with the MMA issue setting the pace,
    // more warps only compete with the pipeline threads for issue slots); 8 otherwise (two per
    // quadrant; for the 256-column NVFP4 tile each holds its 128 accumulator columns in
    // registers: 16 warps would cap registers at 96 and spill).
    static constexpr int kEpiWarps = NVF4 && !SMALLA && BN == 128 ? 4 : 8;
    // NVFP4 tiles 256 columns wide: one accumulator (two of 256 columns would leave no TMEM for
    // the scale factors); its epilogue copies the accumulator to registers and releases it
    // before any arithmetic, so the next tile's MMAs wait only for those TMEM loads.
    static constexpr int kNumAcc = NVF4 && BN == 256 ? 1 : 2;
    static constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
    static constexpr int kACol = SMALLA ? kABoxBytes : kTileBytes;   // A bytes per column block
    static constexpr int kAStage = KB * kACol;
    static constexpr int kBStage = KB * BN * 128;                     // B tile: BN rows of 128 bytes
    static constexpr int kSfStageA = NVF4 ? KB * kSfStageBytes : 0;              // A scale atoms
    static constexpr int kSfStageB = NVF4 ? KB * kSfStageBytes * (BN / 128) : 0; // B: one atom per 128 rows
    static constexpr int kSlack = SMALLA ? kTileBytes - kABoxBytes : 0;
    static constexpr int kElemsPerBlock = NVF4 ? 256 : (KIND == kKindFp8 ? 128 : 64);
    static constexpr int kTmaXPerBlock = (KIND == kKindBf16 || W4) ? 64 : 128;  // tensor-map x units per block
    static constexpr int kStepsPerBlock = 4;                          // MMA K steps per block
    // TMEM columns per stage: 4 per K step for A (128 rows), 4 per 128 rows of B
    static constexpr int kSfColsA = NVF4 ? 16 * KB : 0;
    static constexpr int kSfCols = NVF4 ? 16 * KB * (1 + BN / 128) : 0;
    static constexpr bool kStagedCombine = NVF4 && !SMALLA && STG;    // combine via smem staging
    static constexpr int kStgBytes = kStagedCombine ? kEpiWarps * 4096 : 0;   // one 4 KB buffer per epilogue warp
};

template <int KIND, bool SMALLA, int KB, int BN = kBN, bool STG = false>
constexpr int gemm_smem_bytes(int stages) {
    using C = GemmCfg<KIND, SMALLA, KB, BN, STG>;
    return 1024 + stages * (C::kAStage + C::kBStage + C::kSfStageA + C::kSfStageB) + C::kSlack + 256 +
           stages * C::kRawStage +
           (C::kTables ? static_cast<int>((sizeof(SmemTables) + 15) & ~static_cast<size_t>(15)) : 0) +
           C::kStgBytes + (C::W4 ? 1024 : 0);
}

constexpr int kConvWarps = 6;   // W4A16: warps 2..7 decode the weight tiles

// E2M1 code -> bf16 bits (sign kept; E2M1 values 0, .5, 1, 1.5, 2, 3, 4, 6 are exact in bf16).
__device__ __forceinline__ uint32_t e2m1_bf16_bits(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    const uint32_t mag = e == 0 ? (m ? 0x3F00u : 0u) : (((126u + e) << 7) | (m << 6));
    return mag | ((c & 8u) << 12);
}

// The W4A16 converter: block b of stage `raw` (128 rows x 32 bytes of E2M1 codes, then one
// 512-byte scale atom) -> a 128 x 64 bf16 tile in the SW128 layout at `dst` (16-byte chunk c
// of row r at chunk slot c ^ (r % 8)).  Thread `ct` of `nct` takes (row, 16-element group)
// units; each element is value(code) * value(scale) in bf16, exact.
__device__ __forceinline__ void w4_convert_block(const uint8_t *raw, uint8_t *dst, const uint32_t *lut,
                                                 int ct, int nct) {
    for (int u = ct; u < 128 * 4; u += nct) {
        const int r = u >> 2, grp = u & 3;
        const uint2 codes = *reinterpret_cast<const uint2 *>(raw + r * 32 + grp * 8);
        const uint32_t sfb = raw[4096 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + grp];
        const uint32_t sbits = __float_as_uint(e4m3_to_f32(sfb)) >> 16;   // exact: <= 4 significant bits
        const __nv_bfloat162 sc = __halves2bfloat162(__ushort_as_bfloat16(static_cast<unsigned short>(sbits)),
                                                     __ushort_as_bfloat16(static_cast<unsigned short>(sbits)));
        const uint32_t cw[2] = {codes.x, codes.y};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t byte = (cw[i >> 2] >> (8 * (i & 3))) & 0xFFu;
            uint32_t v = lut[byte];
            __nv_bfloat162 p = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&v), sc);
            o[i] = *reinterpret_cast<uint32_t *>(&p);
        }
        uint8_t *row = dst + r * 128;
        *reinterpret_cast<uint4 *>(row + (((2 * grp) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4 *>(row + (((2 * grp + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// BN: tile width, 128 or (dense kinds without scale factors) 256: a 256-column tile moves
// 48 KB of operands per 64-element K block for twice the outputs of a 128-column one.  64 for
// the bf16 up-projection at decode: twice the CTAs stream the weights, with no split-K.  (NVFP4
// stays at 128: two 256-column accumulators would fill TMEM and leave no room for the scale
// factors, and one accumulator serialises each tile's epilogue with the next tile's MMAs.)
// STG: the staged combine (grouped NVFP4 latent-down at prefill; 32 KB of smem); for the bf16
// GEMM at decode, A staged as fp32 and rounded to bf16 by warps 2-3 (GemmCfg::kAF32).
template <int KIND, bool SMALLA, int KB, int STAGES, int BN = kBN, bool STG = false>
__global__ void __launch_bounds__(GemmCfg<KIND, SMALLA, KB, BN, STG>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs g) {
    using C = GemmCfg<KIND, SMALLA, KB, BN, STG>;
    static_assert(BN == 128 || (BN == 256 && (KIND == kKindBf16 || KIND == kKindFp8)) ||
                      (BN == 256 && KIND == kKindNvf4 && !SMALLA) ||
                      (BN == 64 && KIND == kKindBf16 && SMALLA), "tile width");
    constexpr bool NVF4 = C::NVF4;
    constexpr bool W4 = C::W4;
    constexpr int kEpi0 = C::kEpi0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem;
    uint8_t *sB = sA + STAGES * C::kAStage + C::kSlack;
    uint8_t *sSFA = sB + STAGES * C::kBStage;
    uint8_t *sSFB = sSFA + STAGES * C::kSfStageA;
    uint8_t *sRaw = sSFB + STAGES * C::kSfStageB;             // W4A16: raw weight blocks
    uint64_t *bars = reinterpret_cast<uint64_t *>(sRaw + STAGES * C::kRawStage);
    uint64_t *full = bars, *empty = bars + STAGES, *sfready = bars + 2 * STAGES;
    uint64_t *sffull = bars + 3 * STAGES;   // NVFP4: the stage's scale atoms have landed
    uint64_t *tfull = bars + 4 * STAGES, *tempty = tfull + 2, *drain = tempty + 2;
    uint64_t *cdrain = drain + 1;   // [2]: one per scale copier
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(cdrain + 2);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    SmemTables *tb = reinterpret_cast<SmemTables *>(bars + 256 / 8);
    float4 *stg_all = reinterpret_cast<float4 *>(reinterpret_cast<uint8_t *>(tb) +
                                                 (C::kTables ? ((sizeof(SmemTables) + 15) & ~static_cast<size_t>(15)) : 0));
    uint32_t *lut = reinterpret_cast<uint32_t *>(stg_all);    // W4A16: code byte -> two bf16

    constexpr uint32_t kAccCols = BN;
    constexpr uint32_t kTmemCols = NVF4 ? 512 : 2 * BN;
    constexpr uint32_t kSfCol0 = C::kNumAcc * kAccCols;
    static_assert(!NVF4 || kSfCol0 + STAGES * C::kSfCols <= 512, "TMEM budget");
    static_assert(4 * STAGES + 8 <= 32, "barrier area");
    static_assert(!W4 || kEpi0 == 2 + kConvWarps, "warp roles");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sfready[s], W4 ? kConvWarps : 2);   // scales copied / weights decoded
            mbar_init(&sffull[s], 1);
        }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], C::kEpiWarps); }
        mbar_init(drain, 1);
        mbar_init(&cdrain[0], 1);
        mbar_init(&cdrain[1], 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) { prefetch_tmap(&tmA); prefetch_tmap(&tmB); }
    if (warp == 1) { tmem_alloc(s_tmem, kTmemCols); tmem_relinquish(); }
    auto load_tables = [&]() {
        if (C::kTables && g.grouped) {
            for (int i = threadIdx.x; i <= g.E; i += blockDim.x) {
                tb->mt[i] = __ldg(g.mt_start + i);
                if (i < g.E) tb->cnt[i] = __ldg(g.counts + i);
            }
        }
    };
    constexpr bool kPreload = SMALLA && !W4;
    int npre = 0;           // stages of this CTA's first tile whose B was issued before the wait
    if (kPreload && g.preload) {
        load_tables();
        __syncthreads();    // tables and barrier initialisation visible to the producer warp
        if (warp == 0) {
            const uint32_t leader = elect_leader();
            const int ntiles = g.grouped ? tb->mt[g.E] * g.n_tiles : g.m_tiles * g.n_tiles * g.k_splits;
            if (static_cast<int>(blockIdx.x) < ntiles) {
                const Tile tl = decode_tile(g, tb, blockIdx.x);
                const int K64p = g.K / 64;
                npre = min(STAGES, tl.kt1 - tl.kt0);
                for (int s = 0; s < npre; ++s) {
                    const int kb0 = (tl.kt0 + s) * KB;
                    const uint32_t b_st = smem_u32(sB) + s * C::kBStage;
                    if constexpr (NVF4) {
                        // the stage's arrival, counting the scale atoms of A still to come
                        const int nsteps = min(4 * KB, K64p - 4 * kb0);
                        mbar_arrive_expect_tx_p(leader, &sffull[s], (1 + BN / 128) * nsteps * 512);
                        const uint8_t *sfb_tile = g.sfb + (static_cast<size_t>(tl.e) * g.NB + (tl.n0 >> 7)) * K64p * 512;
                        bulk_load_p(leader, smem_u32(sSFB) + s * C::kSfStageB, sfb_tile + kb0 * 2048, nsteps * 512,
                                    &sffull[s]);
                    }
                    // the stage's arrival, counting the A bytes still to come
                    mbar_arrive_expect_tx_p(leader, &full[s], KB * ((C::kAF32 ? C::kRawBlock : C::kACol) + BN * 128));
#pragma unroll
                    for (int b = 0; b < KB; ++b) {
                        if constexpr (NVF4)
                            tma_load_2d_p(leader, b_st + b * (BN * 128), &tmB, &full[s], 0,
                                          ((tl.e * g.NB + (tl.n0 >> 7)) * g.b_kt + kb0 + b) * 128);
                        else
                            tma_load_2d_p(leader, b_st + b * (BN * 128), &tmB, &full[s],
                                          (kb0 + b) * C::kTmaXPerBlock, tl.b_row0);
                    }
                }
            }
        }
    }
    pdl_wait();      // the previous kernel's outputs (tables, activations) are complete
    pdl_trigger();
    if (W4)
        for (int i = threadIdx.x; i < 256; i += blockDim.x)
            lut[i] = e2m1_bf16_bits(i & 15u) | (e2m1_bf16_bits(i >> 4) << 16);
    if (!(kPreload && g.preload)) load_tables();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // A CTA that allocates all 512 columns (the NVFP4 kernels) always gets lane 0, column 0:
    // a compile-time base lets every TMEM operand stay warp-uniform.
    const uint32_t tmem = kTmemCols == 512 ? 0u : *s_tmem;

    const int num_tiles = g.grouped ? tb->mt[g.E] * g.n_tiles
                                    : g.m_tiles * g.n_tiles * g.k_splits;
    const int K64 = g.K / 64;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // (all lanes run the loop; the elected lane issues: see elect_leader)
        const uint32_t leader = elect_leader();
        int stage = 0;
        uint32_t phase = 0;
        // per stage: ever issued / phase of last issue (a preloaded stage counts as issued)
        uint32_t issued = (1u << npre) - 1u, issued_phase = 0;
        const uint32_t sA0 = smem_u32(sA), sB0 = smem_u32(sB);
        const uint32_t sSFA0 = smem_u32(sSFA), sSFB0 = smem_u32(sSFB);
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x) {
            const Tile tl = decode_tile(g, tb, t);
            const bool first = t == static_cast<int>(blockIdx.x);
            const uint8_t *sfa_tile = NVF4 ? g.sfa + static_cast<size_t>(tl.a_row0 >> 7) * K64 * 512 : nullptr;
            const uint8_t *sfb_tile = (NVF4 || W4) ? g.sfb + (static_cast<size_t>(tl.e) * g.NB + (tl.n0 >> 7)) * K64 * 512 : nullptr;
            for (int kt = tl.kt0; kt < tl.kt1; ++kt) {
                if (!role_wait(&empty[stage], phase ^ 1, s_abort, g.err, g.wait_limit)) break;
                const int kb0 = kt * KB;
                uint64_t *fb = &full[stage];
                const uint32_t a_st = sA0 + stage * C::kAStage, b_st = sB0 + stage * C::kBStage;
                if constexpr (W4) {
                    // activations (bf16), raw E2M1 codes and the scale atom of each 64-element block
                    const int nb = min(KB, K64 - kb0);
                    mbar_arrive_expect_tx_p(leader, fb, nb * (C::kACol + C::kRawBlock));
                    const uint32_t r_st = smem_u32(sRaw) + stage * C::kRawStage;
                    for (int b = 0; b < nb; ++b) {
                        tma_load_2d_p(leader, a_st + b * C::kACol, &tmA, fb, (kb0 + b) * 64, tl.a_row0);
                        // 32 code bytes of 64-element block kb0 + b: a quarter of a tiled box row
                        const int kb = kb0 + b;
                        tma_load_2d_p(leader, r_st + b * C::kRawBlock, &tmB, fb, (kb & 3) * 32,
                                      ((tl.e * g.NB + (tl.n0 >> 7)) * g.b_kt + (kb >> 2)) * 128);
                        bulk_load_p(leader, r_st + b * C::kRawBlock + 4096, sfb_tile + (kb0 + b) * 512, 512, fb);
                    }
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    continue;
                }
                const int nsteps = NVF4 ? min(4 * KB, K64 - 4 * kb0) : 4 * KB;
                // a stage whose B went out before the grid dependency wait (first tile only):
                // its arrivals are made, only A (and A's scale atoms) remain
                const bool pre = first && kt - tl.kt0 < npre;
                if (NVF4) {
                    // the scale atoms first, on their own barrier: they land ahead of the
                    // operand tiles, so their smem -> TMEM copies are off the critical path
                    // (B: the atoms of each 128-row block of the tile, [block][K step][512 B])
                    uint64_t *sb = &sffull[stage];
                    if (!pre) mbar_arrive_expect_tx_p(leader, sb, (1 + BN / 128) * nsteps * 512);
                    bulk_load_p(leader, sSFA0 + stage * C::kSfStageA, sfa_tile + kb0 * 2048, nsteps * 512, sb);
                    // (a 256-column tile whose second half lies past N re-reads the last block,
                    // so no copy leaves the expert's weights; those columns are never stored)
#pragma unroll
                    for (int h = 0; h < BN / 128 && !pre; ++h)
                        bulk_load_p(leader, sSFB0 + stage * C::kSfStageB + h * (4 * KB * 512),
                                    sfb_tile + static_cast<size_t>(min(h, g.NB - 1 - (tl.n0 >> 7))) * K64 * 512 +
                                        kb0 * 2048,
                                    nsteps * 512, sb);
                }
                if (!pre) mbar_arrive_expect_tx_p(leader, fb, KB * ((C::kAF32 ? C::kRawBlock : C::kACol) + BN * 128));
#pragma unroll
                for (int b = 0; b < KB; ++b) {
                    const int kx = (kb0 + b) * C::kTmaXPerBlock;
                    const int kxa = g.a_kwrap > 0 ? kx % g.a_kwrap : kx;
                    if constexpr (C::kAF32)
                        tma_load_2d_p(leader, smem_u32(sRaw) + stage * C::kRawStage + b * C::kRawBlock, &tmA, fb, kx,
                                      tl.a_row0);
                    else
                        tma_load_2d_p(leader, a_st + b * C::kACol, &tmA, fb, kxa, tl.a_row0);
                    if (pre) continue;
                    if (NVF4) {   // weight codes in tile order: box (expert, row block, column block)
#pragma unroll
                        for (int h = 0; h < BN / 128; ++h)
                            tma_load_2d_p(leader, b_st + b * (BN * 128) + h * kTileBytes, &tmB, fb, 0,
                                          ((tl.e * g.NB + min((tl.n0 >> 7) + h, g.NB - 1)) * g.b_kt + kb0 + b) * 128);
                    } else
                        tma_load_2d_p(leader, b_st + b * (BN * 128), &tmB, fb, kx, tl.b_row0);
                }
                issued |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        if (*s_abort) {
            // the last load issued to each stage has landed before the CTA leaves (bounded)
            for (int s = 0; s < STAGES; ++s) {
                if (!((issued >> s) & 1u)) continue;
                const uint32_t p = (issued_phase >> s) & 1u;
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[s], p) && clock64() - t0 < kWaitLimitCycles / 8) {}
                while (NVF4 && !mbar_try_wait(&sffull[s], p) && clock64() - t0 < kWaitLimitCycles / 8) {}
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // (all lanes run the loop; the elected lane issues)
        const uint32_t leader = elect_leader();
        const uint32_t idesc = NVF4 ? idesc_nvf4(kBM, BN)
                                    : (KIND == kKindFp8 ? idesc_f8(kBM, BN) : idesc_bf16(kBM, BN));
        // descriptors of stage 0; a stage adds its byte offset >> 4 to the start address
        const uint64_t adesc0 = sdesc_sw128(smem_u32(sA)), bdesc0 = sdesc_sw128(smem_u32(sB));
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        // Injected fault: `drain` gets its only arrival from the commit after the tile loop, so
        // this wait cannot succeed; it runs out after g.wait_limit cycles and takes the CTA
        // down the timeout path.
        if (g.inject_wait) role_wait(drain, 0, s_abort, g.err, g.wait_limit);
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x, ++it) {
            const Tile tl = decode_tile(g, tb, t);
            const int acc = C::kNumAcc == 2 ? (it & 1) : 0;
            const uint32_t aphase = C::kNumAcc == 2 ? ((it >> 1) & 1) : (it & 1);
            if (!role_wait(&tempty[acc], aphase ^ 1, s_abort, g.err, g.wait_limit)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * kAccCols;
            bool ok = true;
            for (int kt = tl.kt0; kt < tl.kt1; ++kt) {
                if (!role_wait(&full[stage], phase, s_abort, g.err, g.wait_limit)) { ok = false; break; }
                if ((NVF4 || W4 || C::kAF32) && !role_wait(&sfready[stage], phase, s_abort, g.err, g.wait_limit)) { ok = false; break; }
                tc_fence_after();
                const uint64_t ad = adesc0 + ((stage * C::kAStage) >> 4);
                const uint64_t bd = bdesc0 + ((stage * C::kBStage) >> 4);
                const uint32_t acc_flag0 = kt > tl.kt0 ? 1u : 0u;
                if constexpr (NVF4) {
                    const int nsteps = min(4 * KB, K64 - 4 * kt * KB);
                    const uint32_t sf_t = tmem + kSfCol0 + stage * C::kSfCols;
#pragma unroll
                    for (int kk = 0; kk < 4 * KB; ++kk) {
                        if (kk < nsteps)
                            mma_nvf4_p(leader, d_tmem, ad + (((kk >> 2) * C::kACol + (kk & 3) * 32) >> 4),
                                       bd + (((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4), idesc,
                                       sf_t + kk * 4, sf_t + C::kSfColsA + kk * 4 * (BN / 128),
                                       (acc_flag0 | kk) ? 1u : 0u);
                    }
                } else if constexpr (W4) {
                    const int nb = min(KB, K64 - kt * KB);    // 64-element blocks present
                    for (int kk = 0; kk < 4 * nb; ++kk)
                        mma_bf16_p(leader, d_tmem, ad + (((kk >> 2) * C::kACol + (kk & 3) * 32) >> 4),
                                   bd + (((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4), idesc,
                                   (acc_flag0 | kk) ? 1u : 0u);
                } else if constexpr (KIND == kKindFp8) {
#pragma unroll
                    for (int kk = 0; kk < 4 * KB; ++kk)
                        mma_f8_p(leader, d_tmem, ad + (((kk >> 2) * C::kACol + (kk & 3) * 32) >> 4),
                                 bd + (((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4), idesc,
                                 (acc_flag0 | kk) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4 * KB; ++kk)
                        mma_bf16_p(leader, d_tmem, ad + (((kk >> 2) * C::kACol + (kk & 3) * 32) >> 4),
                                   bd + (((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4), idesc,
                                   (acc_flag0 | kk) ? 1u : 0u);
                }
                mma_commit_p(leader, &empty[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            mma_commit_p(leader, &tfull[acc]);
        }
        // all tensor-core work of this CTA is complete before TMEM is released
        mma_commit_p(leader, drain);
        const long long t0 = clock64();
        while (!mbar_try_wait(drain, 0) && clock64() - t0 < kWaitLimitCycles) {}
    } else if (W4 && warp < kEpi0) {
        // ---------------------------------------------------------------- weight decoders
        const int ct = (warp - 2) * 32 + lane;
        int stage = 0;
        uint32_t phase = 0;
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x) {
            const Tile tl = decode_tile(g, tb, t);
            bool ok = true;
            for (int kt = tl.kt0; kt < tl.kt1; ++kt) {
                if (!role_wait(&full[stage], phase, s_abort, g.err, g.wait_limit)) { ok = false; break; }
                const int nb = min(KB, K64 - kt * KB);
                for (int b = 0; b < nb; ++b)
                    w4_convert_block(sRaw + stage * C::kRawStage + b * C::kRawBlock,
                                     sB + stage * C::kBStage + b * (BN * 128), lut, ct, kConvWarps * 32);
                fence_proxy_async();          // the tensor core reads what these threads wrote
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfready[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
        }
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------------- scale copiers
        // (all lanes run the loop; the elected lane issues)
        if (NVF4) {
            const uint32_t leader = elect_leader();
            const bool is_b = warp == 3;
            const uint64_t sfdesc0 = sdesc_sf(smem_u32(is_b ? sSFB : sSFA));
            const uint32_t col_off = is_b ? C::kSfColsA : 0;
            const int nblk = is_b ? BN / 128 : 1;              // 128-row atoms per K step
            const int sf_stage = is_b ? C::kSfStageB : C::kSfStageA;
            int stage = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x) {
                const Tile tl = decode_tile(g, tb, t);
                bool ok = true;
                for (int kt = tl.kt0; kt < tl.kt1; ++kt) {
                    if (!role_wait(&sffull[stage], phase, s_abort, g.err, g.wait_limit)) { ok = false; break; }
                    tc_fence_after();
                    const int nsteps = min(4 * KB, K64 - 4 * kt * KB);
                    const uint32_t sf_t = tmem + kSfCol0 + stage * C::kSfCols + col_off;
                    const uint64_t sfd = sfdesc0 + ((stage * sf_stage) >> 4);
                    // K step kk of 128-row block h: 4 columns at kk * 4 * nblk + 4 h (so a step's
                    // scales of B rows 0..255 sit in 8 consecutive columns), from smem atom (h, kk)
#pragma unroll
                    for (int kk = 0; kk < 4 * KB; ++kk)
                        for (int h = 0; h < nblk; ++h)
                            if (kk < nsteps)
                                tmem_cp_sf_p(leader, sf_t + kk * 4 * nblk + h * 4, sfd + (h * 4 * KB + kk) * (512 >> 4));
                    mma_commit_p(leader, &sfready[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
            }
            // every copy this warp issued is complete before TMEM is released
            mma_commit_p(leader, &cdrain[is_b ? 1 : 0]);
            const long long t0 = clock64();
            while (!mbar_try_wait(&cdrain[is_b ? 1 : 0], 0) && clock64() - t0 < kWaitLimitCycles) {}
        } else if constexpr (C::kAF32) {
            // ------------------------------------------------------------ A converters (fp32 -> bf16)
            // A stage = KB boxes of 8 rows x 64 fp32 (256-byte rows, unswizzled) -> the SW128 bf16
            // A slot (16-byte chunk c of row r at c ^ (r % 8)), round to nearest even as the
            // combine's cast; then the async proxy is fenced and the MMA told ("sfready")
            const int ct = (warp - 2) * 32 + lane;
            int stage = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x) {
                const Tile tl = decode_tile(g, tb, t);
                const bool copy = g.a_copy != nullptr && tl.n0 == 0;
                bool ok = true;
                for (int kt = tl.kt0; kt < tl.kt1; ++kt) {
                    if (!role_wait(&full[stage], phase, s_abort, g.err, g.wait_limit)) { ok = false; break; }
                    const uint8_t *src = sRaw + stage * C::kRawStage;
                    uint8_t *dst = sA + stage * C::kAStage;
                    for (int u = ct; u < KB * kAF32Rows * 8; u += 64) {
                        const int b = u / (kAF32Rows * 8), rem = u - b * (kAF32Rows * 8);
                        const int r = rem >> 3, c = rem & 7;
                        const float4 *f = reinterpret_cast<const float4 *>(src + b * C::kRawBlock + r * 256 + c * 32);
                        const float4 x0 = f[0], x1 = f[1];
                        const uint4 o = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w),
                                                   pack_bf16x2(x1.x, x1.y), pack_bf16x2(x1.z, x1.w));
                        *reinterpret_cast<uint4 *>(dst + b * C::kACol + r * 128 + ((c ^ (r & 7)) << 4)) = o;
                        const int k0 = (kt * KB + b) * 64 + c * 8;
                        if (copy && r < g.a_rows && k0 < g.K)
                            *reinterpret_cast<uint4 *>(g.a_copy + static_cast<int64_t>(tl.a_row0 + r) * g.K + k0) = o;
                    }
                    fence_proxy_async();      // the tensor core reads what these threads wrote
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sfready[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        constexpr int kChunks = BN / 32 / (C::kEpiWarps / 4);    // 32-column chunks per warp and tile
        static_assert(kChunks == 1 || kChunks % 2 == 0, "chunks are loaded singly or in pairs");
        const int ch0 = ((warp - kEpi0) / 4) * kChunks;          // this warp's share of the columns
        const float *rcp_of = (C::kTables && g.grouped && g.epi == EPI_H_QUANT) ? tb->rcp_h : nullptr;
        if (rcp_of) {
            // the h quantizer's table, built by the epilogue warps alone (named barrier 1) so
            // the producer and MMA roles start at once
            for (int i = threadIdx.x - kEpi0 * 32; i < 256; i += C::kEpiWarps * 32)
                tb->rcp_h[i] = quant_rcp_entry(g.q, i);
            asm volatile("bar.sync 1, %0;" ::"r"(C::kEpiWarps * 32) : "memory");
        }
        float4 *stg = stg_all + (warp - kEpi0) * 256;
        int32_t orow[8];
        auto chunk = [&](const Tile &tl, const EpiRow &er, int ch, const uint32_t (&r)[32]) {
            if (ch * 32 >= tl.cols) return;
            if (C::kStagedCombine && g.epi == EPI_COMBINE)
                combine_staged(g, tl, er, ch * 32, r, stg, lane, orow);
            else
                epilogue_chunk(g, tl, er, row, ch * 32, r, rcp_of);
        };
        int it = 0;
        int t = blockIdx.x;
        Tile tl{};
        EpiRow er{};
        if (t < num_tiles) { tl = decode_tile(g, tb, t); er = epilogue_row(g, tl, row); }
        for (; t < num_tiles && !*s_abort; t += gridDim.x, ++it) {
            // The next tile's row scalars (global loads, some dependent) are fetched before this
            // tile is processed, so their latency overlaps this tile's work.
            Tile tn = tl;
            EpiRow en = er;
            if (t + static_cast<int>(gridDim.x) < num_tiles) {
                tn = decode_tile(g, tb, t + gridDim.x);
                en = epilogue_row(g, tn, row);
            }
            const int acc = C::kNumAcc == 2 ? (it & 1) : 0;
            const uint32_t aphase = C::kNumAcc == 2 ? ((it >> 1) & 1) : (it & 1);
            // A warp whose 32 rows are all past the tile's valid rows reads nothing; it still
            // waits for the accumulator before releasing it, which keeps the release phases
            // of all four warps in step.
            const bool live = quad * 32 < tl.rows;
            if (!role_wait(&tfull[acc], aphase, s_abort, g.err, g.wait_limit)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + acc * kAccCols + (static_cast<uint32_t>(quad * 32) << 16);
            if constexpr (C::kNumAcc == 1) {
                // 256-column NVFP4 tile: this warp's accumulator columns go to registers and
                // the accumulator is released at once (the next tile's MMAs wait only for these
                // loads); then the latent-up's h = bf16(relu(alpha acc)^2) and its quantization,
                // or the latent-down's weighted combine
                uint32_t r[kChunks][32];
                if (live) {
#pragma unroll
                    for (int c = 0; c < kChunks; ++c) tmem_ld32(taddr + (ch0 + c) * 32, r[c]);
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
                if constexpr (C::kStagedCombine) {
                    if (live) {
                        combine_rows(er, lane, orow);
#pragma unroll
                        for (int c = 0; c < kChunks; ++c)
                            if ((ch0 + c) * 32 < tl.cols) combine_staged(g, tl, er, (ch0 + c) * 32, r[c], stg, lane, orow);
                    }
                } else if (live && er.valid) {
#pragma unroll
                    for (int c = 0; c < kChunks; c += 2) {
                        if ((ch0 + c + 2) * 32 <= tl.cols)
                            hquant_from_acc(g, tl, row, (ch0 + c) * 32, er.alpha, r[c], r[c + 1], rcp_of);
                    }
                }
                tl = tn;
                er = en;
                continue;
            }
            if (live) {
                if (C::kStagedCombine && g.epi == EPI_COMBINE) combine_rows(er, lane, orow);
                if constexpr (kChunks == 1) {
                    uint32_t r0[32];
                    tmem_ld32(taddr + ch0 * 32, r0);
                    tmem_wait_ld();
                    chunk(tl, er, ch0, r0);
                }
                // two chunks in flight per wait
#pragma unroll 1
                for (int cp = 0; kChunks > 1 && cp < kChunks; cp += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(taddr + (ch0 + cp) * 32, r0);
                    tmem_ld32(taddr + (ch0 + cp + 1) * 32, r1);
                    tmem_wait_ld();
                    if (rcp_of && (ch0 + cp + 2) * 32 <= tl.cols) {
                        hquant_pair(g, tl, er, row, (ch0 + cp) * 32, r0, r1, rcp_of);
                    } else {
                        chunk(tl, er, ch0 + cp, r0);
                        chunk(tl, er, ch0 + cp + 1, r1);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            tl = tn;
            er = en;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace lmoe
