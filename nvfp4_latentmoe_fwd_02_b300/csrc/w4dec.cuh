// w4dec.cuh -- the W4A16 expert GEMMs at decode size (every expert segment has at most 32 rows).
//
// W4A16 form of the experts (NVIDIA AI releases Nemotron 3 Ultra, quantization paragraph):
// bf16 activations times NVFP4 weights, each weight value code * scale exact in bf16.  At
// decode an expert sees a handful of tokens, so the GEMM streams the expert weights once and
// the cost is (a) HBM and (b) decoding 4-bit codes into bf16.  The operands are swapped
// against gemm_kernel: D^T[n][t] = sum_k W[n][k] * X[t][k], so the decoded weights form the
// A operand, held in tensor memory, and the few token rows form the B operand in shared
// memory.  Decoded weights then never touch shared memory: converter warps write them from
// registers into TMEM with tcgen05.st, and tcgen05.mma reads them there (kind::f16, M = 128
// weight rows, N = NT token rows, K = 16 per instruction).
//
// The contraction runs in "chunks" of 256 elements.  Two rings of shared-memory stages:
//   code ring: per chunk the 128 x 128-byte box of E2M1 codes of the tile's 128 weight rows
//              (tile order, 128-byte swizzle: the converters' per-row reads are bank-conflict
//              free) and the four 512-byte scale atoms of those rows; a converter warp copies its
//              32 rows into registers and releases the stage before decoding, so the stages
//              spend their time in flight from HBM, not waiting for the decode;
//   act ring:  per chunk the NT x 64 bf16 activation boxes of the four 64-element blocks (read
//              by the MMAs, released by their commit).
// Both rings have a multiple of G stages, so that each stage is filled for and consumed by one
// group only (see W4Cfg).
//
// G converter groups (G = 3 for NT = 16, 2 for NT = 32).  Chunk q of the CTA's sequence goes
// to group q % G: its four converter warps (one per TMEM lane quadrant) decode the chunk into
// the group's TMEM weight slot (128 columns), and the group's own MMA warp issues the chunk's
// 16 MMAs into the group's accumulator.  A thread issuing tcgen05.mma while three busy warps
// share its SM sub-partition gets a fraction of the issue slots; one issuer per group keeps
// the MMA issue off the critical path.  The epilogue sums the G partial accumulators.
//
// Warp roles (32 (5 G + 6) threads):
//   warps 0..3               epilogue: tcgen05.ld of the accumulators of lane quadrant w, one
//                            thread per weight row (= output column), a loop over the tokens
//   warps 4 .. 4G+3          converters: group (w - 4) / 4, lane quadrant w % 4
//   warp 4G+4                TMA producer of the code ring (elected lane)
//   warp 4G+5                TMA producer of the act ring (elected lane)
//   warps 4G+6 .. 5G+5       MMA issuers, one per group (elected lane); the first allocates TMEM
// TMEM: accumulator (group g, buffer a) at columns (2g + a) NT; weight slot g at 2 G NT + 128 g.
#pragma once
#include "gemm.cuh"

namespace lmoe {

template <int NT>
struct W4Cfg {
    static constexpr int G = NT == 16 ? 3 : 2;              // converter groups = weight slots = MMA issuers
    static constexpr int kConvWarp0 = 4;
    static constexpr int kProdWarp = kConvWarp0 + 4 * G;    // code ring
    static constexpr int kActWarp = kProdWarp + 1;          // act ring
    static constexpr int kMmaWarp0 = kActWarp + 1;
    static constexpr int kWarps = kMmaWarp0 + G;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr uint32_t kSlotCol0 = 2 * G * NT;       // first TMEM column of the weight slots
    static constexpr int kCodeBytes = 128 * 128;            // one tiled code box: 128 rows x 256 elements
    static constexpr int kCodeStage = kCodeBytes + 4 * 512; // + four scale atoms
    static constexpr int kActBlock = NT * 128;              // NT rows x 64 bf16 (one SW128 box)
    static constexpr int kActStage = 4 * kActBlock;
    static constexpr int kStagesC = NT == 16 ? 9 : 8;
    static constexpr int kStagesA = NT == 16 ? 6 : 4;
    static constexpr int kBarBytes = 512;
    // Chunk q fills stage q % S of a ring and is consumed by group q % G.  With S a multiple of G
    // every stage belongs to one group, whose consumers take its fills in order.  Otherwise a
    // consumer that is ahead could wait on a stage whose previous fill (another group's chunk)
    // has not landed yet: the barrier is then one phase short, its parity reads as "complete",
    // and the MMA would read the stage before its data arrived.
    static_assert(kStagesC % G == 0 && kStagesA % G == 0, "each ring stage belongs to one group");
    static_assert(kCodeStage % 1024 == 0 && kActStage % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled boxes");
    static_assert(kSlotCol0 + G * 128 <= 512, "TMEM budget");
};
// Waiting roles sleep on their barrier (mbar_try_wait_sleep) instead of polling.
constexpr uint32_t kW4Sleep = 2000;

template <int NT>
constexpr int w4dec_smem_bytes() {
    using C = W4Cfg<NT>;
    return 1024 + C::kStagesC * C::kCodeStage + C::kStagesA * C::kActStage + C::kBarBytes +
           static_cast<int>((sizeof(SmemTables) + 15) & ~static_cast<size_t>(15));
}

// 32 lanes x 32 consecutive 32-bit TMEM columns from registers (thread i writes lane i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 lanes x 16 columns into registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem)^T, bf16 inputs, fp32 accumulator; A is read from TMEM
// (lane = row of A, column j = elements 2j, 2j + 1 of K).
__device__ __forceinline__ void mma_bf16_ts_p(uint32_t leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(leader)
        : "memory");
}

// Two E4M3 scale bytes (low 16 bits of s) -> f16x2, exact (every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t s) {
    uint32_t r;
    asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(r) : "r"(s));
    return r;
}
// Four bytes of E2M1 code pairs -> four f16x2 (low nibble -> low half), exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&x)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
        : "r"(w));
}
// (code pair as f16x2) * (scale as f16, low half of s) -> bf16x2.  Each product of an E2M1
// value and an E4M3 value has at most 6 significant bits and lies in [2^-10, 2688] (or is
// zero), so the fp32 products are exact and so is their rounding to bf16.
__device__ __forceinline__ uint32_t scale_pair_bf16x2(uint32_t x, uint32_t s) {
    uint32_t d;
    asm("{\n\t.reg .f16 l, h, s, t;\n\t.reg .f32 fl, fh;\n\tmov.b32 {l, h}, %1;\n\tmov.b32 {s, t}, %2;\n\t"
        "fma.rn.f32.f16 fl, l, s, 0f80000000;\n\tfma.rn.f32.f16 fh, h, s, 0f80000000;\n\t"
        "cvt.rn.bf16x2.f32 %0, fh, fl;\n\t}"
        : "=r"(d)
        : "r"(x), "r"(s));
    return d;
}

// One thread decodes the 64 weights of its row in one 64-element block: 32 code bytes (two
// 16-byte pieces, already in registers) and the row's four block scales -> 32 bf16x2.
__device__ __forceinline__ void w4_decode_row64(const uint4 &c0, const uint4 &c1, uint32_t sf4, uint32_t (&o)[32]) {
    const uint32_t s01 = e4m3x2_to_f16x2(sf4 & 0xFFFFu), s23 = e4m3x2_to_f16x2(sf4 >> 16);
    const uint32_t sc[4] = {s01, s01 >> 16, s23, s23 >> 16};   // scale of 16-element group g
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {           // word i: elements 8i .. 8i + 7, group i / 2
        uint32_t x[4];
        e2m1x8_to_f16x2(cw[i], x);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[4 * i + j] = scale_pair_bf16x2(x[j], sc[i >> 1]);
    }
}

// The kernel.  Grouped launch over the expert segments (GemmArgs: tables, sfb, NB, b_kt =
// chunks per tile = k_tiles, epi = EPI_H_BF16 or EPI_COMBINE, out, alpha, and for the combine
// row_slot, route_w, topk, ld_out).  tmX: bf16 activations [R][K], SW128 boxes of 64 x NT;
// tmW: expert codes in tile order, SW128 boxes of 128 bytes x 128 rows.
template <int NT>
__global__ void __launch_bounds__(W4Cfg<NT>::kThreads, 1)
    w4_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const GemmArgs g) {
    using C = W4Cfg<NT>;
    constexpr int SC = C::kStagesC, SA = C::kStagesA, G = C::G;
    static_assert(NT == 16 || NT == 32, "token rows per tile");
    static_assert((2 * SC + 2 * SA + 3 * G + 4) * 8 + 8 <= C::kBarBytes, "barrier area");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *ring_c = smem;                                  // code ring
    uint8_t *ring_a = ring_c + SC * C::kCodeStage;           // act ring
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring_a + SA * C::kActStage);
    uint64_t *fullc = bars, *emptyc = fullc + SC, *fulla = emptyc + SC, *emptya = fulla + SA;
    uint64_t *aready = emptya + SA, *afree = aready + G;
    uint64_t *tfull = afree + G, *tempty = tfull + 2, *drain = tempty + 2;   // drain: one per MMA warp
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(drain + G);
    volatile int *s_abort = reinterpret_cast<volatile int *>(s_tmem + 1);
    SmemTables *tb = reinterpret_cast<SmemTables *>(reinterpret_cast<uint8_t *>(bars) + C::kBarBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC; ++s) { mbar_init(&fullc[s], 1); mbar_init(&emptyc[s], 4); }   // the group's four warps
        for (int s = 0; s < SA; ++s) { mbar_init(&fulla[s], 1); mbar_init(&emptya[s], 1); }   // the MMA commit
        for (int i = 0; i < G; ++i) { mbar_init(&aready[i], 4); mbar_init(&afree[i], 1); mbar_init(&drain[i], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], G); mbar_init(&tempty[a], 4); }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == C::kProdWarp && lane == 0) { prefetch_tmap(&tmW); }
    if (warp == C::kActWarp && lane == 0) { prefetch_tmap(&tmX); }
    if (warp == C::kMmaWarp0) { tmem_alloc(s_tmem, 512); tmem_relinquish(); }
    auto load_tables = [&]() {
        for (int i = threadIdx.x; i <= g.E; i += blockDim.x) {
            tb->mt[i] = __ldg(g.mt_start + i);
            if (i < g.E) tb->cnt[i] = __ldg(g.counts + i);
        }
    };
    const int K64 = g.K / 64;
    const int nch = g.k_tiles;                   // 256-element chunks per tile
    // chunk q of this CTA's sequence (tile it, chunk kt: q = it nch + kt) belongs to group q % G;
    // a group with no chunk in a tile (nch < G) leaves its accumulator of that tile unwritten
    auto takes_part = [&](int it, int grp) { return nch >= G || ((grp - (it * nch) % G) + G) % G < nch; };
    auto sfb_of = [&](const Tile &tl) {
        return g.sfb + (static_cast<size_t>(tl.e) * g.NB + (tl.n0 >> 7)) * K64 * 512;
    };
    // one chunk of codes and scale atoms into code stage s
    auto load_codes = [&](uint32_t leader, int s, const Tile &tl, int kt) {
        const int nb = min(4, K64 - 4 * kt);
        uint8_t *st = ring_c + s * C::kCodeStage;
        mbar_arrive_expect_tx_p(leader, &fullc[s], static_cast<uint32_t>(C::kCodeBytes + nb * 512));
        tma_load_2d_p(leader, smem_u32(st), &tmW, &fullc[s], 0, ((tl.e * g.NB + (tl.n0 >> 7)) * g.b_kt + kt) * 128);
        bulk_load_p(leader, smem_u32(st + C::kCodeBytes), sfb_of(tl) + static_cast<size_t>(kt) * 2048, nb * 512,
                    &fullc[s]);
    };
    // Weights (codes and scale atoms) of the first ring pass go out before the wait on the
    // previous grid: they are static, and the segment tables come from the router, which
    // completed before the previous kernel of the forward began.
    int npre = 0;
    if (g.preload) {
        load_tables();
        __syncthreads();
        if (warp == C::kProdWarp) {
            const uint32_t leader = elect_leader();
            if (static_cast<int>(blockIdx.x) < tb->mt[g.E] * g.n_tiles) {
                const Tile tl = decode_tile(g, tb, blockIdx.x);
                npre = min(SC, nch);
                for (int s = 0; s < npre; ++s) load_codes(leader, s, tl, s);
            }
        }
    }
    pdl_wait();      // the previous kernel's outputs (activations, tables) are complete
    pdl_trigger();
    if (!g.preload) load_tables();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int num_tiles = tb->mt[g.E] * g.n_tiles;

    if (warp == C::kProdWarp || warp == C::kActWarp) {
        // ---------------------------------------------------------------- producers
        const bool codes = warp == C::kProdWarp;
        const int S = codes ? SC : SA;
        uint64_t *full = codes ? fullc : fulla, *empty = codes ? emptyc : emptya;
        const uint32_t leader = elect_leader();
        int stage = 0;
        uint32_t phase = 0, issued = codes ? (1u << npre) - 1u : 0u, issued_phase = 0;
        int q = 0;
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x) {
            const Tile tl = decode_tile(g, tb, t);
            bool ok = true;
            for (int kt = 0; kt < nch; ++kt, ++q) {
                if (!codes || q >= npre) {
                    if (!role_wait(&empty[stage], phase ^ 1, s_abort, g.err, g.wait_limit, kW4Sleep)) { ok = false; break; }
                    if (codes) {
                        load_codes(leader, stage, tl, kt);
                    } else {
                        const int nb = min(4, K64 - 4 * kt);
                        uint8_t *st = ring_a + stage * C::kActStage;
                        mbar_arrive_expect_tx_p(leader, &full[stage], static_cast<uint32_t>(nb * C::kActBlock));
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            if (b < nb)
                                tma_load_2d_p(leader, smem_u32(st + b * C::kActBlock), &tmX, &full[stage],
                                              (4 * kt + b) * 64, tl.a_row0);
                    }
                }
                issued |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == S) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
        }
        if (*s_abort) {
            // the last copies issued to each stage have landed before the CTA leaves (bounded)
            for (int s = 0; s < S; ++s) {
                if (!((issued >> s) & 1u)) continue;
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[s], (issued_phase >> s) & 1u) && clock64() - t0 < kWaitLimitCycles / 8) {}
            }
        }
    } else if (warp >= C::kMmaWarp0) {
        // ---------------------------------------------------------------- MMA issuers (one per group)
        const int grp = warp - C::kMmaWarp0;
        const uint32_t leader = elect_leader();
        const uint32_t idesc = idesc_bf16(kBM, NT);
        const uint64_t bdesc0 = sdesc_sw128(smem_u32(ring_a));
        const uint32_t a0 = tmem + C::kSlotCol0 + grp * 128;
        int q = 0, it = 0;
        // injected fault: drain[0] gets its only arrival after the tile loop, so this wait runs out
        if (g.inject_wait && grp == 0) role_wait(&drain[0], 0, s_abort, g.err, g.wait_limit, kW4Sleep);
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x, ++it) {
            const int acc = it & 1;
            if (!role_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, s_abort, g.err, g.wait_limit, kW4Sleep)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (2 * grp + acc) * NT;
            bool ok = true, first = true;
            for (int kt = 0; kt < nch; ++kt, ++q) {
                if (q % G != grp) continue;
                const int sa = q % SA;
                if (!role_wait(&fulla[sa], (q / SA) & 1, s_abort, g.err, g.wait_limit, kW4Sleep) ||
                    !role_wait(&aready[grp], (q / G) & 1, s_abort, g.err, g.wait_limit, kW4Sleep)) { ok = false; break; }
                tc_fence_after();
                const int nb = min(4, K64 - 4 * kt);
                const uint64_t bd = bdesc0 + ((sa * C::kActStage) >> 4);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    if (kk < 4 * nb)
                        mma_bf16_ts_p(leader, d_tmem, a0 + kk * 8,
                                      bd + (((kk >> 2) * C::kActBlock + (kk & 3) * 32) >> 4), idesc,
                                      (!first || kk) ? 1u : 0u);
                first = false;
                mma_commit_p(leader, &emptya[sa]);
                mma_commit_p(leader, &afree[grp]);
            }
            if (!ok) break;
            if (first) {                           // no chunk of this tile: nothing to wait for
                if (leader) mbar_arrive(&tfull[acc]);
            } else {
                mma_commit_p(leader, &tfull[acc]);
            }
        }
        // all tensor-core work of this warp is complete before TMEM is released
        mma_commit_p(leader, &drain[grp]);
        const long long t0 = clock64();
        while (!mbar_try_wait(&drain[grp], 0) && clock64() - t0 < kWaitLimitCycles) {}
    } else if (warp >= C::kConvWarp0) {
        // ---------------------------------------------------------------- converters
        const int grp = (warp - C::kConvWarp0) >> 2, quad = warp & 3;
        const int r = quad * 32 + lane;                       // weight row of the tile = TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kSlotCol0 + grp * 128;
        int q = 0;
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x) {
            bool ok = true;
            for (int kt = 0; kt < nch; ++kt, ++q) {
                if (q % G != grp) continue;
                const int sc = q % SC;
                if (!role_wait(&fullc[sc], (q / SC) & 1, s_abort, g.err, g.wait_limit, kW4Sleep)) { ok = false; break; }
                const int nb = min(4, K64 - 4 * kt);
                // this row's codes and scales into registers, then the stage goes back to the producer
                const uint8_t *st = ring_c + sc * C::kCodeStage;
                const uint8_t *codes_row = st + r * 128;
                uint4 cv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) cv[j] = *reinterpret_cast<const uint4 *>(codes_row + ((j ^ (r & 7)) << 4));
                uint32_t sf[4];
                const uint8_t *sf_row = st + C::kCodeBytes + (r & 31) * 16 + ((r >> 5) & 3) * 4;
#pragma unroll
                for (int b = 0; b < 4; ++b) sf[b] = b < nb ? *reinterpret_cast<const uint32_t *>(sf_row + b * 512) : 0u;
                __syncwarp();
                if (lane == 0) mbar_arrive(&emptyc[sc]);
                if (!role_wait(&afree[grp], ((q / G) & 1) ^ 1, s_abort, g.err, g.wait_limit, kW4Sleep)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if (b < nb) {
                        uint32_t o[32];
                        w4_decode_row64(cv[2 * b], cv[2 * b + 1], sf[b], o);
                        tmem_st32(lane_base + b * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&aready[grp]);
            }
            if (!ok) break;
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int quad = warp;
        const int row = quad * 32 + lane;                     // weight row = output column n0 + row
        int it = 0;
        for (int t = blockIdx.x; t < num_tiles && !*s_abort; t += gridDim.x, ++it) {
            const Tile tl = decode_tile(g, tb, t);
            // per-token scalars, fetched before the accumulators are ready: lane j holds token j's
            const float alpha = __ldg(g.alpha + tl.e);
            int slot_l = -1;
            float w_l = 0.0f;
            if (g.epi == EPI_COMBINE && lane < tl.rows) {
                slot_l = __ldg(g.row_slot + tl.a_row0 + lane);
                if (slot_l >= 0) w_l = __ldg(g.route_w + slot_l);
            }
            const int acc = it & 1;
            if (!role_wait(&tfull[acc], (it >> 1) & 1, s_abort, g.err, g.wait_limit, kW4Sleep)) break;
            tc_fence_after();
            // the groups' partial accumulators, summed
            uint32_t v[G][NT];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const uint32_t taddr = tmem + (2 * k + acc) * NT + (static_cast<uint32_t>(quad * 32) << 16);
                if (!takes_part(it, k)) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) v[k][j] = 0u;   // +0.0f
                } else if constexpr (NT == 16) {
                    tmem_ld16(taddr, v[k]);
                } else {
                    tmem_ld32(taddr, v[k]);
                }
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            const bool colv = row < tl.cols;
            const int n = tl.n0 + row;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (j >= tl.rows) break;
                float a = __uint_as_float(v[0][j]);
#pragma unroll
                for (int k = 1; k < G; ++k) a = __fadd_rn(a, __uint_as_float(v[k][j]));
                if (g.epi == EPI_H_BF16) {
                    if (colv) {
                        const float u = fmaxf(__fmul_rn(alpha, a), 0.0f);
                        static_cast<__nv_bfloat16 *>(g.out)[static_cast<int64_t>(tl.a_row0 + j) * g.N + n] =
                            __float2bfloat16_rn(__fmul_rn(u, u));
                    }
                } else {
                    const int slot = __shfl_sync(0xffffffffu, slot_l, j);
                    const float ws = __shfl_sync(0xffffffffu, w_l, j);
                    if (colv && slot >= 0)
                        red_add_f32(static_cast<float *>(g.out) + static_cast<int64_t>(slot / g.topk) * g.ld_out + n,
                                    __fmul_rn(ws, __fmul_rn(alpha, a)));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace lmoe
