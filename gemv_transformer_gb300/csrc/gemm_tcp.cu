// gemm_tcp.cu -- persistent tcgen05 GEMM with bf16 X (the workspace path).
//
// Same contraction and epilogue as gemm_tc.cu (cortiq-engine 0.8.49 ae_gemm /
// ae_put: Y = [gelu](X.W^T + bias) [+ old Y]), with X already rounded to bf16
// in a workspace.  What changes is the schedule, built around the facts that a
// 128 x BN tile's output (64-128 KB of f32) takes about as long to write as its
// MMAs take to run, and that the tile count is not a multiple of the SM count:
//
//   * one CTA per SM walks a static list of tiles (tile t -> row block t % RB,
//     column block t / RB, so CTAs running together share W columns in L2);
//   * TMEM holds two accumulators: the MMA warp fills one tile's accumulator
//     while the epilogue warps drain the other, so output writes overlap MMAs;
//   * warps 0 and 1 stream A (X bf16) and B (W) tiles by TMA through a stage
//     ring across tile boundaries, each warp its own operand (a TMA issue holds
//     its thread for a while, so two issuers keep more bytes in flight); a stage
//     spans KS 128-byte swizzle atoms of k (64 bf16 each), since the bytes the
//     TMA unit of one SM delivers per stage grow with the stage size;
//   * warp 2 issues tcgen05.mma (M=128, N=BN, K=16);
//   * pair mode (a cluster of two CTAs on two SMs, cta_group::2): a tile is
//     256 x BN; each CTA stages its own 128 rows of A and BN/2 rows of B, the
//     even-rank CTA issues M = 256 MMAs over both CTAs' shared memory, and each
//     CTA's TMEM receives its 128 rows of the accumulator.  Per SM this halves
//     the operand bytes per MMA flop relative to a 128 x BN tile, and operand
//     delivery (bytes in flight per SM over the L2 latency) is what bounds the
//     one-SM schedule;
//   * helper mode (a cluster of h + 1 CTAs, h = 2 or 3, for shapes with too few
//     tiles to fill the SMs): CTAs 0..h-1 each own one 128 x 128 tile and run
//     the first h / (h + 1) of its k stages; CTA h runs the rest of all h tiles,
//     each into a TMEM accumulator of its own, and as each finishes writes that
//     partial accumulator into the owner tile's block of Y (scratch until the
//     owner's epilogue overwrites it; so Y must not overlap the residual) and
//     signals the owner through a cluster barrier; the owner loads it back into
//     its idle A stage buffers and adds it before its epilogue.  The sum order
//     is fixed, so results are deterministic; e.g. 128 SMs work on 96 tiles
//     instead of 96 SMs;
//   * 16 epilogue warps (4 per TMEM lane quarter) take 32x32 blocks: tcgen05.ld,
//     bias (one coalesced load per block, broadcast by shuffles) and erf-GELU in
//     registers, the block into a 128-byte-swizzled shared buffer, residual added
//     from a TMA load of the same block, and the block written by a TMA store
//     (the hardware clips rows >= n and columns >= m).
// All waits are bounded; an expired wait aborts the CTA's roles, which drain
// their copies and MMAs, meet, free TMEM and return.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_ptx.cuh"
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

using namespace tc;

constexpr int kEpi = 16;                       // epilogue warps
constexpr int kRoles = 3;                      // A producer, B producer, MMA issuer
constexpr int kThreads = (kRoles + kEpi) * 32;
constexpr int kAtomA = BM * BK * 2;            // one 128-row swizzle atom of A: 16 KB
constexpr int kStgBytes = 32 * 32 * 4;         // one 32x32 f32 block

// Schedules: one SM per tile, an SM pair per 256-row tile, or two tile owners
// and a helper per cluster of three.
enum Sched : int { kData = 0, kPair = 1, kHelp = 2 };

template <int BN, int KS, int SCH>
struct PLayout {
    static constexpr bool PAIR = SCH == kPair;
    static constexpr int kBRows = PAIR ? BN / 2 : BN;     // W rows this CTA stages
    static constexpr int kABytes = KS * kAtomA;            // A of a stage
    static constexpr int kBAtom = kBRows * BK * 2;         // one swizzle atom of B
    static constexpr int kBBytes = KS * kBAtom;            // B of a stage
    static constexpr int kFit = (216 * 1024 - kEpi * kStgBytes) / (kABytes + kBBytes);
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static_assert(kStages >= 2, "at least two stages");
    static constexpr size_t kA = 0;
    static constexpr size_t kB = kA + (size_t)kStages * kABytes;
    static constexpr size_t kStg = kB + (size_t)kStages * kBBytes;
    static constexpr size_t kBars = kStg + (size_t)kEpi * kStgBytes;
    // full[S], empty[S], tfull[4], tempty[2], rbar[kEpi], drain, pbar[kEpi], recv[kEpi]
    static constexpr int kNumBars = 2 * kStages + 6 + kEpi + 1 + kEpi + kEpi;
    // Helper mode: a 128 x BN f32 partial accumulator fits the A stage buffers.
    static_assert(SCH != kHelp || (BN == 128 && kStages * kABytes >= BM * BN * 4),
                  "helper hand-over buffer");
    static constexpr size_t kMisc = kBars + kNumBars * sizeof(uint64_t);
    static constexpr size_t kBytes = kMisc + 16 + 1024;
};

// Helper mode: the owners' share of a tile's KB stages.  The helper's share is
// seven eighths of an even split (KB / (h + 1) per tile), since each hand-over
// (a 64 KB store while its next segment streams in) costs it some time (for the
// encoder down projection, KB = 32, h = 3: owners 25 stages; 24 or 26 made the
// whole benchmark step 0.7-0.8 us slower in an A/B on GB300).
__host__ __device__ constexpr int help_split(int KB, int h) {
    return KB - ((7 * KB) / (8 * (h + 1)) > 1 ? (7 * KB) / (8 * (h + 1)) : 1);
}

// DUAL: the epilogue also writes the second output band (columns m.. of Y); a
// separate instantiation, so that kernels without it carry none of its code.
template <int BN, int KS, int SCH, bool DUAL = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcp_kernel(const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap ymap,
                    const __grid_constant__ CUtensorMap rmap,
                    const __grid_constant__ CUtensorMap y2map, const GemmArgs a) {
    // Barriers, tensor memory and descriptors are set up before waiting for the
    // previous grid (they touch nothing it writes); global memory after.
    pdl_launch();
    using L = PLayout<BN, KS, SCH>;
    constexpr bool PAIR = SCH == kPair, HELP = SCH == kHelp;
    static_assert(!(DUAL && HELP), "the helper schedule has no second band");
    constexpr int S = L::kStages;
    constexpr int TM = PAIR ? 2 * BM : BM;  // tile rows
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem + L::kA;
    uint8_t *sB = smem + L::kB;
    uint8_t *sStg = smem + L::kStg;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;   // [4]: helper mode uses one per segment
    uint64_t *tempty = tfull + 4;
    uint64_t *rbar = tempty + 2;
    uint64_t *drain = rbar + kEpi;
    uint64_t *pbar = drain + 1;    // helper mode, in an owner: warp w's partial block loaded
    uint64_t *recv = pbar + kEpi;  // helper mode, in an owner: warp w's partial block is in Y
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Pair and helper modes: CTA `rank` of cluster `unit`; otherwise every CTA is
    // its own unit.
    const uint32_t rank = (PAIR || HELP) ? cluster_ctarank() : 0u;
    const int csize = PAIR ? 2 : (HELP ? (int)cluster_nctarank() : 1);
    const int h = csize - 1;       // helper mode: tile owners per cluster
    const int unit = (int)blockIdx.x / csize;
    const int units = (int)gridDim.x / csize;
    const bool leader = rank == 0;
    const bool helper = HELP && (int)rank == h;
    const int RB = (a.n + TM - 1) / TM, CB = (a.m + BN - 1) / BN;
    const int tiles = RB * CB;
    const int KB = (a.k + KS * BK - 1) / (KS * BK);  // stages per tile
    const uint64_t limit = a.wait_limit;
    // This CTA's work as segments: (tile, k stages [kb0, kb1)), in processing
    // order.  Helper mode: owner r takes stages [0, ks) of tile h * unit + r, the
    // helper stages [ks, KB) of all h tiles.
    const int ks_own = HELP ? help_split(KB, h) : KB;
    int nseg;
    if (HELP) {
        const int left = tiles - h * unit;
        nseg = helper ? (left < h ? left : h) : ((int)rank < left ? 1 : 0);
        if (nseg < 0) nseg = 0;
    } else {
        nseg = unit < tiles ? (tiles - unit + units - 1) / units : 0;
    }
    auto seg_tile = [&](int i) {
        return HELP ? h * unit + (helper ? i : (int)rank) : unit + i * units;
    };
    // TMEM accumulator and tfull barrier of segment i (helper mode: one each).
    auto seg_buf = [&](int i) { return HELP ? i : (i & 1); };
    const int kb0 = helper ? ks_own : 0;
    const int kb1 = (HELP && !helper) ? ks_own : KB;

    if (threadIdx.x == 32) {
        prefetch_tmap(&xmap);
        prefetch_tmap(&wmap);
        prefetch_tmap(&ymap);
        if (a.flags & kResidual) prefetch_tmap(&rmap);
        if (DUAL) prefetch_tmap(&y2map);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // One expect_tx arrival per producer of this CTA; in pair mode the
            // even CTA's producers expect the bytes of both CTAs' copies.
            mbar_init(&full[s], 2);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 4; ++b) mbar_init(&tfull[b], 1);
        for (int b = 0; b < 2; ++b)
            mbar_init(&tempty[b], PAIR ? 2 * kEpi : kEpi);  // both CTAs' epilogue warps
        for (int w = 0; w < kEpi; ++w) mbar_init(&rbar[w], 1);
        mbar_init(drain, 1);
        for (int w = 0; w < kEpi; ++w) mbar_init(&pbar[w], 1);
        for (int w = 0; w < kEpi; ++w) mbar_init(&recv[w], 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    // TMEM: two accumulators of BN f32 columns x 128 lanes (a helper: one per
    // segment, up to three, in a power-of-two allocation).
    constexpr uint32_t kCols = 2 * BN <= 256 ? 256u : 512u;
    const uint32_t ncols = helper ? 512u : kCols;
    if (warp == 2) {
        if (PAIR) {   // one warp of each CTA of the pair allocates collectively
            asm volatile(
                "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                    smem_addr(tmem_slot)),
                "r"(ncols)
                : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile(
                "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                    smem_addr(tmem_slot)),
                "r"(ncols)
                : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncwarp();
    if (PAIR || HELP)
        cluster_sync_all();  // every CTA's barriers exist before any remote arrival
    else
        __syncthreads();
    tc_fence_after();
    // Stage s of one operand: KS swizzle atoms of k at row y (pair mode: the copies
    // of both CTAs complete on the even CTA's full[s]).
    auto load_stage = [&](bool isA, int s, int kb, int y) {
        const CUtensorMap *map = isA ? &xmap : &wmap;
        const int atom = isA ? kAtomA : L::kBAtom;
        const int sbytes = isA ? L::kABytes : L::kBBytes;
        uint8_t *dst = (isA ? sA : sB) + (size_t)s * sbytes;
        if (PAIR) {
            if (leader) mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * sbytes));
            const uint32_t bar = map_to_rank(&full[s], 0);
#pragma unroll
            for (int u = 0; u < KS; ++u)
                tma_load_2d_pair(dst + u * atom, map, (kb * KS + u) * BK, y, bar);
        } else {
            mbar_arrive_expect_tx(&full[s], (uint32_t)sbytes);
#pragma unroll
            for (int u = 0; u < KS; ++u)
                tma_load_2d(dst + u * atom, map, (kb * KS + u) * BK, y, &full[s]);
        }
    };
    auto row_of = [&](bool isA, int t) {
        return isA ? (t % RB) * TM + (PAIR ? (int)rank * BM : 0)
                   : (t / RB) * BN + (PAIR ? (int)rank * L::kBRows : 0);
    };
    // The caller's weights are not written by the previous kernel: the B producer
    // requests its first stage before the grid-dependency wait, while that kernel
    // finishes (X, which it may write, waits).
    const bool b_early = a.w_early && nseg > 0 && kb0 < kb1;
    if (b_early && warp == 1 && lane == 0) load_stage(false, 0, kb0, row_of(false, seg_tile(0)));
    pdl_wait();
    const uint32_t tmem = *tmem_slot;

    if (warp < 2) {
        // --------------------------------------------------------- producers
        // Warp 0 loads A (X rows), warp 1 loads B (W rows); KS atoms per stage.
        if (lane == 0) {
            const bool isA = warp == 0;
            long long q = 0;  // stages issued
            bool ok = true;
            for (int i = 0; i < nseg && ok; ++i) {
                const int y = row_of(isA, seg_tile(i));
                for (int kb = kb0; kb < kb1; ++kb, ++q) {
                    const int s = (int)(q % S);
                    if (q >= S && !wait_or_abort(&empty[s], (uint32_t)(((q / S) - 1) & 1),
                                                 abort_flag, limit, a.status)) {
                        ok = false;
                        break;
                    }
                    if (q == 0 && !isA && b_early) continue;  // issued before the wait
                    load_stage(isA, s, kb, y);
                }
            }
            if (!PAIR || leader) {
                for (long long d = (q > S ? q - S : 0); d < q; ++d)
                    mbar_wait(&full[d % S], (uint32_t)((d / S) & 1), kDrainPolls);
            } else if (!ok) {
                // The odd CTA's copies complete on its peer's barriers, which it
                // cannot poll: after an abort it gives them ample time to land
                // before the final cluster barrier lets the peer exit.  Without
                // an abort every copy is consumed by an MMA before that barrier.
                for (int i = 0; i < 256; ++i) __nanosleep(1000);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && (leader || !PAIR)) {
            constexpr uint32_t idesc = idesc_bf16(TM, BN);
            long long q = 0;
            bool ok = true;
            for (int it = 0; it < nseg && ok; ++it) {
                const int b = seg_buf(it);
                if (!HELP && it >= 2) {
                    const uint32_t ph = (uint32_t)(((it >> 1) - 1) & 1);
                    ok = PAIR ? wait_or_abort_cluster(&tempty[b], ph, abort_flag, limit, a.status)
                              : wait_or_abort(&tempty[b], ph, abort_flag, limit, a.status);
                    if (!ok) break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kb = kb0; kb < kb1; ++kb, ++q) {
                    const int s = (int)(q % S);
                    if (!wait_or_abort(&full[s], (uint32_t)((q / S) & 1), abort_flag, limit,
                                       a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(sA + (size_t)s * L::kABytes);
                    const uint32_t b0 = smem_addr(sB + (size_t)s * L::kBBytes);
#pragma unroll
                    for (int u = 0; u < KS; ++u)
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = smem_desc_sw128(a0 + u * kAtomA + kk * 32);
                            const uint64_t bd = smem_desc_sw128(b0 + u * L::kBAtom + kk * 32);
                            const uint32_t acc = (kb > kb0 || u > 0 || kk > 0) ? 1u : 0u;
                            if (PAIR)
                                tc_mma_pair(d, ad, bd, idesc, acc);
                            else
                                tc_mma(d, ad, bd, idesc, acc);
                        }
                    if (PAIR)
                        tc_commit_pair_mc(&empty[s], 3);  // frees the stage in both CTAs
                    else
                        tc_commit(&empty[s]);
                }
                if (ok) {
                    if (PAIR)
                        tc_commit_pair_mc(&tfull[b], 3);
                    else
                        tc_commit(&tfull[b]);
                }
            }
            // Completes when every MMA issued so far, and the arrivals committed
            // before it, are done: needed after an abort, and in pair mode so
            // that no commit still targets the odd CTA when the pair exits.
            if (PAIR) {
                tc_commit_pair(drain);
                mbar_wait(drain, 0, kDrainPolls);
            } else if (!ok) {
                tc_commit(drain);
                mbar_wait(drain, 0, kDrainPolls);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - kRoles;              // 0..15
        const int q = warp & 3;                    // TMEM lane quarter of this warp
        // A lane quarter's BN columns are 32-column blocks; warp cg of the quarter
        // takes blocks cg, cg + 4, ... (BN = 192: two warps take two, two take one).
        constexpr int NBQ = BN / 32;
        constexpr int NB = (NBQ + 3) / 4;          // blocks per warp at most
        const int cg = ew >> 2;                    // which column group
        uint8_t *stg = sStg + ew * kStgBytes;
        uint32_t rphase = 0;
        bool ok = true;
        bool stored = false;
        bool hfail = false;  // helper mode: a segment could not be served
        const uint32_t tempty_at = PAIR ? map_to_rank(&tempty[0], 0) : 0u;
        for (int it = 0; it < nseg && ok; ++it) {
            const int t = seg_tile(it);
            const int b = seg_buf(it);
            const uint32_t tph = HELP ? 0u : (uint32_t)((it >> 1) & 1);
            if (HELP && helper) {
                // Helper: as each segment's MMAs finish, its partial accumulator goes
                // to the owner tile's block of Y (staging buffer + TMA store); once
                // the store is complete the owner's warp is signalled.  An owner that
                // cannot be served (an expired wait here) is told so: its abort flag
                // is set before the signal.
                const int r = t - h * unit;
                const int hr = (t % RB) * BM + q * 32, hc = (t / RB) * BN + cg * 32;
                // After a failure every later owner is declined too (each is signalled).
                bool serve = !hfail && wait_or_abort(&tfull[b], 0u, abort_flag, limit, a.status);
                serve = __all_sync(0xFFFFFFFFu, serve);
                if (serve) {
                    tc_fence_after();
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + cg * 32),
                              v);
                    if (stored) {
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    fence_proxy_async_smem();  // generic-proxy writes -> TMA store reads
                    __syncwarp();
                    stored = true;
                }
                if (lane == 0) {
                    if (serve) {
                        tma_store_2d(&ymap, hc, hr, stg);
                        bulk_commit();
                        bulk_wait0();                // the block is in Y
                        fence_proxy_async_global();
                    } else {
                        st_cluster_u32(map_to_rank((const void *)abort_flag, (uint32_t)r), 1u);
                    }
                    mbar_arrive_cluster(map_to_rank(&recv[ew], (uint32_t)r));
                }
                __syncwarp();
                if (!serve) hfail = true;
                if (it == nseg - 1 && hfail) ok = false;
                continue;
            }
            const int i0 = (t % RB) * TM + (PAIR ? (int)rank * BM : 0);
            const int jt = (t / RB) * BN;          // the tile's first column
            const int j0 = jt + cg * 32;           // this warp's first block
            const int r0 = i0 + q * 32;            // first row of this warp's blocks
            // Everything that does not need the accumulator is fetched while the
            // MMAs still run: this warp's bias values (lane c holds column c of
            // each block) and the first block's old Y (residual) by TMA.
            float bl[NB];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const int jc = jt + (cg + 4 * u) * 32 + lane;
                bl[u] = ((a.flags & kBias) && cg + 4 * u < NBQ && jc < a.m) ? __ldg(a.bias + jc)
                                                                              : 0.f;
            }
            // The staging block is free once the previous store has read it.
            if (stored) {
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
            }
            if ((a.flags & kResidual) && lane == 0) {
                mbar_arrive_expect_tx(&rbar[ew], (uint32_t)kStgBytes);
                tma_load_2d(stg, &rmap, j0, r0, &rbar[ew]);
            }
            bool got = wait_or_abort(&tfull[b], tph, abort_flag, limit, a.status);
            got = __all_sync(0xFFFFFFFFu, got);
            if (HELP && nseg > 0) {
                // Owner: the helper always signals (its partial is in Y, or it set
                // this CTA's abort flag), so this wait is long but always ends.  The
                // partial comes back by TMA into the A stage buffers, idle once this
                // CTA's MMAs are done.
                bool in = false;
                for (uint64_t i = 0; i < kDrainPolls && !in; ++i) in = mbar_try_wait_cluster(&recv[ew], 0u);
                in = __all_sync(0xFFFFFFFFu, in);
                got = got && in && *abort_flag == 0u;
                if (got) {
                    if (lane == 0) {
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(&pbar[ew], (uint32_t)kStgBytes);
                        tma_load_2d(sA + ew * kStgBytes, &ymap, j0, r0, &pbar[ew]);
                    }
                    bool w = mbar_wait(&pbar[ew], 0u, limit);
                    w = __all_sync(0xFFFFFFFFu, w);
                    if (!w) {
                        if (lane == 0) {
                            if (!*abort_flag) record_status(a.status, kStTimeout);
                            *abort_flag = 1u;
                            mbar_wait(&pbar[ew], 0u, kDrainPolls);
                        }
                        __syncwarp();
                        got = false;
                    }
                }
            }
            if (!got) {
                if ((a.flags & kResidual) && lane == 0)
                    mbar_wait(&rbar[ew], rphase, kDrainPolls);  // the copy lands first
                __syncwarp();
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                if (!ok || cg + 4 * u >= NBQ) break;
                const int jb = jt + (cg + 4 * u) * 32;
                if (u > 0) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                    if ((a.flags & kResidual) && lane == 0) {
                        mbar_arrive_expect_tx(&rbar[ew], (uint32_t)kStgBytes);
                        tma_load_2d(stg, &rmap, jb, r0, &rbar[ew]);
                    }
                }
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) +
                              (uint32_t)(b * BN + (cg + 4 * u) * 32),
                          v);
                if (HELP) {  // + the helper's part: k stages [ks, KB) after [0, ks)
                    const uint8_t *pp = sA + ew * kStgBytes + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 pv =
                            *reinterpret_cast<const float4 *>(pp + ((j ^ (lane & 7)) << 4));
                        v[4 * j] += pv.x;
                        v[4 * j + 1] += pv.y;
                        v[4 * j + 2] += pv.z;
                        v[4 * j + 3] += pv.w;
                    }
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float bc = __shfl_sync(0xFFFFFFFFu, bl[u], c);
                    float x = v[c];
                    if (a.flags & kBias) x += bc;
                    v[c] = a.alpha * activate(x, a.flags);
                }
                if (a.flags & kResidual) {
                    bool w = mbar_wait(&rbar[ew], rphase, limit);
                    w = __all_sync(0xFFFFFFFFu, w);
                    if (!w) {
                        if (lane == 0) {
                            if (!*abort_flag) record_status(a.status, kStTimeout);
                            *abort_flag = 1u;
                            mbar_wait(&rbar[ew], rphase, kDrainPolls);
                        }
                        __syncwarp();
                        ok = false;
                        break;
                    }
                    rphase ^= 1u;
                }
                // Row `lane` of the block, 16-byte chunk j stored at chunk j ^ (lane % 8).
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float4 *p = reinterpret_cast<float4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
                    float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    if (a.flags & kResidual) {
                        const float4 r = *p;
                        o.x += r.x; o.y += r.y; o.z += r.z; o.w += r.w;
                    }
                    *p = o;
                }
                fence_proxy_async_smem();  // generic-proxy writes -> TMA store reads
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&ymap, jb, r0, stg);
                    bulk_commit();
                }
                stored = true;
                if (DUAL && jb < a.dual) {
                    // The second band: the same sums + bias2, no activation, alpha or
                    // residual, at column m + jb (the map clips columns past dual).
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) +
                                  (uint32_t)(b * BN + (cg + 4 * u) * 32),
                              v);
                    if (HELP) {
                        const uint8_t *pp = sA + ew * kStgBytes + lane * 128;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 pv =
                                *reinterpret_cast<const float4 *>(pp + ((j ^ (lane & 7)) << 4));
                            v[4 * j] += pv.x;
                            v[4 * j + 1] += pv.y;
                            v[4 * j + 2] += pv.z;
                            v[4 * j + 3] += pv.w;
                        }
                    }
                    const float b2 = jb + lane < a.dual ? __ldg(a.bias2 + jb + lane) : 0.f;
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[c] += __shfl_sync(0xFFFFFFFFu, b2, c);
                    if (lane == 0) bulk_wait_read0();  // the block above has left stg
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&y2map, jb, r0, stg);
                        bulk_commit();
                    }
                }
            }
            // This accumulator may be refilled.
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) {
                if (PAIR)  // the even CTA's MMA warp waits for both CTAs' epilogues
                    mbar_arrive_cluster(tempty_at + (uint32_t)(b * sizeof(uint64_t)));
                else
                    mbar_arrive(&tempty[b]);
            }
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }
    __syncwarp();  // every role's lanes meet before the block-wide barrier
    tc_fence_before();
    if (PAIR || HELP)
        cluster_sync_all();  // no CTA leaves while another may still signal or write it
    else
        __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(ncols)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                         "r"(ncols)
                         : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                            cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_2d(CUtensorMap &map, CUtensorMapDataType dt, int esize, const void *base, int cols,
               int rows, int box_cols, int box_rows, int ld = 0) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld > 0 ? ld : cols) * esize};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(&map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `csize` CTAs of `kern` that the device holds at once, or 0 (cached
// per device and cluster size).
template <typename Kernel>
int max_clusters(Kernel kern, int smem, int csize, const DeviceInfo &dev) {
    static std::atomic<int> cached[8][64];
    std::atomic<int> &c = cached[csize & 7][dev.ordinal & 63];
    int v = c.load(std::memory_order_acquire);
    if (v != 0) return v < 0 ? 0 : v;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        c.store(-1, std::memory_order_release);
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(csize * (dev.sm_count / csize)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        clusters = 0;
    }
    c.store(clusters > 0 ? clusters : -1, std::memory_order_release);
    return clusters;
}

template <int BN, int KS, int SCH, bool DUAL = false>
cudaError_t launch_bn(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                      cudaStream_t stream, int clusters = 0) {
    using L = PLayout<BN, KS, SCH>;
    constexpr int TM = SCH == kPair ? 2 * BM : BM;
    static std::atomic<unsigned long long> smem_set{0};
    CUtensorMap wmap, xmap, ymap, rmap, y2map;
    if (!encode_2d(wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W, a.k, a.m, BK, L::kBRows) ||
        !encode_2d(xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xb, a.k, a.n, BK, BM) ||
        !encode_2d(ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.Y, a.m, a.n, 32, 32, a.ldy))
        return cudaErrorInvalidValue;
    if (a.flags & kResidual) {
        if (!encode_2d(rmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.R, a.m, a.n, 32, 32, a.ldy))
            return cudaErrorInvalidValue;
    } else {
        rmap = ymap;  // unused
    }
    if (DUAL) {  // the second band: columns m .. m + dual of each row of Y
        if (!encode_2d(y2map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.Y + a.m, a.dual, a.n, 32, 32,
                       a.ldy))
            return cudaErrorInvalidValue;
    } else {
        y2map = ymap;  // unused
    }
    auto kern = gemm_tcp_kernel<BN, KS, SCH, DUAL>;
    static_assert(L::kBytes <= 227 * 1024, "shared memory budget");
    cudaError_t err = ensure_smem(kern, (int)L::kBytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    const long long tiles = (long long)((a.n + TM - 1) / TM) * ((a.m + BN - 1) / BN);
    if (SCH == kData) {
        const int grid = (int)(tiles < dev.sm_count ? tiles : dev.sm_count);
        return launch_pdl(kern, dim3(grid), dim3(kThreads), L::kBytes, stream, wmap, xmap, ymap,
                          rmap, y2map, a);
    }
    // Pair mode: up to `clusters` pairs walk the tiles.  Helper mode: `clusters`
    // is h, one cluster of h + 1 CTAs per h tiles.
    const int csize = SCH == kPair ? 2 : clusters + 1;
    const long long nc =
        SCH == kPair ? (tiles < clusters ? tiles : clusters) : (tiles + clusters - 1) / clusters;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(csize * nc));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, wmap, xmap, ymap, rmap, y2map, a);
}

}  // namespace

bool gemm_tcp_supported(const GemmArgs &a) {
    // TMA stores need 16-byte aligned rows of Y (and of the residual, and of the
    // second band at column m).
    if (a.m % 4 != 0 || a.ldy % 4 != 0 || ((uintptr_t)a.Y & 15u)) return false;
    if ((a.flags & kResidual) && ((uintptr_t)a.R & 15u)) return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_gemm_tcp(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                            cudaStream_t stream) {
    // Schedule with the smallest estimate of
    //   rounds x (64-k steps x step time + epi / 2) + epi / 2,
    // rounds = tiles per SM (or SM pair, or cluster) rounded up; the step times
    // are measured on GB300 (128 x 128 on one SM 0.275 us and 128 x 256 0.45 us,
    // both bound by operand delivery; 256 x 256 on an SM pair 0.33 us, bound by
    // the MMA, and 256 x 192 taken as three quarters of that); epi = the time to drain one tile's accumulator, 1.5 us per
    // 128 x 128 f32 block of output per SM (twice that with an exp- or erf-based
    // activation), about half of which overlaps the next tile's MMAs.  The helper
    // schedule with h owners runs the owners' share of the steps of a 128 x 128
    // tile plus about 1 us of hand-over, when all its clusters fit at once.
    const double ks = (double)((a.k + BK - 1) / BK);
    const double e = (a.flags & (kGelu | kSilu | kTanh)) ? 3.0 : 1.5;
    const long long rows = (a.n + BM - 1) / BM, rows2 = (a.n + 2 * BM - 1) / (2 * BM);
    const long long sm = dev.sm_count;
    auto est = [&](long long tiles, long long units, double steps, double step, double epi) {
        const double rounds = (double)((tiles + units - 1) / units);
        return rounds * (steps * step + 0.5 * epi) + 0.5 * epi;
    };
    const long long tiles128 = rows * ((a.m + 127) / 128);
    const double t128 = est(tiles128, sm, ks, 0.275, e);
    const double t256 = est(rows * ((a.m + 255) / 256), sm, ks, 0.45, 2 * e);
    double best = t128 < t256 ? t128 : t256;
    int pick = t128 < t256 ? 0 : 1;
    using LP = PLayout<256, 1, kPair>;
    using LH = PLayout<128, 2, kHelp>;
    int pairs = 0;
    if (a.n > BM) {
        pairs = max_clusters(gemm_tcp_kernel<256, 1, kPair>, (int)LP::kBytes, 2, dev);
        if (pairs > 0) {
            // An exp- or erf-based epilogue competes with the pair's MMA-bound
            // mainloop more than with a one-SM tile's operand-bound one (measured
            // on the encoder up projection): charge it twice.
            const double pe = (a.flags & (kGelu | kSilu | kTanh)) ? 2.0 * e : e;
            const double tp = est(rows2 * ((a.m + 255) / 256), pairs, ks, 0.33, 2 * pe);
            if (tp < best) {
                best = tp;
                pick = 2;
            }
            // 256 x 192 pair tiles: three quarters of the MMA work per step.
            const double tq = est(rows2 * ((a.m + 191) / 192), pairs, ks, 0.25, 1.5 * pe);
            if (tq < best) {
                best = tq;
                pick = 4;
            }
        }
    }
    const long long kb128 = (a.k + 2 * BK - 1) / (2 * BK);  // 128-k stages
    // The helper schedule parks partial sums in Y: only when Y is not the residual,
    // and only without a second band.
    const size_t ybytes = (size_t)a.n * a.ldy * sizeof(float);
    const uintptr_t y0 = (uintptr_t)a.Y, r0 = (uintptr_t)a.R;
    const bool y_free = !(a.flags & kResidual) || r0 + ybytes <= y0 || y0 + ybytes <= r0;
    int owners = 0;
    for (int hh = 2; hh <= 3 && y_free && a.dual == 0 && kb128 >= hh + 1 && tiles128 >= hh;
         ++hh) {
        // Only when every cluster is resident at once (one round).
        const int fit = max_clusters(gemm_tcp_kernel<128, 2, kHelp>, (int)LH::kBytes, hh + 1, dev);
        const long long need = (tiles128 + hh - 1) / hh;
        if (fit <= 0 || need > fit) continue;
        const double steps = 2.0 * (double)help_split((int)kb128, hh);
        const double th = est(need, need, steps, 0.275, e) + 1.0;
        if (th < best) {
            best = th;
            pick = 3;
            owners = hh;
        }
    }
    if (a.dual > 0) {
        switch (pick) {
            case 1: return launch_bn<256, 1, kData, true>(a, xb, dev, stream);
            case 2: return launch_bn<256, 1, kPair, true>(a, xb, dev, stream, pairs);
            case 4: return launch_bn<192, 1, kPair, true>(a, xb, dev, stream, pairs);
            default: return launch_bn<128, 2, kData, true>(a, xb, dev, stream);
        }
    }
    switch (pick) {
        case 1: return launch_bn<256, 1, kData>(a, xb, dev, stream);
        case 2: return launch_bn<256, 1, kPair>(a, xb, dev, stream, pairs);
        case 3: return launch_bn<128, 2, kHelp>(a, xb, dev, stream, owners);
        case 4: return launch_bn<192, 1, kPair>(a, xb, dev, stream, pairs);
        default: return launch_bn<128, 2, kData>(a, xb, dev, stream);
    }
}

}  // namespace wq
