// gemv_mma.cu -- small-n GEMV and routed MoE matvec on the tensor cores.
//
// Computes the same contraction as gemv_stream.cu (hanzo-ml 0.11.13
// src/wgpu_backend.rs matvec_q8_0_gpu / matvec_q4_0_gpu / moe_matvec_gpu, with the
// cortiq-engine 0.8.49 ae_put epilogue) for Q8_0/Q4_0 weights with k % 256 == 0.
//
// Why tensor cores for an HBM-bound op: with f32 FMAs every weight costs a
// decode, an X load and one FMA per token, which issues more instructions than
// the SM can retire while HBM streams 4-8 weights per SM-cycle.  Here the
// weights' integer codes (exact in bf16) are decoded in registers straight into
// the A fragments of mma.sync.m16n8k16 (no shared-memory round trip for the
// decoded operand), and X is split exactly into three bf16 terms
// x = x1 + x2 + x3 (8 + 8 + 8 significant bits: every product is exact and the
// f32 accumulation is the only rounding).  The columns of the MMA are
// (split, token) pairs, so one decoded weight tile serves every token and split.
// The block scale d is applied once per 32-weight block per row (an f32x2 FMA
// on the MMA's partial sums), as in the block definition w = d*q.
//
// Data movement: a stage holds one 512-weight chunk of every row of the CTA's
// current row group, loaded by a producer warp as one tall TMA box (2-D tensor
// map over the byte image; two boxes for Q8_0), since a TMA request's cost is
// per request and tall boxes keep HBM streaming at full rate.  The producer is a
// warp of its own because a TMA issue blocks its thread while the engine takes
// the box.  Each of the 16 consumer warps owns one 32-weight block of every
// stage, prefetches its X one stage ahead, builds its B fragments once and
// applies them to all row tiles of the group.
//
// Column layouts of the MMA (n = tokens of a pass): for 1-2 tokens the three
// splits of each token are packed into one n-tile (column s*P + i); for 3-8
// tokens n-tile s holds split s of token i in column i, so a thread's three
// n-tile results are the same token's three splits and one accumulator chain
// sums them; 9-16 tokens use six n-tiles the same way (two token halves).
// The partial sums of the 16 warps are reduced in shared memory in a fixed
// order (deterministic) and the epilogue (bias, erf-GELU, residual) is fused
// into the store.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

constexpr int kCW = 16;                  // consumer warps (one block of each chunk each)
constexpr int kThreads = (kCW + 1) * 32; // + one producer warp
constexpr int kBlocks = 16;              // blocks (of 32 weights) per chunk
constexpr int kMaxSlots = 256;
constexpr int kRedBufs = 4;              // partial-sum buffers of the ordered reduction

// A stage holds, for every row of the group, the 16 blocks (512 weights) of one
// chunk, loaded as NBOX tall TMA boxes (the box inner size is at most 256 u16, so
// Q8_0's 544-byte chunk row takes two boxes of 8 blocks).
template <int WT>
struct Fmt;
template <>
struct Fmt<kQ4_0> {
    static constexpr int BB = 18;     // block bytes
    static constexpr int BOXB = 16;   // blocks per box row
    static constexpr int NBOX = 1;
    static constexpr int ROWB = 288;  // bytes per box row
};
template <>
struct Fmt<kQ8_0> {
    static constexpr int BB = 34;
    static constexpr int BOXB = 8;
    static constexpr int NBOX = 2;
    static constexpr int ROWB = 272;
};

// Accumulator columns per row of the reduction buffer: 8 (one n-tile), 16 when wide.
template <bool WIDE>
struct Cols {
    static constexpr int C = WIDE ? 16 : 8;
};

template <int WT, bool WIDE, int T>
struct Layout {
    static constexpr int kTileBytes = 16 * Fmt<WT>::ROWB;       // one tile, one box
    static constexpr int kBoxBytes = T * kTileBytes;            // the group's rows, one box
    static constexpr int kStageBytes = Fmt<WT>::NBOX * kBoxBytes;
    static constexpr int kRedBytes = kRedBufs * T * 16 * Cols<WIDE>::C * 4;
    static constexpr int kBudget = 200 * 1024 - kRedBytes;
    static constexpr int kStages = (kBudget / kStageBytes) > 8 ? 8 : (kBudget / kStageBytes);
    static_assert(kStages >= 2, "at least two stages");
};

// ------------------------------------------------------------------ helpers --

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The three exact bf16 terms of a pair of f32 values, packed (lo, hi) per term.
__device__ __forceinline__ void split3(float a, float b, uint32_t &p1, uint32_t &p2,
                                       uint32_t &p3) {
    p1 = pack_bf16x2_rn(a, b);
    a -= __uint_as_float(p1 << 16);
    b -= __uint_as_float(p1 & 0xFFFF0000u);
    p2 = pack_bf16x2_rn(a, b);
    a -= __uint_as_float(p2 << 16);
    b -= __uint_as_float(p2 & 0xFFFF0000u);
    p3 = pack_bf16x2_rn(a, b);
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A.B with a zero accumulator input.
__device__ __forceinline__ void mma_bf16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// acc[0..1] += d0 * p[0..1]; acc[2..3] += d1 * p[2..3] (packed f32x2 FMAs).
__device__ __forceinline__ void scale_acc(float (&acc)[4], const float (&p)[4], float d0,
                                          float d1) {
    unsigned long long a01, a23, p01, p23, dd0, dd1;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a01) : "f"(acc[0]), "f"(acc[1]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(a23) : "f"(acc[2]), "f"(acc[3]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(p01) : "f"(p[0]), "f"(p[1]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(p23) : "f"(p[2]), "f"(p[3]));
    asm("mov.b64 %0, {%1, %1};" : "=l"(dd0) : "f"(d0));
    asm("mov.b64 %0, {%1, %1};" : "=l"(dd1) : "f"(d1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a01) : "l"(dd0), "l"(p01));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a23) : "l"(dd1), "l"(p23));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[0]), "=f"(acc[1]) : "l"(a01));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2]), "=f"(acc[3]) : "l"(a23));
}

__device__ __forceinline__ uint32_t sub_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Q4_0: the four bytes v = qs[4t..4t+3] of one row give, for the two MMA k-steps of
// the block, A registers (low nibbles: elements 4t..4t+3; high: 16+4t..16+4t+3).
// Each bf16x2 holds elements (j, j+2) of its nibble group: 0x4300 | q is 128 + q
// exactly, and subtracting 136 leaves q - 8.
__device__ __forceinline__ void decode_q4(uint32_t v, uint32_t &lo02, uint32_t &lo13,
                                          uint32_t &hi02, uint32_t &hi13) {
    const uint32_t m = 0x000F000Fu, magic = 0x43004300u, off = 0x43084308u;  // 136, 136
    lo02 = sub_bf16x2((v & m) | magic, off);
    lo13 = sub_bf16x2(((v >> 8) & m) | magic, off);
    hi02 = sub_bf16x2(((v >> 4) & m) | magic, off);
    hi13 = sub_bf16x2(((v >> 12) & m) | magic, off);
}

// Q8_0: eight signed bytes -> four bf16x2 (pairs (0,1), (2,3), (4,5), (6,7)), exact.
__device__ __forceinline__ void decode_q8(uint32_t v0, uint32_t v1, uint32_t (&r)[4]) {
    float f[8];
    s8x4_to_f32(v0, f[0], f[1], f[2], f[3]);
    s8x4_to_f32(v1, f[4], f[5], f[6], f[7]);
    r[0] = pack_bf16x2_rn(f[0], f[1]);
    r[1] = pack_bf16x2_rn(f[2], f[3]);
    r[2] = pack_bf16x2_rn(f[4], f[5]);
    r[3] = pack_bf16x2_rn(f[6], f[7]);
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}

// ------------------------------------------------------------ job schedule --
//
// Work units are 16-row tiles; GEMV: tiles 0..ceil(m/16) of the one matrix; MoE:
// tiles of the active experts in order (expert a owns units [a*tpe, (a+1)*tpe)).
// A CTA takes a contiguous range of units and processes it in row groups of at
// most T tiles that never straddle an expert; every group is run once per pass
// of at most P tokens.

struct Sched {
    int n_act;          // MoE: active experts; GEMV: 1
    int tpe;            // tiles per expert (GEMV: per matrix)
    long long u0, u1;   // this CTA's unit range
};

template <int T>
__device__ __forceinline__ int group_tiles(const Sched &sc, long long u) {
    const long long end_e = (u / sc.tpe + 1) * sc.tpe;
    long long e = u + T;
    if (e > end_e) e = end_e;
    if (e > sc.u1) e = sc.u1;
    return (int)(e - u);
}

template <int WT, bool MOE, bool WIDE, int T>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap_t,
                    const __grid_constant__ CUtensorMap wmap_1, const StreamArgs a) {
    using L = Layout<WT, WIDE, T>;
    constexpr int S = L::kStages;
    constexpr int C = Cols<WIDE>::C;
    constexpr int P_MAX = WIDE ? 16 : 8;   // tokens per pass
    constexpr int NT = WIDE ? 6 : 3;       // n-tiles at most
    constexpr int NH = WIDE ? 2 : 1;       // tokens per thread in the split-major layout
    constexpr int NA = NH;                 // accumulator groups per tile
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * L::kStageBytes);  // [4][T*16][C]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + kRedBufs * T * 16 * C);
    uint64_t *empty = full + S;
    unsigned long long *s_key = reinterpret_cast<unsigned long long *>(empty + S);
    int *s_sorted = reinterpret_cast<int *>(s_key + kMaxSlots);
    int *s_seg = s_sorted + kMaxSlots;
    int *s_act = s_seg + kMaxSlots + 1;
    int *s_nact = s_act + kMaxSlots;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(s_nact + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int m = a.m, k = a.k;
    const int nb = k / 32;                          // blocks per row
    const int KC = (nb + kBlocks - 1) / kBlocks;    // chunks per row (last may be half)
    const uint64_t limit = a.wait_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    Sched sc;
    sc.tpe = (m + 15) / 16;
    if (MOE) {
        const int Sl = a.n * a.topk;
        const unsigned long long big = 1ull << 62;
        for (int q = threadIdx.x; q < Sl; q += blockDim.x) {
            const int e = a.ids[q];
            const bool ok = e >= 0 && e < a.n_experts;
            if (!ok && blockIdx.x == 0) record_status(a.status, kStBadExpert);
            s_key[q] = ok ? ((unsigned long long)e << 16) | (unsigned)q : big | (unsigned)q;
        }
        __syncthreads();
        for (int q = threadIdx.x; q < Sl; q += blockDim.x) {
            const unsigned long long kq = s_key[q];
            int r = 0;
            for (int q2 = 0; q2 < Sl; ++q2) r += s_key[q2] < kq;
            s_sorted[r] = q;
        }
        __syncthreads();
        if (warp == 0) {  // segment starts of the sorted slots, by ballot and prefix count
            int na = 0;
            for (int base = 0; base < Sl; base += 32) {
                const int r = base + lane;
                bool valid = false, start = false;
                int e = 0;
                if (r < Sl) {
                    const unsigned long long kr = s_key[s_sorted[r]];
                    valid = !(kr & big);
                    e = (int)(kr >> 16);
                    start = valid && (r == 0 || (int)(s_key[s_sorted[r - 1]] >> 16) != e);
                }
                const unsigned sm = __ballot_sync(0xFFFFFFFFu, start);
                if (start) {
                    const int idx = na + __popc(sm & ((1u << lane) - 1u));
                    s_seg[idx] = r;
                    s_act[idx] = e;
                }
                na += __popc(sm);
                const unsigned vm = __ballot_sync(0xFFFFFFFFu, valid);
                if (vm != 0xFFFFFFFFu) {  // the first invalid slot ends the valid ones
                    if (lane == 0) {
                        s_seg[na] = base + __popc(vm);
                        *s_nact = na;
                    }
                    break;
                }
                if (base + 32 >= Sl && lane == 0) {
                    s_seg[na] = Sl;
                    *s_nact = na;
                }
            }
        }
        __syncthreads();
        sc.n_act = *s_nact;
    } else {
        __syncthreads();
        sc.n_act = 1;
    }
    const long long units = (long long)sc.n_act * sc.tpe;
    sc.u0 = units * blockIdx.x / gridDim.x;
    sc.u1 = units * (blockIdx.x + 1) / gridDim.x;

    auto group_tokens = [&](long long u, int &seg0) -> int {
        if (!MOE) {
            seg0 = 0;
            return a.n;
        }
        const int ai = (int)(u / sc.tpe);
        seg0 = s_seg[ai];
        return s_seg[ai + 1] - seg0;
    };
    auto tile_row = [&](long long u) -> int {
        const int ai = (int)(u / sc.tpe), j = (int)(u % sc.tpe) * 16;
        return MOE ? s_act[ai] * m + j : j;
    };

    if (warp == kCW) {
        // ------------------------------------------------------------ producer
        // A full group is one tall box per NBOX (T tiles of rows); a short group
        // takes one 16-row box per tile.
        if (lane == 0) {
            const uint64_t policy = l2_evict_first();
            long long q = 0;
            bool ok = true;
            for (long long u = sc.u0; u < sc.u1 && ok;) {
                const int nt = group_tiles<T>(sc, u);
                int seg0;
                const int ntok = group_tokens(u, seg0);
                for (int p0 = 0; p0 < ntok && ok; p0 += P_MAX) {
                    for (int c = 0; c < KC; ++c, ++q) {
                        const int s = (int)(q % S);
                        if (q >= S) {
                            const uint32_t par = (uint32_t)(((q / S) - 1) & 1);
                            bool w = mbar_test_wait(&empty[s], par);
                            for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                                w = mbar_try_wait(&empty[s], par);
                            if (!w) {
                                if (!*abort_flag) record_status(a.status, kStTimeout);
                                *abort_flag = 1u;
                                ok = false;
                                break;
                            }
                        }
                        mbar_arrive_expect_tx(&full[s],
                                              (uint32_t)(Fmt<WT>::NBOX * nt * L::kTileBytes));
                        uint8_t *dst = stages + (size_t)s * L::kStageBytes;
                        for (int bx = 0; bx < Fmt<WT>::NBOX; ++bx) {
                            const int x = (c * Fmt<WT>::NBOX + bx) * (Fmt<WT>::ROWB / 2);
                            if (nt == T) {
                                tma_load_2d(dst + bx * L::kBoxBytes, &wmap_t, x, tile_row(u),
                                            &full[s], policy);
                            } else {
                                for (int tt = 0; tt < nt; ++tt)
                                    tma_load_2d(dst + bx * L::kBoxBytes + tt * L::kTileBytes,
                                                &wmap_1, x, tile_row(u + tt), &full[s], policy);
                            }
                        }
                    }
                }
                u += nt;
            }
            for (long long d = (q > S ? q - S : 0); d < q; ++d)
                mbar_wait(&full[d % S], (uint32_t)((d / S) & 1), kDrainPolls);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    long long q = 0;
    bool ok = true;
    for (long long u = sc.u0; u < sc.u1 && ok;) {
        const int ntiles = group_tiles<T>(sc, u);
        int seg0;
        const int ntok_all = group_tokens(u, seg0);
        const int ai = (int)(u / sc.tpe);
        const int e = MOE ? s_act[ai] : 0;
        const int row0 = (int)(u % sc.tpe) * 16;
        for (int p0 = 0; p0 < ntok_all && ok; p0 += P_MAX) {
            const int ntok = min(P_MAX, ntok_all - p0);
            // packed: 1-2 tokens, column g = split (g / P) of token (g % P), one n-tile;
            // else split-major: n-tile s, column g = token g (+8 for the second half).
            const bool packed = !WIDE && ntok <= 2;
            const int P = packed ? ntok : (WIDE ? 16 : 8);
            int xrow[NH];
            bool tok_ok[NH];
            int col_s = 0;  // packed: which split this thread's column carries
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const int i = packed ? g % P : h * 8 + g;
                tok_ok[h] = packed ? (g < 3 * P) : (i < ntok);
                const int r = p0 + (tok_ok[h] ? i : 0);
                xrow[h] = MOE ? s_sorted[seg0 + r] / a.topk : r;
            }
            if (packed) col_s = g / P;

            float acc[T][NA][4];
#pragma unroll
            for (int tt = 0; tt < T; ++tt)
#pragma unroll
                for (int j = 0; j < NA; ++j)
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[tt][j][r] = 0.f;

            // X of this warp's block of a chunk.
            auto load_x = [&](int c, float (&xv)[1][NH][8]) {
#pragma unroll
                for (int hb = 0; hb < 1; ++hb) {
                    const int blk = c * kBlocks + warp;
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        float4 u0v = make_float4(0.f, 0.f, 0.f, 0.f), u1v = u0v;
                        if (blk < nb && tok_ok[h]) {
                            const float *xp = a.X + (size_t)xrow[h] * k + (size_t)blk * 32;
                            if (WT == kQ4_0) {
                                u0v = __ldg(reinterpret_cast<const float4 *>(xp + 4 * t));
                                u1v = __ldg(reinterpret_cast<const float4 *>(xp + 16 + 4 * t));
                            } else {
                                u0v = __ldg(reinterpret_cast<const float4 *>(xp + 8 * t));
                                u1v = __ldg(reinterpret_cast<const float4 *>(xp + 8 * t + 4));
                            }
                        }
                        xv[hb][h][0] = u0v.x; xv[hb][h][1] = u0v.y;
                        xv[hb][h][2] = u0v.z; xv[hb][h][3] = u0v.w;
                        xv[hb][h][4] = u1v.x; xv[hb][h][5] = u1v.y;
                        xv[hb][h][6] = u1v.z; xv[hb][h][7] = u1v.w;
                    }
                }
            };
            float xcur[1][NH][8];
            load_x(0, xcur);

            for (int c = 0; c < KC; ++c, ++q) {
                float xnext[1][NH][8];
                if (c + 1 < KC) load_x(c + 1, xnext);
                const int s = (int)(q % S);
                bool w = mbar_test_wait(&full[s], (uint32_t)((q / S) & 1));
                for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                    w = mbar_try_wait(&full[s], (uint32_t)((q / S) & 1));
                w = __all_sync(0xFFFFFFFFu, w);
                if (!w) {
                    if (lane == 0) {
                        if (!*abort_flag) record_status(a.status, kStTimeout);
                        *abort_flag = 1u;
                    }
                    ok = false;
                    break;
                }
#pragma unroll
                for (int hb = 0; hb < 1; ++hb) {
                    const int wb = warp;             // block within the chunk (0..15)
                    const int blk = c * kBlocks + wb;
                    if (blk >= nb) continue;
                    // Exact 3-term split of X, pairs in the element order of the A decode.
                    uint32_t sp[NH][4][3];
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const float *xv = xcur[hb][h];
                        if (WT == kQ4_0) {  // pairs (0,2), (1,3) of each nibble group
                            split3(xv[0], xv[2], sp[h][0][0], sp[h][0][1], sp[h][0][2]);
                            split3(xv[1], xv[3], sp[h][1][0], sp[h][1][1], sp[h][1][2]);
                            split3(xv[4], xv[6], sp[h][2][0], sp[h][2][1], sp[h][2][2]);
                            split3(xv[5], xv[7], sp[h][3][0], sp[h][3][1], sp[h][3][2]);
                        } else {            // pairs (0,1), (2,3), (4,5), (6,7)
                            split3(xv[0], xv[1], sp[h][0][0], sp[h][0][1], sp[h][0][2]);
                            split3(xv[2], xv[3], sp[h][1][0], sp[h][1][1], sp[h][1][2]);
                            split3(xv[4], xv[5], sp[h][2][0], sp[h][2][1], sp[h][2][2]);
                            split3(xv[6], xv[7], sp[h][3][0], sp[h][3][1], sp[h][3][2]);
                        }
                    }
                    // B fragments [k-step][n-tile][reg]: k-step 0 uses pairs 0,1; k-step 1 pairs 2,3.
                    uint32_t bf[2][NT][2];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
                            for (int rr = 0; rr < 2; ++rr) {
                                const int pr = ks * 2 + rr;
                                uint32_t v;
                                if (WIDE) {
                                    v = sp[nt & 1][pr][nt >> 1];          // n-tile = 2 * split + half
                                } else if (packed) {
                                    v = col_s == 0 ? sp[0][pr][0] : (col_s == 1 ? sp[0][pr][1] : sp[0][pr][2]);
                                } else {
                                    v = sp[0][pr][nt];                    // n-tile = split
                                }
                                bf[ks][nt][rr] = v;
                            }
                        }
                    }
                    const uint8_t *st = stages + (size_t)s * L::kStageBytes +
                                        (wb / Fmt<WT>::BOXB) * L::kBoxBytes +
                                        (wb % Fmt<WT>::BOXB) * Fmt<WT>::BB;
#pragma unroll
                    for (int tt = 0; tt < T; ++tt) {
                        if (tt < ntiles) {
                            const uint8_t *r0p = st + tt * L::kTileBytes + g * Fmt<WT>::ROWB;
                            const uint8_t *r1p = r0p + 8 * Fmt<WT>::ROWB;
                            const float d0 = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(r0p));
                            const float d1 = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(r1p));
                            uint32_t a1[4], a2[4];  // A of k-step 0 and 1
                            if (WT == kQ4_0) {
                                const uint32_t v0 = ld_u32_a2(r0p + 2 + 4 * t);
                                const uint32_t v1 = ld_u32_a2(r1p + 2 + 4 * t);
                                decode_q4(v0, a1[0], a1[2], a2[0], a2[2]);
                                decode_q4(v1, a1[1], a1[3], a2[1], a2[3]);
                            } else {
                                uint32_t q0[4], q1[4];
                                decode_q8(ld_u32_a2(r0p + 2 + 8 * t), ld_u32_a2(r0p + 6 + 8 * t), q0);
                                decode_q8(ld_u32_a2(r1p + 2 + 8 * t), ld_u32_a2(r1p + 6 + 8 * t), q1);
                                a1[0] = q0[0]; a1[2] = q0[1]; a1[1] = q1[0]; a1[3] = q1[1];
                                a2[0] = q0[2]; a2[2] = q0[3]; a2[1] = q1[2]; a2[3] = q1[3];
                            }
                            if (packed) {
                                float part[4];
                                mma_bf16_z(part, a1, bf[0][0][0], bf[0][0][1]);
                                mma_bf16(part, a2, bf[1][0][0], bf[1][0][1]);
                                scale_acc(acc[tt][0], part, d0, d1);
                            } else {
                                // The three splits of a token sit in the same thread and
                                // column of three n-tiles: one accumulator chain sums them.
#pragma unroll
                                for (int h = 0; h < NH; ++h) {
                                    float part[4];
#pragma unroll
                                    for (int sp_i = 0; sp_i < 3; ++sp_i) {
                                        const int nt = WIDE ? 2 * sp_i + h : sp_i;
                                        if (sp_i == 0)
                                            mma_bf16_z(part, a1, bf[0][nt][0], bf[0][nt][1]);
                                        else
                                            mma_bf16(part, a1, bf[0][nt][0], bf[0][nt][1]);
                                        mma_bf16(part, a2, bf[1][nt][0], bf[1][nt][1]);
                                    }
                                    scale_acc(acc[tt][h], part, d0, d1);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                    for (int j = 0; j < 8; ++j) xcur[0][h][j] = xnext[0][h][j];
            }
            // Every consumer warp gets here, aborted or not; the flag read after the
            // barrier is the same in all of them, so they leave (or go on) together.
            consumers_sync();
            ok = *abort_flag == 0u;
            if (!ok) break;

            // Ordered reduction: warp w adds into buffer w % 4, in 4 rounds.
            const int RT = T * 16 * C;
            for (int rnd = 0; rnd < kCW / kRedBufs; ++rnd) {
                if (warp / kRedBufs == rnd) {
                    float *buf = red + (warp % kRedBufs) * RT;
#pragma unroll
                    for (int tt = 0; tt < T; ++tt) {
                        if (tt < ntiles) {
#pragma unroll
                            for (int j = 0; j < NA; ++j) {
#pragma unroll
                                for (int r = 0; r < 4; ++r) {
                                    const int row = tt * 16 + g + (r >= 2 ? 8 : 0);
                                    const int col = j * 8 + 2 * t + (r & 1);
                                    float *dst = &buf[row * C + col];
                                    *dst = (rnd == 0) ? acc[tt][j][r] : *dst + acc[tt][j][r];
                                }
                            }
                        }
                    }
                }
                consumers_sync();
            }
            const int R = ntiles * 16;
            for (int idx = threadIdx.x; idx < R * ntok; idx += kCW * 32) {
                const int i = idx / R, r = idx % R;
                const int row = row0 + r;
                if (row < m) {
                    float v = 0.f;
#pragma unroll
                    for (int b = 0; b < kRedBufs; ++b) {
                        const float *rp = red + b * RT + r * C;
                        v += packed ? (rp[i] + rp[P + i]) + rp[2 * P + i] : rp[i];
                    }
                    const int yrow = MOE ? s_sorted[seg0 + p0 + i] : p0 + i;
                    const size_t o = (size_t)yrow * m + row;
                    const float *bj = a.bias + (MOE ? (size_t)e * m + row : (size_t)row);
                    a.Y[o] = epilogue(v, a.flags, bj, a.R + o);
                }
            }
            consumers_sync();
        }
        u += ntiles;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                            cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int WT, bool WIDE, int T>
constexpr size_t smem_bytes() {
    using L = Layout<WT, WIDE, T>;
    return (size_t)L::kStages * L::kStageBytes + L::kRedBytes + 2 * L::kStages * sizeof(uint64_t) +
           kMaxSlots * sizeof(unsigned long long) + (3 * kMaxSlots + 4) * sizeof(int) + 16;
}

bool make_map(CUtensorMap &map, const StreamArgs &a, int wtype, long long rows, int box_rows) {
    auto encode = encode_fn();
    if (!encode) return false;
    const size_t rb = row_bytes(wtype, a.k);
    const int box = wtype == kQ4_0 ? Fmt<kQ4_0>::ROWB : Fmt<kQ8_0>::ROWB;
    const cuuint64_t dims[2] = {(cuuint64_t)(rb / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)rb};
    const cuuint32_t boxd[2] = {(cuuint32_t)(box / 2), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(a.W), dims,
                  strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int WT, bool MOE, bool WIDE, int T>
cudaError_t launch_inst(const StreamArgs &a, long long rows, int grid, const DeviceInfo &dev,
                        cudaStream_t stream) {
    static std::atomic<unsigned long long> smem_set{0};
    CUtensorMap map_t, map_1;
    if (!make_map(map_t, a, WT, rows, T * 16) || !make_map(map_1, a, WT, rows, 16))
        return cudaErrorInvalidValue;
    auto kern = gemv_mma_kernel<WT, MOE, WIDE, T>;
    constexpr size_t bytes = smem_bytes<WT, WIDE, T>();
    static_assert(bytes <= 227 * 1024, "shared memory budget");
    cudaError_t err = ensure_smem(kern, (int)bytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, bytes, stream>>>(map_t, map_1, a);
    return cudaGetLastError();
}

template <int WT>
cudaError_t launch_gemv_wt(const StreamArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    const long long tiles = (a.m + 15) / 16;
    const int grid = (int)(tiles < dev.sm_count ? tiles : dev.sm_count);
    const long long per = (tiles + grid - 1) / grid;  // tiles per CTA (max)
    if (a.n > 8) return launch_inst<WT, false, true, 3>(a, a.m, grid, dev, stream);
    if (per <= 2) return launch_inst<WT, false, false, 2>(a, a.m, grid, dev, stream);
    if (per <= 4) return launch_inst<WT, false, false, 4>(a, a.m, grid, dev, stream);
    return launch_inst<WT, false, false, 6>(a, a.m, grid, dev, stream);
}

}  // namespace

bool mma_gemv_supported(int wtype, int k) {
    return (wtype == kQ4_0 || wtype == kQ8_0) && k % 256 == 0 && encode_fn() != nullptr;
}

cudaError_t launch_mma_gemv(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                            cudaStream_t stream) {
    return wtype == kQ4_0 ? launch_gemv_wt<kQ4_0>(a, dev, stream)
                          : launch_gemv_wt<kQ8_0>(a, dev, stream);
}

cudaError_t launch_mma_moe(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                           cudaStream_t stream) {
    const long long rows = (long long)a.n_experts * a.m;
    const int grid = dev.sm_count;
    return wtype == kQ4_0 ? launch_inst<kQ4_0, true, false, 6>(a, rows, grid, dev, stream)
                          : launch_inst<kQ8_0, true, false, 4>(a, rows, grid, dev, stream);
}

}  // namespace wq
