// gemv_mma.cu -- small-n GEMV and routed MoE matvec on the tensor cores.
//
// Computes the same contraction as gemv_stream.cu (hanzo-ml 0.11.13
// src/wgpu_backend.rs matvec_q8_0_gpu / matvec_q4_0_gpu / moe_matvec_gpu, with the
// cortiq-engine 0.8.49 ae_put epilogue) for Q8_0/Q4_0 weights with k % 256 == 0.
//
// Why tensor cores for an HBM-bound op: with f32 FMAs every weight costs a
// decode, an X load and one FMA per token, which issues more instructions than
// the SM can retire while HBM streams 4-8 weights per SM-cycle.  Here the
// weights' integer codes (exact in f16) are decoded in registers straight into
// the A fragments of mma.sync.m16n8k16 (no shared-memory round trip for the
// decoded operand): a mask-and-or places each 4- or 8-bit code in the mantissa of
// an f16 magic number and one packed f16 subtract (or fma) removes the bias, two
// weights per instruction.  X is brought into f16 range by a power of two per
// (token, 32-block) -- chosen from the block's largest |x| -- and split into two
// f16 terms x ~ x1 + x2 with |x - x1 - x2| <= 2^-22 |x| (elements below 2^-17 of
// their block's largest |x| keep an absolute error of at most 2^-39 of it, f16's
// subnormal floor).  Every product of a code and a term is exact in the f32
// accumulation, so the result is within 2^-22 sum|x||w| plus f32 rounding of the
// sums -- far inside the 1e-5 sum|x||w| contract.  The columns of the MMA are
// (term, token) pairs, so one decoded weight tile serves every token and term.
// The block scale d times the power of two's inverse is applied once per 32-weight
// block per row, on the MMA's partial sums, as in the block definition w = d*q.
//
// Data movement: a stage holds one chunk (CW blocks of 32 weights) of every row
// of the CTA's current row group, loaded by a producer warp as one tall TMA box
// (3-D tensor map over the byte image; two boxes for a 16-block Q8_0 chunk),
// since a TMA request's cost is per request and tall boxes keep HBM streaming at
// full rate.  The producer is a warp of its own because a TMA issue blocks its
// thread while the engine takes the box.  Each of the CW consumer warps owns one
// block of every stage, builds its B fragments once and applies them to all row
// tiles of the group.  GEMV runs one CTA of 16 consumer warps per SM; MoE two CTAs
// of 8, so that one CTA's reduction and epilogue overlap the other's chunks.
//
// Column layouts of the MMA (n = tokens of a pass): for 1-4 tokens the two terms
// of each token are packed into one n-tile (column s*P + i); for 5-8 tokens
// n-tile s holds term s of token i in column i, so a thread's two n-tile results
// are the same token's two terms and one accumulator chain sums them; 9-16
// tokens use four n-tiles the same way (two token halves).
// The partial sums of the 16 warps are reduced in shared memory in a fixed
// order (deterministic) and the epilogue (bias, erf-GELU, residual) is fused
// into the store.
//
// MoE routing: the n_tok * topk slots are taken in windows of at most 256; for
// each window every CTA sorts the window's slots by (expert, slot) in shared
// memory and runs over the touched experts' row tiles, so a selected expert's
// weights are read once per window however many of its slots the window holds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "tile_sched.cuh"

namespace wq {
namespace {

// CW consumer warps per CTA, each owning one 32-weight block of every chunk, so a
// chunk is CW blocks: 16 (one CTA per SM, 512-weight chunks) or 8 (two CTAs per SM,
// 256-weight chunks, so that one CTA's reduction and epilogue overlap the other's
// chunk arithmetic).
template <int CW>
struct Warps {
    static constexpr int kThreads = (CW + 1) * 32;          // + one producer warp
    static constexpr int kCtas = CW == 16 ? 1 : 2;          // resident per SM
    static constexpr int kXChunkBytes = CW * 32 * 4;        // one token's X for one chunk (f32)
    static constexpr int kSmemBudget = (CW == 16 ? 200 : 108) * 1024;  // stages + reduction
};

// A stage holds, for every row of the group, the NB blocks of one chunk, loaded as
// NBOX tall TMA boxes (the box inner size is at most 256 u16, so Q8_0's 544-byte
// row of a 16-block chunk takes two boxes of 8 blocks).
template <int WT, int NB>
struct Fmt;
template <int NB>
struct Fmt<kQ4_0, NB> {
    static constexpr int BB = 18;        // block bytes
    static constexpr int BOXB = NB;      // blocks per box row
    static constexpr int NBOX = 1;
    static constexpr int ROWB = 18 * NB; // bytes per box row
};
template <int NB>
struct Fmt<kQ8_0, NB> {
    static constexpr int BB = 34;
    static constexpr int BOXB = 8;
    static constexpr int NBOX = NB / 8;
    static constexpr int ROWB = 272;
};

// Column layouts of a pass (see the file comment):
//   kPacked  1-4 tokens, the two terms of each token in one n-tile;
//   kSplit8  up to 8 tokens, n-tile s = term s, column = token;
//   kSplit16 up to 16 tokens, four n-tiles (two token halves);
//   kMixed   up to 8 tokens, packed when a pass has at most 4 (MoE: token counts
//            per expert vary from pass to pass).
enum PassMode : int { kPacked = 0, kSplit8 = 1, kSplit16 = 2, kMixed = 3 };

template <int MODE>
struct Mode {
    static constexpr bool WIDE = MODE == kSplit16;
    static constexpr int P_MAX = MODE == kPacked ? 4 : (WIDE ? 16 : 8);  // tokens per pass
    static constexpr int C = WIDE ? 16 : 8;     // accumulator columns per reduction row
    static constexpr int NT = WIDE ? 4 : 2;     // n-tiles at most
    static constexpr int NH = WIDE ? 2 : 1;     // token halves per thread (split layouts)
};

template <int WT, int MODE, int T, int CW>
struct Layout {
    using F = Fmt<WT, CW>;
    static constexpr int kBudgetAll = Warps<CW>::kSmemBudget;
    static constexpr int kTileBytes = 16 * F::ROWB;             // one tile, one box
    static constexpr int kBoxBytes = T * kTileBytes;            // the group's rows, one box
    static constexpr int kWBytes = F::NBOX * kBoxBytes;         // weights of a stage
    static constexpr int kStageBytes = kWBytes + Mode<MODE>::P_MAX * Warps<CW>::kXChunkBytes;
    // epilogue inputs staged at the start of a pass: residual [P_MAX][T*16], bias [T*16]
    static constexpr int kEpiBytes = (T * 16 * Mode<MODE>::P_MAX + T * 16) * 4;
    // per consumer warp: two tokens x two terms x four threads x 16 bytes of B
    // fragments, then 16 zero bytes for the padding columns
    static constexpr int kCoopBytes = MODE == kPacked ? CW * 272 : 0;
    // Partial-sum buffers of the ordered reduction: 8 (two rounds of warps, three
    // barriers per pass) when they cost no pipeline stage, else 4 (four rounds).
    static constexpr int stages_with(int bufs) {
        return (kBudgetAll - bufs * T * 16 * Mode<MODE>::C * 4 - kEpiBytes - kCoopBytes) /
               kStageBytes;
    }
    static constexpr int kRedBufs =
        (stages_with(8) >= 8 || stages_with(8) == stages_with(4)) ? 8 : 4;
    static constexpr int kRedBytes = kRedBufs * T * 16 * Mode<MODE>::C * 4;
    static constexpr int kBudget = kBudgetAll - kRedBytes - kEpiBytes - kCoopBytes;
    static constexpr int kStages = (kBudget / kStageBytes) > 8 ? 8 : (kBudget / kStageBytes);
    static_assert(kStages >= 2, "at least two stages");
};

// ------------------------------------------------------------------ helpers --

__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void unpack_f16x2(uint32_t p, float &lo, float &hi) {
    unsigned short l, h;
    asm("mov.b32 {%0, %1}, %2;" : "=h"(l), "=h"(h) : "r"(p));
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(l));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(h));
}

// The two f16 terms of a pair of f32 values with |v| < 2^15, packed (lo, hi) per
// term: t1 = f16(v), t2 = f16(v - t1) (the subtraction is exact), so
// |v - t1 - t2| <= 2^-22 |v| while t2 is a normal f16, and <= 2^-25 below that.
__device__ __forceinline__ void split2(float a, float b, uint32_t &p1, uint32_t &p2) {
    float a1, b1;
    p1 = pack_f16x2_rn(a, b);
    unpack_f16x2(p1, a1, b1);
    p2 = pack_f16x2_rn(a - a1, b - b1);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A.B with a zero accumulator input.
__device__ __forceinline__ void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// acc[0..1] += (d0 * inv0, d0 * inv1) * p[0..1]; acc[2..3] += (d1 * inv0, d1 * inv1) * p[2..3].
__device__ __forceinline__ void scale_acc(float (&acc)[4], const float (&p)[4], float d0,
                                          float d1, float inv0, float inv1) {
    acc[0] = fmaf(d0 * inv0, p[0], acc[0]);
    acc[1] = fmaf(d0 * inv1, p[1], acc[1]);
    acc[2] = fmaf(d1 * inv0, p[2], acc[2]);
    acc[3] = fmaf(d1 * inv1, p[3], acc[3]);
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// (a & b) | c as one three-input logic instruction (written out because the
// compiler otherwise issues the AND and the OR separately here).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Q4_0: the four code bytes v = qs[4t..4t+3] of one row -> the A registers of the
// block's two MMA k-steps, as exact f16 (q - 8).  Low nibbles (elements 4t..4t+3):
// 0x6400 | q is 1024 + q, minus 1032.  High nibbles (elements 16+4t..16+4t+3) sit
// four bits up: 0x6400 | 16q is 1024 + 16q, times 1/16 minus 72 (one exact fma).
// Each register pairs elements (j, j+2): l02 = (4t, 4t+2), l13 = (4t+1, 4t+3),
// h02 = (16+4t, 18+4t), h13 = (17+4t, 19+4t).
__device__ __forceinline__ void decode_q4(uint32_t v, uint32_t &l02, uint32_t &l13,
                                          uint32_t &h02, uint32_t &h13) {
    const uint32_t v8 = v >> 8;
    const uint32_t one16 = 0x2C002C00u, m72 = 0xD480D480u, c1032 = 0x64086408u;
    l02 = hsub2(and_or(v, 0x000F000Fu, 0x64006400u), c1032);
    l13 = hsub2(and_or(v8, 0x000F000Fu, 0x64006400u), c1032);
    h02 = hfma2(and_or(v, 0x00F000F0u, 0x64006400u), one16, m72);
    h13 = hfma2(and_or(v8, 0x00F000F0u, 0x64006400u), one16, m72);
}

// Q8_0: four signed code bytes v = qs[j..j+3] -> f16 pairs (j, j+2) and (j+1, j+3),
// exact: the byte biased to unsigned becomes the low byte of 0x64xx = 1024 + u, and
// 1024 + u - 1152 = u - 128 is the signed code.
__device__ __forceinline__ void decode_q8(uint32_t v, uint32_t &p02, uint32_t &p13) {
    const uint32_t u = v ^ 0x80808080u;
    p02 = hsub2(__byte_perm(u, 0x64646464u, 0x4240), 0x64806480u);
    p13 = hsub2(__byte_perm(u, 0x64646464u, 0x4341), 0x64806480u);
}

// The power of two s = 2^e that brings a block's largest |x| into [2^14, 2^15)
// (so every scaled value is below f16's 65504), and 1/s; e is clamped to
// [-113, 126] so both stay normal f32.
__device__ __forceinline__ void block_scale_bits(uint32_t mx_bits, float &s, float &inv) {
    const int E = (int)((mx_bits >> 23) & 0xFFu);
    const int sb = min(253, max(1, 268 - E));
    s = __uint_as_float((uint32_t)sb << 23);
    inv = __uint_as_float((uint32_t)(254 - sb) << 23);
}

__device__ __forceinline__ void block_scale(float mx, float &s, float &inv) {
    block_scale_bits(__float_as_uint(mx), s, inv);
}

// f32 -> f16 bits (round to nearest even) and back.
__device__ __forceinline__ uint16_t f16_rn(float v) {
    unsigned short h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
    return h;
}
__device__ __forceinline__ float f16_f32(uint16_t h) {
    float v;
    asm("cvt.f32.f16 %0, %1;" : "=f"(v) : "h"(h));
    return v;
}

// 4-byte global -> shared copy that does not hold a register (completes at
// cp_async_wait_all).
__device__ __forceinline__ void cp_async4(float *dst, const float *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}


// Tensor maps of the weight image, one per box height: the group's T tiles, and
// 4, 2 and 1 tiles, from which a shorter group's rows are composed (binary
// decomposition of its tile count), so that a short group moves only its own rows.
struct WMaps {
    CUtensorMap full, b4, b2, b1;
};

template <int WT, bool MOE, int MODE, int T, int CW>
__global__ void __launch_bounds__(Warps<CW>::kThreads, Warps<CW>::kCtas)
    gemv_mma_kernel(const __grid_constant__ WMaps wm, const StreamArgs a) {
    // The barriers and the weight map's descriptor are set up before waiting for
    // the previous grid (they touch nothing it writes); global memory after.
    pdl_launch();
    using L = Layout<WT, MODE, T, CW>;
    using MD = Mode<MODE>;
    using F = typename L::F;
    constexpr int kCW = CW;                                   // consumer warps
    constexpr int kBlocks = CW;                               // blocks per chunk
    constexpr int kXChunkBytes = Warps<CW>::kXChunkBytes;
    constexpr int S = L::kStages;
    constexpr bool WIDE = MD::WIDE;
    constexpr int C = MD::C;
    constexpr int P_MAX = MD::P_MAX;
    constexpr int NT = MD::NT;
    constexpr int NH = MD::NH;
    constexpr int NA = NH;                 // accumulator groups per tile
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * L::kStageBytes);  // [4][T*16][C]
    float *s_res = red + L::kRedBufs * T * 16 * C;   // [P_MAX][T*16]
    float *s_bias = s_res + T * 16 * P_MAX;           // [T*16]
    uint8_t *s_coop = reinterpret_cast<uint8_t *>(s_bias + T * 16);  // [CW][272], 16-aligned
    uint64_t *full = reinterpret_cast<uint64_t *>(s_coop + L::kCoopBytes);
    uint64_t *empty = full + S;
    unsigned long long *s_key = reinterpret_cast<unsigned long long *>(empty + S);
    int *s_sorted = reinterpret_cast<int *>(s_key + kMaxSlots);
    int *s_seg = s_sorted + kMaxSlots;
    int *s_act = s_seg + kMaxSlots + 1;
    int *s_nact = s_act + kMaxSlots;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(s_nact + 1);
    // the producer's count of stages issued, kept here between routing windows so
    // that it occupies no register of the consumer warps
    long long *s_q = reinterpret_cast<long long *>(((uintptr_t)(s_nact + 2) + 7) & ~(uintptr_t)7);
    int *s_wcnt = reinterpret_cast<int *>(s_q + 1);  // per-warp counts of the routing scan [32]

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
        *s_q = 0;
        fence_mbar_init();
    }
    if (L::kCoopBytes > 0 && warp < kCW && lane < 4)
        reinterpret_cast<uint32_t *>(s_coop + warp * 272 + 256)[lane] = 0u;
    if (threadIdx.x == kCW * 32)  // the producer's thread
    {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.full)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.b1)) : "memory");
        if (T > 2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.b2)) : "memory");
        if (T > 4) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.b4)) : "memory");
    }
    // The weight boxes of one stage: a full group is one tall box per NBOX (T tiles
    // of rows); a shorter one is composed of boxes of 4, 2 and 1 tiles, each tile
    // landing where it would in a full box.  Rows past the matrix's end are
    // zero-filled by the TMA unit; they are computed and never stored.
    auto issue_w = [&](uint8_t *dst, uint64_t *bar, int nt, int c, int trow, int tmat,
                       uint64_t policy) {
        for (int bx = 0; bx < F::NBOX; ++bx) {
            const int x = (c * F::NBOX + bx) * (F::ROWB / 2);
            uint8_t *bd = dst + bx * L::kBoxBytes;
            if (nt == T) {
                tma_load_3d(bd, &wm.full, x, trow, tmat, bar, policy);
            } else {
                int t0 = 0;
                if (T > 4 && (nt & 4)) {
                    tma_load_3d(bd, &wm.b4, x, trow, tmat, bar, policy);
                    t0 = 4;
                }
                if (T > 2 && (nt & 2)) {
                    tma_load_3d(bd + t0 * L::kTileBytes, &wm.b2, x, trow + 16 * t0, tmat, bar,
                                policy);
                    t0 += 2;
                }
                if (nt & 1)
                    tma_load_3d(bd + t0 * L::kTileBytes, &wm.b1, x, trow + 16 * t0, tmat, bar,
                                policy);
            }
        }
    };
    auto chunk_bytes = [&](int nt, int c, uint32_t &wbytes, uint32_t &xbytes) {
        // X of one token for the chunk (256 or 512 floats); the group's weight rows
        xbytes = (uint32_t)min(kBlocks * 32, k - c * kBlocks * 32) * 4u;
        wbytes = nt == T ? (uint32_t)L::kWBytes : (uint32_t)(F::NBOX * nt * L::kTileBytes);
    };
    // GEMV: no kernel of this library writes a weight image, so the producer requests
    // the weight boxes of its first stage before the grid-dependency wait, while the
    // previous kernel finishes; its X follows after the wait (the stage barrier
    // expects both).  One stage measured best: with all S stages the first X copy
    // queues behind every early box (benchmark step 164.4 us with one, 164.5 with
    // two, 166.9 with all, 167.8 with none).  MoE rows depend on the ids, which are
    // read after the wait.
    constexpr int kEarly = 1;
    int early = 0;  // stages whose weight boxes went out before the wait
    if constexpr (!MOE) {
        __syncthreads();  // the stage barriers are initialised
        if (threadIdx.x == kCW * 32) {
            Sched s0;
            s0.tpe = (m + 15) / 16;
            s0.n_act = 1;
            split_units(s0);
            const uint64_t policy = l2_evict_first();
            for (Walk wk(s0); wk.more() && early < kEarly;) {
                const int nt = wk.template group<T>();
                for (int p0 = 0; p0 < a.n && early < kEarly; p0 += P_MAX) {
                    const int npass = min(P_MAX, a.n - p0);
                    for (int c = 0; c < KC && early < kEarly; ++c, ++early) {
                        uint32_t wbytes, xbytes;
                        chunk_bytes(nt, c, wbytes, xbytes);
                        mbar_arrive_expect_tx(&full[early], wbytes + npass * xbytes);
                        issue_w(stages + (size_t)early * L::kStageBytes, &full[early], nt, c,
                                wk.tl * 16, 0, policy);
                    }
                }
                wk.advance(nt);
            }
        }
    }
    pdl_wait();
    Sched sc;
    sc.tpe = (m + 15) / 16;
    const int S_all = MOE ? a.n * a.topk : 0;
    const int n_win = MOE ? (S_all + kMaxSlots - 1) / kMaxSlots : 1;
    // Ring positions, carried across routing windows.
    int qs = 0;            // consumers: stage of the next chunk
    uint32_t qph = 0u;     // its fill parity
    bool ok = true;        // consumers: no wait ran out

    for (int win = 0; win < n_win; ++win) {
    if (MOE) {
        const int base = win * kMaxSlots;
        route_window(a, base, min(kMaxSlots, S_all - base),
                     RouteSmem{s_key, s_sorted, s_seg, s_act, s_nact, s_wcnt});
    }
    __syncthreads();
    if (*abort_flag) break;  // the same in every thread after the barrier
    sc.n_act = MOE ? *s_nact : 1;
    // GEMV: contiguous ranges of tiles.  MoE: groups dealt out by cost (DealWalk);
    // the routing keys are no longer needed, so their space holds the experts' order.
    int *s_order = reinterpret_cast<int *>(s_key);
    if constexpr (MOE) {
        order_by_slots(s_seg, sc.n_act, s_order);
        __syncthreads();
    } else {
        split_units(sc);
    }
    auto make_walk = [&]() {
        if constexpr (MOE)
            return DealWalk<T>(sc, s_order);
        else
            return Walk(sc);
    };

    if (warp == kCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t policy = l2_evict_first();
            long long q = *s_q;                 // stages issued so far
            int s = (int)(q % S);               // the next one's ring slot
            uint32_t wrap = (uint32_t)((q / S) & 1);  // and the parity of its round
            bool pok = true;
            for (auto wk = make_walk(); wk.more() && pok;) {
                const int nt = wk.template group<T>();
                const int seg0 = MOE ? s_seg[wk.ai] : 0;
                const int ntok = MOE ? s_seg[wk.ai + 1] - seg0 : a.n;
                const int trow = wk.tl * 16, tmat = MOE ? s_act[wk.ai] : 0;
                for (int p0 = 0; p0 < ntok && pok; p0 += P_MAX) {
                    const int npass = min(P_MAX, ntok - p0);
                    // X rows of the pass's tokens (MoE: the token of a slot is slot / topk).
                    int tok[MOE ? P_MAX : 1];
                    if constexpr (MOE) {
    #pragma unroll
                        for (int i = 0; i < P_MAX; ++i)
                            tok[i] = i < npass ? s_sorted[seg0 + p0 + i] / a.topk : 0;
                    }
                    for (int c = 0; c < KC; ++c, ++q) {
                        if (q >= S) {  // wait until the consumers released the slot's previous round
                            const uint32_t par = wrap ^ 1u;
                            bool w = mbar_test_wait(&empty[s], par);
                            for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                                w = mbar_try_wait(&empty[s], par);
                            if (!w) {
                                if (!*abort_flag) record_status(a.status, kStTimeout);
                                *abort_flag = 1u;
                                pok = false;
                                break;
                            }
                        }
                        uint32_t wbytes, xbytes;
                        chunk_bytes(nt, c, wbytes, xbytes);
                        uint8_t *dst = stages + (size_t)s * L::kStageBytes;
                        if (q >= early) {
                            mbar_arrive_expect_tx(&full[s], wbytes + npass * xbytes);
                            issue_w(dst, &full[s], nt, c, trow, tmat, policy);
                        }
    #pragma unroll
                        for (int i = 0; i < P_MAX; ++i)
                            if (i < npass)
                                bulk_g2s_nohint(dst + L::kWBytes + i * kXChunkBytes,
                                                a.X + (size_t)(MOE ? tok[MOE ? i : 0] : p0 + i) * k +
                                                    (size_t)c * kBlocks * 32,
                                                xbytes, &full[s]);
                        if (++s == S) {
                            s = 0;
                            wrap ^= 1u;
                        }
                    }
                }
                wk.advance(nt);
            }
            *s_q = q;
        }
        __syncwarp();
    } else {

    // ---------------------------------------------------------------- consumers
    for (auto wk = make_walk(); wk.more() && ok;) {
        const int ntiles = wk.template group<T>();
        const int seg0 = MOE ? s_seg[wk.ai] : 0;
        const int ntok_all = MOE ? s_seg[wk.ai + 1] - seg0 : a.n;
        const int e = MOE ? s_act[wk.ai] : 0;
        const int row0 = wk.tl * 16;
        for (int p0 = 0; p0 < ntok_all && ok; p0 += P_MAX) {
            const int ntok = min(P_MAX, ntok_all - p0);
            // One pass over the group's chunks; the column layout is a compile-time
            // choice so the tile loop carries no layout branches.
            auto pass = [&](auto pk, auto ck) {
                // packed: 1-4 tokens, column g = term (g % 2) of token (g / 2), one n-tile
                // (a thread's two accumulator columns are one token's two terms);
                // else split-major: n-tile s, column g = token g (+8 for the second half).
                constexpr bool packed = decltype(pk)::value;
                // one- and two-token packed passes: each lane splits one element of its
                // block per token and the warp shares the B fragments through s_coop
                constexpr bool COOP = packed && decltype(ck)::value && L::kCoopBytes > 0;
                const int P = packed ? ntok : (WIDE ? 16 : 8);
                int xslot[NH];  // the token slot of this thread's B column in the stage
                bool tok_ok[NH];
                int col_s = 0;  // packed: which split this thread's column carries
    #pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const int i = packed ? g >> 1 : h * 8 + g;
                    tok_ok[h] = packed ? (g < 2 * P) : (i < ntok);
                    xslot[h] = tok_ok[h] ? i : 0;
                }
                if (packed) col_s = g & 1;
                int coop_w = 0, coop_r = 256;  // u16 index of lane's write; byte offset of the read
                if constexpr (COOP) {
                    const int j = lane;
                    const int tt = WT == kQ4_0 ? (j & 15) >> 2 : j >> 3;
                    const int w = WT == kQ4_0 ? j & 3 : j & 7;
                    const int pair = WT == kQ4_0 ? 2 * (j >> 4) + (w & 1) : 2 * (w >> 2) + (w & 1);
                    const int half = WT == kQ4_0 ? w >> 1 : (w >> 1) & 1;
                    coop_w = tt * 8 + pair * 2 + half;
                    if (g < 2 * P) coop_r = (g * 4 + t) * 16;  // [token][term][t] = [g][t]
                }

                // Stage this pass's bias and residual values in shared memory now, so the
                // epilogue does not wait on global loads (same index map as the epilogue).
                {
                    const int R = ntiles * 16;
                    for (int idx = threadIdx.x; idx < R * ntok; idx += kCW * 32) {
                        const int i = idx / R, r = idx % R, row = row0 + r;
                        if (row < m) {
                            if (a.flags & kResidual) {
                                const int yrow = MOE ? s_sorted[seg0 + p0 + i] : p0 + i;
                                cp_async4(&s_res[idx], a.R + (size_t)yrow * (MOE ? m : a.ldy) + row);
                            }
                            if (i == 0 && (a.flags & kBias))
                                cp_async4(&s_bias[r], a.bias + (MOE ? (size_t)e * m + row : (size_t)row));
                        }
                    }
                    cp_async_commit();
                }
                float acc[T][NA][4];
    #pragma unroll
                for (int tt = 0; tt < T; ++tt)
    #pragma unroll
                    for (int j = 0; j < NA; ++j)
    #pragma unroll
                        for (int r = 0; r < 4; ++r) acc[tt][j][r] = 0.f;

                // The warp's block sits at the same offset in every stage; its code bytes
                // start 4-byte aligned when the block's byte offset is 2 mod 4.
                const int wb = warp;
                const bool qs_aligned = ((F::BB * (wb % F::BOXB)) & 3) == 2;
                const int blk_off = (wb / F::BOXB) * L::kBoxBytes +
                                    (wb % F::BOXB) * F::BB + g * F::ROWB;

                for (int c = 0; c < KC; ++c) {
                    const int s = qs;
                    const uint32_t par = qph;
                    if (++qs == S) {
                        qs = 0;
                        qph ^= 1u;
                    }
                    bool w = mbar_test_wait(&full[s], par);
                    for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                        w = mbar_try_wait(&full[s], par);
                    w = __all_sync(0xFFFFFFFFu, w);
                    if (!w) {
                        if (lane == 0) {
                            if (!*abort_flag) record_status(a.status, kStTimeout);
                            *abort_flag = 1u;
                        }
                        ok = false;
                        break;
                    }
                    if (c * kBlocks + wb < nb) {
                        // B: each token's block scaled by a power of two (block_scale), then
                        // split into two f16 terms; pairs in the A decode's order.
                        uint32_t bf[2][NT][2];
                        float inv0[NH], inv1[NH];
                        if constexpr (COOP) {
                            // Lane j takes element j of the block for each token: scale, split,
                            // and store both terms at the fragment slot that wants them
                            // ([token][term][thread t][pair][half], f16).
                            const float *xb = reinterpret_cast<const float *>(
                                stages + (size_t)s * L::kStageBytes + L::kWBytes) + wb * 32 + lane;
                            uint16_t *cw = reinterpret_cast<uint16_t *>(s_coop + wb * 272) + coop_w;
                            float invp[2];
                            auto split_one = [&](int p) {
                                const float x = xb[p * (kXChunkBytes / 4)];
                                const uint32_t mb =
                                    __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(x) & 0x7FFFFFFFu);
                                float sc;
                                block_scale_bits(mb, sc, invp[p]);
                                const float xs = x * sc;
                                const uint16_t h1 = f16_rn(xs);
                                cw[p * 64] = h1;
                                cw[p * 64 + 32] = f16_rn(xs - f16_f32(h1));
                            };
                            split_one(0);
                            if (ntok > 1)
                                split_one(1);
                            else
                                invp[1] = invp[0];
                            __syncwarp();
                            const uint4 bv = *reinterpret_cast<const uint4 *>(s_coop + wb * 272 + coop_r);
                            bf[0][0][0] = bv.x;
                            bf[0][0][1] = bv.y;
                            bf[1][0][0] = bv.z;
                            bf[1][0][1] = bv.w;
                            inv0[0] = t == 0 ? invp[0] : invp[1];  // the columns of token t
                            inv1[0] = inv0[0];
                        } else {
                            uint32_t sp[NH][4][2];
                            float inv_own[NH];
                            const uint8_t *xst = stages + (size_t)s * L::kStageBytes + L::kWBytes;
    #pragma unroll
                            for (int h = 0; h < NH; ++h) {
                                // This thread's 8 values of its column's token, in the A decode's
                                // order (zeros for a padding column).
                                float xv[8];
                                float4 u0v = make_float4(0.f, 0.f, 0.f, 0.f), u1v = u0v;
                                if (tok_ok[h]) {
                                    const float *xp = reinterpret_cast<const float *>(
                                        xst + xslot[h] * kXChunkBytes) + wb * 32;
                                    u0v = *reinterpret_cast<const float4 *>(xp + (WT == kQ4_0 ? 4 * t : 8 * t));
                                    u1v = *reinterpret_cast<const float4 *>(xp + (WT == kQ4_0 ? 16 + 4 * t : 8 * t + 4));
                                }
                                xv[0] = u0v.x; xv[1] = u0v.y; xv[2] = u0v.z; xv[3] = u0v.w;
                                xv[4] = u1v.x; xv[5] = u1v.y; xv[6] = u1v.z; xv[7] = u1v.w;
                                float mx = 0.f;
    #pragma unroll
                                for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(xv[j]));
                                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
                                mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
                                float sc;
                                block_scale(mx, sc, inv_own[h]);
                                float xs[8];
    #pragma unroll
                                for (int j = 0; j < 8; ++j) xs[j] = xv[j] * sc;
                                split2(xs[0], xs[2], sp[h][0][0], sp[h][0][1]);
                                split2(xs[1], xs[3], sp[h][1][0], sp[h][1][1]);
                                split2(xs[4], xs[6], sp[h][2][0], sp[h][2][1]);
                                split2(xs[5], xs[7], sp[h][3][0], sp[h][3][1]);
                            }
                            // 1/scale of the accumulator columns 2t and 2t+1: that of the threads
                            // whose B column they are (g = 2t, 2t+1).
    #pragma unroll
                            for (int h = 0; h < NH; ++h) {
                                inv0[h] = __shfl_sync(0xFFFFFFFFu, inv_own[h], 8 * t);
                                inv1[h] = packed ? inv0[h]  // packed: both columns are token t's
                                                 : __shfl_sync(0xFFFFFFFFu, inv_own[h], 8 * t + 4);
                            }
                            // B fragments [k-step][n-tile][reg]: k-step 0 uses pairs 0,1; k-step 1 pairs 2,3.
    #pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
    #pragma unroll
                                for (int ks = 0; ks < 2; ++ks) {
    #pragma unroll
                                    for (int rr = 0; rr < 2; ++rr) {
                                        const int pr = ks * 2 + rr;
                                        uint32_t v;
                                        if (WIDE) {
                                            v = sp[nt & 1][pr][nt >> 1];  // n-tile = 2 * term + half
                                        } else if (packed) {
                                            v = col_s == 0 ? sp[0][pr][0] : sp[0][pr][1];
                                        } else {
                                            v = sp[0][pr][nt];            // n-tile = term
                                        }
                                        bf[ks][nt][rr] = v;
                                    }
                                }
                            }
                        }
                        const uint8_t *st = stages + (size_t)s * L::kStageBytes + blk_off;
                        // Only the group's tiles are loaded and computed.
                        auto tiles = [&](auto aligned, auto whole) {
                            constexpr bool AL = decltype(aligned)::value;
                            constexpr bool FULL = decltype(whole)::value;
    #pragma unroll
                            for (int tt = 0; tt < T; ++tt) {
                                if (!FULL && tt >= ntiles) break;
                                const uint8_t *r0p = st + tt * L::kTileBytes;
                                const uint8_t *r1p = r0p + 8 * F::ROWB;
                                const float d0 = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(r0p));
                                const float d1 = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(r1p));
                                uint32_t a1[4], a2[4];  // A of k-step 0 and 1
                                if (WT == kQ4_0) {
                                    uint32_t v0, v1;
                                    if (AL) {
                                        v0 = *reinterpret_cast<const uint32_t *>(r0p + 2 + 4 * t);
                                        v1 = *reinterpret_cast<const uint32_t *>(r1p + 2 + 4 * t);
                                    } else {
                                        const uint32_t *w0 = reinterpret_cast<const uint32_t *>(r0p + 4 * t);
                                        const uint32_t *w1 = reinterpret_cast<const uint32_t *>(r1p + 4 * t);
                                        v0 = __funnelshift_r(w0[0], w0[1], 16);
                                        v1 = __funnelshift_r(w1[0], w1[1], 16);
                                    }
                                    decode_q4(v0, a1[0], a1[2], a2[0], a2[2]);
                                    decode_q4(v1, a1[1], a1[3], a2[1], a2[3]);
                                } else {
                                    uint32_t v00, v01, v10, v11;  // bytes 8t.., 8t+4.. of rows g, g+8
                                    if (AL) {
                                        const uint32_t *w0 = reinterpret_cast<const uint32_t *>(r0p + 2 + 8 * t);
                                        const uint32_t *w1 = reinterpret_cast<const uint32_t *>(r1p + 2 + 8 * t);
                                        v00 = w0[0]; v01 = w0[1];
                                        v10 = w1[0]; v11 = w1[1];
                                    } else {
                                        const uint32_t *w0 = reinterpret_cast<const uint32_t *>(r0p + 8 * t);
                                        const uint32_t *w1 = reinterpret_cast<const uint32_t *>(r1p + 8 * t);
                                        const uint32_t x0 = w0[0], x1 = w0[1], x2 = w0[2];
                                        const uint32_t y0 = w1[0], y1 = w1[1], y2 = w1[2];
                                        v00 = __funnelshift_r(x0, x1, 16);
                                        v01 = __funnelshift_r(x1, x2, 16);
                                        v10 = __funnelshift_r(y0, y1, 16);
                                        v11 = __funnelshift_r(y1, y2, 16);
                                    }
                                    decode_q8(v00, a1[0], a1[2]);
                                    decode_q8(v01, a2[0], a2[2]);
                                    decode_q8(v10, a1[1], a1[3]);
                                    decode_q8(v11, a2[1], a2[3]);
                                }
                                if (packed) {
                                    // columns 2t, 2t + 1: token t's two terms, one scale;
                                    // accumulators [0] and [1] hold rows g and g + 8
                                    float part[4];
                                    mma_f16_z(part, a1, bf[0][0][0], bf[0][0][1]);
                                    mma_f16(part, a2, bf[1][0][0], bf[1][0][1]);
                                    acc[tt][0][0] = fmaf(d0 * inv0[0], part[0] + part[1], acc[tt][0][0]);
                                    acc[tt][0][1] = fmaf(d1 * inv0[0], part[2] + part[3], acc[tt][0][1]);
                                } else {
                                    // The two terms of a token sit in the same thread and column
                                    // of two n-tiles: one accumulator chain sums them.
    #pragma unroll
                                    for (int h = 0; h < NH; ++h) {
                                        float part[4];
    #pragma unroll
                                        for (int sp_i = 0; sp_i < 2; ++sp_i) {
                                            const int nt = WIDE ? 2 * sp_i + h : sp_i;
                                            if (sp_i == 0)
                                                mma_f16_z(part, a1, bf[0][nt][0], bf[0][nt][1]);
                                            else
                                                mma_f16(part, a1, bf[0][nt][0], bf[0][nt][1]);
                                            mma_f16(part, a2, bf[1][nt][0], bf[1][nt][1]);
                                        }
                                        scale_acc(acc[tt][h], part, d0, d1, inv0[h], inv1[h]);
                                    }
                                }
                            }
                        };
                        using Yes = std::true_type;
                        using No = std::false_type;
                        if (ntiles == T) {  // (a separate copy keeps the full group's schedule)
                            if (qs_aligned)
                                tiles(Yes{}, Yes{});
                            else
                                tiles(No{}, Yes{});
                        } else {
                            if (qs_aligned)
                                tiles(Yes{}, No{});
                            else
                                tiles(No{}, No{});
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
                // Ordered reduction: warp w adds into buffer w % NB, in kCW / NB rounds.
                // Round 0 needs no barrier before it (the buffers were last read before
                // the previous pass's final barrier); an aborted warp's writes are
                // harmless, as the pass ends at the next barrier.
                constexpr int NB = L::kRedBufs;
                const int RT = T * 16 * C;
                auto round = [&](int rnd) {
                    if (warp / NB != rnd) return;
                    float *buf = red + (warp % NB) * RT;
    #pragma unroll
                    for (int tt = 0; tt < T; ++tt) {
                        if (tt < ntiles) {
                            if (packed) {  // token t of rows g, g + 8 in column t
    #pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    float *dst = &buf[(tt * 16 + g + 8 * r) * C + t];
                                    *dst = (rnd == 0) ? acc[tt][0][r] : *dst + acc[tt][0][r];
                                }
                            } else {
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
                };
                round(0);
                cp_async_wait_all();  // staged bias/residual: visible to all after the barrier
                // Every consumer warp gets here, aborted or not, and all of them get the
                // same answer, so they leave (or go on) together (lane 0 of a warp that
                // gave up has set the flag itself).
                ok = !consumers_sync_any<CW>(*abort_flag != 0u);
                if (!ok) return;
                for (int rnd = 1; rnd < kCW / NB; ++rnd) {
                    round(rnd);
                    consumers_sync<CW>();
                }
                const int R = ntiles * 16;
                for (int idx = threadIdx.x; idx < R * ntok; idx += kCW * 32) {
                    const int i = idx / R, r = idx % R;
                    const int row = row0 + r;
                    if (row < m) {
                        float v = 0.f;
    #pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            const float *rp = red + b * RT + r * C;
                            v += rp[i];  // packed: the token's two terms already summed
                        }
                        const int yrow = MOE ? s_sorted[seg0 + p0 + i] : p0 + i;
                        // MoE has no second band: its rows are m wide.
                        float *yp = a.Y + (size_t)yrow * (MOE ? m : a.ldy) + row;
                        *yp = epilogue_vals(v, a.flags, s_bias[r], s_res[idx], a.alpha);
                        if (!MOE && row < a.dual) yp[m] = v + a.bias2[row];  // the raw second band
                    }
                }
                consumers_sync<CW>();
            };
            using Y = std::true_type;
            using N = std::false_type;
            if constexpr (MODE == kPacked) {
                if (ntok <= 2)
                    pass(Y{}, Y{});
                else
                    pass(Y{}, N{});
            } else if constexpr (MODE == kMixed) {
                // (MoE: with eight consumer warps per CTA the shared split's longer
                // dependency chain per chunk costs more than it saves; measured)
                if (ntok <= 4)
                    pass(Y{}, N{});
                else
                    pass(N{}, N{});
            } else {
                pass(N{}, N{});
            }
        }
        wk.advance(ntiles);
    }
    }  // consumers
    // The window's routing tables are rewritten by the next window: every thread is
    // done with them here.  (Consumers that gave up skipped the rest of the window;
    // no window is started after an abort.)
    if (n_win > 1) __syncthreads();
    }  // windows
    if (warp == kCW && lane == 0) {
        // Drain copies that no consumer waited for (only after an abort).
        const long long q = *s_q;
        for (long long d = (q > S ? q - S : 0); d < q; ++d)
            mbar_wait(&full[d % S], (uint32_t)((d / S) & 1), kDrainPolls);
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

template <int WT, int MODE, int T, int CW>
constexpr size_t smem_bytes() {
    using L = Layout<WT, MODE, T, CW>;
    return (size_t)L::kStages * L::kStageBytes + L::kRedBytes + L::kEpiBytes + L::kCoopBytes +
           2 * L::kStages * sizeof(uint64_t) +
           kMaxSlots * sizeof(unsigned long long) + (3 * kMaxSlots + 4 + 32) * sizeof(int) + 32;
}

// The weight image as a 3-D tensor [matrices][m][row bytes] (one matrix for a GEMV,
// the experts for MoE): a box that runs past a matrix's last row reads nothing
// there (the rows are out of bounds and zero-filled), so a short row group at an
// expert's end does not fetch the next expert's rows.
bool make_map(CUtensorMap &map, const StreamArgs &a, int wtype, long long matrices, int box_rows,
              int box) {
    auto encode = encode_fn();
    if (!encode) return false;
    const size_t rb = row_bytes(wtype, a.k);
    const cuuint64_t dims[3] = {(cuuint64_t)(rb / 2), (cuuint64_t)a.m, (cuuint64_t)matrices};
    const cuuint64_t strides[2] = {(cuuint64_t)rb, (cuuint64_t)rb * a.m};
    const cuuint32_t boxd[3] = {(cuuint32_t)(box / 2), (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint8_t *>(a.W), dims,
                  strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int WT, bool MOE, int MODE, int T, int CW = 16>
cudaError_t launch_inst(const StreamArgs &a, long long matrices, int grid, const DeviceInfo &dev,
                        cudaStream_t stream) {
    static std::atomic<unsigned long long> smem_set{0};
    WMaps maps;
    constexpr int rb = Fmt<WT, CW>::ROWB;
    if (!make_map(maps.full, a, WT, matrices, T * 16, rb) ||
        !make_map(maps.b4, a, WT, matrices, (T > 4 ? 4 : T) * 16, rb) ||
        !make_map(maps.b2, a, WT, matrices, (T > 2 ? 2 : T) * 16, rb) ||
        !make_map(maps.b1, a, WT, matrices, 16, rb))
        return cudaErrorInvalidValue;
    auto kern = gemv_mma_kernel<WT, MOE, MODE, T, CW>;
    constexpr size_t bytes = smem_bytes<WT, MODE, T, CW>();
    static_assert(Warps<CW>::kCtas * (bytes + 1024) <= 228 * 1024, "CTAs per SM");
    static_assert(bytes <= 227 * 1024, "shared memory budget");
    cudaError_t err = ensure_smem(kern, (int)bytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    if (Warps<CW>::kCtas > 1) {  // the largest shared-memory carve-out, so that both fit
        static std::atomic<unsigned long long> carve_set{0};
        const unsigned long long bit = 1ull << (dev.ordinal & 63);
        if (!(carve_set.load(std::memory_order_acquire) & bit)) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
            if (err != cudaSuccess) return err;
            carve_set.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    return launch_pdl(kern, dim3(grid), dim3(Warps<CW>::kThreads), bytes, stream, maps, a);
}

template <int WT, int MODE>
cudaError_t launch_gemv_mode(const StreamArgs &a, int grid, long long per, const DeviceInfo &dev,
                             cudaStream_t stream) {
    if (per <= 2) return launch_inst<WT, false, MODE, 2>(a, 1, grid, dev, stream);
    if (per <= 4) return launch_inst<WT, false, MODE, 4>(a, 1, grid, dev, stream);
    return launch_inst<WT, false, MODE, 6>(a, 1, grid, dev, stream);
}

template <int WT>
cudaError_t launch_gemv_wt(const StreamArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    const long long tiles = (a.m + 15) / 16;
    const int grid = (int)(tiles < dev.sm_count ? tiles : dev.sm_count);
    const long long per = (tiles + grid - 1) / grid;  // tiles per CTA (max)
    if (a.n > 8) return launch_inst<WT, false, kSplit16, 3>(a, 1, grid, dev, stream);
    if (a.n > 4) return launch_gemv_mode<WT, kSplit8>(a, grid, per, dev, stream);
    return launch_gemv_mode<WT, kPacked>(a, grid, per, dev, stream);
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
    // Two CTAs of eight consumer warps per SM, with 128-row (Q4_0) or 96-row (Q8_0)
    // groups: measured on GB300 against one CTA of sixteen warps (6 % less time for
    // both formats at 16 tokens x top-6 of 64 experts, 1408 x 2048 each).  Groups
    // half as tall when at most that many active experts (the slots, or the bank)
    // give too few full groups to go round: the fewer rounds x (tiles + 7) (a pass
    // over a group costs about seven tiles' worth of work besides its tiles).
    const long long matrices = a.n_experts;
    const int grid = dev.sm_count * Warps<8>::kCtas;
    const long long slots = (long long)a.n * a.topk;
    const long long nact = slots < a.n_experts ? slots : a.n_experts;
    const long long tpe = (a.m + 15) / 16;
    auto est = [&](long long t) {
        const long long groups = nact * ((tpe + t - 1) / t);
        return (groups + grid - 1) / grid * (t + 7);
    };
    if (wtype == kQ4_0)
        return est(4) < est(8) ? launch_inst<kQ4_0, true, kMixed, 4, 8>(a, matrices, grid, dev, stream)
                               : launch_inst<kQ4_0, true, kMixed, 8, 8>(a, matrices, grid, dev, stream);
    return est(3) < est(6) ? launch_inst<kQ8_0, true, kMixed, 3, 8>(a, matrices, grid, dev, stream)
                           : launch_inst<kQ8_0, true, kMixed, 6, 8>(a, matrices, grid, dev, stream);
}

}  // namespace wq
