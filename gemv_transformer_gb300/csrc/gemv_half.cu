// gemv_half.cu -- small-n GEMV with bf16-pair or F16 weights on the tensor cores.
//
// Computes the same contraction as gemv_stream.cu for 16-bit float weights
// (cortiq-engine 0.8.49 AudioEncoder::gemm / ae_gemm: W as bf16 pairs, Y (=|+=)
// X.W^T with the ae_put epilogue; wavo's F16 weights and Pass::gemv for the small-n
// call), for 1 <= n <= 16 and k % 256 == 0.
//
// A bf16 or f16 weight is exact as an operand of mma.sync.m16n8k16 (bf16 x bf16 or
// f16 x f16 -> f32), so the weights are not decoded at all: a producer warp streams
// 16-row tiles by TMA into shared memory in the 128-byte-swizzled layout, and
// ldmatrix hands each warp its A fragments directly.  X is split into terms of the
// weights' type after scaling each token's 64-element slice of a chunk by a power
// of two: bf16, three terms, x ~ t1 + t2 + t3 with |x - t1 - t2 - t3| <= 2^-24 |x|
// (each term the next 8 bits of the significand; the scale keeps the third term a
// normal number); f16, two terms with the slice's largest |x| scaled into [2^14,
// 2^15), |x - t1 - t2| <= 2^-22 |x| (below 2^-17 of that largest |x| an absolute
// 2^-39 of it, f16's subnormal floor).  Every product of a weight and a term is
// exact in f32, and the terms of a token occupy separate n-tiles whose MMAs add
// into one partial sum per slice; the slice's partial sums are multiplied by the
// inverse power of two into the f32 accumulator (one rounding per 64 elements of
// k), so the result is within 2^-22 sum|x||w| plus f32 rounding of the sums --
// inside the 1e-5 sum|x||w| contract.
//
// Work: every CTA takes groups of T 16-row tiles; the producer warp loads a chunk
// of 256 k for the whole group per stage (four 64-element TMA boxes of T*16 rows,
// plus the chunk of X of every token by bulk copies).  Its T * KS consumer warps
// each own one tile and one of KS slices of every chunk's k.  Per chunk all
// consumer warps first build the B fragments in shared memory together (one warp
// per token and 64-element slice: its block maximum, scale and three-term split,
// written in fragment order) and meet at a barrier; then each warp runs its tile
// over its slices: per 16-k step one ldmatrix.x4 and, per token half and term, one
// 8-byte fragment load and one MMA, the three terms in three accumulators so that
// the MMAs do not wait on one another.  At the end of a group the KS partial sums
// of a tile are added in slice order in shared memory (deterministic) and the
// epilogue is fused into the store.  The B buffer is double-buffered: the barrier
// of chunk c is passed only after every warp has finished chunk c - 1, so chunk
// c + 1 may reuse chunk c - 1's buffer.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "wq_device.cuh"
#include "wq_internal.h"
#include "tile_sched.cuh"

namespace wq {
namespace {

constexpr int kChunk = 256;              // k per stage
constexpr int kBoxK = 64;                // k per TMA box: 128 bytes, the swizzle span
constexpr int kParts = kChunk / kBoxK;   // 64-element slices per chunk
constexpr int kKSteps = kChunk / 16;     // MMA k-steps per chunk
constexpr int kBudget = 200 * 1024;      // stages + B fragments

// The X terms of each weight type: bf16 three (scaled to 2^62), f16 two (scaled to
// 2^14, below f16's largest finite value).
template <int WT>
struct Terms {
    static constexpr int kN = WT == kBF16 ? 3 : 2;
    static constexpr int kTarget = WT == kBF16 ? 62 : 14;  // log2 of the scaled largest |x|
};

// T tiles per group; KS slices of each chunk's k (a warp per tile and slice); NH
// halves of eight tokens (n <= 8 NH).
template <int WT, int T, int KS, int NH>
struct BL {
    static constexpr int TN = Terms<WT>::kN;
    static constexpr int kCW = T * KS;                    // consumer warps
    static constexpr int kPP = kParts / KS;               // 64-element slices per warp
    static constexpr int kThreads = (kCW + 1) * 32;
    static constexpr int kBoxBytes = T * 16 * 128;        // T*16 rows x 64 bf16
    static constexpr int kWBytes = kParts * kBoxBytes;
    static constexpr int kXBytes = NH * 8 * kChunk * 4;   // f32 X of up to 8 * NH tokens
    static constexpr int kStageBytes = kWBytes + kXBytes;
    // B fragments of one chunk, u32 [k-step][term][half][lane][2], and the slices'
    // inverse scales, f32 [part][token]
    static constexpr int kFragWords = kKSteps * TN * NH * 32 * 2;
    static constexpr int kInvWords = kParts * 16;
    static constexpr int kBufWords = kFragWords + kInvWords;
    // the tiles' partial sums per slice, f32 [KS][T][lane][NH * 4]
    static constexpr int kRedWords = KS > 1 ? KS * T * 32 * NH * 4 : 0;
    static constexpr int kFit = (kBudget - 2 * kBufWords * 4 - kRedWords * 4) / kStageBytes;
    static constexpr int kStages = kFit > 8 ? 8 : kFit;
    static_assert(kStages >= 2, "at least two stages");
    static_assert(kStageBytes % 1024 == 0 && kBoxBytes % 1024 == 0, "swizzle atoms");
    static constexpr size_t kBytes = (size_t)kStages * kStageBytes + 2 * kBufWords * 4 +
                                     kRedWords * 4 + 2 * kStages * 8 + 16 + 1024;
};

__device__ __forceinline__ uint16_t bf16_rn(float v) {
    unsigned short h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
    return h;
}

__device__ __forceinline__ float bf16_val(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ uint16_t f16_rn(float v) {
    unsigned short h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
    return h;
}

__device__ __forceinline__ float f16_val(uint16_t h) {
    float v;
    asm("cvt.f32.f16 %0, %1;" : "=f"(v) : "h"(h));
    return v;
}

// A term of the weights' type, rounded to nearest even, and its value.
template <int WT>
__device__ __forceinline__ uint16_t term_rn(float v) {
    return WT == kBF16 ? bf16_rn(v) : f16_rn(v);
}
template <int WT>
__device__ __forceinline__ float term_val(uint16_t h) {
    return WT == kBF16 ? bf16_val(h) : f16_val(h);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += A.B (bf16 or f16 operands, f32 accumulation).
template <int WT>
__device__ __forceinline__ void mma_16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
    if (WT == kBF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}


// The B fragments of one chunk for tokens [0, nt): one warp per (token, 64-element
// slice) scales by a power of two, splits into TN terms and stores each term where
// its fragment wants it; lane 0 keeps the slice's inverse scale.
template <class L, int WT, int NH, int CW>
__device__ __forceinline__ void build_b(const uint8_t *st, uint32_t *fb, float *invb, int nt,
                                        int warp, int lane) {
    constexpr int TN = L::TN;
    // B: one warp per (token, 64-element slice): scale by a power of two,
    // split into TN terms, store each where its fragment wants it.
    const float *xs = reinterpret_cast<const float *>(st + L::kWBytes);
    uint16_t *f16 = reinterpret_cast<uint16_t *>(fb);
    for (int it = warp; it < nt * kParts; it += CW) {
        const int tok = it / kParts, p = it % kParts;
        const float x0 = xs[tok * kChunk + p * kBoxK + lane];
        const float x1 = xs[tok * kChunk + p * kBoxK + 32 + lane];
        const uint32_t mb = __reduce_max_sync(
            0xFFFFFFFFu, max(__float_as_uint(x0) & 0x7FFFFFFFu,
                             __float_as_uint(x1) & 0x7FFFFFFFu));
        // sc = 2^(sb - 127) with the slice's largest |x| * sc in [2^target,
        // 2^(target + 1)) (E is that |x|'s biased exponent); sb kept in [1,
        // 253] so that sc and 1/sc are normal.
        const int E = (int)((mb >> 23) & 0xFFu);
        const int sb = min(253, max(1, 254 + Terms<WT>::kTarget - E));
        const float sc = __uint_as_float((uint32_t)sb << 23);
        if (lane == 0) invb[p * 16 + tok] = __uint_as_float((uint32_t)(254 - sb) << 23);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float xv = (e ? x1 : x0) * sc;
            const uint16_t h1 = term_rn<WT>(xv);
            const float r1 = xv - term_val<WT>(h1);
            const uint16_t h2 = term_rn<WT>(r1);
            // element kc of the chunk -> k-step kk, register reg of thread
            // (g = token % 8, tt), low or high half
            const int kc = p * kBoxK + e * 32 + lane;
            const int kk = kc >> 4, r = kc & 15;
            const int reg = r >> 3, tt = (r & 7) >> 1, half = r & 1;
            const int ln = (tok & 7) * 4 + tt;
            const int i0 = (((kk * TN * NH + (tok >> 3)) * 32 + ln) * 2 + reg) * 2 + half;
            f16[i0] = h1;                   // term 0
            f16[i0 + NH * 128] = h2;        // term 1: + NH * 32 lanes * 2 regs * 2
            if (TN == 3)                    // term 2
                f16[i0 + 2 * NH * 128] = term_rn<WT>(r1 - term_val<WT>(h2));
        }
    }
}

// This warp's 64-element slices of one chunk for the 16 rows of its tile, added
// into acc (rows g, g + 8 x tokens 2t, 2t + 1 of each half).
template <class L, int WT, int NH>
__device__ __forceinline__ void tile_chunk(const uint8_t *st, const uint32_t *fb,
                                           const float *invb, float (&acc)[NH][4], int tw,
                                           int sw, int lane, int t) {
    constexpr int TN = L::TN;
    // The tile: 16 rows over this warp's 64-element slices of the chunk, a
    // partial sum per slice (per term, added after the slice's MMAs).
#pragma unroll 1
    for (int p = sw * L::kPP; p < (sw + 1) * L::kPP; ++p) {
        float part[NH][TN][4];
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int term = 0; term < TN; ++term)
#pragma unroll
                for (int r = 0; r < 4; ++r) part[h][term][r] = 0.f;
        const uint8_t *box = st + p * L::kBoxBytes;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = p * 4 + k4;
            // ldmatrix.x4: matrices (rows 0-7, k 0-7), (8-15, 0-7), (0-7, 8-15),
            // (8-15, 8-15) of the tile: lane l gives row (l & 8) + (l & 7) of
            // matrix l / 8, 16-byte chunk 2 * k4 + l / 16, swizzled by row.
            const int mi = lane >> 3;
            const int row = tw * 16 + ((mi & 1) << 3) + (lane & 7);
            const int ch = 2 * k4 + (mi >> 1);
            uint32_t A[4];
            ldmatrix_x4(A, smem_addr(box + row * 128 + ((ch ^ (row & 7)) << 4)));
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int term = 0; term < TN; ++term) {
                    const uint2 b = *reinterpret_cast<const uint2 *>(
                        fb + (((kk * TN + term) * NH + h) * 32 + lane) * 2);
                    mma_16<WT>(part[h][term], A, b.x, b.y);
                }
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            const float2 iv = *reinterpret_cast<const float2 *>(invb + p * 16 + h * 8 + 2 * t);
            float v[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                v[r] = TN == 3 ? (part[h][0][r] + part[h][1][r]) + part[h][TN - 1][r]
                               : part[h][0][r] + part[h][1][r];
            acc[h][0] = fmaf(iv.x, v[0], acc[h][0]);
            acc[h][1] = fmaf(iv.y, v[1], acc[h][1]);
            acc[h][2] = fmaf(iv.x, v[2], acc[h][2]);
            acc[h][3] = fmaf(iv.y, v[3], acc[h][3]);
        }
    }
}

template <int WT, int T, int KS, int NH>
__global__ void __launch_bounds__(BL<WT, T, KS, NH>::kThreads, 1)
    gemv_half_kernel(const __grid_constant__ CUtensorMap wmap, const StreamArgs a) {
    // Barriers and the descriptor are set up before waiting for the previous grid
    // (they touch nothing it writes); global memory after.
    pdl_launch();
    using L = BL<WT, T, KS, NH>;
    constexpr int S = L::kStages;
    constexpr int CW = L::kCW;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *stages = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // swizzle atoms: 1 KB
    uint32_t *bufs = reinterpret_cast<uint32_t *>(stages + (size_t)S * L::kStageBytes);
    float *red = reinterpret_cast<float *>(bufs + 2 * L::kBufWords);
    uint64_t *full = reinterpret_cast<uint64_t *>(red + L::kRedWords);
    uint64_t *empty = full + S;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(empty + S);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int tw = warp % T, sw = warp / T;  // consumers: tile and k slice of this warp
    const int n = a.n, m = a.m, k = a.k;
    const int KC = k / kChunk;
    const int groups = ((m + 15) / 16 + T - 1) / T;
    const uint64_t limit = a.wait_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (threadIdx.x == CW * 32)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
    // Both B buffers start at zero: the columns of tokens >= n are never written.
    for (int i = threadIdx.x; i < 2 * L::kBufWords; i += blockDim.x) bufs[i] = 0u;
    __syncthreads();
    // No kernel of this library writes a weight image, so the producer requests the
    // weight boxes of its first stage before the grid-dependency wait, while the
    // previous kernel finishes; its X follows after the wait (the stage barrier
    // expects both).  One stage, as in the quantised GEMV: with more, the first X
    // copy queues behind the early boxes.
    constexpr int kEarly = 1;
    int early = 0;  // stages whose weight boxes went out before the wait
    if (threadIdx.x == CW * 32) {
        const uint64_t policy = l2_evict_first();
        for (int grp = blockIdx.x; grp < groups && early < kEarly; grp += gridDim.x)
            for (int c = 0; c < KC && early < kEarly; ++c, ++early) {
                uint8_t *dst = stages + (size_t)early * L::kStageBytes;
                mbar_arrive_expect_tx(&full[early], (uint32_t)(L::kWBytes + n * kChunk * 4));
                for (int b = 0; b < kParts; ++b)
                    tma_load_2d(dst + b * L::kBoxBytes, &wmap, c * kChunk + b * kBoxK,
                                grp * T * 16, &full[early], policy);
            }
    }
    pdl_wait();

    if (warp == CW) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t policy = l2_evict_first();
            long long q = 0;
            int s = 0;
            uint32_t wrap = 0u;
            bool ok = true;
            for (int grp = blockIdx.x; grp < groups && ok; grp += gridDim.x) {
                const int row0 = grp * T * 16;
                for (int c = 0; c < KC; ++c, ++q) {
                    if (q >= S) {  // the consumers released the slot's previous round
                        bool w = mbar_test_wait(&empty[s], wrap ^ 1u);
                        for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                            w = mbar_try_wait(&empty[s], wrap ^ 1u);
                        if (!w) {
                            if (!*abort_flag) record_status(a.status, kStTimeout);
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                    }
                    uint8_t *dst = stages + (size_t)s * L::kStageBytes;
                    if (q >= early) {
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(L::kWBytes + n * kChunk * 4));
                        for (int b = 0; b < kParts; ++b)
                            tma_load_2d(dst + b * L::kBoxBytes, &wmap, c * kChunk + b * kBoxK,
                                        row0, &full[s], policy);
                    }
                    for (int i = 0; i < n; ++i)
                        bulk_g2s_nohint(dst + L::kWBytes + i * kChunk * 4,
                                   a.X + (size_t)i * k + (size_t)c * kChunk, kChunk * 4, &full[s]);
                    if (++s == S) {
                        s = 0;
                        wrap ^= 1u;
                    }
                }
            }
            // Drain copies no consumer waited for (only after an abort).
            for (long long d = (q > S ? q - S : 0); d < q; ++d)
                mbar_wait(&full[d % S], (uint32_t)((d / S) & 1), kDrainPolls);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    long long q = 0;
    int s = 0;
    uint32_t ph = 0u;
    for (int grp = blockIdx.x; grp < groups; grp += gridDim.x) {
        const int row0 = grp * T * 16;
        float acc[NH][4];
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[h][r] = 0.f;
        for (int c = 0; c < KC; ++c, ++q) {
            bool w = mbar_test_wait(&full[s], ph);
            for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i) w = mbar_try_wait(&full[s], ph);
            w = __all_sync(0xFFFFFFFFu, w);
            if (!w && lane == 0) {
                if (!*abort_flag) record_status(a.status, kStTimeout);
                *abort_flag = 1u;
            }
            // Every consumer warp meets here each chunk, timed out or not, and all of
            // them get the same answer (lane 0 of a warp that gave up set the flag).
            const uint8_t *st = stages + (size_t)s * L::kStageBytes;
            uint32_t *fb = bufs + (int)(q & 1) * L::kBufWords;
            float *invb = reinterpret_cast<float *>(fb + L::kFragWords);
            if (w) build_b<L, WT, NH, CW>(st, fb, invb, n, warp, lane);
            if (consumers_sync_any<CW>(*abort_flag != 0u)) return;
            tile_chunk<L, WT, NH>(st, fb, invb, acc, tw, sw, lane, t);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        // The tile's slices, added in slice order by the warp of slice 0 (its own
        // first); each thread's values sit in a lane slot of its own.
        if (KS > 1) {
            float *mine = red + ((sw * T + tw) * 32 + lane) * (NH * 4);
            if (sw > 0) {
#pragma unroll
                for (int h = 0; h < NH; ++h)
#pragma unroll
                    for (int r = 0; r < 4; ++r) mine[h * 4 + r] = acc[h][r];
            }
            consumers_sync<CW>();
            if (sw == 0) {
#pragma unroll 1
                for (int s2 = 1; s2 < KS; ++s2) {
                    const float *o = red + ((s2 * T + tw) * 32 + lane) * (NH * 4);
#pragma unroll
                    for (int h = 0; h < NH; ++h)
#pragma unroll
                        for (int r = 0; r < 4; ++r) acc[h][r] += o[h * 4 + r];
                }
            }
        }
        if (sw != 0) continue;  // (the next group's chunk barriers order the slots' reuse)
        // Epilogue: thread (g, t) holds rows g, g + 8 of its tile for tokens 2t, 2t + 1
        // of each half.
#pragma unroll
        for (int h = 0; h < NH; ++h)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int row = row0 + tw * 16 + g + (r >= 2 ? 8 : 0);
                const int tok = h * 8 + 2 * t + (r & 1);
                if (row < m && tok < n) {
                    float *yp = a.Y + (size_t)tok * a.ldy + row;
                    const float bj = (a.flags & kBias) ? a.bias[row] : 0.f;
                    const float rij = (a.flags & kResidual) ? a.R[(size_t)tok * a.ldy + row] : 0.f;
                    *yp = epilogue_vals(acc[h][r], a.flags, bj, rij, a.alpha);
                    if (row < a.dual) yp[m] = acc[h][r] + a.bias2[row];  // the raw second band
                }
            }
    }
}

// Tensor maps of a weight bank [E][m][k]: boxes of the group's T tiles, and of 2 and
// 1 tiles, from which a shorter group's rows are composed (rows past an expert's m
// read as zero: the bank is a 3-D tensor).
struct BankMaps {
    CUtensorMap full, b2, b1;
};

// The routed MoE matvec (hanzo-ml 0.11.13 moe_matvec_gpu) with bf16 or F16 weights:
// y[s] = W[ids[s]] . x[s / topk] for every slot s, through the epilogue.  The
// arithmetic per chunk is the GEMV kernel's (build_b, tile_chunk); around it, each
// window of kMaxSlots slots is routed in shared memory (route_window) and the CTAs
// take the active experts' 16-row tiles in groups of T (never across an expert),
// dealt out by cost (DealWalk), once per pass of up to eight of the expert's
// slots.  Output row s of Y and of the residual is slot s's; bias row e of [E][m]
// is expert e's.
//
// A wait that runs out sets the CTA's abort flag: the consumers leave their pass
// together (the answer of consumers_sync_any), the producer stops issuing, no window
// is routed after it, and the producer drains its copies in flight at the end --
// no thread leaves while others still wait at a barrier that counts it.
template <int WT, int T, int KS>
__global__ void __launch_bounds__(BL<WT, T, KS, 1>::kThreads, 1)
    moe_half_kernel(const __grid_constant__ BankMaps wm, const StreamArgs a) {
    pdl_launch();
    using L = BL<WT, T, KS, 1>;
    constexpr int S = L::kStages;
    constexpr int CW = L::kCW;
    static_assert(L::kThreads >= kMaxSlots, "routing: one thread per slot of a window");
    static_assert(T == 1 || T == 2 || T == 4, "short groups are composed of 2- and 1-tile boxes");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *stages = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint32_t *bufs = reinterpret_cast<uint32_t *>(stages + (size_t)S * L::kStageBytes);
    float *red = reinterpret_cast<float *>(bufs + 2 * L::kBufWords);
    uint64_t *full = reinterpret_cast<uint64_t *>(red + L::kRedWords);
    uint64_t *empty = full + S;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(empty + S);
    // the producer's count of stages issued, kept here between windows so that it
    // occupies no register of the consumer warps
    long long *s_q = reinterpret_cast<long long *>(empty + S) + 1;
    RouteSmem rs;
    rs.key = reinterpret_cast<unsigned long long *>(s_q + 1);
    rs.sorted = reinterpret_cast<int *>(rs.key + kMaxSlots);
    rs.seg = rs.sorted + kMaxSlots;
    rs.act = rs.seg + kMaxSlots + 1;
    rs.nact = rs.act + kMaxSlots;
    rs.wcnt = rs.nact + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int tw = warp % T, sw = warp / T;
    const int m = a.m, k = a.k;
    const int KC = k / kChunk;
    const uint64_t limit = a.wait_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        *abort_flag = 0u;
        *s_q = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == CW * 32) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.full)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.b1)) : "memory");
        if (T > 2) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wm.b2)) : "memory");
    }
    for (int i = threadIdx.x; i < 2 * L::kBufWords; i += blockDim.x) bufs[i] = 0u;
    pdl_wait();

    Sched sc;
    sc.tpe = (m + 15) / 16;
    const int S_all = a.n * a.topk;
    const int n_win = (S_all + kMaxSlots - 1) / kMaxSlots;
    // consumers: ring position of the next chunk, carried across windows
    long long q = 0;
    int s = 0;
    uint32_t ph = 0u;
    bool ok = true;

    for (int win = 0; win < n_win; ++win) {
        const int base = win * kMaxSlots;
        __syncthreads();  // the previous window's tables are no longer read
        route_window(a, base, min(kMaxSlots, S_all - base), rs);
        __syncthreads();
        if (*abort_flag) break;  // the same in every thread: no one writes it here
        sc.n_act = *rs.nact;
        // the groups dealt out by cost; the experts' order takes the routing keys' space
        int *s_order = reinterpret_cast<int *>(rs.key);
        order_by_slots(rs.seg, sc.n_act, s_order);
        __syncthreads();

        if (warp == CW) {
            // ------------------------------------------------------------ producer
            if (lane == 0) {
                const uint64_t policy = l2_evict_first();
                long long qp = *s_q;
                int sp = (int)(qp % S);
                uint32_t wrap = (uint32_t)((qp / S) & 1);
                bool pok = true;
                for (DealWalk<T> wk(sc, s_order); wk.more() && pok;) {
                    const int nt = wk.template group<T>();
                    const int seg0 = rs.seg[wk.ai];
                    const int ntok = rs.seg[wk.ai + 1] - seg0;
                    const int trow = wk.tl * 16, ex = rs.act[wk.ai];
                    for (int p0 = 0; p0 < ntok && pok; p0 += 8) {
                        const int npass = min(8, ntok - p0);
                        int tok[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            tok[i] = i < npass ? rs.sorted[seg0 + p0 + i] / a.topk : 0;
                        for (int c = 0; c < KC; ++c, ++qp) {
                            if (qp >= S) {  // the consumers released the slot's previous round
                                bool w = mbar_test_wait(&empty[sp], wrap ^ 1u);
                                for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                                    w = mbar_try_wait(&empty[sp], wrap ^ 1u);
                                if (!w) {
                                    if (!*abort_flag) record_status(a.status, kStTimeout);
                                    *abort_flag = 1u;
                                    pok = false;
                                    break;
                                }
                            }
                            uint8_t *dst = stages + (size_t)sp * L::kStageBytes;
                            mbar_arrive_expect_tx(&full[sp], (uint32_t)(kParts * nt * 16 * 128 +
                                                                        npass * kChunk * 4));
                            for (int b = 0; b < kParts; ++b) {
                                const int x = c * kChunk + b * kBoxK;
                                uint8_t *bd = dst + b * L::kBoxBytes;
                                if (nt == T) {
                                    tma_load_3d(bd, &wm.full, x, trow, ex, &full[sp], policy);
                                } else {  // tile tt of the group lands where it would in a full box
                                    int t0 = 0;
                                    if (T > 2 && (nt & 2)) {
                                        tma_load_3d(bd, &wm.b2, x, trow, ex, &full[sp], policy);
                                        t0 = 2;
                                    }
                                    if (nt & 1)
                                        tma_load_3d(bd + t0 * 16 * 128, &wm.b1, x, trow + 16 * t0,
                                                    ex, &full[sp], policy);
                                }
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                if (i < npass)
                                    bulk_g2s_nohint(dst + L::kWBytes + i * kChunk * 4,
                                               a.X + (size_t)tok[i] * k + (size_t)c * kChunk,
                                               kChunk * 4, &full[sp]);
                            if (++sp == S) {
                                sp = 0;
                                wrap ^= 1u;
                            }
                        }
                    }
                    wk.advance(nt);
                }
                *s_q = qp;
            }
            __syncwarp();
        } else {
            // ------------------------------------------------------------ consumers
            for (DealWalk<T> wk(sc, s_order); wk.more() && ok;) {
                const int nt = wk.template group<T>();
                const int seg0 = rs.seg[wk.ai];
                const int ntok = rs.seg[wk.ai + 1] - seg0;
                const int row0 = wk.tl * 16, ex = rs.act[wk.ai];
                for (int p0 = 0; p0 < ntok && ok; p0 += 8) {
                    const int npass = min(8, ntok - p0);
                    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
                    for (int c = 0; c < KC; ++c, ++q) {
                        bool w = mbar_test_wait(&full[s], ph);
                        for (uint64_t i = 1; !w && i < limit && !*abort_flag; ++i)
                            w = mbar_try_wait(&full[s], ph);
                        w = __all_sync(0xFFFFFFFFu, w);
                        if (!w && lane == 0) {
                            if (!*abort_flag) record_status(a.status, kStTimeout);
                            *abort_flag = 1u;
                        }
                        const uint8_t *st = stages + (size_t)s * L::kStageBytes;
                        uint32_t *fb = bufs + (int)(q & 1) * L::kBufWords;
                        float *invb = reinterpret_cast<float *>(fb + L::kFragWords);
                        if (w) build_b<L, WT, 1, CW>(st, fb, invb, npass, warp, lane);
                        if (consumers_sync_any<CW>(*abort_flag != 0u)) {
                            ok = false;
                            break;
                        }
                        if (tw < nt) tile_chunk<L, WT, 1>(st, fb, invb, acc, tw, sw, lane, t);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&empty[s]);
                        if (++s == S) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (KS > 1) {  // the tile's slices, added in slice order
                        float *mine = red + ((sw * T + tw) * 32 + lane) * 4;
                        if (sw > 0)
#pragma unroll
                            for (int r = 0; r < 4; ++r) mine[r] = acc[0][r];
                        consumers_sync<CW>();
                        if (sw == 0) {
#pragma unroll 1
                            for (int s2 = 1; s2 < KS; ++s2) {
                                const float *o = red + ((s2 * T + tw) * 32 + lane) * 4;
#pragma unroll
                                for (int r = 0; r < 4; ++r) acc[0][r] += o[r];
                            }
                        }
                    }
                    if (sw != 0 || tw >= nt) continue;
                    // Epilogue: rows g, g + 8 of the tile for the pass's slots 2t, 2t + 1.
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = row0 + tw * 16 + g + (r >= 2 ? 8 : 0);
                        const int i = 2 * t + (r & 1);
                        if (row < m && i < npass) {
                            const size_t yo = (size_t)rs.sorted[seg0 + p0 + i] * m + row;
                            const float bj = (a.flags & kBias) ? a.bias[(size_t)ex * m + row] : 0.f;
                            const float rij = (a.flags & kResidual) ? a.R[yo] : 0.f;
                            a.Y[yo] = epilogue_vals(acc[0][r], a.flags, bj, rij, a.alpha);
                        }
                    }
                }
                wk.advance(nt);
            }
        }
    }
    if (warp == CW && lane == 0) {
        // Drain copies that no consumer waited for (only after an abort).
        const long long qp = *s_q;
        for (long long d = (qp > S ? qp - S : 0); d < qp; ++d)
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

template <int WT, int T, int KS, int NH>
cudaError_t launch_t(const StreamArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    using L = BL<WT, T, KS, NH>;
    static std::atomic<unsigned long long> smem_set{0};
    auto encode = encode_fn();
    if (!encode) return cudaErrorInvalidValue;
    // W as a 2-D tensor of 16-bit elements [m][k]; boxes of 64 elements x T*16 rows,
    // 128-byte swizzle (rows past m read as zero).
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)a.k, (cuuint64_t)a.m};
    const cuuint64_t strides[1] = {(cuuint64_t)a.k * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBoxK, (cuuint32_t)(T * 16)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(a.W), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    auto kern = gemv_half_kernel<WT, T, KS, NH>;
    static_assert(L::kBytes <= 227 * 1024, "shared memory budget");
    cudaError_t err = ensure_smem(kern, (int)L::kBytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    const long long groups = ((a.m + 15) / 16 + T - 1) / T;
    const int grid = (int)(groups < dev.sm_count ? groups : dev.sm_count);
    return launch_pdl(kern, dim3(grid), dim3(L::kThreads), L::kBytes, stream, map, a);
}

// A weight bank as a 3-D tensor of 16-bit elements [E][m][k]: boxes of 64 elements x
// `rows` rows of one matrix, 128-byte swizzle.
bool make_bank_map(CUtensorMap &map, const StreamArgs &a, int rows) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)a.k, (cuuint64_t)a.m, (cuuint64_t)a.n_experts};
    const cuuint64_t strides[2] = {(cuuint64_t)a.k * 2, (cuuint64_t)a.m * a.k * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kBoxK, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint8_t *>(a.W), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Routing tables and the producer's stage count after the GEMV kernel's layout.
constexpr size_t kRouteBytes = 8 + kMaxSlots * 8 + (3 * kMaxSlots + 2 + kMaxSlots / 32) * 4;

template <int WT, int T, int KS>
cudaError_t launch_moe_t(const StreamArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    using L = BL<WT, T, KS, 1>;
    static std::atomic<unsigned long long> smem_set{0};
    BankMaps maps;
    if (!make_bank_map(maps.full, a, T * 16) || !make_bank_map(maps.b2, a, (T > 2 ? 2 : T) * 16) ||
        !make_bank_map(maps.b1, a, 16))
        return cudaErrorInvalidValue;
    auto kern = moe_half_kernel<WT, T, KS>;
    constexpr size_t bytes = L::kBytes + kRouteBytes;
    static_assert(bytes <= 227 * 1024, "shared memory budget");
    cudaError_t err = ensure_smem(kern, (int)bytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(dev.sm_count), dim3(L::kThreads), bytes, stream, maps, a);
}

}  // namespace

namespace {
template <int WT>
cudaError_t launch_wt(const StreamArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    // T tiles per group: about one group per SM (the groups of a CTA share nothing);
    // k slices so that 8-16 consumer warps hide the latencies of each warp's MMAs.
    const long long tiles = (a.m + 15) / 16;
    const long long per = (tiles + dev.sm_count - 1) / dev.sm_count;
    if (a.n > 8) {
        if (per <= 2) return launch_t<WT, 2, 4, 2>(a, dev, stream);
        return launch_t<WT, 4, 2, 2>(a, dev, stream);
    }
    if (per <= 2) return launch_t<WT, 2, 4, 1>(a, dev, stream);
    if (per <= 4) return launch_t<WT, 4, 4, 1>(a, dev, stream);
    if (per <= 6) return launch_t<WT, 6, 2, 1>(a, dev, stream);
    return launch_t<WT, 8, 2, 1>(a, dev, stream);
}
}  // namespace

bool half_gemv_supported(int wtype, int n, int k) {
    return (wtype == kBF16 || wtype == kF16) && n >= 1 && n <= 16 && k % kChunk == 0 &&
           encode_fn() != nullptr;
}

cudaError_t launch_half_gemv(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                             cudaStream_t stream) {
    return wtype == kBF16 ? launch_wt<kBF16>(a, dev, stream) : launch_wt<kF16>(a, dev, stream);
}

bool half_moe_supported(int wtype, int k) {
    return (wtype == kBF16 || wtype == kF16) && k % kChunk == 0 && encode_fn() != nullptr;
}

cudaError_t launch_half_moe(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                            cudaStream_t stream) {
    // Four 16-row tiles per group and two k slices: eight consumer warps, 288 threads
    // (routing wants one per slot of a window).
    return wtype == kBF16 ? launch_moe_t<kBF16, 4, 2>(a, dev, stream)
                          : launch_moe_t<kF16, 4, 2>(a, dev, stream);
}

}  // namespace wq
