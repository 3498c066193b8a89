// gemm_tc.cu -- large-n GEMM on the 5th-generation tensor cores (tcgen05).
//
// Computes cortiq-engine 0.8.49 ae_gemm's Y[n.m] (=|+=) X[n.k] . W[m.k]^T (+bias)
// (gelu) with W bf16 pairs (exact) and X rounded to bf16 (round to nearest
// even), products and sums in the tensor core's f32 accumulator, and the ae_put
// epilogue (+bias, erf-GELU, +old Y) fused into the TMEM read-back.  The page's
// kernel runs f32 FMAs on 128x128 register tiles; this one is a tcgen05 kernel:
//
//   warp 0      TMA producer: W tiles [BN rows][64 k] (bf16, 128-byte swizzle)
//   warp 1      TMEM owner + MMA issuer (one thread): tcgen05.mma kind::f16,
//               M = 128 (X rows) x N = BN (W rows) x K = 16, f32 accumulator in TMEM
//   warps 2..17 converters: load X f32 rows (coalesced, four k-blocks in flight
//               in registers: the register file holds the X data in flight that
//               shared memory, full of operand stages, cannot), round to bf16 and
//               store them in the 128-byte-swizzled K-major layout the tensor core
//               reads (no extra HBM pass for X); afterwards the same warps are the
//               epilogue: tcgen05.ld of the accumulator, bias and GELU in
//               registers, then each 32x32 block goes through shared memory so
//               that residual loads and Y stores are whole 128-byte rows.
//
// A/B stages are a 4-deep ring guarded by mbarriers; every wait is bounded.  A
// wait that runs out sets the CTA's abort flag and WQ_ERR_DEVICE_TIMEOUT; every
// role then stops, the producer drains its TMA copies, the MMA thread waits for
// its MMAs, all threads meet, TMEM is freed and the CTA returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

using namespace tc;
constexpr int kStages = 4;
constexpr int kConvWarps = 16;  // X converters (fused path); they are also the epilogue
constexpr int kEpiWarps = 8;    // epilogue warps of the path with X already in bf16

// Warps after the producer and MMA warps: converters+epilogue, or epilogue only.
template <bool ATMA>
struct Roles {
    static constexpr int kWork = ATMA ? kEpiWarps : kConvWarps;
    static constexpr int kThreads = (2 + kWork) * 32;
};
constexpr int kABytes = BM * BK * 2;  // 16 KB

template <int BN>
struct Smem {
    static constexpr int kBBytes = BN * BK * 2;
    static constexpr size_t kA = 0;
    static constexpr size_t kB = kA + (size_t)kStages * kABytes;
    static constexpr size_t kBars = kB + (size_t)kStages * kBBytes;
    // a_full[S], b_full[S], empty[S], acc_full, drain
    static constexpr size_t kMisc = kBars + (3 * kStages + 2) * sizeof(uint64_t);
    static constexpr size_t kBytes = kMisc + 16 + 1024;  // + tmem slot, abort flag; + alignment
};

// ATMA: X arrives already rounded to bf16 (a workspace written by x_to_bf16) and is
// loaded by TMA like W; otherwise the converter warps round it from f32.
template <int BN, bool ATMA>
__global__ void __launch_bounds__(Roles<ATMA>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const GemmArgs a) {
    pdl_enter();
    using L = Smem<BN>;
    constexpr int NW = Roles<ATMA>::kWork;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled operand tiles.
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem + L::kA;
    uint8_t *sB = smem + L::kB;
    uint64_t *a_full = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *b_full = a_full + kStages;
    uint64_t *empty = b_full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *drain = acc_full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = blockIdx.y * BM, j0 = blockIdx.x * BN;
    const int KB = (a.k + BK - 1) / BK;
    const uint64_t limit = a.wait_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&a_full[s], kConvWarps);
            mbar_init(&b_full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {  // TMEM: BN f32 columns x 128 lanes
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(tmem_slot)),
            "r"(BN)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int kb = 0;
            for (; kb < KB; ++kb) {
                const int s = kb % kStages;
                if (kb >= kStages &&
                    !wait_or_abort(&empty[s], ((kb / kStages) - 1) & 1, abort_flag, limit,
                                   a.status))
                    break;
                if (ATMA) {
                    mbar_arrive_expect_tx(&b_full[s], (uint32_t)(kABytes + L::kBBytes));
                    tma_load_2d(sA + (size_t)s * kABytes, &xmap, kb * BK, i0, &b_full[s]);
                } else {
                    mbar_arrive_expect_tx(&b_full[s], (uint32_t)L::kBBytes);
                }
                tma_load_2d(sB + (size_t)s * L::kBBytes, &wmap, kb * BK, j0, &b_full[s]);
            }
            // Drain: the last kStages loads issued may still be in flight.
            for (int d = (kb > kStages ? kb - kStages : 0); d < kb; ++d)
                mbar_wait(&b_full[d % kStages], (d / kStages) & 1, kDrainPolls);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(BM, BN);
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++kb) {
                const int s = kb % kStages;
                const uint32_t ph = (kb / kStages) & 1;
                ok = (ATMA || wait_or_abort(&a_full[s], ph, abort_flag, limit, a.status)) &&
                     wait_or_abort(&b_full[s], ph, abort_flag, limit, a.status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_addr(sA + (size_t)s * kABytes);
                const uint32_t b0 = smem_addr(sB + (size_t)s * L::kBBytes);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    tc_mma(tmem, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32),
                           idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&empty[s]);
            }
            if (ok) {
                tc_commit(acc_full);
            } else {
                tc_commit(drain);  // completes when every MMA issued so far is done
                mbar_wait(drain, 0, kDrainPolls);
            }
        }
    } else {
        // ----------------------------------------------------- X converters
        const int cw = warp - 2;          // 0..15: rows 8cw .. 8cw+7 of the tile
        const int half = lane >> 4;       // which of the two rows of one load step
        const int c4 = lane & 15;         // float4 index within the row's 64 k
        bool ok = true;
        const int KBc = ATMA ? 0 : KB;    // k-blocks this warp converts
        float4 b0[4], b1[4], b2[4], b3[4];  // k-blocks kb .. kb+3 (three loads in flight)
        auto load_block = [&](int kb, float4(&dst)[4]) {
            const int col = kb * BK + 4 * c4;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int row = i0 + cw * 8 + 2 * it + half;
                if (row < a.n && col < a.k)
                    dst[it] = __ldg(reinterpret_cast<const float4 *>(a.X + (size_t)row * a.k + col));
                else
                    dst[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        // Convert block kb from `cur` into stage kb % kStages, after starting the
        // load of block kb + 3 into `pre`.
        auto step = [&](int kb, const float4(&cur)[4], float4(&pre)[4]) -> bool {
            const int s = kb % kStages;
            if (kb + 3 < KB) load_block(kb + 3, pre);
            if (kb >= kStages &&
                !wait_or_abort(&empty[s], ((kb / kStages) - 1) & 1, abort_flag, limit, a.status))
                return false;
            uint8_t *tile = sA + (size_t)s * kABytes;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int r = cw * 8 + 2 * it + half;  // row within the tile
                const uint32_t lo = pack_bf16x2(cur[it].x, cur[it].y);
                const uint32_t hi = pack_bf16x2(cur[it].z, cur[it].w);
                const int chunk = c4 >> 1;                         // 16-byte chunk of the row
                const uint32_t off = r * 128 + ((chunk ^ (r & 7)) << 4) + ((c4 & 1) << 3);
                *reinterpret_cast<uint2 *>(tile + off) = make_uint2(lo, hi);
            }
            fence_proxy_async_smem();  // generic-proxy stores -> tensor core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[s]);
            return true;
        };
        if (KBc > 0) load_block(0, b0);
        if (KBc > 1) load_block(1, b1);
        if (KBc > 2) load_block(2, b2);
        for (int kb = 0; kb < KBc && ok; kb += 4) {
            ok = step(kb, b0, b3);
            if (ok && kb + 1 < KBc) ok = step(kb + 1, b1, b0);
            if (ok && kb + 2 < KBc) ok = step(kb + 2, b2, b1);
            if (ok && kb + 3 < KBc) ok = step(kb + 3, b3, b2);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && wait_or_abort(acc_full, 0, abort_flag, limit, a.status)) {
            tc_fence_after();
            const int q = warp & 3;                  // TMEM lane quarter of this warp
            constexpr int CW = BN / (NW / 4);        // columns per warp
            const int cg = cw >> 2;                  // which group of CW columns
            constexpr int kStage = 36;               // staging row stride (floats)
            // The operand stages are idle now: every MMA has completed.
            float *stg = reinterpret_cast<float *>(smem) + cw * 32 * kStage;
            // 16-byte stores where every row of Y (and of the residual, and the second
            // band at column m) starts 16-byte aligned.
            const bool vec = ((a.ldy | a.m) & 3) == 0 && ((uintptr_t)a.Y & 15u) == 0 &&
                             (!(a.flags & kResidual) || ((uintptr_t)a.R & 15u) == 0);
            for (int c0 = cg * CW; c0 < (cg + 1) * CW; c0 += 32) {
                const int jb = j0 + c0;
                // Band 0: epi(sums) into columns < m; band 1 (blocks left of dual): the
                // same sums + bias2, no activation, alpha or residual, at column m + j.
                for (int band = 0; band < (jb < a.dual ? 2 : 1); ++band) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
                    if (band == 1) {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            v[c] += (jb + c < a.dual) ? __ldg(a.bias2 + jb + c) : 0.f;
                    } else if (a.flags & (kBias | kActs)) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            float t = v[c];
                            if (a.flags & kBias) t += (jb + c < a.m) ? __ldg(a.bias + jb + c) : 0.f;
                            v[c] = a.alpha * activate(t, a.flags);
                        }
                    }
                    // Row `lane` of the 32x32 block into shared memory...
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(&stg[lane * kStage + c]) =
                            make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
                    __syncwarp();
                    // ...then four rows of 128 bytes per warp instruction to global.
                    const int lim = band ? a.dual : a.m;
                    const bool res = !band && (a.flags & kResidual);
                    float *yb = a.Y + (band ? a.m : 0);
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = it * 4 + (lane >> 3), cc = (lane & 7) * 4;
                        const int row = i0 + q * 32 + rr, col = jb + cc;
                        if (row >= a.n || col >= lim) continue;
                        float4 o = *reinterpret_cast<const float4 *>(&stg[rr * kStage + cc]);
                        const size_t off = (size_t)row * a.ldy + col;
                        if (vec && col + 4 <= lim) {
                            if (res) {
                                const float4 r4 = *reinterpret_cast<const float4 *>(a.R + off);
                                o.x += r4.x; o.y += r4.y; o.z += r4.z; o.w += r4.w;
                            }
                            *reinterpret_cast<float4 *>(yb + off) = o;
                        } else {
                            const float ov[4] = {o.x, o.y, o.z, o.w};
                            for (int e = 0; e < 4 && col + e < lim; ++e)
                                yb[off + e] = ov[e] + (res ? a.R[off + e] : 0.f);
                        }
                    }
                    __syncwarp();
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN)
                     : "memory");
    }
}

// ----------------------------------------------------------- host side --

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

bool encode_bf16_map(CUtensorMap &map, const void *base, int cols, int rows, int box_rows) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool ATMA>
cudaError_t launch_bn(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                      cudaStream_t stream) {
    static std::atomic<unsigned long long> smem_set{0};
    CUtensorMap wmap, xmap;
    if (!encode_bf16_map(wmap, a.W, a.k, a.m, BN)) return cudaErrorInvalidValue;
    if (ATMA) {
        if (!encode_bf16_map(xmap, xb, a.k, a.n, BM)) return cudaErrorInvalidValue;
    } else {
        xmap = wmap;  // unused
    }
    auto kern = gemm_tc_kernel<BN, ATMA>;
    cudaError_t err = ensure_smem(kern, (int)Smem<BN>::kBytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    dim3 grid((a.m + BN - 1) / BN, (a.n + BM - 1) / BM);
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    return launch_pdl(kern, grid, dim3(Roles<ATMA>::kThreads), Smem<BN>::kBytes, stream, wmap, xmap, a);
}

// X f32 -> bf16, round to nearest even (the rounding the fused path applies).
// The copy is bound by bytes in flight: each thread first requests `upt` <= kXU
// 16-byte pieces with cp.async into shared memory (no registers held while they
// are in flight, so four CTAs of up to 48 KB keep up to ~190 KB per SM
// outstanding), then converts its own pieces and stores them.  upt is the least
// that covers X with four CTAs per SM, so that a small X still spreads over
// every SM.
constexpr int kXU = 12;
constexpr int kXThreads = 256;
constexpr int kXSmem = kXThreads * kXU * 16;
__global__ void __launch_bounds__(kXThreads) x_to_bf16_kernel(const float4 *__restrict__ x,
                                                              uint2 *__restrict__ xb, size_t n4,
                                                              int upt) {
    pdl_enter();
    extern __shared__ float4 xs[];
    const size_t per_cta = (size_t)kXThreads * upt;
    for (size_t base = (size_t)blockIdx.x * per_cta; base < n4; base += (size_t)gridDim.x * per_cta) {
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            const size_t i = base + (size_t)u * kXThreads + threadIdx.x;
            if (u < upt && i < n4)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                 smem_addr(&xs[u * kXThreads + threadIdx.x])),
                             "l"(x + i)
                             : "memory");
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
#pragma unroll
        for (int u = 0; u < kXU; ++u) {
            const size_t i = base + (size_t)u * kXThreads + threadIdx.x;
            if (u < upt && i < n4) {
                const float4 v = xs[u * kXThreads + threadIdx.x];
                xb[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
            }
        }
    }
}

template <bool ATMA>
cudaError_t launch_tc(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                      cudaStream_t stream) {
    // Pick the tile width with the smaller (waves x tile time); ties go to 256,
    // whose X tile is shared by twice the columns.
    const long long rows = (a.n + BM - 1) / BM;
    const long long w256 = (rows * ((a.m + 255) / 256) + dev.sm_count - 1) / dev.sm_count;
    const long long w128 = (rows * ((a.m + 127) / 128) + dev.sm_count - 1) / dev.sm_count;
    if (w256 * 2 <= w128) return launch_bn<256, ATMA>(a, xb, dev, stream);
    return launch_bn<128, ATMA>(a, xb, dev, stream);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs &a, const DeviceInfo &dev, cudaStream_t stream) {
    return launch_tc<false>(a, nullptr, dev, stream);
}

size_t gemm_tc_workspace_bytes(int n, int k) { return ((size_t)n * k * 2 + 255) & ~(size_t)255; }

// Quantised W -> bf16 [m][k]: each dequantised weight d*q (Q8_0) or d*(q-8) (Q4_0),
// exact in f32, rounded to the nearest bf16 (ties to even).  One thread per
// 32-weight block; a block starts 2-byte aligned, so it is read as 16-bit words.
template <int WT>
__global__ void w_to_bf16_kernel(const uint8_t *__restrict__ W, int m, int k,
                                 uint4 *__restrict__ wb) {
    pdl_enter();
    const int nb = k / 32;
    const long long blocks = (long long)m * nb;
    const size_t rb = row_bytes(WT, k);
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < blocks;
         u += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(u / nb), b = (int)(u % nb);
        const uint16_t *bp = reinterpret_cast<const uint16_t *>(
            W + (size_t)j * rb + (size_t)b * (WT == kQ8_0 ? 34 : 18));
        const float d = half_bits_to_f32(bp[0]);
        float w[32];
        if (WT == kQ8_0) {
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const uint32_t v = bp[1 + h];
                w[2 * h] = d * (float)(int8_t)(v & 0xFFu);
                w[2 * h + 1] = d * (float)(int8_t)(v >> 8);
            }
        } else {
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const uint32_t v = bp[1 + h];  // bytes 2h, 2h+1 of the 16 code bytes
                w[2 * h] = d * (float)((int)(v & 0xFu) - 8);
                w[2 * h + 1] = d * (float)((int)((v >> 8) & 0xFu) - 8);
                w[16 + 2 * h] = d * (float)((int)((v >> 4) & 0xFu) - 8);
                w[16 + 2 * h + 1] = d * (float)((int)(v >> 12) - 8);
            }
        }
        uint4 *o = wb + ((size_t)j * k + (size_t)b * 32) / 8;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            o[c] = make_uint4(pack_bf16x2(w[8 * c], w[8 * c + 1]), pack_bf16x2(w[8 * c + 2], w[8 * c + 3]),
                              pack_bf16x2(w[8 * c + 4], w[8 * c + 5]), pack_bf16x2(w[8 * c + 6], w[8 * c + 7]));
    }
}

// Quantised W -> bf16 [m][k] when a row is a whole number of 16-byte words
// (k % 256 == 0): a CTA takes a row at a time, loads its blocks with coalesced
// 16-byte loads into shared memory, and each thread then decodes 8-weight pieces
// c = threadIdx.x + 256 u (block c / 4, quarter c % 4) and stores them, so that a
// warp's store covers 512 contiguous bytes.  Same values as w_to_bf16_kernel.
template <int WT>
__global__ void __launch_bounds__(256) w_rows_to_bf16_kernel(const uint8_t *__restrict__ W,
                                                             int m, int k,
                                                             uint4 *__restrict__ wb) {
    pdl_enter();
    extern __shared__ uint4 rowbuf[];
    const size_t rb = row_bytes(WT, k);
    const int words = (int)(rb / 16);
    const int pieces = k / 8;
    const uint8_t *sb = reinterpret_cast<const uint8_t *>(rowbuf);
    for (int j = blockIdx.x; j < m; j += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(W + (size_t)j * rb);
        for (int w = threadIdx.x; w < words; w += blockDim.x) rowbuf[w] = __ldg(src + w);
        __syncthreads();
        for (int c = threadIdx.x; c < pieces; c += blockDim.x) {
            const int b = c >> 2, qt = c & 3;
            const uint8_t *bp = sb + (size_t)b * (WT == kQ8_0 ? 34 : 18);
            const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
            float w[8];
            if (WT == kQ8_0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) w[e] = d * (float)(int8_t)bp[2 + 8 * qt + e];
            } else {  // quarter qt: low (qt < 2) or high nibbles of code bytes 8 (qt & 1) ..
                const uint8_t *cb = bp + 2 + 8 * (qt & 1);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t byte = cb[e];
                    const int code = qt < 2 ? (int)(byte & 15u) : (int)(byte >> 4);
                    w[e] = d * (float)(code - 8);
                }
            }
            wb[(size_t)j * pieces + c] =
                make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                           pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
        }
        __syncthreads();  // the row buffer is refilled next
    }
}

// F16 / F32 W -> bf16 [m][k], each element rounded to the nearest bf16 (ties to
// even).  One thread per 8 weights (k % 8 == 0, rows 16-byte aligned).
template <int WT>
__global__ void wf_to_bf16_kernel(const uint8_t *__restrict__ W, int m, int k,
                                  uint4 *__restrict__ wb) {
    pdl_enter();
    const long long units = (long long)m * (k / 8);
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        float w[8];
        if (WT == kF16) {
            const uint4 v = reinterpret_cast<const uint4 *>(W)[u];  // 8 halves
            const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                w[2 * e] = half_bits_to_f32(h[e]);
                w[2 * e + 1] = half_bits_to_f32(h[e] >> 16);
            }
        } else {
            const float4 a = reinterpret_cast<const float4 *>(W)[2 * u];
            const float4 b = reinterpret_cast<const float4 *>(W)[2 * u + 1];
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        }
        wb[u] = make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                           pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
    }
}

size_t gemm_tc_w_workspace_bytes(int m, int k) {
    return ((size_t)m * k * 2 + 255) & ~(size_t)255;
}

cudaError_t launch_gemm_tc_ws(const GemmArgs &a, int wtype, void *workspace,
                              const DeviceInfo &dev, cudaStream_t stream, bool x_ready) {
    GemmArgs g = a;
    g.w_early = wtype == kBF16;  // else W is the bf16 copy the next kernel writes
    if (wtype != kBF16) {
        // The weights first: bf16 after X in the workspace, then the bf16 GEMM.
        uint8_t *wb = static_cast<uint8_t *>(workspace) + gemm_tc_workspace_bytes(a.n, a.k);
        const bool plain = wtype == kF16 || wtype == kF32;
        const long long units = (long long)a.m * (a.k / (plain ? 8 : 32));
        long long grid = (units + 255) / 256;
        if (grid > (long long)dev.sm_count * 8) grid = (long long)dev.sm_count * 8;
        uint4 *wo = reinterpret_cast<uint4 *>(wb);
        cudaError_t err;
        const bool rows16 = !plain && a.k % 256 == 0 && ((uintptr_t)a.W & 15u) == 0;
        if (rows16) {  // whole rows through shared memory: coalesced loads and stores
            // The row buffer's size follows k: above the default 48 KB the limit is
            // raised for this call (never lowered, so other sizes stay launchable).
            const int rbytes = (int)row_bytes(wtype, a.k);
            long long g = a.m < dev.sm_count * 8 ? a.m : (long long)dev.sm_count * 8;
            auto kern = wtype == kQ8_0 ? w_rows_to_bf16_kernel<kQ8_0> : w_rows_to_bf16_kernel<kQ4_0>;
            err = rbytes > 48 * 1024
                      ? cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             rbytes)
                      : cudaSuccess;
            if (err == cudaSuccess)
                err = launch_pdl(kern, dim3((unsigned)g), dim3(256), rbytes, stream, a.W, a.m, a.k,
                                 wo);
            if (err != cudaSuccess) return err;
        } else switch (wtype) {
        case kQ8_0:
            err = launch_pdl(w_to_bf16_kernel<kQ8_0>, dim3((unsigned)grid), dim3(256), 0, stream,
                             a.W, a.m, a.k, wo);
            break;
        case kF16:
            err = launch_pdl(wf_to_bf16_kernel<kF16>, dim3((unsigned)grid), dim3(256), 0, stream,
                             a.W, a.m, a.k, wo);
            break;
        case kF32:
            err = launch_pdl(wf_to_bf16_kernel<kF32>, dim3((unsigned)grid), dim3(256), 0, stream,
                             a.W, a.m, a.k, wo);
            break;
        default:
            err = launch_pdl(w_to_bf16_kernel<kQ4_0>, dim3((unsigned)grid), dim3(256), 0, stream,
                             a.W, a.m, a.k, wo);
        }
        if (err != cudaSuccess) return err;
        g.W = wb;
    }
    if (!x_ready) {  // else the workspace already holds bf16 X (e.g. a fused LayerNorm)
        const size_t n4 = (size_t)a.n * a.k / 4;
        const long long cap = (long long)dev.sm_count * 4;  // resident at once
        const size_t round = (size_t)cap * kXThreads;          // float4s per piece per thread
        const int upt = (int)std::min<size_t>(kXU, std::max<size_t>(1, (n4 + round - 1) / round));
        const size_t per_cta = (size_t)kXThreads * upt;
        long long blocks = (long long)((n4 + per_cta - 1) / per_cta);
        if (blocks > cap) blocks = cap;
        static std::atomic<unsigned long long> smem_set{0};
        cudaError_t err = ensure_smem(x_to_bf16_kernel, kXSmem, dev, smem_set);
        if (err != cudaSuccess) return err;
        err = launch_pdl(x_to_bf16_kernel, dim3((unsigned)blocks), dim3(kXThreads), kXSmem, stream,
                         reinterpret_cast<const float4 *>(a.X),
                         reinterpret_cast<uint2 *>(workspace), n4, upt);
        if (err != cudaSuccess) return err;
    }
    if (gemm_tcp_supported(g)) return launch_gemm_tcp(g, workspace, dev, stream);
    return launch_tc<true>(g, workspace, dev, stream);
}

}  // namespace wq
