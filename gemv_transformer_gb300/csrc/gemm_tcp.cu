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

template <int BN, int KS>
struct PLayout {
    static constexpr int kABytes = KS * kAtomA;            // A of a stage
    static constexpr int kBBytes = KS * BN * BK * 2;       // B of a stage
    static constexpr int kFit = (216 * 1024 - kEpi * kStgBytes) / (kABytes + kBBytes);
    static constexpr int kStages = kFit > 6 ? 6 : kFit;
    static_assert(kStages >= 2, "at least two stages");
    static constexpr size_t kA = 0;
    static constexpr size_t kB = kA + (size_t)kStages * kABytes;
    static constexpr size_t kStg = kB + (size_t)kStages * kBBytes;
    static constexpr size_t kBars = kStg + (size_t)kEpi * kStgBytes;
    // full[S], empty[S], tfull[2], tempty[2], rbar[kEpi], drain
    static constexpr int kNumBars = 2 * kStages + 4 + kEpi + 1;
    static constexpr size_t kMisc = kBars + kNumBars * sizeof(uint64_t);
    static constexpr size_t kBytes = kMisc + 16 + 1024;
};

template <int BN, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcp_kernel(const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap xmap,
                    const __grid_constant__ CUtensorMap ymap,
                    const __grid_constant__ CUtensorMap rmap, const GemmArgs a) {
    pdl_enter();
    using L = PLayout<BN, KS>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t *sA = smem + L::kA;
    uint8_t *sB = smem + L::kB;
    uint8_t *sStg = smem + L::kStg;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *rbar = tempty + 2;
    uint64_t *drain = rbar + kEpi;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RB = (a.n + BM - 1) / BM, CB = (a.m + BN - 1) / BN;
    const int tiles = RB * CB;
    const int KB = (a.k + KS * BK - 1) / (KS * BK);  // stages per tile
    const uint64_t limit = a.wait_limit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 2);  // one expect_tx arrival per producer
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpi);
        }
        for (int w = 0; w < kEpi; ++w) mbar_init(&rbar[w], 1);
        mbar_init(drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 2) {  // TMEM: two accumulators of BN f32 columns x 128 lanes
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(tmem_slot)),
            "r"(2 * BN)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 2) {
        // --------------------------------------------------------- producers
        // Warp 0 loads A (X rows), warp 1 loads B (W rows); KS atoms per stage.
        if (lane == 0) {
            const bool isA = warp == 0;
            const CUtensorMap *map = isA ? &xmap : &wmap;
            const int atom = isA ? kAtomA : BN * BK * 2;
            uint8_t *base = isA ? sA : sB;
            const int sbytes = isA ? L::kABytes : L::kBBytes;
            long long q = 0;  // stages issued
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int y = isA ? (t % RB) * BM : (t / RB) * BN;
                for (int kb = 0; kb < KB; ++kb, ++q) {
                    const int s = (int)(q % S);
                    if (q >= S && !wait_or_abort(&empty[s], (uint32_t)(((q / S) - 1) & 1),
                                                 abort_flag, limit, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], (uint32_t)sbytes);
                    uint8_t *dst = base + (size_t)s * sbytes;
#pragma unroll
                    for (int u = 0; u < KS; ++u)
                        tma_load_2d(dst + u * atom, map, (kb * KS + u) * BK, y, &full[s]);
                }
            }
            for (long long d = (q > S ? q - S : 0); d < q; ++d)
                mbar_wait(&full[d % S], (uint32_t)((d / S) & 1), kDrainPolls);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(BM, BN);
            long long q = 0;
            int it = 0;  // local tile index
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++it) {
                const int b = it & 1;
                if (it >= 2 && !wait_or_abort(&tempty[b], (uint32_t)(((it >> 1) - 1) & 1),
                                              abort_flag, limit, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kb = 0; kb < KB; ++kb, ++q) {
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
                        for (int kk = 0; kk < BK / 16; ++kk)
                            tc_mma(d, smem_desc_sw128(a0 + u * kAtomA + kk * 32),
                                   smem_desc_sw128(b0 + u * (BN * BK * 2) + kk * 32), idesc,
                                   (kb > 0 || u > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[s]);
                }
                if (ok) tc_commit(&tfull[b]);
            }
            if (!ok) {
                tc_commit(drain);  // completes when every MMA issued so far is done
                mbar_wait(drain, 0, kDrainPolls);
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - kRoles;              // 0..15
        const int q = warp & 3;                    // TMEM lane quarter of this warp
        constexpr int CW = BN / (kEpi / 4);        // columns per warp per tile
        const int cg = ew >> 2;                    // which column group
        uint8_t *stg = sStg + ew * kStgBytes;
        uint32_t rphase = 0;
        bool ok = true;
        bool stored = false;
        int it = 0;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++it) {
            const int b = it & 1;
            const int i0 = (t % RB) * BM, j0 = (t / RB) * BN;
            const int r0 = i0 + q * 32;            // first row of this warp's blocks
            if (!wait_or_abort(&tfull[b], (uint32_t)((it >> 1) & 1), abort_flag, limit,
                               a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            for (int c0 = cg * CW; c0 < (cg + 1) * CW && ok; c0 += 32) {
                const int jb = j0 + c0;
                const float bl = ((a.flags & kBias) && jb + lane < a.m) ? __ldg(a.bias + jb + lane)
                                                                         : 0.f;
                // The staging block is free once the previous store has read it.
                if (stored) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
                }
                if (a.flags & kResidual) {  // old Y block into the staging buffer
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&rbar[ew], (uint32_t)kStgBytes);
                        tma_load_2d(stg, &rmap, jb, r0, &rbar[ew]);
                    }
                }
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c0), v);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float bc = __shfl_sync(0xFFFFFFFFu, bl, c);
                    float x = v[c];
                    if (a.flags & kBias) x += bc;
                    v[c] = activate(x, a.flags);
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
            }
            // This accumulator may be refilled.
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&tempty[b]);
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }
    __syncwarp();  // every role's lanes meet before the block-wide barrier
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(2 * BN)
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
               int rows, int box_cols, int box_rows) {
    auto encode = encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(&map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int KS>
cudaError_t launch_bn(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                      cudaStream_t stream) {
    using L = PLayout<BN, KS>;
    static std::atomic<unsigned long long> smem_set{0};
    CUtensorMap wmap, xmap, ymap, rmap;
    if (!encode_2d(wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.W, a.k, a.m, BK, BN) ||
        !encode_2d(xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xb, a.k, a.n, BK, BM) ||
        !encode_2d(ymap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.Y, a.m, a.n, 32, 32))
        return cudaErrorInvalidValue;
    if (a.flags & kResidual) {
        if (!encode_2d(rmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.R, a.m, a.n, 32, 32))
            return cudaErrorInvalidValue;
    } else {
        rmap = ymap;  // unused
    }
    auto kern = gemm_tcp_kernel<BN, KS>;
    static_assert(L::kBytes <= 227 * 1024, "shared memory budget");
    cudaError_t err = ensure_smem(kern, (int)L::kBytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    const long long tiles =
        (long long)((a.n + BM - 1) / BM) * ((a.m + BN - 1) / BN);
    const int grid = (int)(tiles < dev.sm_count ? tiles : dev.sm_count);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), L::kBytes, stream, wmap, xmap, ymap,
                      rmap, a);
}

}  // namespace

bool gemm_tcp_supported(const GemmArgs &a) {
    // TMA stores need 16-byte aligned rows of Y (and of the residual).
    if (a.m % 4 != 0 || ((uintptr_t)a.Y & 15u)) return false;
    if ((a.flags & kResidual) && ((uintptr_t)a.R & 15u)) return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_gemm_tcp(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                            cudaStream_t stream) {
    // Tile width: the one with fewer (tiles per SM, rounded up) x tile time.
    const long long rows = (a.n + BM - 1) / BM;
    const long long w256 = (rows * ((a.m + 255) / 256) + dev.sm_count - 1) / dev.sm_count;
    const long long w128 = (rows * ((a.m + 127) / 128) + dev.sm_count - 1) / dev.sm_count;
    if (w256 * 2 <= w128) return launch_bn<256, 1>(a, xb, dev, stream);
    return launch_bn<128, 2>(a, xb, dev, stream);
}

}  // namespace wq
