// gemv_stream.cu -- weight-streaming GEMV and routed MoE matvec (small n).
//
// What it computes (hanzo-ml 0.11.13 src/wgpu_backend.rs, matvec_q8_0_gpu /
// matvec_q4_0_gpu: y = Wq * x read straight from the GGML blocks; moe_matvec_gpu:
// y[s, r] = sum_k W[ids[s], r, k] x[s, k] in one dispatch; cortiq-engine 0.8.49
// ae_put for the epilogue):
//     Y[i][j] = epi( sum_t X[i][t] * W[j][t] )
//
// Design.  The work is HBM-bound: every weight byte is read exactly once per
// call.  The grid has one CTA per SM; every warp owns a contiguous range of
// "row jobs" (a W row and the X rows it multiplies) and streams that range
// through its own ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier), so each SM keeps ~100 KB of weight
// reads in flight without tying up registers.  A row is cut into pieces of at
// most 2.3 KB; the lanes of the warp decode a piece from shared memory (4 or 8
// weights per lane step, lanes of one block adjacent so the X loads coalesce),
// multiply in f32 and reduce with shuffles in a fixed order (deterministic).
// Scales are applied once per lane step (the block's 4 or 8 products are summed
// first, then multiplied by d), which is exact up to f32 rounding of the sums.
//
// MoE: the routed slots are taken in windows of at most 256; for each window
// each CTA sorts the window's slots by (expert, slot) in shared memory, and the
// row jobs run over (active expert, row), so a selected expert's weights are
// read once per window no matter how many of its slots the window holds.
#include "wq_device.cuh"
#include "wq_internal.h"
#include "tile_sched.cuh"

namespace wq {
namespace {

constexpr int kWarps = 16;
constexpr int kStages = 4;
constexpr int kStageBytes = 2336;  // largest piece (2304 B) + 16 B head + 16 B tail

// Weights per piece: Q8_0 64 blocks (2176 B), Q4_0 128 blocks (2304 B), bf16 2048 B.
template <int WT>
struct Piece;
template <>
struct Piece<kQ8_0> {
    static constexpr int elems = 2048;
};
template <>
struct Piece<kQ4_0> {
    static constexpr int elems = 4096;
};
template <>
struct Piece<kBF16> {
    static constexpr int elems = 1024;
};
template <>
struct Piece<kF16> {
    static constexpr int elems = 1024;
};
template <>
struct Piece<kF32> {
    static constexpr int elems = 512;
};

constexpr size_t kSmemStages = (size_t)kWarps * kStages * kStageBytes;
constexpr size_t kSmemBars = (size_t)kWarps * kStages * sizeof(uint64_t);
constexpr size_t kSmemTot = (size_t)kWarps * kMaxSlots * sizeof(float);
constexpr size_t kSmemMoe = (size_t)kMaxSlots * sizeof(unsigned long long) +  // keys
                            (size_t)(3 * kMaxSlots + 3 + kMaxSlots / 32) * sizeof(int);
constexpr size_t kSmemBytes = kSmemStages + kSmemBars + kSmemTot + kSmemMoe;

template <int WT, bool MOE, int NT>
__global__ void __launch_bounds__(kWarps * 32, 1) stream_kernel(const StreamArgs a) {
    pdl_enter();
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kSmemStages);
    float *tot_all = reinterpret_cast<float *>(smem + kSmemStages + kSmemBars);
    unsigned long long *s_key =
        reinterpret_cast<unsigned long long *>(smem + kSmemStages + kSmemBars + kSmemTot);
    int *s_sorted = reinterpret_cast<int *>(s_key + kMaxSlots);  // slots sorted by expert
    int *s_seg = s_sorted + kMaxSlots;                          // segment starts (+ end)
    int *s_act = s_seg + kMaxSlots + 1;                         // expert of each segment
    int *s_nact = s_act + kMaxSlots;                            // number of segments
    volatile unsigned *s_abort = reinterpret_cast<volatile unsigned *>(s_nact + 1);
    int *s_wcnt = s_nact + 2;                                   // routing: per-warp counts

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k = a.k, m = a.m;
    constexpr int PE = Piece<WT>::elems;
    const size_t rb = row_bytes(WT, k);
    const int P = (k + PE - 1) / PE;  // pieces per row

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWarps * kStages; ++i) mbar_init(&bars[i], 1);
        *s_abort = 0u;
        fence_mbar_init();
    }
    __syncthreads();  // every warp's barriers are initialised
    uint8_t *my_stages = stages + (size_t)warp * kStages * kStageBytes;
    uint64_t *my_bars = bars + warp * kStages;
    float *tot = tot_all + warp * kMaxSlots;
    const uint64_t policy = l2_evict_first();
    // MoE slots are routed in windows of at most kMaxSlots; every warp's ring of
    // stages carries on from one window to the next (pieces streamed so far).
    const int S_all = MOE ? a.n * a.topk : 0;
    const int n_win = MOE ? (S_all + kMaxSlots - 1) / kMaxSlots : 1;
    long long ibase = 0;

    for (int win = 0; win < n_win; ++win) {
        long long n_jobs;
        if (MOE) {
            const int base = win * kMaxSlots;
            route_window(a, base, min(kMaxSlots, S_all - base),
                         RouteSmem{s_key, s_sorted, s_seg, s_act, s_nact, s_wcnt});
            __syncthreads();
            if (*s_abort) break;  // the same in every thread after the barrier
            n_jobs = (long long)(*s_nact) * m;
        } else {
            n_jobs = m;
        }

        const long long wt = (long long)gridDim.x * kWarps;
        const long long gw = (long long)blockIdx.x * kWarps + warp;
        const long long j0 = n_jobs * gw / wt, j1 = n_jobs * (gw + 1) / wt;
        const long long total = (j1 - j0) * P;  // pieces this warp streams in this window

        // Byte range of piece i of this warp's stream: [off, off + len) of W.
        auto piece_range = [&](long long i, size_t &off, uint32_t &len, int &elems) {
            const long long job = j0 + i / P;
            const int p = (int)(i % P);
            size_t row_off;
            if (MOE) {
                const int ai = (int)(job / m), j = (int)(job % m);
                row_off = ((size_t)s_act[ai] * m + j) * rb;
            } else {
                row_off = (size_t)job * rb;
            }
            elems = min(PE, k - p * PE);
            off = row_off + row_bytes(WT, p * PE);
            len = (uint32_t)row_bytes(WT, elems);
        };
        auto issue = [&](long long i) {
            size_t off;
            uint32_t len;
            int elems;
            piece_range(i, off, len, elems);
            const size_t a0 = off & ~(size_t)15;
            const uint32_t bytes = (uint32_t)(((off + len + 15) & ~(size_t)15) - a0);
            const int s = (int)((ibase + i) % kStages);
            mbar_arrive_expect_tx(&my_bars[s], bytes);
            bulk_g2s(my_stages + (size_t)s * kStageBytes, a.W + a0, bytes, &my_bars[s], policy);
        };

        if (lane == 0) {
            fence_proxy_async_smem();  // the previous window's reads of the stages come first
            for (long long i = 0; i < total && i < kStages; ++i) issue(i);
        }

        bool failed = false;
        for (long long i = 0; i < total; ++i) {
            const long long ig = ibase + i;
            const int s = (int)(ig % kStages);
            bool ok = mbar_wait(&my_bars[s], (uint32_t)((ig / kStages) & 1), a.wait_limit);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                if (lane == 0) {
                    record_status(a.status, kStTimeout);
                    *s_abort = 1u;
                }
                // Drain this warp's copies in flight before leaving.
                const long long issued = min(total, i + kStages);
                for (long long ii = i; ii < issued; ++ii)
                    mbar_wait(&my_bars[(ibase + ii) % kStages],
                              (uint32_t)(((ibase + ii) / kStages) & 1), kDrainPolls);
                failed = true;
                break;
            }

            size_t off;
            uint32_t len;
            int elems;
            piece_range(i, off, len, elems);
            const uint8_t *pc = my_stages + (size_t)s * kStageBytes + (off & 15);
            const long long job = j0 + i / P;
            const int p = (int)(i % P);
            int j, e = 0, seg0 = 0, ns;
            if (MOE) {
                const int ai = (int)(job / m);
                j = (int)(job % m);
                e = s_act[ai];
                seg0 = s_seg[ai];
                ns = s_seg[ai + 1] - seg0;
            } else {
                j = (int)job;
                ns = a.n;
            }
            const int xoff = p * PE;
            for (int g0 = 0; g0 < ns; g0 += NT) {
                const int ng = min(NT, ns - g0);
                const float *xr[NT];
    #pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const int r = g0 + (t < ng ? t : 0);
                    const int xrow = MOE ? s_sorted[seg0 + r] / a.topk : r;
                    xr[t] = a.X + (size_t)xrow * k + xoff;
                }
                float acc[NT];
    #pragma unroll
                for (int t = 0; t < NT; ++t) acc[t] = 0.f;

                if (WT == kQ8_0) {
                    const int units = elems >> 2;  // 4 weights per lane step
                    for (int u = lane; u < units; u += 32) {
                        const int blk = u >> 3, within = (u & 7) << 2;
                        const uint8_t *bp = pc + blk * 34;
                        const float d = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(bp));
                        float w0, w1, w2, w3;
                        s8x4_to_f32(ld_u32_a2(bp + 2 + within), w0, w1, w2, w3);
                        const int xe = blk * 32 + within;
    #pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (t < ng) {
                                const float4 x = __ldg(reinterpret_cast<const float4 *>(xr[t] + xe));
                                float part = w0 * x.x;
                                part = fmaf(w1, x.y, part);
                                part = fmaf(w2, x.z, part);
                                part = fmaf(w3, x.w, part);
                                acc[t] = fmaf(d, part, acc[t]);
                            }
                        }
                    }
                } else if (WT == kQ4_0) {
                    const int units = elems >> 3;  // 8 weights (4 bytes) per lane step
                    for (int u = lane; u < units; u += 32) {
                        const int blk = u >> 2, jb = (u & 3) << 2;
                        const uint8_t *bp = pc + blk * 18;
                        const float d = half_bits_to_f32(*reinterpret_cast<const uint16_t *>(bp));
                        const uint32_t v = ld_u32_a2(bp + 2 + jb);
                        float l0, l1, l2, l3, h0, h1, h2, h3;
                        u4x4_to_f32_m8(v & 0x0F0F0F0Fu, l0, l1, l2, l3);
                        u4x4_to_f32_m8((v >> 4) & 0x0F0F0F0Fu, h0, h1, h2, h3);
                        const int xe = blk * 32 + jb;
    #pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (t < ng) {
                                const float4 xl = __ldg(reinterpret_cast<const float4 *>(xr[t] + xe));
                                const float4 xh =
                                    __ldg(reinterpret_cast<const float4 *>(xr[t] + xe + 16));
                                float part = l0 * xl.x;
                                part = fmaf(l1, xl.y, part);
                                part = fmaf(l2, xl.z, part);
                                part = fmaf(l3, xl.w, part);
                                part = fmaf(h0, xh.x, part);
                                part = fmaf(h1, xh.y, part);
                                part = fmaf(h2, xh.z, part);
                                part = fmaf(h3, xh.w, part);
                                acc[t] = fmaf(d, part, acc[t]);
                            }
                        }
                    }
                } else {  // bf16 pairs, f16 or f32 elements
                    const int units = elems >> 2;  // 4 weights per lane step
                    for (int u = lane; u < units; u += 32) {
                        float w0, w1, w2, w3;
                        if (WT == kF32) {
                            const float4 wv = *reinterpret_cast<const float4 *>(pc + (size_t)u * 16);
                            w0 = wv.x; w1 = wv.y; w2 = wv.z; w3 = wv.w;
                        } else if (WT == kF16) {
                            const uint2 wv = *reinterpret_cast<const uint2 *>(pc + (size_t)u * 8);
                            w0 = half_bits_to_f32(wv.x); w1 = half_bits_to_f32(wv.x >> 16);
                            w2 = half_bits_to_f32(wv.y); w3 = half_bits_to_f32(wv.y >> 16);
                        } else {
                            const uint2 wv = *reinterpret_cast<const uint2 *>(pc + (size_t)u * 8);
                            w0 = bf16_lo(wv.x); w1 = bf16_hi(wv.x);
                            w2 = bf16_lo(wv.y); w3 = bf16_hi(wv.y);
                        }
    #pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (t < ng) {
                                const float4 x = __ldg(reinterpret_cast<const float4 *>(xr[t] + 4 * u));
                                float part = w0 * x.x;
                                part = fmaf(w1, x.y, part);
                                part = fmaf(w2, x.z, part);
                                part = fmaf(w3, x.w, part);
                                acc[t] += part;
                            }
                        }
                    }
                }
    #pragma unroll
                for (int t = 0; t < NT; ++t) {
                    if (t < ng) {
                        const float v = warp_sum(acc[t]);
                        if (lane == 0) tot[g0 + t] = (p == 0) ? v : tot[g0 + t] + v;
                    }
                }
            }
            __syncwarp();
            // The stage is free: refill it with piece i + kStages.
            if (lane == 0 && i + kStages < total) {
                fence_proxy_async_smem();
                issue(i + kStages);
            }
            if (p == P - 1) {  // row done: epilogue and store
                for (int r = lane; r < ns; r += 32) {
                    const int yrow = MOE ? s_sorted[seg0 + r] : r;
                    const size_t o = (size_t)yrow * a.ldy + j;
                    const float *bj = a.bias + (MOE ? (size_t)e * m + j : (size_t)j);
                    a.Y[o] = epilogue(tot[r], a.flags, bj, a.R + o, a.alpha);
                    if (j < a.dual) a.Y[o + m] = tot[r] + a.bias2[j];  // the raw second band
                }
            }
            __syncwarp();
        }
        if (failed) break;
        ibase += total;
        // The window's routing tables are rewritten by the next window.
        if (n_win > 1) __syncthreads();
    }
}

template <int WT, bool MOE, int NT>
cudaError_t launch_one(const StreamArgs &a, int grid, const DeviceInfo &dev, cudaStream_t stream) {
    static std::atomic<unsigned long long> smem_set{0};
    auto kern = stream_kernel<WT, MOE, NT>;
    cudaError_t err = ensure_smem(kern, (int)kSmemBytes, dev, smem_set);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(grid), dim3(kWarps * 32), kSmemBytes, stream, a);
}

template <int WT>
cudaError_t launch_gemv_wt(const StreamArgs &a, int grid, const DeviceInfo &dev,
                           cudaStream_t stream) {
    if (a.n <= 1) return launch_one<WT, false, 1>(a, grid, dev, stream);
    if (a.n <= 2) return launch_one<WT, false, 2>(a, grid, dev, stream);
    if (a.n <= 4) return launch_one<WT, false, 4>(a, grid, dev, stream);
    return launch_one<WT, false, 8>(a, grid, dev, stream);
}

}  // namespace

cudaError_t launch_stream_gemv(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                               cudaStream_t stream) {
    const long long need = ((long long)a.m + kWarps - 1) / kWarps;
    const int grid = (int)(need < dev.sm_count ? need : dev.sm_count);
    switch (wtype) {
    case kBF16: return launch_gemv_wt<kBF16>(a, grid, dev, stream);
    case kF16: return launch_gemv_wt<kF16>(a, grid, dev, stream);
    case kF32: return launch_gemv_wt<kF32>(a, grid, dev, stream);
    case kQ8_0: return launch_gemv_wt<kQ8_0>(a, grid, dev, stream);
    default: return launch_gemv_wt<kQ4_0>(a, grid, dev, stream);
    }
}

cudaError_t launch_stream_moe(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                              cudaStream_t stream) {
    const long long slots = (long long)a.n * a.topk;
    const long long need = (slots * a.m + kWarps - 1) / kWarps;
    const int grid = (int)(need < dev.sm_count ? need : dev.sm_count);
    switch (wtype) {
    case kBF16: return launch_one<kBF16, true, 4>(a, grid, dev, stream);
    case kF16: return launch_one<kF16, true, 4>(a, grid, dev, stream);
    case kF32: return launch_one<kF32, true, 4>(a, grid, dev, stream);
    case kQ8_0: return launch_one<kQ8_0, true, 4>(a, grid, dev, stream);
    default: return launch_one<kQ4_0, true, 4>(a, grid, dev, stream);
    }
}

}  // namespace wq
