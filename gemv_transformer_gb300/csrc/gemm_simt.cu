// gemm_simt.cu -- tiled f32-FMA GEMM for any n, all three weight formats.
//
// Computes cortiq-engine 0.8.49 ae_gemm's Y[n.m] (=|+=) X[n.k] . W[m.k]^T (+bias)
// (gelu) with exact f32 products (W decoded bit-exactly, X as given), and the
// masked store of ae_store (nothing outside [n][m] is written).
//
// Tile 64 (X rows) x 64 (W rows) x 32 (k), 256 threads, 4x4 outputs per thread.
// W tiles are decoded into f32 in shared memory as they are loaded (one 32-weight
// block per row per k step for Q8_0/Q4_0).  Each k step's 32 products are summed
// into a fresh partial that is then added to the running total, which bounds the
// serial f32 chain per output to k/32 + 32 terms.
//
// Grids smaller than one wave (small n and m, e.g. n = 32, m = 512) instead run
// gemm_rows_kernel when k <= 2048: 32 x 8 output blocks, one per CTA, each with
// the whole k loop (one warp per W row, one lane per X row).  With larger k they
// run gemm_splitk_kernel: 32 x 32 output tiles, the k steps of a tile split across
// the KS CTAs of a thread-block cluster (KS <= 8), each CTA summing its steps the
// same way; each CTA then adds the KS partials of one slice of the tile, in rank
// order, through distributed shared memory (deterministic) and applies the
// epilogue.
#include <cooperative_groups.h>

#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

// Eight consecutive weights t0..t0+7 (t0 % 8 == 0) of one W row, exact in f32.
template <int WT>
__device__ __forceinline__ void decode8(const uint8_t *row, int t0, float (&w)[8]) {
    if (WT == kF16) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + (size_t)2 * t0);
        w[0] = half_bits_to_f32(v.x); w[1] = half_bits_to_f32(v.x >> 16);
        w[2] = half_bits_to_f32(v.y); w[3] = half_bits_to_f32(v.y >> 16);
        w[4] = half_bits_to_f32(v.z); w[5] = half_bits_to_f32(v.z >> 16);
        w[6] = half_bits_to_f32(v.w); w[7] = half_bits_to_f32(v.w >> 16);
    } else if (WT == kF32) {
        const float4 v0 = *reinterpret_cast<const float4 *>(row + (size_t)4 * t0);
        const float4 v1 = *reinterpret_cast<const float4 *>(row + (size_t)4 * t0 + 16);
        w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
        w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
    } else if (WT == kBF16) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + (size_t)2 * t0);
        w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x);
        w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
        w[4] = bf16_lo(v.z); w[5] = bf16_hi(v.z);
        w[6] = bf16_lo(v.w); w[7] = bf16_hi(v.w);
    } else if (WT == kQ8_0) {
        const uint8_t *bp = row + (size_t)34 * (t0 / 32);
        const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
        for (int e = 0; e < 8; ++e) w[e] = d * (float)(int8_t)bp[2 + (t0 & 31) + e];
    } else {
        const uint8_t *bp = row + (size_t)18 * (t0 / 32);
        const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
        for (int e = 0; e < 8; ++e) {
            const int t = (t0 & 31) + e;
            const uint32_t byte = bp[2 + (t & 15)];
            const int code = (t < 16) ? (int)(byte & 15u) : (int)(byte >> 4);
            w[e] = d * (float)(code - 8);
        }
    }
}


constexpr int TI = 64, TJ = 64, TK = 32;

template <int WT>
__device__ __forceinline__ void load_w_tile(const GemmArgs &a, int j0, int kk, int tid,
                                            float (*ws)[TJ + 4]) {
    const int r = tid >> 2, q = tid & 3;  // row of the tile, eighth of the k step
    const int j = j0 + r;
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = 0.f;
    if (j < a.m) {
        const uint8_t *row = a.W + (size_t)j * row_bytes(WT, a.k);
        if (WT == kBF16 || WT == kF16 || WT == kF32) {
            const int t0 = kk + 8 * q;
            if (t0 < a.k) decode8<WT>(row, t0, w);  // k % 8 == 0: all eight or none
        } else if (WT == kQ8_0) {
            const uint8_t *bp = row + (size_t)34 * (kk / 32);
            const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = d * (float)(int8_t)bp[2 + 8 * q + e];
        } else {
            const uint8_t *bp = row + (size_t)18 * (kk / 32);
            const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = 8 * q + e;  // element of the block
                const uint32_t byte = bp[2 + (t & 15)];
                const int code = (t < 16) ? (int)(byte & 15u) : (int)(byte >> 4);
                w[e] = d * (float)(code - 8);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ws[8 * q + e][r] = w[e];
}

// DUAL: also the second output band (columns m.. of Y); a separate instantiation,
// so that kernels without it carry none of its code.
template <int WT, bool DUAL>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const GemmArgs a) {
    pdl_enter();
    __shared__ float xs[TK][TI + 4];
    __shared__ float ws[TK][TJ + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int i0 = blockIdx.y * TI, j0 = blockIdx.x * TJ;
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;

    for (int kk = 0; kk < a.k; kk += TK) {
        {  // X tile, transposed into xs[k][i]
            const int r = tid >> 2, c0 = (tid & 3) * 8;
            const int i = i0 + r;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = kk + c0 + e;
                xs[c0 + e][r] = (i < a.n && t < a.k) ? __ldg(a.X + (size_t)i * a.k + t) : 0.f;
            }
        }
        load_w_tile<WT>(a, j0, kk, tid, ws);
        __syncthreads();
        float part[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) part[u][v] = 0.f;
#pragma unroll 8
        for (int t = 0; t < TK; ++t) {
            const float4 xv = *reinterpret_cast<const float4 *>(&xs[t][ty * 4]);
            const float4 wv = *reinterpret_cast<const float4 *>(&ws[t][tx * 4]);
            const float xa[4] = {xv.x, xv.y, xv.z, xv.w};
            const float wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) part[u][v] = fmaf(xa[u], wa[v], part[u][v]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) acc[u][v] += part[u][v];
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = i0 + ty * 4 + u;
        if (i >= a.n) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int j = j0 + tx * 4 + v;
            if (j >= a.m) continue;
            const size_t o = (size_t)i * a.ldy + j;
            a.Y[o] = epilogue(acc[u][v], a.flags, a.bias + j, a.R + o, a.alpha);
            if (DUAL && j < a.dual) a.Y[o + a.m] = acc[u][v] + a.bias2[j];  // the raw second band
        }
    }
}

// ------------------------------------------------------------ split-k --

constexpr int SK = 32;  // tile rows (X) = tile rows (W) = k step

// Four consecutive weights 4q..4q+3 of the 32-step at kk of row j, decoded to f32.
template <int WT>
__device__ __forceinline__ void load_w4(const GemmArgs &a, int j, int kk, int q, float (&w)[4]) {
    w[0] = w[1] = w[2] = w[3] = 0.f;
    if (j >= a.m || kk + 4 * q >= a.k) return;
    const uint8_t *row = a.W + (size_t)j * row_bytes(WT, a.k);
    if (WT == kBF16) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + (size_t)2 * (kk + 4 * q));
        w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x);
        w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    } else if (WT == kF16) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + (size_t)2 * (kk + 4 * q));
        w[0] = half_bits_to_f32(v.x); w[1] = half_bits_to_f32(v.x >> 16);
        w[2] = half_bits_to_f32(v.y); w[3] = half_bits_to_f32(v.y >> 16);
    } else if (WT == kF32) {
        const float4 v = *reinterpret_cast<const float4 *>(row + (size_t)4 * (kk + 4 * q));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if (WT == kQ8_0) {
        const uint8_t *bp = row + (size_t)34 * (kk / 32);
        const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = d * (float)(int8_t)bp[2 + 4 * q + e];
    } else {
        const uint8_t *bp = row + (size_t)18 * (kk / 32);
        const float d = half_bits_to_f32((uint32_t)bp[0] | ((uint32_t)bp[1] << 8));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = 4 * q + e;  // element of the block
            const uint32_t byte = bp[2 + (t & 15)];
            const int code = (t < 16) ? (int)(byte & 15u) : (int)(byte >> 4);
            w[e] = d * (float)(code - 8);
        }
    }
}

template <int WT, bool DUAL>
__global__ void __launch_bounds__(256) gemm_splitk_kernel(const GemmArgs a, int steps_per_rank) {
    pdl_enter();
    namespace cg = cooperative_groups;
    __shared__ float xs[SK][SK + 4];   // [k][i]
    __shared__ float ws[SK][SK + 4];   // [k][j]
    __shared__ float red[SK * SK];     // this CTA's partial tile, [i][j]
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int i0 = blockIdx.y * SK, j0 = blockIdx.x * SK;
    const int rank = (int)cluster.block_rank();
    const int KS = (int)cluster.num_blocks();
    const int nsteps = (a.k + SK - 1) / SK;
    const int s0 = rank * steps_per_rank, s1 = min(nsteps, s0 + steps_per_rank);

    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    for (int st = s0; st < s1; ++st) {
        const int kk = st * SK;
        {   // X tile: row r, elements 4q..4q+3 (k % 4 == 0: a float4 is all in or all out)
            const int r = tid >> 3, q = tid & 7, i = i0 + r, t = kk + 4 * q;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < a.n && t < a.k)
                v = __ldg(reinterpret_cast<const float4 *>(a.X + (size_t)i * a.k + t));
            xs[4 * q + 0][r] = v.x; xs[4 * q + 1][r] = v.y;
            xs[4 * q + 2][r] = v.z; xs[4 * q + 3][r] = v.w;
        }
        {
            const int r = tid >> 3, q = tid & 7;
            float w[4];
            load_w4<WT>(a, j0 + r, kk, q, w);
#pragma unroll
            for (int e = 0; e < 4; ++e) ws[4 * q + e][r] = w[e];
        }
        __syncthreads();
        float part[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 8
        for (int t = 0; t < SK; ++t) {
            const float2 xv = *reinterpret_cast<const float2 *>(&xs[t][2 * ty]);
            const float2 wv = *reinterpret_cast<const float2 *>(&ws[t][2 * tx]);
            part[0][0] = fmaf(xv.x, wv.x, part[0][0]);
            part[0][1] = fmaf(xv.x, wv.y, part[0][1]);
            part[1][0] = fmaf(xv.y, wv.x, part[1][0]);
            part[1][1] = fmaf(xv.y, wv.y, part[1][1]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int v = 0; v < 2; ++v) acc[u][v] += part[u][v];
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int v = 0; v < 2; ++v) red[(2 * ty + u) * SK + 2 * tx + v] = acc[u][v];
    cluster.sync();
    // Every rank finishes a slice of the tile: the partials of ranks 0..KS-1, added
    // in rank order (deterministic), loaded from their shared memory all at once.
    const int slice = (SK * SK + KS - 1) / KS;
    const int end = min(SK * SK, (rank + 1) * slice);
    for (int idx = rank * slice + tid; idx < end; idx += 256) {
        float p[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) p[r] = r < KS ? cluster.map_shared_rank(red, r)[idx] : 0.f;
        float sum = p[0];
#pragma unroll
        for (int r = 1; r < 8; ++r)
            if (r < KS) sum += p[r];
        const int i = i0 + idx / SK, j = j0 + idx % SK;
        if (i < a.n && j < a.m) {
            const size_t o = (size_t)i * a.ldy + j;
            a.Y[o] = epilogue(sum, a.flags, a.bias + j, a.R + o, a.alpha);
            if (DUAL && j < a.dual) a.Y[o + a.m] = sum + a.bias2[j];  // the raw second band
        }
    }
    cluster.sync();  // every rank keeps its shared memory until all slices are read
}

// Small grids with moderate k: one warp per W row and one lane per X row (32 x 8
// outputs per CTA), the whole k loop in one CTA -- no cluster, no cross-CTA
// reduction, so a call costs little more than its launch and two passes over
// shared memory.  X and W are staged in chunks of RK values of k (W decoded
// exactly into f32), all of a chunk's loads in flight at once; each lane sums each
// chunk in four interleaved chains that are then added in a fixed order
// (deterministic).
constexpr int RK = 256;

template <int WT, bool DUAL>
__global__ void __launch_bounds__(256) gemm_rows_kernel(const GemmArgs a) {
    pdl_enter();
    __shared__ __align__(16) float xs[32][RK + 4];  // [token][k], padded: conflict-free float4 reads
    __shared__ __align__(16) float ws[8][RK];       // [row][k], read as a warp broadcast
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = blockIdx.y * 32, j0 = blockIdx.x * 8;
    const size_t rb = row_bytes(WT, a.k);
    const int i = i0 + lane, j = j0 + warp;
    // The epilogue's inputs are requested first, so their latency overlaps the loop.
    const bool out = i < a.n && j < a.m;
    const size_t o = (size_t)i * a.ldy + j;
    const float bj = (out && (a.flags & kBias)) ? __ldg(a.bias + j) : 0.f;
    const float rij = (out && (a.flags & kResidual)) ? a.R[o] : 0.f;  // may alias Y: plain load
    float acc = 0.f;
    for (int k0 = 0; k0 < a.k; k0 += RK) {
        {   // X: row r, float4s q, q + 8, q + 16, q + 24 of the chunk (k % 4 == 0)
            const int r = tid >> 3, q = tid & 7, i = i0 + r;
#pragma unroll
            for (int u = 0; u < RK / 32; ++u) {
                const int t = k0 + 4 * (q + 8 * u);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < a.n && t < a.k)
                    v = __ldg(reinterpret_cast<const float4 *>(a.X + (size_t)i * a.k + t));
                *reinterpret_cast<float4 *>(&xs[r][4 * (q + 8 * u)]) = v;
            }
        }
        if (tid < 8 * (RK / 8)) {   // W: row r, eight weights from t0 (k % 8 == 0)
            const int r = tid / (RK / 8), g = tid % (RK / 8), j = j0 + r, t0 = k0 + 8 * g;
            float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (j < a.m && t0 < a.k) decode8<WT>(a.W + (size_t)j * rb, t0, w);
            *reinterpret_cast<float4 *>(&ws[r][8 * g]) = make_float4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<float4 *>(&ws[r][8 * g + 4]) = make_float4(w[4], w[5], w[6], w[7]);
        }
        __syncthreads();
        float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
#pragma unroll 16
        for (int t = 0; t < RK; t += 4) {
            const float4 xv = *reinterpret_cast<const float4 *>(&xs[lane][t]);
            const float4 wv = *reinterpret_cast<const float4 *>(&ws[warp][t]);
            c0 = fmaf(xv.x, wv.x, c0);
            c1 = fmaf(xv.y, wv.y, c1);
            c2 = fmaf(xv.z, wv.z, c2);
            c3 = fmaf(xv.w, wv.w, c3);
        }
        acc += (c0 + c1) + (c2 + c3);
        __syncthreads();
    }
    if (out) {
        a.Y[o] = epilogue_vals(acc, a.flags, bj, rij, a.alpha);
        if (DUAL && j < a.dual) a.Y[o + a.m] = acc + a.bias2[j];  // the raw second band
    }
}

template <int WT>
cudaError_t launch_rows_wt(const GemmArgs &a, cudaStream_t stream) {
    const dim3 grid((unsigned)((a.m + 7) / 8), (unsigned)((a.n + 31) / 32));
    if (a.dual > 0) return launch_pdl(gemm_rows_kernel<WT, true>, grid, dim3(256), 0, stream, a);
    return launch_pdl(gemm_rows_kernel<WT, false>, grid, dim3(256), 0, stream, a);
}

template <int WT>
cudaError_t launch_splitk_wt(const GemmArgs &a, int tiles_m, int tiles_n, int ks, int spr,
                             cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)tiles_m, (unsigned)tiles_n, (unsigned)ks);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)ks;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (a.dual > 0) return cudaLaunchKernelEx(&cfg, gemm_splitk_kernel<WT, true>, a, spr);
    return cudaLaunchKernelEx(&cfg, gemm_splitk_kernel<WT, false>, a, spr);
}

template <int WT>
__global__ void dequant_kernel(int m, int k, const uint8_t *W, float *out) {
    pdl_enter();
    // One thread per 8 weights.
    const long long units = (long long)m * (k / 8);
    const size_t rb = row_bytes(WT, k);
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(u / (k / 8));
        const int t0 = (int)(u % (k / 8)) * 8;
        float w[8];
        decode8<WT>(W + (size_t)j * rb, t0, w);
        float *o = out + (size_t)j * k + t0;
        for (int e = 0; e < 8; ++e) o[e] = w[e];
    }
}

// Embedding row gather (wavo 0.3.0 src/gpu/mod.rs, Recorder::embed):
// out[t][j] = W[ids[t]][j] + pos[t][j] + bias[j], in that order, f32.  One thread
// per 8 values (with VEC, pos, bias and out are 16-byte aligned and moved as
// float4); an id outside [0, rows) leaves its row unwritten and records the
// bad-index status (once, by the row's first thread).
template <int WT, bool VEC>
__global__ void embed_kernel(int n_ids, int rows, int k, const uint8_t *W, const int32_t *ids,
                             const float *pos, const float *bias, float *out, unsigned *status) {
    pdl_enter();
    const long long units = (long long)n_ids * (k / 8);
    const size_t rb = row_bytes(WT, k);
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(u / (k / 8));
        const int t0 = (int)(u % (k / 8)) * 8;
        const int id = ids[t];
        if (id < 0 || id >= rows) {
            if (t0 == 0) record_status(status, kStBadIndex);
            continue;
        }
        float w[8];
        decode8<WT>(W + (size_t)id * rb, t0, w);
        float *o = out + (size_t)t * k + t0;
        const float *p = pos ? pos + (size_t)t * k + t0 : nullptr;
        if (VEC) {
            float pv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            float bv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (p) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
                const float4 c = __ldg(reinterpret_cast<const float4 *>(p) + 1);
                pv[0] = a.x; pv[1] = a.y; pv[2] = a.z; pv[3] = a.w;
                pv[4] = c.x; pv[5] = c.y; pv[6] = c.z; pv[7] = c.w;
            }
            if (bias) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(bias + t0));
                const float4 c = __ldg(reinterpret_cast<const float4 *>(bias + t0) + 1);
                bv[0] = a.x; bv[1] = a.y; bv[2] = a.z; bv[3] = a.w;
                bv[4] = c.x; bv[5] = c.y; bv[6] = c.z; bv[7] = c.w;
            }
            float v[8];
            for (int e = 0; e < 8; ++e) {
                v[e] = w[e];
                if (p) v[e] += pv[e];
                if (bias) v[e] += bv[e];
            }
            reinterpret_cast<float4 *>(o)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4 *>(o)[1] = make_float4(v[4], v[5], v[6], v[7]);
        } else {
            for (int e = 0; e < 8; ++e) {
                float v = w[e];
                if (p) v += p[e];
                if (bias) v += bias[t0 + e];
                o[e] = v;
            }
        }
    }
}

template <bool DUAL>
cudaError_t launch_simt(const GemmArgs &a, int wtype, dim3 grid, cudaStream_t stream) {
    switch (wtype) {
    case kBF16: return launch_pdl(gemm_simt_kernel<kBF16, DUAL>, grid, dim3(256), 0, stream, a);
    case kF16: return launch_pdl(gemm_simt_kernel<kF16, DUAL>, grid, dim3(256), 0, stream, a);
    case kF32: return launch_pdl(gemm_simt_kernel<kF32, DUAL>, grid, dim3(256), 0, stream, a);
    case kQ8_0: return launch_pdl(gemm_simt_kernel<kQ8_0, DUAL>, grid, dim3(256), 0, stream, a);
    default: return launch_pdl(gemm_simt_kernel<kQ4_0, DUAL>, grid, dim3(256), 0, stream, a);
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs &a, int wtype, const DeviceInfo &dev,
                             cudaStream_t stream) {
    dim3 grid((a.m + TJ - 1) / TJ, (a.n + TI - 1) / TI);
    if ((long long)grid.x * grid.y < dev.sm_count && a.k <= 2048 &&
        (long long)(a.n + 31) / 32 <= 65535) {
        // Under one wave, moderate k: one CTA per 32 x 8 block of outputs, whole k.
        switch (wtype) {
        case kBF16: return launch_rows_wt<kBF16>(a, stream);
        case kF16: return launch_rows_wt<kF16>(a, stream);
        case kF32: return launch_rows_wt<kF32>(a, stream);
        case kQ8_0: return launch_rows_wt<kQ8_0>(a, stream);
        default: return launch_rows_wt<kQ4_0>(a, stream);
        }
    }
    if ((long long)grid.x * grid.y < dev.sm_count) {
        // Under one wave: split k across a cluster so that about one wave of CTAs runs.
        const long long tm = (a.m + SK - 1) / SK, tn = (a.n + SK - 1) / SK;
        const int nsteps = (a.k + SK - 1) / SK;
        long long ks = dev.sm_count / (tm * tn);
        if (ks > 8) ks = 8;
        if (ks > nsteps) ks = nsteps;
        if (ks < 1) ks = 1;
        const int spr = (nsteps + (int)ks - 1) / (int)ks;
        ks = (nsteps + spr - 1) / spr;  // no rank without steps
        if (tn <= 65535) {
            switch (wtype) {
            case kBF16: return launch_splitk_wt<kBF16>(a, (int)tm, (int)tn, (int)ks, spr, stream);
            case kF16: return launch_splitk_wt<kF16>(a, (int)tm, (int)tn, (int)ks, spr, stream);
            case kF32: return launch_splitk_wt<kF32>(a, (int)tm, (int)tn, (int)ks, spr, stream);
            case kQ8_0: return launch_splitk_wt<kQ8_0>(a, (int)tm, (int)tn, (int)ks, spr, stream);
            default: return launch_splitk_wt<kQ4_0>(a, (int)tm, (int)tn, (int)ks, spr, stream);
            }
        }
    }
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    return a.dual > 0 ? launch_simt<true>(a, wtype, grid, stream)
                      : launch_simt<false>(a, wtype, grid, stream);
}

cudaError_t launch_dequant(int wtype, int m, int k, const uint8_t *W, float *out,
                           cudaStream_t stream) {
    const long long units = (long long)m * (k / 8);
    long long blocks = (units + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3((unsigned)blocks), dim3(256), 0, stream, m, k, W, out);
    };
    switch (wtype) {
    case kBF16: return go(dequant_kernel<kBF16>);
    case kF16: return go(dequant_kernel<kF16>);
    case kF32: return go(dequant_kernel<kF32>);
    case kQ8_0: return go(dequant_kernel<kQ8_0>);
    default: return go(dequant_kernel<kQ4_0>);
    }
}

cudaError_t launch_embed(int n_ids, int rows, int k, int wtype, const uint8_t *W,
                         const int32_t *ids, const float *pos, const float *bias, float *out,
                         const DeviceInfo &dev, cudaStream_t stream) {
    const long long units = (long long)n_ids * (k / 8);
    long long blocks = (units + 255) / 256;
    const long long cap = (long long)dev.sm_count * 8;
    if (blocks > cap) blocks = cap;
    auto a16 = [](const void *q) { return ((uintptr_t)q & 15u) == 0; };
    const bool vec = a16(out) && (!pos || a16(pos)) && (!bias || a16(bias));
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3((unsigned)blocks), dim3(256), 0, stream, n_ids, rows, k, W,
                          ids, pos, bias, out, dev.status);
    };
    switch (wtype) {
    case kBF16: return vec ? go(embed_kernel<kBF16, true>) : go(embed_kernel<kBF16, false>);
    case kF16: return vec ? go(embed_kernel<kF16, true>) : go(embed_kernel<kF16, false>);
    case kF32: return vec ? go(embed_kernel<kF32, true>) : go(embed_kernel<kF32, false>);
    case kQ8_0: return vec ? go(embed_kernel<kQ8_0, true>) : go(embed_kernel<kQ8_0, false>);
    default: return vec ? go(embed_kernel<kQ4_0, true>) : go(embed_kernel<kQ4_0, false>);
    }
}

}  // namespace wq
