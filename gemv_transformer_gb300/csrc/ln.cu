// ln.cu -- row LayerNorm written into a GEMM workspace (the pass before wq_gemm_ln_ws).
//
// cortiq-engine 0.8.49 src/gpu_wgpu/nemotron_audio.rs, kernel ae_ln: per row of
// X [n][k], mean = sum x / k, var = sum (x - mean)^2 / k, and
//     y = (x - mean) / sqrt(var + 1e-5) * g + b      (gb = [g (k) | b (k)]).
// One 128-thread block per row (many rows in flight per SM): each thread sums a
// strided slice of the row, the partial sums are added by a fixed butterfly of
// shuffles and then the four warp sums in order (deterministic), and the row is
// read three times (mean, variance, output), the later passes from L1/L2.  The
// output is f32, or bf16 rounded to nearest even for the tensor-core GEMM.
#include "tc_ptx.cuh"
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {
namespace {

__device__ __forceinline__ float warp_sum_bfly(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

constexpr int kLnThreads = 128;  // one block per row

// Sum over the block in a fixed order: each warp's butterfly, then the four warp
// sums added 0, 1, 2, 3 (every thread gets the same, deterministic, value).
__device__ __forceinline__ float block_sum(float v, float *s_part) {
    v = warp_sum_bfly(v);
    const int warp = threadIdx.x >> 5;
    __syncthreads();  // s_part free (a previous sum has been read)
    if ((threadIdx.x & 31) == 0) s_part[warp] = v;
    __syncthreads();
    return ((s_part[0] + s_part[1]) + s_part[2]) + s_part[3];
}

template <bool BF16_OUT>
__global__ void __launch_bounds__(kLnThreads) ln_rows_kernel(const float *__restrict__ X,
                                                             const float *__restrict__ gb, int n,
                                                             int k, void *__restrict__ out) {
    pdl_enter();
    __shared__ float s_part[kLnThreads / 32];
    const int k4 = k / 4;  // k % 4 == 0 for every weight format (k % 8 or k % 32)
    for (long long row = blockIdx.x; row < n; row += gridDim.x) {
        const float4 *x4 = reinterpret_cast<const float4 *>(X + (size_t)row * k);
        float s = 0.f;
#pragma unroll 4
        for (int j = threadIdx.x; j < k4; j += kLnThreads) {
            const float4 v = __ldg(x4 + j);
            s += (v.x + v.y) + (v.z + v.w);
        }
        const float mean = block_sum(s, s_part) / (float)k;
        float q = 0.f;
#pragma unroll 4
        for (int j = threadIdx.x; j < k4; j += kLnThreads) {
            const float4 v = __ldg(x4 + j);
            const float a = v.x - mean, b = v.y - mean, c = v.z - mean, d = v.w - mean;
            q += (a * a + b * b) + (c * c + d * d);
        }
        const float rstd = 1.0f / sqrtf(block_sum(q, s_part) / (float)k + 1e-5f);
        const float4 *g4 = reinterpret_cast<const float4 *>(gb);
        const float4 *b4 = reinterpret_cast<const float4 *>(gb + k);
#pragma unroll 4
        for (int j = threadIdx.x; j < k4; j += kLnThreads) {
            const float4 v = __ldg(x4 + j), g = __ldg(g4 + j), bb = __ldg(b4 + j);
            const float y0 = (v.x - mean) * rstd * g.x + bb.x, y1 = (v.y - mean) * rstd * g.y + bb.y;
            const float y2 = (v.z - mean) * rstd * g.z + bb.z, y3 = (v.w - mean) * rstd * g.w + bb.w;
            if (BF16_OUT) {
                reinterpret_cast<uint2 *>(out)[(size_t)row * k4 + j] =
                    make_uint2(tc::pack_bf16x2(y0, y1), tc::pack_bf16x2(y2, y3));
            } else {
                reinterpret_cast<float4 *>(out)[(size_t)row * k4 + j] = make_float4(y0, y1, y2, y3);
            }
        }
    }
}

}  // namespace

cudaError_t launch_layer_norm(const float *X, const float *gb, int n, int k, void *out,
                              bool bf16_out, const DeviceInfo &dev, cudaStream_t stream) {
    long long blocks = n;  // one row per block
    if (blocks > (long long)dev.sm_count * 64) blocks = (long long)dev.sm_count * 64;
    if (blocks < 1) blocks = 1;
    return bf16_out ? launch_pdl(ln_rows_kernel<true>, dim3((unsigned)blocks), dim3(kLnThreads), 0,
                                 stream, X, gb, n, k, out)
                    : launch_pdl(ln_rows_kernel<false>, dim3((unsigned)blocks), dim3(kLnThreads), 0,
                                 stream, X, gb, n, k, out);
}

}  // namespace wq
