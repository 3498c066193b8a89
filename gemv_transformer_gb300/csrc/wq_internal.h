// wq_internal.h -- host-side declarations shared by libwq's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/wq.h"

namespace wq {

// Arguments of the weight-streaming kernels (plain GEMV and routed MoE).
struct StreamArgs {
    const float *X;        // [n][k] (GEMV) or [n_tok][k] (MoE)
    const uint8_t *W;      // [m][row_bytes] or bank [E][m][row_bytes]
    const float *bias;     // [m] or [E][m]
    const float *R;        // residual, [n][m] or [slots][m]
    float *Y;              // [n][m] or [slots][m]
    const int32_t *ids;    // MoE: [n_tok][topk]
    int n;                 // GEMV: rows of X; MoE: n_tok
    int m, k;
    unsigned flags;
    int topk, n_experts;   // MoE only
    unsigned *status;      // device status word
    unsigned long long wait_limit;
    float alpha = 1.0f;    // scale of the contribution before the residual
    int ldy = 0;           // row stride of Y and R: m + dual (MoE: m)
    int dual = 0;          // GEMV: columns j < dual also stored as acc + bias2[j] at m + j
    const float *bias2 = nullptr;  // [dual]
};

struct GemmArgs {
    const float *X;
    const uint8_t *W;
    const float *bias;
    const float *R;
    float *Y;
    int n, m, k;
    unsigned flags;
    unsigned *status;
    unsigned long long wait_limit;
    float alpha = 1.0f;    // scale of the contribution before the residual
    int ldy = 0;           // row stride of Y and R: m + dual
    int dual = 0;          // columns j < dual also stored as acc + bias2[j] at m + j
    const float *bias2 = nullptr;  // [dual]
    // W is the caller's weight image (not a workspace copy written by the kernel
    // launched just before): its first tiles may be requested before the wait for
    // that kernel.
    bool w_early = false;
};

struct DeviceInfo {
    int ordinal;
    int sm_count;
    unsigned *status;  // address of this device's status word
};

// Raise a kernel's dynamic shared memory limit once per device.  `done` holds one
// bit per device ordinal (< 64) and belongs to the kernel.
template <typename Kernel>
cudaError_t ensure_smem(Kernel kern, int bytes, const DeviceInfo &dev,
                        std::atomic<unsigned long long> &done) {
    const unsigned long long bit = 1ull << (dev.ordinal & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return err;
}

// Host-side argument checks shared by the wq_gemm family (no device work).
wq_status check_gemm_args(int n, int m, int k, int wtype, unsigned flags, const float *X,
                          const void *W, const float *bias, const float *residual,
                          const float *Y);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream finishes; it waits for it in pdl_enter()
// before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Facts about the current device (SM count cached per ordinal; the status word's
// address looked up each time).  Returns false on a CUDA error.
bool device_info(DeviceInfo &out);
unsigned long long wait_limit();

cudaError_t launch_stream_gemv(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                               cudaStream_t stream);
cudaError_t launch_stream_moe(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                              cudaStream_t stream);
bool mma_gemv_supported(int wtype, int k);
// bf16 or F16 weights, 1 <= n <= 16, k % 256 == 0: the tensor-core GEMV of gemv_half.cu.
bool half_gemv_supported(int wtype, int n, int k);
cudaError_t launch_half_gemv(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                             cudaStream_t stream);
// bf16 / F16 routed MoE matvec on the tensor cores (k % 256 == 0).
bool half_moe_supported(int wtype, int k);
cudaError_t launch_half_moe(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                            cudaStream_t stream);
cudaError_t launch_mma_gemv(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                            cudaStream_t stream);
cudaError_t launch_mma_moe(const StreamArgs &a, int wtype, const DeviceInfo &dev,
                           cudaStream_t stream);
cudaError_t launch_gemm_simt(const GemmArgs &a, int wtype, const DeviceInfo &dev,
                             cudaStream_t stream);
cudaError_t launch_gemm_tc(const GemmArgs &a, const DeviceInfo &dev, cudaStream_t stream);
size_t gemm_tc_workspace_bytes(int n, int k);
bool gemm_tcp_supported(const GemmArgs &a);
cudaError_t launch_gemm_tcp(const GemmArgs &a, const void *xb, const DeviceInfo &dev,
                            cudaStream_t stream);
size_t gemm_tc_w_workspace_bytes(int m, int k);
cudaError_t launch_gemm_tc_ws(const GemmArgs &a, int wtype, void *workspace,
                              const DeviceInfo &dev, cudaStream_t stream, bool x_ready = false);
cudaError_t launch_layer_norm(const float *X, const float *gb, int n, int k, void *out,
                              bool bf16_out, const DeviceInfo &dev, cudaStream_t stream);
cudaError_t launch_dequant(int wtype, int m, int k, const uint8_t *W, float *out,
                           cudaStream_t stream);
cudaError_t launch_embed(int n_ids, int rows, int k, int wtype, const uint8_t *W,
                         const int32_t *ids, const float *pos, const float *bias, float *out,
                         const DeviceInfo &dev, cudaStream_t stream);

}  // namespace wq
