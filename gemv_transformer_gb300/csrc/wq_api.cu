// wq_api.cu -- the extern "C" entry points of libwq (declared in include/wq.h).
//
// Host-side only: argument checks (hanzo-ml 0.11.13 src/wgpu_backend.rs refuses,
// in matvec_q*_gpu, a k that 32 does not divide and an x shorter than k, and in
// moe_matvec_gpu, fewer ids than rows), routing to a kernel, and the sticky device
// status word
// (wavo 0.3.0 src/gpu/mod.rs keeps the first device error and reports it on the
// next call).  Nothing here computes; every step of the contraction runs in the
// kernels.
#include <cmath>
#include <mutex>

#include "../../include/wq.h"
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {

// One status word per device (each device has its own copy of module globals).
__device__ unsigned g_status = 0u;

namespace {
constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitPolls = 1ull << 22;
std::mutex g_mu;
int g_sm_count[kMaxDevices];  // per ordinal, 0 until first asked
unsigned long long g_wait_limit = kDefaultWaitPolls;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

wq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? WQ_OK : WQ_ERR_CUDA; }

bool shape_ok(int wtype, int m, int k) {
    if (m <= 0 || k <= 0) return false;
    if (wtype == kBF16) return k % 8 == 0;
    if (wtype == kQ8_0 || wtype == kQ4_0) return k % 32 == 0;
    if (wtype == kF16 || wtype == kF32) return k % 8 == 0;
    return false;
}

// Common checks of wq_gemm / wq_gemv.
wq_status check_common(int n, int m, int k, int wtype, unsigned flags, const float *X,
                       const void *W, const float *bias, const float *residual, const float *Y) {
    if (n <= 0 || !shape_ok(wtype, m, k)) return WQ_ERR_INVALID_ARG;
    if (flags & ~(unsigned)(WQ_EPILOGUE_FLAGS | WQ_TC_BF16)) return WQ_ERR_INVALID_ARG;
    const unsigned acts = flags & (WQ_GELU | WQ_SILU | WQ_RELU | WQ_TANH);
    if (acts & (acts - 1)) return WQ_ERR_INVALID_ARG;  // more than one activation
    if (!X || !W || !Y) return WQ_ERR_INVALID_ARG;
    if ((flags & WQ_BIAS) && !bias) return WQ_ERR_INVALID_ARG;
    if ((flags & WQ_RESIDUAL) && !residual) return WQ_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W)) return WQ_ERR_INVALID_ARG;
    return WQ_OK;
}

// The epilogue's parts beyond the flags (wavo 0.3.0 src/gpu/mod.rs): the scale of
// Epilogue::Residual(a), and the `dual` outputs of Gpu::linear, written a second
// time after the m others with their own bias and no epilogue.
struct Extra {
    float alpha = 1.0f;
    int dual = 0;
    const float *bias2 = nullptr;
};
}  // namespace

wq_status check_gemm_args(int n, int m, int k, int wtype, unsigned flags, const float *X,
                          const void *W, const float *bias, const float *residual,
                          const float *Y) {
    return check_common(n, m, k, wtype, flags, X, W, bias, residual, Y);
}

bool device_info(DeviceInfo &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    // The status word's address is looked up on every call (a host-side lookup
    // that allocates nothing), not cached: after a cudaDeviceReset the module is
    // loaded again in a new context and the word may sit elsewhere.
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return false;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_sm_count[dev] &&
            cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess) {
            g_sm_count[dev] = 0;
            return false;
        }
        out.sm_count = g_sm_count[dev];
    }
    out.ordinal = dev;
    out.status = static_cast<unsigned *>(p);
    return true;
}

unsigned long long wait_limit() {
    std::lock_guard<std::mutex> lock(g_mu);
    return g_wait_limit;
}

namespace {
// The fields every contraction call shares; Y and the residual have rows of
// m + dual values.
template <typename Args>
void fill_args(Args &a, int n, int m, int k, unsigned flags, const float *X, const void *W,
               const float *bias, const float *residual, float *Y, const DeviceInfo &dev,
               const Extra &ex) {
    a.X = X;
    a.W = static_cast<const uint8_t *>(W);
    a.bias = bias;
    a.R = residual;
    a.Y = Y;
    a.n = n;
    a.m = m;
    a.k = k;
    a.flags = flags & WQ_EPILOGUE_FLAGS;
    a.status = dev.status;
    a.wait_limit = wait_limit();
    a.alpha = ex.alpha;
    a.ldy = m + ex.dual;
    a.dual = ex.dual;
    a.bias2 = ex.bias2;
}
}  // namespace

}  // namespace wq

using namespace wq;

extern "C" {

size_t wq_weight_bytes(int wtype, int m, int k) {
    if (!shape_ok(wtype, m, k)) return 0;
    const size_t b = row_bytes(wtype, k) * (size_t)m;
    return (b + 15) & ~(size_t)15;
}

static wq_status gemv_impl(int n, int m, int k, int wtype, unsigned flags, const float *X,
                           const void *W, const float *bias, const float *residual, float *Y,
                           wq_stream_t stream, const Extra &ex = Extra()) {
    DeviceInfo dv;
    if (!device_info(dv)) return WQ_ERR_CUDA;
    const DeviceInfo *dev = &dv;
    StreamArgs a{};
    fill_args(a, n, m, k, flags, X, W, bias, residual, Y, *dev, ex);
    if (mma_gemv_supported(wtype, k))
        return cuda_status(launch_mma_gemv(a, wtype, *dev, (cudaStream_t)stream));
    if (half_gemv_supported(wtype, n, k))
        return cuda_status(launch_half_gemv(a, wtype, *dev, (cudaStream_t)stream));
    return cuda_status(launch_stream_gemv(a, wtype, *dev, (cudaStream_t)stream));
}

wq_status wq_gemv(int n, int m, int k, int wtype, unsigned flags, const float *X, const void *W,
                  const float *bias, const float *residual, float *Y, wq_stream_t stream) {
    wq_status s = check_common(n, m, k, wtype, flags, X, W, bias, residual, Y);
    if (s != WQ_OK) return s;
    if (n > WQ_GEMV_MAX_N || (flags & WQ_TC_BF16)) return WQ_ERR_INVALID_ARG;
    return gemv_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, stream);
}

// wq_gemm after its argument checks.
static wq_status gemm_impl(int n, int m, int k, int wtype, unsigned flags, const float *X,
                           const void *W, const float *bias, const float *residual, float *Y,
                           wq_stream_t stream, const Extra &ex) {
    if (n <= WQ_GEMV_MAX_N)
        return gemv_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, stream, ex);
    // Tensor cores with quantised W need the bf16 copy of W: wq_gemm_ws.
    if ((flags & WQ_TC_BF16) && wtype != kBF16) return WQ_ERR_UNSUPPORTED;
    DeviceInfo dv;
    if (!device_info(dv)) return WQ_ERR_CUDA;
    const DeviceInfo *dev = &dv;
    GemmArgs a{};
    fill_args(a, n, m, k, flags, X, W, bias, residual, Y, *dev, ex);
    if (flags & WQ_TC_BF16) return cuda_status(launch_gemm_tc(a, *dev, (cudaStream_t)stream));
    return cuda_status(launch_gemm_simt(a, wtype, *dev, (cudaStream_t)stream));
}

wq_status wq_gemm(int n, int m, int k, int wtype, unsigned flags, const float *X, const void *W,
                  const float *bias, const float *residual, float *Y, wq_stream_t stream) {
    wq_status s = check_common(n, m, k, wtype, flags, X, W, bias, residual, Y);
    if (s != WQ_OK) return s;
    return gemm_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, stream, Extra());
}

size_t wq_gemm_workspace_bytes(int n, int m, int k, int wtype, unsigned flags) {
    if (n <= 0 || !shape_ok(wtype, m, k)) return 0;
    if (!(flags & WQ_TC_BF16) || n <= WQ_GEMV_MAX_N) return 0;
    const size_t x = gemm_tc_workspace_bytes(n, k);
    return wtype == kBF16 ? x : x + gemm_tc_w_workspace_bytes(m, k);
}

// wq_gemm_ws after the common argument checks.
static wq_status gemm_ws_impl(int n, int m, int k, int wtype, unsigned flags, const float *X,
                              const void *W, const float *bias, const float *residual, float *Y,
                              void *workspace, size_t workspace_bytes, wq_stream_t stream,
                              const Extra &ex) {
    const size_t need = wq_gemm_workspace_bytes(n, m, k, wtype, flags);
    if (need == 0)
        return gemm_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, stream, ex);
    if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < need)
        return WQ_ERR_INVALID_ARG;
    DeviceInfo dv;
    if (!device_info(dv)) return WQ_ERR_CUDA;
    const DeviceInfo *dev = &dv;
    GemmArgs a{};
    fill_args(a, n, m, k, flags, X, W, bias, residual, Y, *dev, ex);
    return cuda_status(launch_gemm_tc_ws(a, wtype, workspace, *dev, (cudaStream_t)stream));
}

wq_status wq_gemm_ws(int n, int m, int k, int wtype, unsigned flags, const float *X,
                     const void *W, const float *bias, const float *residual, float *Y,
                     void *workspace, size_t workspace_bytes, wq_stream_t stream) {
    wq_status s = check_common(n, m, k, wtype, flags, X, W, bias, residual, Y);
    if (s != WQ_OK) return s;
    return gemm_ws_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, workspace,
                        workspace_bytes, stream, Extra());
}

wq_status wq_gemm_dual(int n, int m, int k, int dual, int wtype, unsigned flags, float alpha,
                       const float *X, const void *W, const float *bias, const float *bias2,
                       const float *residual, float *Y, void *workspace, size_t workspace_bytes,
                       wq_stream_t stream) {
    wq_status s = check_common(n, m, k, wtype, flags, X, W, bias, residual, Y);
    if (s != WQ_OK) return s;
    if (!std::isfinite(alpha)) return WQ_ERR_INVALID_ARG;
    if (dual < 0 || dual > m || (dual > 0 && !bias2)) return WQ_ERR_INVALID_ARG;
    if ((long long)m + dual > 0x7FFFFFFFll) return WQ_ERR_INVALID_ARG;  // the row stride is an int
    const Extra ex{alpha, dual, dual > 0 ? bias2 : nullptr};
    if (!workspace)
        return gemm_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, stream, ex);
    return gemm_ws_impl(n, m, k, wtype, flags, X, W, bias, residual, Y, workspace,
                        workspace_bytes, stream, ex);
}

wq_status wq_gemm_alpha(int n, int m, int k, int wtype, unsigned flags, float alpha,
                        const float *X, const void *W, const float *bias, const float *residual,
                        float *Y, void *workspace, size_t workspace_bytes, wq_stream_t stream) {
    return wq_gemm_dual(n, m, k, 0, wtype, flags, alpha, X, W, bias, nullptr, residual, Y,
                        workspace, workspace_bytes, stream);
}

size_t wq_gemm_ln_workspace_bytes(int n, int m, int k, int wtype, unsigned flags) {
    if (n <= 0 || !shape_ok(wtype, m, k)) return 0;
    const size_t tc = wq_gemm_workspace_bytes(n, m, k, wtype, flags);
    if (tc) return tc;                                   // bf16 LN(X) (+ bf16 W)
    return ((size_t)n * k * 4 + 255) & ~(size_t)255;     // f32 LN(X)
}

wq_status wq_gemm_ln_ws(int n, int m, int k, int wtype, unsigned flags, const float *X,
                        const float *ln_gb, const void *W, const float *bias,
                        const float *residual, float *Y, void *workspace,
                        size_t workspace_bytes, wq_stream_t stream) {
    wq_status s = check_common(n, m, k, wtype, flags, X, W, bias, residual, Y);
    if (s != WQ_OK) return s;
    if (!ln_gb) return WQ_ERR_INVALID_ARG;
    const size_t need = wq_gemm_ln_workspace_bytes(n, m, k, wtype, flags);
    if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < need)
        return WQ_ERR_INVALID_ARG;
    if ((const void *)residual == workspace || (const void *)Y == workspace)
        return WQ_ERR_INVALID_ARG;
    DeviceInfo dv;
    if (!device_info(dv)) return WQ_ERR_CUDA;
    const DeviceInfo *dev = &dv;
    const bool tc = wq_gemm_workspace_bytes(n, m, k, wtype, flags) != 0;
    cudaError_t err = launch_layer_norm(X, ln_gb, n, k, workspace, tc, *dev, (cudaStream_t)stream);
    if (err != cudaSuccess) return WQ_ERR_CUDA;
    if (!tc)  // the f32 normalised rows feed the exact f32 paths, as wq_gemm
        return wq_gemm(n, m, k, wtype, flags & ~(unsigned)WQ_TC_BF16,
                       static_cast<const float *>(workspace), W, bias, residual, Y, stream);
    GemmArgs a{};
    // X is not read: the GEMM takes the bf16 rows from the workspace.
    fill_args(a, n, m, k, flags, X, W, bias, residual, Y, *dev, Extra());
    return cuda_status(launch_gemm_tc_ws(a, wtype, workspace, *dev, (cudaStream_t)stream, true));
}

wq_status wq_moe_gemv(int n_tok, int topk, int n_experts, int m, int k, int wtype,
                      unsigned flags, const float *X, const void *Wbank, const int32_t *ids,
                      const float *bias, const float *residual, float *Y, wq_stream_t stream) {
    if (topk <= 0 || n_experts <= 0 || !ids) return WQ_ERR_INVALID_ARG;
    wq_status s = check_common(n_tok, m, k, wtype, flags, X, Wbank, bias, residual, Y);
    if (s != WQ_OK) return s;
    if (flags & WQ_TC_BF16) return WQ_ERR_INVALID_ARG;
    if ((long long)m * n_experts > 0x7FFFFFFFll) return WQ_ERR_INVALID_ARG;
    if ((long long)n_tok * topk > 0x7FFFFFFFll) return WQ_ERR_INVALID_ARG;
    DeviceInfo dv;
    if (!device_info(dv)) return WQ_ERR_CUDA;
    const DeviceInfo *dev = &dv;
    StreamArgs a{};
    fill_args(a, n_tok, m, k, flags, X, Wbank, bias, residual, Y, *dev, Extra());
    a.ids = ids;
    a.topk = topk;
    a.n_experts = n_experts;
    if (mma_gemv_supported(wtype, k))
        return cuda_status(launch_mma_moe(a, wtype, *dev, (cudaStream_t)stream));
    if (half_moe_supported(wtype, k))
        return cuda_status(launch_half_moe(a, wtype, *dev, (cudaStream_t)stream));
    return cuda_status(launch_stream_moe(a, wtype, *dev, (cudaStream_t)stream));
}

wq_status wq_dequantize(int wtype, int m, int k, const void *W, float *out, wq_stream_t stream) {
    if (!shape_ok(wtype, m, k) || !W || !out || !aligned16(W)) return WQ_ERR_INVALID_ARG;
    return cuda_status(
        launch_dequant(wtype, m, k, static_cast<const uint8_t *>(W), out, (cudaStream_t)stream));
}

wq_status wq_embed(int n_ids, int rows, int k, int wtype, const void *W, const int32_t *ids,
                   const float *pos, const float *bias, float *out, wq_stream_t stream) {
    if (n_ids <= 0 || !shape_ok(wtype, rows, k) || !W || !ids || !out || !aligned16(W))
        return WQ_ERR_INVALID_ARG;
    DeviceInfo dv;
    if (!device_info(dv)) return WQ_ERR_CUDA;
    const DeviceInfo *dev = &dv;
    return cuda_status(launch_embed(n_ids, rows, k, wtype, static_cast<const uint8_t *>(W), ids,
                                    pos, bias, out, *dev, (cudaStream_t)stream));
}

wq_status wq_get_device_status(wq_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return WQ_ERR_CUDA;
    unsigned v = 0;
    const unsigned zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return WQ_ERR_CUDA;
    if (v != 0 && cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess)
        return WQ_ERR_CUDA;
    return (wq_status)v;
}

const char *wq_status_string(int status) {
    switch (status) {
    case WQ_OK: return "ok";
    case WQ_ERR_INVALID_ARG: return "invalid argument";
    case WQ_ERR_UNSUPPORTED: return "unsupported request";
    case WQ_ERR_CUDA: return "CUDA runtime error";
    case WQ_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case WQ_ERR_BAD_EXPERT: return "expert id out of range";
    case WQ_ERR_TOO_LARGE: return "request exceeds the fixed scratch size";
    case WQ_ERR_BAD_INDEX: return "embedding row id out of range";
    default: return "unknown status";
    }
}

void wq_set_wait_limit(uint64_t polls) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_wait_limit = polls ? (unsigned long long)polls : kDefaultWaitPolls;
}

}  // extern "C"
