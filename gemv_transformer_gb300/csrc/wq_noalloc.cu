// wq_noalloc.cu -- wq_gemm_noalloc: the workspace tensor-core GEMM with its bf16
// copy of X held in a fixed, statically reserved device array instead of a
// caller buffer.
//
// Who needs it: callers that may not allocate device memory at call time and
// have no buffer of their own to lend -- code running where an allocation could
// block, fail, or be forbidden (a real-time serving loop with a frozen memory
// budget, a plug-in host that owns the allocator, an embedded runtime with no
// allocator at all).  Nothing here allocates: no cudaMalloc/cudaFree, no
// allocating library routine.  The array below is part of the library's device
// image; the CUDA runtime reserves it when it loads this module on a device.
#include <mutex>

#include "../../include/wq.h"
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {

// The rounded X (bf16 [n][k], row-major).  Every byte a call reads is written by
// the same call first (the rounding pass covers all n*k elements and the GEMM's
// tensor map stops at row n; rows past it are zero-filled by the TMA unit, not
// read), so nothing here has to start at zero.  One copy per device.
__device__ __align__(256) unsigned char g_noalloc_scratch[WQ_GEMM_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_na_mu;
void *g_na_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per ordinal

// Looks the array's address up once per device, with that device current (the
// caller's).  Returns nullptr if the lookup fails.
void *scratch_ptr(int ordinal) {
    if (ordinal < 0 || ordinal >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_ptr[ordinal]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress((void **)&p, g_noalloc_scratch) != cudaSuccess || !p)
            return nullptr;
        g_na_ptr[ordinal] = p;
    }
    return g_na_ptr[ordinal];
}
}  // namespace
}  // namespace wq

using namespace wq;

extern "C" wq_status wq_gemm_noalloc(int n, int m, int k, int wtype, unsigned flags,
                                     const float *X, const void *W, const float *bias,
                                     const float *residual, float *Y, wq_stream_t stream) {
    const wq_status s = check_gemm_args(n, m, k, wtype, flags, X, W, bias, residual, Y);
    if (s != WQ_OK) return s;
    const size_t need = wq_gemm_workspace_bytes(n, m, k, wtype, flags);
    if (need == 0)  // this route takes no scratch: plain wq_gemm
        return wq_gemm(n, m, k, wtype, flags, X, W, bias, residual, Y, stream);
    if (need > (size_t)WQ_GEMM_NOALLOC_SCRATCH_BYTES) return WQ_ERR_TOO_LARGE;
    int ordinal = -1;
    if (cudaGetDevice(&ordinal) != cudaSuccess) return WQ_ERR_CUDA;
    void *scratch = scratch_ptr(ordinal);
    if (!scratch) return WQ_ERR_CUDA;
    return wq_gemm_ws(n, m, k, wtype, flags, X, W, bias, residual, Y, scratch,
                      (size_t)WQ_GEMM_NOALLOC_SCRATCH_BYTES, stream);
}
