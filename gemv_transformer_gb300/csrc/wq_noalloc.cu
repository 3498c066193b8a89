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
#include "../../include/wq.h"
#include "wq_device.cuh"
#include "wq_internal.h"

namespace wq {

// The rounded X (bf16 [n][k], row-major), followed for Q8_0/Q4_0/F16/F32 weights
// by the rounded W (bf16 [m][k]).  Every byte a call reads is written by the same
// call first (the rounding passes cover all n*k and m*k elements and the GEMM's
// tensor maps stop at rows n and m; rows past them are zero-filled by the TMA
// unit, not read), so nothing here has to start at zero.  One copy per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[WQ_GEMM_NOALLOC_SCRATCH_BYTES];

namespace {
// The array's device address on the current device.  Host code cannot use the
// symbol itself (it names a host-side stand-in), so the address is looked up;
// this is a host-side table lookup that allocates nothing.  It is repeated on
// every call rather than cached, so that a context created after a
// cudaDeviceReset (which loads the module again, possibly elsewhere) is never
// given a stale address.  Returns nullptr if the lookup fails.
void *scratch_ptr() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    return p;
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
    void *scratch = scratch_ptr();
    if (!scratch) return WQ_ERR_CUDA;
    return wq_gemm_ws(n, m, k, wtype, flags, X, W, bias, residual, Y, scratch,
                      (size_t)WQ_GEMM_NOALLOC_SCRATCH_BYTES, stream);
}
