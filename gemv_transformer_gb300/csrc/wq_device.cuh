// wq_device.cuh -- device helpers shared by libwq's kernels (sm_103a).
//
// Storage formats (decoded here, bit-exact):
//   bf16 pairs   cortiq-engine 0.8.49 src/gpu_wgpu/nemotron_audio.rs, ae_gemm:
//                element 2c = f32 bits (w << 16), element 2c+1 = f32 bits (w & 0xFFFF0000).
//   Q8_0         hanzo-ml 0.11.13 src/wgpu_backend.rs, matvec_q8_0_gpu: 34-byte
//                blocks, little-endian f16 d then 32 int8 q; w = d*q.
//   Q4_0         hanzo-ml 0.11.13, matvec_q4_0_gpu: 18-byte blocks, f16 d then 16
//                bytes; element t < 16 = low nibble of byte t, t >= 16 = high
//                nibble of byte t-16; w = d*(q-8).
//   F16 / F32    wavo 0.3.0 src/gpu/mod.rs, Linear (pipeline index 0 / 1): IEEE
//                binary16 / binary32 elements, row after row.
// Epilogue       cortiq-engine ae_put: +bias, erf-GELU, +old Y, in that order.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wq {

enum WType : int { kBF16 = 0, kQ8_0 = 1, kQ4_0 = 2, kF16 = 3, kF32 = 4 };
enum Flag : unsigned { kBias = 1u, kGelu = 2u, kResidual = 4u, kSilu = 8u, kRelu = 16u, kTanh = 32u };
constexpr unsigned kActs = kGelu | kSilu | kRelu | kTanh;  // at most one per call
enum DevStatus : unsigned { kStTimeout = 4u, kStBadExpert = 5u, kStBadIndex = 7u };

// Bytes of one row of k weights in each format.
__host__ __device__ __forceinline__ size_t row_bytes(int wt, int k) {
    switch (wt) {
    case kBF16: case kF16: return (size_t)2 * k;
    case kF32: return (size_t)4 * k;
    case kQ8_0: return (size_t)34 * (k / 32);
    default: return (size_t)18 * (k / 32);
    }
}

// First error wins; later ones are dropped.
__device__ __forceinline__ void record_status(unsigned *st, unsigned code) {
    atomicCAS(st, 0u, code);
}

// ------------------------------------------------------------------ decode --

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Four signed bytes of v -> f32, exact.  Each byte is biased to unsigned and
// placed in the mantissa of 2^23; subtracting 2^23 + 128 leaves the value.
__device__ __forceinline__ void s8x4_to_f32(uint32_t v, float &a, float &b, float &c, float &d) {
    const uint32_t u = v ^ 0x80808080u;
    const float off = 8388736.0f;  // 2^23 + 128
    a = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440)) - off;
    b = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441)) - off;
    c = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7442)) - off;
    d = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7443)) - off;
}

// Four 4-bit codes (one per byte, 0..15) of v -> f32 (q - 8), exact.
__device__ __forceinline__ void u4x4_to_f32_m8(uint32_t v, float &a, float &b, float &c,
                                               float &d) {
    const float off = 8388616.0f;  // 2^23 + 8
    a = __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440)) - off;
    b = __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7441)) - off;
    c = __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7442)) - off;
    d = __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7443)) - off;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 32-bit value from two 16-bit-aligned halves (shared memory).
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t *p) {
    const uint16_t *h = reinterpret_cast<const uint16_t *>(p);
    return (uint32_t)h[0] | ((uint32_t)h[1] << 16);
}

// ---------------------------------------------------------------- epilogue --

__device__ __forceinline__ float gelu_erf(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752440f));
}

// The activation of the epilogue (wavo 0.3.0 src/gpu/mod.rs, enum Epilogue: Gelu,
// Silu v/(1+exp(-v)), Relu max(v, 0), Tanh); none when no activation flag is set.
__device__ __forceinline__ float activate(float v, unsigned flags) {
    if (!(flags & kActs)) return v;
    if (flags & kGelu) return gelu_erf(v);
    if (flags & kSilu) return v / (1.0f + expf(-v));
    if (flags & kRelu) return fmaxf(v, 0.0f);
    return tanhf(v);
}

// acc -> Y value.  `res` is read only with kResidual.  alpha scales the
// contribution before the residual is added (wavo 0.3.0 src/gpu/mod.rs,
// Epilogue::Residual(a): the biased product times a is added to the old output;
// 1 otherwise, which leaves every value unchanged).
__device__ __forceinline__ float epilogue(float acc, unsigned flags, const float *bias_j,
                                          const float *res_ij, float alpha) {
    float v = acc;
    if (flags & kBias) v += __ldg(bias_j);
    v = alpha * activate(v, flags);
    if (flags & kResidual) v += *res_ij;  // may alias Y: plain load
    return v;
}

// The same, with the bias and residual values already loaded (e.g. staged in
// shared memory); each is used only when its flag is set.
__device__ __forceinline__ float epilogue_vals(float acc, unsigned flags, float bias_j,
                                               float res_ij, float alpha) {
    float v = acc;
    if (flags & kBias) v += bias_j;
    v = alpha * activate(v, flags);
    if (flags & kResidual) v += res_ij;
    return v;
}

// ------------------------------------------------ programmatic dependent launch --

// First statement of every kernel.  Lets the next kernel on the stream (launched
// with programmatic serialization) be scheduled now, then waits until every grid
// this one depends on has completed and its memory is visible: nothing below
// touches global memory before that, so the ordering is that of a plain launch;
// only launch latency and CTA setup overlap the previous kernel's tail.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The two halves of pdl_enter() for kernels that first set up on-chip state
// (barriers, tensor memory) that no earlier grid touches: the setup then
// overlaps the previous kernel's tail, and every thread calls pdl_wait()
// before its first global-memory access.
__device__ __forceinline__ void pdl_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------- mbarrier + bulk copy --

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking check of the phase with `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with `parity`: one non-blocking check, then up to
// limit - 1 polls that may each suspend the thread for a short while.  With
// limit == 1 only the non-blocking check is made.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit) {
    if (mbar_test_wait(bar, parity)) return true;
    for (uint64_t i = 1; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Polls used when draining copies after a failed wait (not shortened by the
// diagnostic wait limit, so a drain outlives a deliberately short wait).
constexpr uint64_t kDrainPolls = 1ull << 24;

// Global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read once per call (weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace wq
