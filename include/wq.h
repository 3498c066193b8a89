/*
 * wq.h -- C ABI of libwq: the weight-format contraction on one GPU
 *
 *     Y[n][m] (=|+=) epi( X[n][k] . W[m][k]^T )
 *
 * with W stored as bf16 pairs, GGML Q8_0 blocks or GGML Q4_0 blocks, dequantised
 * on the fly, accumulated in f32, and a fused epilogue (bias, erf-GELU,
 * residual add); plus the routed MoE matvec over one expert weight bank.
 *
 * Sources of each operation (page title, item):
 *   - wq_gemm: cortiq-engine 0.8.49, src/gpu_wgpu/nemotron_audio.rs,
 *     AudioEncoder::gemm and its kernel ae_gemm (Y[n][m] set or accumulated from
 *     X[n][k] . W[m][k]^T, optional bias and GELU, W as bf16 pairs), epilogue
 *     ae_put, masked store ae_store;
 *     wavo 0.3.0, src/gpu/mod.rs, Pass::gemm (Q8_0 weights).
 *   - wq_gemv: hanzo-ml 0.11.13, src/wgpu_backend.rs, matvec_q8_0_gpu /
 *     matvec_q4_0_gpu (y[nout] = Wq x[k] with the raw GGML blocks read in place);
 *     wavo 0.3.0, Pass::gemv (one activation row).
 *   - wq_moe_gemv: hanzo-ml 0.11.13, moe_matvec_gpu (y[s][r] = sum over k of
 *     W[ids[s]][r][k] x[s][k] over one bank [E][rows][k], router gather and
 *     expert matvec in one dispatch).
 *   - wq_gemm_alpha: wavo 0.3.0, src/gpu/mod.rs, Epilogue::Residual(a)
 *     (c += alpha (a W^T + b)) on the routes of wq_gemm / wq_gemm_ws.
 *   - wq_gemm_dual: wavo 0.3.0, src/gpu/mod.rs, Gpu::linear (dual outputs).
 *   - wq_dequantize: the block formats themselves (same pages).
 *   - wq_embed: wavo 0.3.0, src/gpu/mod.rs, Recorder::embed (table row ids[i]
 *     plus a position row plus the table's bias, k values each) and its test
 *     gemv_and_embed.
 *   - wq_get_device_status: wavo 0.3.0, Gpu "failure" (the first device error is
 *     reported by the next call) and its completion marks.
 *
 * Conventions shared by every call
 *   - Index names: n = rows of X (tokens), m = rows of W (outputs), k = inner.
 *   - All tensor pointers are DEVICE pointers owned by the caller.  libwq never
 *     allocates, frees or retains them, and allocates no device memory itself
 *     (the one fixed array of wq_gemm_noalloc is part of its device image).
 *   - Calls are asynchronous and ordered on `stream` (NULL = the legacy default
 *     stream).  They return once the work is launched.  A returned error means
 *     nothing was launched and no output was touched.
 *   - X is f32 row-major [n][k] and must be 16-byte aligned.
 *   - W is the storage-format byte image [m][row_bytes], 16-byte aligned, and its
 *     buffer must hold at least wq_weight_bytes(wtype, m, k) bytes: the format's
 *     size rounded up to a multiple of 16.  The padding is read, never used.
 *   - W is read as constant data: a call may start reading W before the kernel
 *     launched just before it on the same stream has finished (libwq's kernels use
 *     programmatic dependent launch and request their first weight tiles ahead of
 *     the wait for that kernel), so that kernel must not write W.  libwq's own
 *     kernels never write a weight image; a weight image produced on the device
 *     needs any other launch, an event wait or a synchronisation in between.
 *   - bias is f32 [m] (read when WQ_BIAS is set, else ignored, may be NULL).
 *   - residual is f32 [n][m] (read when WQ_RESIDUAL is set); it may equal Y, which
 *     gives the in-place "Y +=" form.  No other argument may overlap Y.
 *   - Y is f32 row-major [n][m].  Exactly the n*m elements of Y are written;
 *     nothing before or after them.
 *   - Device-side faults detected by a kernel (a bounded wait that ran out, an
 *     expert id out of range) do not trap: they are recorded in a sticky per-device
 *     status word that wq_get_device_status() reports and clears.
 *   - Results are deterministic: the same call on the same inputs gives the same
 *     bits.
 */
#ifndef WQ_H
#define WQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define WQ_API __attribute__((visibility("default")))
#else
#define WQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without including CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *wq_stream_t;

/* Weight storage formats. */
typedef enum {
    WQ_BF16 = 0, /* bf16 pairs: u32 word c of a row = element 2c | element 2c+1 << 16;
                    i.e. row-major little-endian bf16 [m][k]; k % 8 == 0 */
    WQ_Q8_0 = 1, /* 34-byte blocks of 32 weights along k: f16 d (LE), int8 q[32];
                    w = d*q; k % 32 == 0 */
    WQ_Q4_0 = 2, /* 18-byte blocks of 32 weights: f16 d (LE), 16 bytes; element t<16
                    = low nibble of byte t, t>=16 = high nibble of byte t-16;
                    w = d*(q-8); k % 32 == 0 */
    WQ_F16 = 3,  /* wavo 0.3.0 src/gpu/mod.rs Linear type 1: IEEE binary16 [m][k],
                    little-endian; k % 8 == 0 */
    WQ_F32 = 4   /* wavo Linear type 0: IEEE binary32 [m][k]; k % 8 == 0 */
} wq_wtype;

/* Epilogue flags, the bit values and order of cortiq-engine's ae_put:
 * v = acc; if BIAS v += bias[j]; if GELU v = 0.5 v (1 + erf(v / sqrt 2));
 * if RESIDUAL v += residual[i][j]; Y[i][j] = v.
 * SILU, RELU and TANH are wavo 0.3.0's other Epilogue activations (src/gpu/mod.rs,
 * enum Epilogue): v / (1 + exp(-v)), max(v, 0), tanh(v), in GELU's place.  At
 * most one of GELU, SILU, RELU, TANH per call (else WQ_ERR_INVALID_ARG); wavo's
 * GeluResidual is GELU | RESIDUAL. */
enum {
    WQ_BIAS = 1u,
    WQ_GELU = 2u,
    WQ_RESIDUAL = 4u,
    WQ_SILU = 8u,
    WQ_RELU = 16u,
    WQ_TANH = 32u,
    WQ_EPILOGUE_FLAGS = 63u,
    /* n > WQ_GEMV_MAX_N only: run the contraction on the tcgen05 tensor cores with
     * X rounded to bf16 (round to nearest even) and f32 accumulation; quantised
     * weights are dequantised and rounded to bf16 the same way (wq_gemm_ws and
     * wq_gemm_noalloc only).  Without it every path multiplies exact f32
     * products; smaller n ignore it (the GEMV kernels are exact). */
    WQ_TC_BF16 = 256u
};

typedef enum {
    WQ_OK = 0,
    WQ_ERR_INVALID_ARG = 1,    /* bad size, null pointer, misalignment, bad flag */
    WQ_ERR_UNSUPPORTED = 2,    /* valid request this build has no kernel for */
    WQ_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
    WQ_ERR_DEVICE_TIMEOUT = 4, /* a kernel's bounded wait ran out (device status) */
    WQ_ERR_BAD_EXPERT = 5,     /* an expert id outside [0, n_experts) (device status) */
    WQ_ERR_TOO_LARGE = 6,      /* wq_gemm_noalloc: the call needs more than its fixed scratch */
    WQ_ERR_BAD_INDEX = 7       /* wq_embed: a row id outside [0, rows) (device status) */
} wq_status;

/* Largest n that wq_gemv accepts. */
#define WQ_GEMV_MAX_N 16
/* wq_moe_gemv routes its n_tok * topk slots in windows of this many: a selected
 * expert's weights are read once per window that routes slots to it.  Not a
 * limit on n_tok * topk. */
#define WQ_MOE_WINDOW_SLOTS 256

/*
 * Y = epi(X . W^T) for any n >= 1 (cortiq-engine ae_gemm semantics).
 * Routing: n <= WQ_GEMV_MAX_N goes to the weight-streaming GEMV kernels (as
 * wq_gemv); otherwise WQ_TC_BF16 with WQ_BF16 weights runs the tcgen05 kernel,
 * and everything else the f32-FMA tiled kernel.
 * Errors: WQ_ERR_INVALID_ARG for n, m, k <= 0; k % 32 != 0 (Q8_0/Q4_0) or
 * k % 8 != 0 (bf16, f16, f32); null X, W or Y; null bias/residual when its flag
 * is set; X or W not 16-byte aligned; unknown flag bits or wtype.
 * WQ_ERR_UNSUPPORTED for WQ_TC_BF16 with a wtype other than WQ_BF16 and
 * n > WQ_GEMV_MAX_N (that needs the bf16 copy of W in a workspace: wq_gemm_ws;
 * f16/f32 elements, like d*q, are rounded to the nearest bf16 there).
 * WQ_ERR_CUDA if the launch fails.
 */
WQ_API wq_status wq_gemm(int n, int m, int k, int wtype, unsigned flags, const float *X, const void *W,
                  const float *bias, const float *residual, float *Y, wq_stream_t stream);

/*
 * wq_gemm with a caller-provided device workspace, which lets the tensor-core path
 * round X to bf16 once in a separate pass (into the workspace) and then feed both
 * operands to the tcgen05 kernel by TMA; that is faster than rounding X inside the
 * GEMM, where the f32 X in flight does not fit on chip.  The results are
 * identical to wq_gemm's (same rounding, same accumulation order per output).
 * With WQ_TC_BF16 and Q8_0/Q4_0 weights (the quantised large-n GEMM, e.g. a
 * prompt of many tokens through GGML weights) W is dequantised into the
 * workspace as well, each weight d*q (or d*(q-8)) rounded to the nearest bf16,
 * and the same tcgen05 kernel runs on the bf16 copy; both operands are then
 * within 2^-8 of their exact values, inside the 8e-3 sum|x||w| contract of
 * WQ_TC_BF16.
 * workspace: device memory of at least wq_gemm_workspace_bytes(n, m, k, wtype,
 * flags) bytes, 256-byte aligned, not overlapping any other argument; it is
 * overwritten and may be reused once the stream has passed this call.  When that
 * size is 0 the workspace is not touched and may be NULL.
 * Errors: as wq_gemm, plus WQ_ERR_INVALID_ARG for a missing, misaligned or too
 * small workspace when one is needed.
 */
WQ_API wq_status wq_gemm_ws(int n, int m, int k, int wtype, unsigned flags, const float *X,
                            const void *W, const float *bias, const float *residual, float *Y,
                            void *workspace, size_t workspace_bytes, wq_stream_t stream);

/* Workspace bytes wq_gemm_ws needs for this call when it takes the tensor-core
 * path (WQ_TC_BF16, n > WQ_GEMV_MAX_N): 2*n*k rounded up to 256 (bf16 X), plus
 * 2*m*k rounded up to 256 (bf16 W) for Q8_0/Q4_0 weights; else 0.  0 also for an
 * invalid shape. */
WQ_API size_t wq_gemm_workspace_bytes(int n, int m, int k, int wtype, unsigned flags);

/* Size of the fixed device scratch array behind wq_gemm_noalloc (one per device). */
#define WQ_GEMM_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * wq_gemm_ws without a caller workspace, for callers that may not allocate device
 * memory and have no buffer to lend: code on a path where an allocation could
 * block or fail (a serving loop with a frozen memory budget), a host application
 * that owns the device allocator, a runtime with no allocator.  None of the pages
 * this library follows has a counterpart; it is a library convenience.
 * The bf16 copy of X (and of W, for quantised weights) lives in a statically
 * reserved device array of WQ_GEMM_NOALLOC_SCRATCH_BYTES (16 MiB) per device, so
 * the tensor-core route takes wq_gemm_workspace_bytes(...) <= 16 MiB (bf16
 * weights: n*k <= 8,388,608, e.g. 1500 x 4096).  The call allocates
 * nothing, by any route.  Nothing in the array needs to start at zero: each call
 * writes every byte it later reads.
 * Set-up: every call looks up the array's address on the current device (a
 * host-side lookup that allocates nothing); the first call on a device may load
 * the library's device image there, so make that first call before any stream
 * capture begins.
 * Concurrency: all calls on one device share the one array.  Calls ordered on one
 * stream are safe; calls that may overlap in time (different streams without an
 * ordering between them, or different host threads) race on it and give wrong
 * results: serialise them, or use wq_gemm_ws with a buffer per stream.
 * Routes without scratch (wq_gemm_workspace_bytes(...) == 0) run as wq_gemm.
 * Results are identical to wq_gemm_ws's.
 * Errors: as wq_gemm_ws, plus WQ_ERR_TOO_LARGE when wq_gemm_workspace_bytes(n, m,
 * k, wtype, flags) > WQ_GEMM_NOALLOC_SCRATCH_BYTES (nothing is launched).
 */
WQ_API wq_status wq_gemm_noalloc(int n, int m, int k, int wtype, unsigned flags, const float *X,
                                 const void *W, const float *bias, const float *residual, float *Y,
                                 wq_stream_t stream);

/*
 * Y = epi( LayerNorm(X) . W^T ): the row LayerNorm of cortiq-engine 0.8.49
 * src/gpu_wgpu/nemotron_audio.rs, kernel ae_ln (y = (x - mean) / sqrt(var + 1e-5)
 * * g + b per row, biased variance), fused into the pass that prepares X for the
 * contraction -- the encoder block's "LN, then projection".
 * ln_gb: f32 [2*k] on the device, gamma (k values) then beta (k values), as the
 * kernel's weight buffer.  Everything else as wq_gemm_ws.  The normalised rows are
 * written to the workspace (f32; bf16, rounded to nearest even, on the
 * tensor-core route) and the contraction reads them from there.
 * workspace: at least wq_gemm_ln_workspace_bytes(...) bytes, 256-byte aligned,
 * overlapping no other argument.
 * Errors: as wq_gemm_ws, plus WQ_ERR_INVALID_ARG for a null ln_gb.
 */
WQ_API wq_status wq_gemm_ln_ws(int n, int m, int k, int wtype, unsigned flags, const float *X,
                               const float *ln_gb, const void *W, const float *bias,
                               const float *residual, float *Y, void *workspace,
                               size_t workspace_bytes, wq_stream_t stream);

/* Workspace bytes wq_gemm_ln_ws needs: wq_gemm_workspace_bytes(...) on the
 * tensor-core route, else 4*n*k (the f32 normalised rows), rounded up to 256.
 * 0 for an invalid shape. */
WQ_API size_t wq_gemm_ln_workspace_bytes(int n, int m, int k, int wtype, unsigned flags);

/*
 * Same contract as wq_gemm for small n (1 <= n <= WQ_GEMV_MAX_N): the
 * HBM-bound path that streams each weight byte once (hanzo-ml matvec_q*_gpu).
 * WQ_TC_BF16 is rejected (WQ_ERR_INVALID_ARG).
 */
WQ_API wq_status wq_gemv(int n, int m, int k, int wtype, unsigned flags, const float *X, const void *W,
                  const float *bias, const float *residual, float *Y, wq_stream_t stream);

/*
 * Routed MoE matvec (hanzo-ml moe_matvec_gpu), one launch:
 *   Y[t][s][j] = epi( X[t] . Wbank[ids[t][s]][j]^T ),  t < n_tok, s < topk, j < m.
 * X f32 [n_tok][k]; Wbank byte image [n_experts][m][row_bytes] (16-byte aligned,
 * at least wq_weight_bytes(wtype, n_experts * m, k) bytes); ids int32
 * [n_tok][topk] on the device; bias f32 [n_experts][m] (per expert, WQ_BIAS);
 * residual f32 [n_tok*topk][m] (WQ_RESIDUAL, may equal Y); Y f32 [n_tok][topk][m].
 * The slots are routed in windows of WQ_MOE_WINDOW_SLOTS consecutive slots; each
 * selected expert's weights are read once per window whatever the number of the
 * window's slots routed to it (once per call when n_tok * topk <= 256).
 * n_tok * topk may be any value up to 2^31 - 1.  With topk = 1 and X holding
 * one row per slot this is the page's per-slot form.  An id outside [0, n_experts) leaves that slot's Y row
 * unwritten and sets WQ_ERR_BAD_EXPERT in the device status.
 * Errors: as wq_gemm, plus null ids, topk or n_experts <= 0, n_tok * topk or
 * m * n_experts above 2^31 - 1, WQ_TC_BF16 (all WQ_ERR_INVALID_ARG).
 */
WQ_API wq_status wq_moe_gemv(int n_tok, int topk, int n_experts, int m, int k, int wtype,
                      unsigned flags, const float *X, const void *Wbank, const int32_t *ids,
                      const float *bias, const float *residual, float *Y, wq_stream_t stream);

/* Bytes a W buffer of m rows must hold: 2mk (bf16), 34mk/32 (Q8_0) or 18mk/32
 * (Q4_0), rounded up to a multiple of 16.  0 for an invalid wtype/shape. */
WQ_API size_t wq_weight_bytes(int wtype, int m, int k);

/* out[m][k] (f32, device) = the dequantised weights, bit-exact (d*q and d*(q-8)
 * are exact in f32).  Same W contract as wq_gemm.  Asynchronous on `stream`. */
WQ_API wq_status wq_dequantize(int wtype, int m, int k, const void *W, float *out, wq_stream_t stream);

/* wq_gemm / wq_gemm_ws with the epilogue's contribution scaled by alpha before
 * the residual is added: wavo 0.3.0 src/gpu/mod.rs, Epilogue::Residual(a), which
 * accumulates alpha times the biased product into c:
 *   Y[i][j] = (WQ_RESIDUAL ? residual[i][j] : 0) + alpha * act(X.W^T + bias),
 * the product and sum in f32.  workspace NULL: the routes of wq_gemm; otherwise
 * those of wq_gemm_ws, with the same workspace rules.  alpha = 1 gives results
 * bit-identical to wq_gemm / wq_gemm_ws.
 * Errors: as wq_gemm / wq_gemm_ws, plus WQ_ERR_INVALID_ARG for a NaN or infinite
 * alpha. */
WQ_API wq_status wq_gemm_alpha(int n, int m, int k, int wtype, unsigned flags, float alpha,
                               const float *X, const void *W, const float *bias,
                               const float *residual, float *Y, void *workspace,
                               size_t workspace_bytes, wq_stream_t stream);

/*
 * wq_gemm_alpha with `dual` outputs: wavo 0.3.0 src/gpu/mod.rs, Gpu::linear (a
 * bias with `dual` more values than rows has the first `dual` outputs written a
 * second time after the others, with those biases: one q projection with two
 * position biases) and its gemm test (the extra columns carry no epilogue):
 *   Y[i][j]     = (WQ_RESIDUAL ? residual[i][j] : 0) + alpha * act(X.W^T + bias)[i][j],  j < m
 *   Y[i][m + j] = (X.W^T)[i][j] + bias2[j],                                           j < dual
 * Y and residual: f32 [n][m + dual], row stride m + dual (residual may equal Y;
 * its columns m.. are not read).  bias2: f32 [dual] on the device, required when
 * dual > 0.  0 <= dual <= m; dual = 0 is wq_gemm_alpha.  Both bands come from one
 * accumulation: W is read once, and Y[i][m + j] - bias2[j] is bit-identical to the
 * sum that feeds column j.  workspace NULL: the routes of wq_gemm; otherwise those
 * of wq_gemm_ws, with the same workspace rules.
 * Errors: as wq_gemm_alpha, plus WQ_ERR_INVALID_ARG for dual < 0, dual > m, a null
 * bias2 with dual > 0, or m + dual above 2^31 - 1.
 */
WQ_API wq_status wq_gemm_dual(int n, int m, int k, int dual, int wtype, unsigned flags,
                              float alpha, const float *X, const void *W, const float *bias,
                              const float *bias2, const float *residual, float *Y,
                              void *workspace, size_t workspace_bytes, wq_stream_t stream);

/* Embedding row gather: for t < n_ids and j < k,
 *   out[t][j] = W[ids[t]][j] + pos[t][j] + bias[j]
 * (f32; the dequantised weight, exact in f32, then + pos, then + bias).
 * W: a table of `rows` rows of k weights in format wtype, same contract as
 *    wq_gemm (16-byte aligned; k % 8 == 0 for bf16, k % 32 == 0 for Q8_0/Q4_0).
 * ids: int32 [n_ids].  An id outside [0, rows) leaves row t of out unwritten and
 *    records WQ_ERR_BAD_INDEX in the device status.
 * pos: f32 [n_ids][k] (the page's position rows, one per id) or NULL;
 * bias: f32 [k] or NULL; out: f32 [n_ids][k].
 * Errors: WQ_ERR_INVALID_ARG for n_ids <= 0, rows <= 0, a bad k or wtype, null
 * W, ids or out, W not 16-byte aligned.  Asynchronous on `stream`. */
WQ_API wq_status wq_embed(int n_ids, int rows, int k, int wtype, const void *W,
                          const int32_t *ids, const float *pos, const float *bias, float *out,
                          wq_stream_t stream);

/* Synchronises `stream`, then returns and clears the current device's sticky
 * status word: WQ_OK, WQ_ERR_DEVICE_TIMEOUT, WQ_ERR_BAD_EXPERT or
 * WQ_ERR_BAD_INDEX (the first recorded since the last call); WQ_ERR_CUDA if the
 * synchronisation fails. */
WQ_API wq_status wq_get_device_status(wq_stream_t stream);

/* Static English text for a status code. */
WQ_API const char *wq_status_string(int status);

/* Diagnostics: the number of polls after which a kernel's wait on an mbarrier
 * gives up, records WQ_ERR_DEVICE_TIMEOUT, drains its own copies in flight,
 * releases what it holds and returns.  0 restores the default (about seconds).
 * Affects launches made after the call, on every device. */
WQ_API void wq_set_wait_limit(uint64_t polls);

#ifdef __cplusplus
}
#endif
#endif /* WQ_H */
