"""Seeded synthetic inputs for the weight-format contraction.

This module only *draws* inputs and *encodes* them in the storage formats the
contraction reads (bf16 pairs, GGML Q8_0 blocks, GGML Q4_0 blocks).  It holds
none of the contraction's arithmetic: no dequantisation, no dot products, no
epilogue.  Both sides of every parity check take their inputs from here: the
f64 oracle under ``oracle/`` and the CUDA library under
``gemv_transformer_gb300/``.  Neither of those imports the other.

Storage formats, as the pages define them:

* bf16 pairs (cortiq-engine 0.8.49, src/gpu_wgpu/nemotron_audio.rs, kernel
  ``ae_gemm``): W is an array of u32 words; word c of row j holds element 2c in
  its low 16 bits and element 2c+1 in its high 16 bits.  On a little-endian
  machine that is byte-identical to row-major bf16 ``[m][k]``.
* Q8_0 (hanzo-ml 0.11.13, src/wgpu_backend.rs, ``matvec_q8_0_gpu``, 34-byte
  blocks; wavo 0.3.0, src/gpu/mod.rs, ``upload_linear`` and the test
  quantiser, which writes the f16 scale with ``to_le_bytes``): per 32 weights
  along k, a little-endian f16 scale ``d`` then 32 int8 ``qs``; value d*q.
* Q4_0 (hanzo-ml 0.11.13, ``matvec_q4_0_gpu``, which reads the blocks as stored; the
  nibble order is not on the pages, it is the one the Q4_0 workload fixes): per
  32 weights, a little-endian f16 scale then 16 bytes; element j < 16 is the
  low nibble of byte j, element j >= 16 the high nibble of byte j-16; value
  d*(q-8).

Every generator takes a seed; the same seed gives the same bytes.
"""
from __future__ import annotations

import numpy as np

WTYPE_BF16 = 0
WTYPE_Q8_0 = 1
WTYPE_Q4_0 = 2
WTYPE_F16 = 3
WTYPE_F32 = 4

QK = 32  # weights per quantisation block along k
Q8_0_BLOCK_BYTES = 34
Q4_0_BLOCK_BYTES = 18


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_f32(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return (g.standard_normal(shape) * std).astype(np.float32)


def f16_bits(values) -> np.ndarray:
    """IEEE binary16 bit patterns of ``values`` (numpy's round-to-nearest-even)."""
    return np.asarray(values, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits_rne(values) -> np.ndarray:
    """bf16 bit patterns of f32 ``values`` rounded to nearest, ties to even.

    Used only to *draw* bf16 weights ("W = bf16(N(0, sigma))").
    """
    u = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(values, dtype=np.float32))
    r[nan] = 0x7FC0
    return r


def bf16_pairs(bits: np.ndarray) -> np.ndarray:
    """Pack bf16 bit patterns ``[m][k]`` (k even) into the u32-pair byte image.

    Word c of a row = element 2c (low half) | element 2c+1 << 16, stored
    little-endian.  Returns ``uint8 [m][2k]``.
    """
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    m, k = bits.shape
    assert k % 2 == 0
    lo = bits[:, 0::2].astype(np.uint32)
    hi = bits[:, 1::2].astype(np.uint32)
    words = (lo | (hi << 16)).astype("<u4")
    return words.view(np.uint8).reshape(m, 2 * k)


def encode_q8_0(d_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Q8_0 byte image from scale bits ``[m][k/32]`` and int8 ``q [m][k]``."""
    d_bits = np.ascontiguousarray(d_bits, dtype=np.uint16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    m, k = q.shape
    nb = k // QK
    assert d_bits.shape == (m, nb) and k % QK == 0
    out = np.empty((m, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0] = (d_bits & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d_bits >> 8).astype(np.uint8)
    out[:, :, 2:] = q.view(np.uint8).reshape(m, nb, QK)
    return out.reshape(m, nb * Q8_0_BLOCK_BYTES)


def encode_q4_0(d_bits: np.ndarray, q4: np.ndarray) -> np.ndarray:
    """Q4_0 byte image from scale bits ``[m][k/32]`` and 4-bit codes ``q4 [m][k]`` in 0..15."""
    d_bits = np.ascontiguousarray(d_bits, dtype=np.uint16)
    q4 = np.ascontiguousarray(q4, dtype=np.uint8)
    m, k = q4.shape
    nb = k // QK
    assert d_bits.shape == (m, nb) and k % QK == 0
    assert int(q4.max(initial=0)) < 16
    blk = q4.reshape(m, nb, QK)
    out = np.empty((m, nb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0] = (d_bits & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d_bits >> 8).astype(np.uint8)
    out[:, :, 2:] = blk[:, :, :16] | (blk[:, :, 16:] << 4)
    return out.reshape(m, nb * Q4_0_BLOCK_BYTES)


def weight_bytes(wtype: int, m: int, k: int) -> int:
    if wtype == WTYPE_BF16:
        return 2 * m * k
    if wtype == WTYPE_Q8_0:
        return Q8_0_BLOCK_BYTES * m * (k // QK)
    if wtype == WTYPE_Q4_0:
        return Q4_0_BLOCK_BYTES * m * (k // QK)
    if wtype == WTYPE_F16:
        return 2 * m * k
    if wtype == WTYPE_F32:
        return 4 * m * k
    raise ValueError(wtype)


def draw_bf16_weights(g, m, k, std):
    """bf16 W ``[m][k]`` = bf16_rne(N(0, std)) as the u32-pair byte image."""
    return bf16_pairs(bf16_bits_rne(normal_f32(g, (m, k), std)))


def draw_q8_0_weights(g, m, k, d_lo=1e-3, d_hi=1e-2, q_lo=-127, q_hi=127):
    """Q8_0 W: d = f16(U[d_lo, d_hi]), q integer U[q_lo, q_hi]."""
    nb = k // QK
    d = f16_bits(g.uniform(d_lo, d_hi, size=(m, nb)))
    q = g.integers(q_lo, q_hi + 1, size=(m, k), dtype=np.int16).astype(np.int8)
    return encode_q8_0(d, q)


def draw_q4_0_weights(g, m, k, d_lo=1e-3, d_hi=1e-2):
    """Q4_0 W: d = f16(U[d_lo, d_hi]); the 16 nibble bytes uniform over 0..255."""
    nb = k // QK
    d = f16_bits(g.uniform(d_lo, d_hi, size=(m, nb)))
    out = np.empty((m, nb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0] = (d & 0xFF).astype(np.uint8)
    out[:, :, 1] = (d >> 8).astype(np.uint8)
    out[:, :, 2:] = g.integers(0, 256, size=(m, nb, 16), dtype=np.int16).astype(np.uint8)
    return out.reshape(m, nb * Q4_0_BLOCK_BYTES)


def draw_f16_weights(g, m, k, std):
    """W = f16(N(0, std)) (numpy's round-to-nearest-even), the byte image [m][2k]."""
    return f16_bits(normal_f32(g, (m, k), std)).view(np.uint8).reshape(m, 2 * k)


def draw_f32_weights(g, m, k, std):
    """W = N(0, std) in f32, the byte image [m][4k]."""
    return normal_f32(g, (m, k), std).view(np.uint8).reshape(m, 4 * k)


def draw_weights(g, wtype, m, k, std=0.05):
    if wtype == WTYPE_BF16:
        return draw_bf16_weights(g, m, k, std)
    if wtype == WTYPE_Q8_0:
        return draw_q8_0_weights(g, m, k)
    if wtype == WTYPE_Q4_0:
        return draw_q4_0_weights(g, m, k)
    if wtype == WTYPE_F16:
        return draw_f16_weights(g, m, k, std)
    if wtype == WTYPE_F32:
        return draw_f32_weights(g, m, k, std)
    raise ValueError(wtype)


def moe_ids(g, n_tok: int, topk: int, n_experts: int) -> np.ndarray:
    """Per token, ``topk`` distinct expert ids drawn uniformly (partial Fisher-Yates)."""
    assert topk <= n_experts
    ids = np.empty((n_tok, topk), dtype=np.int32)
    for t in range(n_tok):
        perm = np.arange(n_experts, dtype=np.int64)
        for s in range(topk):
            j = s + int(g.integers(0, n_experts - s))
            perm[s], perm[j] = perm[j], perm[s]
            ids[t, s] = perm[s]
    return ids


# ---------------------------------------------------------------------------
# The five workloads.  Each returns a dict of numpy arrays plus the shape and
# flag fields; weights are uint8 byte images in their storage format.
# Flag bits: 1 bias, 2 erf-GELU, 4 residual add (cortiq-engine ``ae_put``).
# ---------------------------------------------------------------------------

FLAG_BIAS, FLAG_GELU, FLAG_RESIDUAL = 1, 2, 4


def workload_bf16_gemm(seed=1, n=32, m=512, k=256):
    """bf16-weight GEMM with bias + GELU, f32 FMA path."""
    g = rng(seed)
    return dict(name=f"bf16_gemm_n{n}_m{m}_k{k}", kind="gemm", wtype=WTYPE_BF16, n=n, m=m, k=k,
                flags=FLAG_BIAS | FLAG_GELU,
                X=normal_f32(g, (n, k)), W=draw_bf16_weights(g, m, k, 0.05),
                bias=normal_f32(g, (m,), 0.1), residual=None)


def workload_q8_0_gemv(seed=2, n=1, m=4096, k=4096):
    """Q8_0 GEMV, no epilogue."""
    g = rng(seed)
    return dict(name=f"q8_0_gemv_n{n}_m{m}_k{k}", kind="gemv", wtype=WTYPE_Q8_0, n=n, m=m, k=k,
                flags=0, W=draw_q8_0_weights(g, m, k), X=normal_f32(g, (n, k)),
                bias=None, residual=None)


def workload_float_gemv(seed=10, wtype=WTYPE_BF16, n=1, m=4096, k=4096):
    """A one-token GEMV through unquantised weights (bf16 pairs, or wavo's F16 / F32
    elements), N(0, 0.03), with a bias: the weight-streaming kernel's workload."""
    g = rng(seed * 10 + wtype)
    tag = {WTYPE_BF16: "bf16", WTYPE_F16: "f16", WTYPE_F32: "f32"}[wtype]
    return dict(name=f"{tag}_gemv_n{n}_m{m}_k{k}", kind="gemv", wtype=wtype, n=n, m=m, k=k,
                flags=FLAG_BIAS, W=draw_weights(g, wtype, m, k, 0.03), X=normal_f32(g, (n, k)),
                bias=normal_f32(g, (m,), 0.1), residual=None)


def workload_q4_0_gemv(seed=3, n=1, m=14336, k=4096):
    """Q4_0 small-batch GEMV with a residual add of Y0."""
    g = rng(seed * 100 + n)
    return dict(name=f"q4_0_gemv_n{n}_m{m}_k{k}", kind="gemv", wtype=WTYPE_Q4_0, n=n, m=m, k=k,
                flags=FLAG_RESIDUAL, W=draw_q4_0_weights(g, m, k), X=normal_f32(g, (n, k)),
                bias=None, residual=normal_f32(g, (n, m)))


def workload_encoder_gemms(seed=4, n=1500, d=1024, inter=4096):
    """The three bf16 GEMMs of an encoder block, tensor-core path with X rounded to bf16.

    qkv: [n, d] x [3d, d]^T + bias; MLP up: [n, d] x [inter, d]^T + bias, GELU;
    MLP down: [n, inter] x [d, inter]^T + bias + residual.
    """
    g = rng(seed)
    out = []
    for tag, m, k, flags in (("qkv", 3 * d, d, FLAG_BIAS),
                             ("up", inter, d, FLAG_BIAS | FLAG_GELU),
                             ("down", d, inter, FLAG_BIAS | FLAG_RESIDUAL)):
        out.append(dict(name=f"bf16_tc_{tag}_n{n}_m{m}_k{k}", kind="gemm_tc", wtype=WTYPE_BF16,
                        n=n, m=m, k=k, flags=flags,
                        X=normal_f32(g, (n, k)), W=draw_bf16_weights(g, m, k, 0.03),
                        bias=normal_f32(g, (m,), 0.1),
                        residual=normal_f32(g, (n, m)) if flags & FLAG_RESIDUAL else None))
    return out


def workload_moe(seed=5, n_experts=64, m=1408, k=2048, n_tok=16, topk=6, wtype=WTYPE_Q4_0):
    """MoE routed GEMV over one weight bank ``[E][m][k]`` (Q4_0 unless ``wtype``
    says otherwise)."""
    g = rng(seed)
    bank = draw_weights(g, wtype, n_experts * m, k).reshape(n_experts, m, -1)
    tag = {WTYPE_Q4_0: "q4_0", WTYPE_Q8_0: "q8_0", WTYPE_BF16: "bf16", WTYPE_F16: "f16",
           WTYPE_F32: "f32"}[wtype]
    return dict(name=f"moe_{tag}_E{n_experts}_m{m}_k{k}_t{n_tok}x{topk}", kind="moe",
                wtype=wtype, n_tok=n_tok, topk=topk, n_experts=n_experts, m=m, k=k,
                flags=0, W=bank, X=normal_f32(g, (n_tok, k)),
                ids=moe_ids(g, n_tok, topk, n_experts), bias=None, residual=None)


def workload_quant_prefill(seed=6, wtype=WTYPE_Q4_0, n=512, m=14336, k=4096):
    """A prompt of n tokens through one quantised projection on the tensor cores
    (the large-n row after the five workloads): X ~ N(0,1), GGML weights as above."""
    g = rng(seed * 10 + wtype)
    tag = "q4_0" if wtype == WTYPE_Q4_0 else "q8_0"
    return dict(name=f"{tag}_tc_prefill_n{n}_m{m}_k{k}", kind="gemm_tc", wtype=wtype, n=n, m=m,
                k=k, flags=0, W=draw_weights(g, wtype, m, k), X=normal_f32(g, (n, k)),
                bias=None, residual=None)


def workload_ln_qkv(seed=7, n=1500, d=1024):
    """The encoder block's first step: row LayerNorm of X, then the fused qkv
    projection with bias on the tensor cores (X with a mean and a scale; gamma
    ~ N(1, 0.1), beta ~ N(0, 0.1))."""
    g = rng(seed)
    return dict(name=f"ln_bf16_tc_qkv_n{n}_m{3 * d}_k{d}", kind="gemm_ln_tc", wtype=WTYPE_BF16,
                n=n, m=3 * d, k=d, flags=FLAG_BIAS, X=normal_f32(g, (n, d), 3.0) + np.float32(1.5),
                ln_gb=np.concatenate([normal_f32(g, (d,), 0.1) + np.float32(1.0),
                                      normal_f32(g, (d,), 0.1)]),
                W=draw_bf16_weights(g, 3 * d, d, 0.03), bias=normal_f32(g, (3 * d,), 0.1),
                residual=None)


def workload_dual_q(seed=9, n=1500, d=1024, dual=True):
    """A q projection whose bias carries a second set of d values (wavo's dual
    outputs: one q with two position biases): 1500 rows of X ~ N(0,1) through a
    bf16 d x d weight (N(0, 0.03)) on the tensor cores, bias and second bias
    N(0, 0.1); Y has 2d columns.  With dual=False the same call without the
    second band."""
    g = rng(seed)
    tag = "dual" if dual else "plain"
    return dict(name=f"{tag}_bf16_tc_q_n{n}_m{d}_k{d}", kind="gemm_dual_tc", wtype=WTYPE_BF16,
                n=n, m=d, k=d, dual=d if dual else 0, flags=FLAG_BIAS, X=normal_f32(g, (n, d)),
                W=draw_bf16_weights(g, d, d, 0.03), bias=normal_f32(g, (d,), 0.1),
                bias2=normal_f32(g, (d,), 0.1), residual=None)


def workload_embed(seed=8, wtype=WTYPE_BF16, rows=32000, k=4096, n_ids=512):
    """The token embedding of a 512-token prompt: rows ids[t] drawn uniformly from
    a vocabulary table (32,000 x 4,096, the table's format as for the weights
    above), plus one position row per token (N(0,1)) and the table's bias
    (N(0, 0.1))."""
    g = rng(seed * 10 + wtype)
    tag = {WTYPE_BF16: "bf16", WTYPE_Q8_0: "q8_0", WTYPE_Q4_0: "q4_0"}[wtype]
    return dict(name=f"embed_{tag}_V{rows}_k{k}_n{n_ids}", kind="embed", wtype=wtype, n=n_ids,
                m=rows, k=k, flags=FLAG_BIAS, W=draw_weights(g, wtype, rows, k),
                ids=g.integers(0, rows, size=n_ids).astype(np.int32),
                X=normal_f32(g, (n_ids, k)), bias=normal_f32(g, (k,), 0.1), residual=None)
