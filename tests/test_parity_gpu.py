"""GPU parity: the CUDA path, called through the C ABI, against the f64 oracle.

Small shapes span several pieces/tiles and ragged tails; the full workloads are
checked at their real sizes.  Dequantised weights must be bit-exact; Y must be
within tau * L * sum|x||w| (+ epilogue rounding, see helpers.py) with tau = 1e-5
on the f32-FMA paths.  Outputs sit between guard zones that must stay intact.
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16, Q8_0, Q4_0 = wq.WQ_BF16, wq.WQ_Q8_0, wq.WQ_Q4_0
BIAS, GELU, RES = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    yield
    status_ok()


def run_gemm(fn, n, m, k, wtype, flags, X, img, bias=None, R=None, inplace=False):
    Xd, Wd = dev(X), weights_dev(img, wtype, m, k)
    bd = dev(bias) if bias is not None else None
    if inplace:
        out = Guarded(n * m, R)
        Rd = out.view
    else:
        out = Guarded(n * m)
        Rd = dev(R) if R is not None else None
    st = fn(n, m, k, wtype, flags, Xd, Wd, bd, Rd, out.view)
    wq.check(st, fn.__name__)
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def case(seed, wtype, n, m, k, flags):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wtype, m, k)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & RES else None
    return X, img, bias, R


def check_against_oracle(oracle_mod, fn, wtype, n, m, k, flags, seed=0, inplace=False):
    X, img, bias, R = case(seed, wtype, n, m, k, flags)
    Y = run_gemm(fn, n, m, k, wtype, flags, X, img, bias, R, inplace=inplace)
    Yref, S = oracle_mod.gemm(n, m, k, wtype, flags, X, img, bias=bias, residual=R)
    return assert_within(Y, Yref, S, TAU, gelu=bool(flags & GELU), bias=bias, R=R,
                         what=f"{fn.__name__} wtype={wtype} n={n} m={m} k={k} flags={flags}")


# ------------------------------------------------------------------ GEMV --

GEMV_SHAPES = [(1, 1, 32), (1, 37, 64), (2, 130, 96), (3, 513, 4128), (4, 300, 2080),
               (5, 77, 8224), (8, 1000, 512), (9, 64, 256), (16, 129, 4160)]


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
@pytest.mark.parametrize("shape", GEMV_SHAPES)
def test_gemv_quantized(oracle_mod, wtype, shape):
    n, m, k = shape
    check_against_oracle(oracle_mod, wq.wq_gemv, wtype, n, m, k, 0, seed=n * 31 + m)


# k % 256 == 0 takes the tensor-core GEMV (X scaled per 32-block, exact 3-term f16 split).
MMA_SHAPES = [(1, 1, 256), (1, 17, 512), (2, 300, 256), (3, 64, 768), (4, 1000, 1024),
              (5, 33, 256), (6, 100, 512), (8, 129, 2048), (9, 50, 512), (12, 16, 256),
              (16, 257, 1024), (7, 4100, 256)]


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
@pytest.mark.parametrize("shape", MMA_SHAPES)
def test_gemv_tensor_core_path(oracle_mod, wtype, shape):
    n, m, k = shape
    check_against_oracle(oracle_mod, wq.wq_gemv, wtype, n, m, k, BIAS | RES, seed=7 * n + m)


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
@pytest.mark.parametrize("n", [1, 2, 5, 12])
def test_gemv_tensor_core_wide_range_x(oracle_mod, wtype, n):
    """X spanning 2^-60 .. 2^60 (far outside f16), a zero block, a block of values
    near 2^100 and an f32 subnormal: the per-block power-of-two scaling must keep every
    product exact to the tolerance."""
    m, k = 300, 1024
    g = synth.rng(90 + n)
    X = synth.normal_f32(g, (n, k)) * np.exp2(g.integers(-60, 61, size=(n, k))).astype(np.float32)
    X[:, 64:96] = 0.0                                   # a zero block
    X[:, 128:160] = synth.normal_f32(g, (n, 32)) * np.float32(2.0 ** 100)  # huge block
    X[:, 200] = np.float32(1e-40)                       # an f32 subnormal
    img = synth.draw_weights(g, wtype, m, k)
    Y = run_gemm(wq.wq_gemv, n, m, k, wtype, 0, X, img)
    Yref, S = oracle_mod.gemm(n, m, k, wtype, 0, X, img)
    assert_within(Y, Yref, S, TAU, what=f"wide-range X wtype={wtype} n={n}")


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
@pytest.mark.parametrize("n,m,k", [(1, 151936, 4096),   # a vocabulary-sized output projection
                                   (4, 2048, 16384)])   # a long reduction
def test_gemv_at_size_limits(oracle_mod, wtype, n, m, k):
    """Large m and large k through the tensor-core GEMV; the oracle checks bands of
    rows at both ends and in the middle."""
    g = synth.rng(m + k + wtype)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wtype, m, k)
    Y = run_gemm(wq.wq_gemv, n, m, k, wtype, 0, X, img)
    assert np.isfinite(Y).all()
    for j0 in (0, m // 2 - 40, m - 96):
        rows = (j0, j0 + 96)
        Yref, S = oracle_mod.gemm(n, m, k, wtype, 0, X, img, rows=rows)
        sl = slice(*rows)
        assert_within(Y[:, sl], Yref[:, sl], S[:, sl], TAU, what=f"size limits rows {rows}")


@pytest.mark.parametrize("shape", [(1, 1, 8), (1, 37, 16), (2, 130, 1032), (3, 300, 2056),
                                   (4, 65, 4104), (8, 200, 520), (16, 33, 1000)])
def test_gemv_bf16(oracle_mod, shape):
    n, m, k = shape
    check_against_oracle(oracle_mod, wq.wq_gemv, BF16, n, m, k, 0, seed=n * 31 + m)


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("flags", [BIAS, GELU, BIAS | GELU, RES, BIAS | RES, BIAS | GELU | RES])
def test_gemv_epilogues(oracle_mod, wtype, flags):
    check_against_oracle(oracle_mod, wq.wq_gemv, wtype, 3, 261, 2048, flags, seed=flags)


ACTS = [wq.WQ_SILU, wq.WQ_RELU, wq.WQ_TANH]


@pytest.mark.parametrize("act", ACTS, ids=["silu", "relu", "tanh"])
@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("fn,n,k", [(wq.wq_gemv, 3, 512), (wq.wq_gemv, 2, 96),
                                    (wq.wq_gemm, 40, 256)], ids=["gemv-mma", "gemv-ragged", "simt"])
def test_wavo_activations(oracle_mod, act, wtype, fn, n, k):
    """wavo's Silu / Relu / Tanh epilogues, with bias and residual (bias, act, residual)."""
    m = 130
    X, img, bias, R = case(act + n + wtype, wtype, n, m, k, BIAS | RES)
    Y = run_gemm(fn, n, m, k, wtype, BIAS | RES | act, X, img, bias, R)
    Yref, S = oracle_mod.gemm(n, m, k, wtype, BIAS | RES | act, X, img, bias=bias, residual=R)
    assert_within(Y, Yref, S, TAU, gelu=True, bias=bias, R=R,
                  what=f"{fn.__name__} act={act} wtype={wtype} n={n} k={k}")


@pytest.mark.parametrize("act", ACTS, ids=["silu", "relu", "tanh"])
def test_moe_activations(oracle_mod, act):
    nt, tk, E, m, k = 5, 3, 9, 70, 512
    g = synth.rng(act)
    X = synth.normal_f32(g, (nt, k))
    img = synth.draw_weights(g, Q4_0, E * m, k)
    ids = synth.moe_ids(g, nt, tk, E)
    Y = Guarded(nt * tk * m)
    wq.check(wq.wq_moe_gemv(nt, tk, E, m, k, Q4_0, act, dev(X), weights_dev(img, Q4_0, E * m, k),
                            dev(ids), None, None, Y.view), "moe")
    torch.cuda.synchronize()
    status_ok()
    Yref, S = oracle_mod.moe(nt, tk, E, m, k, Q4_0, act, X, img, ids)
    assert_within(Y.result(), Yref, S, TAU, gelu=True, what=f"moe act={act}")


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_gemv_residual_in_place(oracle_mod, wtype):
    check_against_oracle(oracle_mod, wq.wq_gemv, wtype, 4, 190, 1024, BIAS | GELU | RES,
                         seed=9, inplace=True)


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_gemm_small_n_routes_to_gemv(oracle_mod, wtype):
    check_against_oracle(oracle_mod, wq.wq_gemm, wtype, 16, 100, 512, BIAS | GELU, seed=4)


# ------------------------------------------------------------ SIMT GEMM --

@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
# Grids under one wave take the cluster split-k kernel; (700, 900, 96) fills a
# wave of 64 x 64 tiles and takes the plain tiled kernel.
@pytest.mark.parametrize("shape", [(17, 64, 32), (32, 65, 96), (100, 200, 256), (129, 31, 544),
                                   (17, 40, 8192), (33, 512, 256), (700, 900, 96)])
def test_gemm_simt(oracle_mod, wtype, shape):
    n, m, k = shape
    check_against_oracle(oracle_mod, wq.wq_gemm, wtype, n, m, k, BIAS | GELU, seed=n + m)


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_gemm_simt_residual_in_place(oracle_mod, wtype):
    check_against_oracle(oracle_mod, wq.wq_gemm, wtype, 70, 130, 160 if wtype == BF16 else 192,
                         BIAS | RES, seed=3, inplace=True)


def test_gemm_bf16_ragged_k(oracle_mod):
    check_against_oracle(oracle_mod, wq.wq_gemm, BF16, 40, 72, 200, BIAS, seed=8)


# ---------------------------------------------------------------- dequant --

@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("mk", [(1, 32), (7, 96), (300, 4128)])
def test_dequantize_bit_exact(oracle_mod, wtype, mk):
    m, k = mk
    img = synth.draw_weights(synth.rng(m + k), wtype, m, k)
    out = Guarded(m * k)
    wq.check(wq.wq_dequantize(wtype, m, k, weights_dev(img, wtype, m, k), out.view))
    got = out.result().reshape(m, k)
    want = oracle_mod.dequant(wtype, m, k, img)
    assert (got.astype(np.float64) == want).all()


def test_dequantize_hand_blocks(oracle_mod):
    """The worked Q8_0 codes under a subnormal and a negative scale, and all Q4_0 codes."""
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(2, 128)
    for dbits, unit in ((0x0001, 2.0 ** -24), (0xBC00, -1.0), (0x2000, 2.0 ** -7)):
        img = synth.encode_q8_0(np.full((2, 4), dbits, np.uint16), codes)
        out = Guarded(256)
        wq.check(wq.wq_dequantize(Q8_0, 2, 128, weights_dev(img, Q8_0, 2, 128), out.view))
        assert (out.result().reshape(2, 128) == codes.astype(np.float64) * unit).all()
    q4 = (np.arange(32)[None, :] + np.arange(16)[:, None]) % 16
    img = synth.encode_q4_0(np.full((16, 1), 0x4000, np.uint16), q4.astype(np.uint8))
    out = Guarded(16 * 32)
    wq.check(wq.wq_dequantize(Q4_0, 16, 32, weights_dev(img, Q4_0, 16, 32), out.view))
    assert (out.result().reshape(16, 32) == 2.0 * (q4 - 8)).all()


# -------------------------------------------------------- exact brute force --

@pytest.mark.parametrize("fn", [wq.wq_gemv, wq.wq_gemm])
@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_integer_exact(oracle_mod, fn, wtype):
    """Small-integer X and power-of-two scales: every sum is exact in f32, so the
    GPU result must equal the oracle bit for bit in any summation order."""
    n = 5 if fn is wq.wq_gemv else 40
    m, k = 70, 256
    g = synth.rng(77)
    X = g.integers(-3, 4, size=(n, k)).astype(np.float32)
    if wtype == BF16:
        img = synth.bf16_pairs(synth.bf16_bits_rne((g.integers(-8, 9, size=(m, k)) * 0.5)
                                                   .astype(np.float32)))
    else:
        d = synth.f16_bits(np.ldexp(1.0, g.integers(-6, -2, size=(m, k // 32))))
        img = (synth.encode_q8_0(d, g.integers(-128, 128, size=(m, k)).astype(np.int8))
               if wtype == Q8_0 else
               synth.encode_q4_0(d, g.integers(0, 16, size=(m, k)).astype(np.uint8)))
    Y = run_gemm(fn, n, m, k, wtype, 0, X, img)
    Yref, _ = oracle_mod.gemm(n, m, k, wtype, 0, X, img)
    assert (Y.astype(np.float64) == Yref).all()


def test_wavo_probe_closed_form():
    """wavo's probe_tensor shape: c[r][j] = j % 32 + r % 32 exactly (both paths)."""
    n, m, k = 130, 64, 32
    a = np.array([[x + r % 32 for x in range(k)] for r in range(n)], np.float32)
    onehot = np.array([[1 if x == j % 32 else 0 for x in range(k)] for j in range(m)])
    img = synth.encode_q8_0(np.full((m, 1), 0x3C00, np.uint16), onehot.astype(np.int8))
    want = np.array([[j % 32 + r % 32 for j in range(m)] for r in range(n)], np.float32)
    Y = run_gemm(wq.wq_gemm, n, m, k, Q8_0, BIAS, a, img, bias=np.zeros(m, np.float32))
    assert (Y == want).all()
    Y = run_gemm(wq.wq_gemv, 16, m, k, Q8_0, BIAS, a[:16], img, bias=np.zeros(m, np.float32))
    assert (Y == want[:16]).all()


# -------------------------------------------------------------------- MoE --

def run_moe(n_tok, topk, E, m, k, wtype, flags, X, bank, ids, bias=None, R=None):
    out = Guarded(n_tok * topk * m)
    st = wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, flags, dev(X),
                        weights_dev(bank, wtype, E * m, k), dev(ids),
                        dev(bias) if bias is not None else None,
                        dev(R) if R is not None else None, out.view)
    wq.check(st, "wq_moe_gemv")
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("cfg", [(1, 1, 1, 33, 64), (3, 2, 5, 70, 256), (16, 6, 64, 140, 2048),
                                 (8, 3, 4, 257, 4160), (32, 8, 16, 40, 96)])
def test_moe(oracle_mod, wtype, cfg):
    n_tok, topk, E, m, k = cfg
    if wtype == BF16:
        k = k + 8 if k % 32 == 0 else k
    g = synth.rng(sum(cfg) + wtype)
    bank = synth.draw_weights(g, wtype, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = synth.moe_ids(g, n_tok, topk, E)
    flags = BIAS | GELU | RES
    bias = synth.normal_f32(g, (E, m), 0.1)
    R = synth.normal_f32(g, (n_tok * topk, m))
    Y = run_moe(n_tok, topk, E, m, k, wtype, flags, X, bank, ids, bias, R).result()
    status_ok()
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wtype, flags, X, bank, ids, bias=bias,
                             residual=R)
    bias_rows = bias[ids.reshape(-1)]
    assert_within(Y.reshape(Yref.shape), Yref, S, TAU, gelu=True, bias=None,
                  R=np.abs(R) + np.abs(bias_rows), what=f"moe {cfg}")


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
def test_moe_many_slots_per_expert(oracle_mod, wtype):
    """About 64 slots per expert: the tensor-core MoE path runs several token passes."""
    n_tok, topk, E, m, k = 32, 8, 4, 70, 512
    g = synth.rng(31 + wtype)
    bank = synth.draw_weights(g, wtype, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = np.stack([g.integers(0, E, size=topk) for _ in range(n_tok)]).astype(np.int32)
    bias = synth.normal_f32(g, (E, m), 0.1)
    Y = run_moe(n_tok, topk, E, m, k, wtype, BIAS, X, bank, ids, bias).result()
    status_ok()
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wtype, BIAS, X, bank, ids, bias=bias)
    assert_within(Y.reshape(Yref.shape), Yref, S, TAU, R=np.abs(bias[ids.reshape(-1)]),
                  what="moe many slots")


def test_moe_repeated_expert_and_bad_id(oracle_mod):
    """A token may route twice to one expert; a bad id sets the device status and
    leaves only its own slot's row unwritten."""
    n_tok, topk, E, m, k = 4, 3, 6, 50, 64
    g = synth.rng(12)
    bank = synth.draw_q4_0_weights(g, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = np.array([[1, 1, 2], [5, 0, 1], [3, 9, 3], [2, 2, 2]], np.int32)  # 9 is out of range
    out = run_moe(n_tok, topk, E, m, k, Q4_0, 0, X, bank, ids)
    assert wq.wq_get_device_status() == wq.WQ_ERR_BAD_EXPERT
    status_ok()  # cleared by the read
    Y = out.result().reshape(n_tok * topk, m)
    bad = 2 * topk + 1
    assert (Y[bad].view(np.int32) == -1).all()
    good = [q for q in range(n_tok * topk) if q != bad]
    ids_ok = ids.copy()
    ids_ok[2, 1] = 0
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, Q4_0, 0, X, bank, ids_ok)
    assert_within(Y[good], Yref[good], S[good], TAU, what="moe repeated ids")


def test_moe_scaled_identity_routing():
    """Expert e = (e+1)*2^-6 * I: Y[t][s] is (ids[t][s]+1)*2^-6 * X[t] rounded once to f32."""
    E, k, n_tok, topk = 8, 64, 5, 3
    imgs = []
    for e in range(E):
        d = np.full((k, k // 32), synth.f16_bits((e + 1) * 2.0 ** -6)[()], np.uint16)
        q = np.zeros((k, k), np.int8)
        np.fill_diagonal(q, 1)
        imgs.append(synth.encode_q8_0(d, q))
    bank = np.stack(imgs)
    g = synth.rng(5)
    X = synth.normal_f32(g, (n_tok, k))
    ids = synth.moe_ids(g, n_tok, topk, E)
    Y = run_moe(n_tok, topk, E, k, k, Q8_0, 0, X, bank, ids).result().reshape(n_tok, topk, k)
    want = (ids[:, :, None] + 1) * 2.0 ** -6 * X[:, None, :].astype(np.float64)
    assert (Y == want.astype(np.float32)).all()


# ------------------------------------------------------------ determinism --

@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_bit_identical_reruns(wtype):
    n, m, k = 8, 1500, 2048
    X, img, bias, _ = case(21, wtype, n, m, k, BIAS)
    Y1 = run_gemm(wq.wq_gemv, n, m, k, wtype, BIAS, X, img, bias)
    Y2 = run_gemm(wq.wq_gemv, n, m, k, wtype, BIAS, X, img, bias)
    assert (Y1.view(np.int32) == Y2.view(np.int32)).all()


# ------------------------------------------------------- bounded waits --

@pytest.mark.parametrize("wtype,n,m,k", [(Q4_0, 4, 14336, 8192),   # tensor-core GEMV
                                         (BF16, 1, 4096, 16384),    # bf16 tensor-core GEMV
                                         (BF16, 1, 4096, 16392)])   # streaming GEMV
def test_wait_limit_expires_without_hang(oracle_mod, wtype, n, m, k):
    """A one-poll wait limit makes the stage waits give up as soon as a stage is not
    yet filled: the kernel records WQ_ERR_DEVICE_TIMEOUT, drains its copies and
    returns; the context stays usable and the next call (default limit) is correct.
    The shapes need many stage refills per CTA, so some wait finds its stage empty
    (each attempt is harmless either way; a few are allowed)."""
    X, img, _, _ = case(5, wtype, n, m, k, 0)
    Xd, Wd = dev(X), weights_dev(img, wtype, m, k)
    Y = torch.zeros(n * m, device="cuda")
    seen = []
    wq.wq_set_wait_limit(1)
    try:
        for _ in range(5):
            wq.check(wq.wq_gemv(n, m, k, wtype, 0, Xd, Wd, None, None, Y))
            seen.append(wq.wq_get_device_status())
            if seen[-1] == wq.WQ_ERR_DEVICE_TIMEOUT:
                break
    finally:
        wq.wq_set_wait_limit(0)
    assert wq.WQ_ERR_DEVICE_TIMEOUT in seen, seen
    assert set(seen) <= {wq.WQ_OK, wq.WQ_ERR_DEVICE_TIMEOUT}
    assert wq.wq_get_device_status() == wq.WQ_OK
    wq.check(wq.wq_gemv(n, m, k, wtype, 0, Xd, Wd, None, None, Y))
    status_ok()
    rows = (0, 256)
    Yref, S = oracle_mod.gemm(n, m, k, wtype, 0, X, img, rows=rows)
    got = Y.cpu().numpy().reshape(n, m)
    assert_within(got[:, :256], Yref[:, :256], S[:, :256], TAU)


@pytest.mark.parametrize("wtype", [Q4_0, BF16])  # tensor-core MoE: quantized / bf16 bank
def test_moe_wait_limit_expires_without_hang(oracle_mod, wtype):
    """The same with the routed MoE kernels, over two routing windows: a wait that
    gives up must not strand the other warps of its CTA at a barrier, in this window
    or the next; the next call (default limit) is correct."""
    n_tok, topk, E, m, k = 64, 8, 8, 4096, 4096
    g = synth.rng(6 + wtype)
    bank = synth.draw_weights(g, wtype, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = synth.moe_ids(g, n_tok, topk, E)
    Xd, Wd, idd = dev(X), weights_dev(bank, wtype, E * m, k), dev(ids)
    Y = torch.zeros(n_tok * topk * m, device="cuda")
    seen = []
    wq.wq_set_wait_limit(1)
    try:
        for _ in range(5):
            wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, 0, Xd, Wd, idd, None, None, Y))
            seen.append(wq.wq_get_device_status())
            if seen[-1] == wq.WQ_ERR_DEVICE_TIMEOUT:
                break
    finally:
        wq.wq_set_wait_limit(0)
    assert wq.WQ_ERR_DEVICE_TIMEOUT in seen, seen
    assert set(seen) <= {wq.WQ_OK, wq.WQ_ERR_DEVICE_TIMEOUT}
    assert wq.wq_get_device_status() == wq.WQ_OK
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, 0, Xd, Wd, idd, None, None, Y))
    status_ok()
    q0, q1 = 300, 306  # slots of the second window
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wtype, 0, X, bank, ids, slots=(q0, q1))
    got = Y.cpu().numpy().reshape(n_tok * topk, m)
    assert_within(got[q0:q1], Yref[q0:q1], S[q0:q1], TAU)
