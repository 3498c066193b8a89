"""GPU parity of the tensor-core GEMV for bf16-pair weights (gemv_bf16.cu), which
wq_gemv and the small-n wq_gemm take for bf16 weights when k % 256 == 0
(cortiq-engine 0.8.49 AudioEncoder::gemm: W as bf16 pairs; hanzo-ml-style small-n
calls).  X is scaled by a power of two per token and 64-element slice and split
into three bf16 terms; every check is against the f64 oracle at tau = 1e-5.
The group sizes of the kernel (2, 4, 6 or 8 tiles of 16 rows per CTA, one or two
halves of eight tokens) follow m and n, so the shapes below reach each of them."""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16 = wq.WQ_BF16
BIAS, GELU, RES = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run(n, m, k, flags, X, img, bias=None, R=None, fn=None):
    fn = fn or wq.wq_gemv
    out = Guarded(n * m)
    st = fn(n, m, k, BF16, flags, dev(X), weights_dev(img, BF16, m, k),
            dev(bias) if bias is not None else None, dev(R) if R is not None else None, out.view)
    wq.check(st, fn.__name__)
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def check(oracle_mod, n, m, k, flags, X, img, bias=None, R=None, rows=None, what="", fn=None):
    Y = run(n, m, k, flags, X, img, bias, R, fn)
    assert np.isfinite(Y).all()
    Yref, S = oracle_mod.gemm(n, m, k, BF16, flags, X, img, bias=bias, residual=R, rows=rows)
    sl = slice(*rows) if rows else slice(None)
    assert_within(Y[:, sl], Yref[:, sl], S[:, sl], TAU, gelu=bool(flags & GELU),
                  bias=None if bias is None else bias[sl], R=None if R is None else R[:, sl],
                  what=what)


# m and n that select each group size: tiles per SM <= 2, 4, 6 and more (8), with
# one half of tokens (n <= 8) or two (n <= 16); ragged m and n in each.
GROUPS = [(1, 4000, 1024), (3, 9000, 512), (8, 14336, 256), (2, 20000, 768),
          (9, 3000, 512), (16, 9000, 256), (12, 515, 1280)]


@pytest.mark.parametrize("n,m,k", GROUPS)
def test_group_sizes(oracle_mod, n, m, k):
    g = synth.rng(n * 7 + m)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, BF16, m, k)
    bias = synth.normal_f32(g, (m,), 0.1)
    R = synth.normal_f32(g, (n, m))
    check(oracle_mod, n, m, k, BIAS | RES, X, img, bias, R, what=f"bf16 mma n={n} m={m} k={k}")


@pytest.mark.parametrize("n", [1, 5, 12])
def test_wide_range_x(oracle_mod, n):
    """X spanning 2^-60 .. 2^60, a zero slice, a slice near 2^100 and an f32
    subnormal: the power-of-two scaling per 64-element slice keeps the three terms
    normal and every product exact to the tolerance."""
    m, k = 300, 1024
    g = synth.rng(190 + n)
    X = synth.normal_f32(g, (n, k)) * np.exp2(g.integers(-60, 61, size=(n, k))).astype(np.float32)
    X[:, 64:128] = 0.0                                                         # a zero slice
    X[:, 256:320] = synth.normal_f32(g, (n, 64)) * np.float32(2.0 ** 100)    # a huge slice
    X[:, 400] = np.float32(1e-40)                                              # f32 subnormal
    img = synth.draw_weights(g, BF16, m, k)
    check(oracle_mod, n, m, k, 0, X, img, what=f"wide-range X n={n}")


@pytest.mark.parametrize("scale", [2.0 ** -120, 2.0 ** -100, 2.0 ** 110])
def test_tiny_and_huge_x(oracle_mod, scale):
    """X entirely near the bottom (below where an unscaled third bf16 term would be
    subnormal) or near the top of the f32 range."""
    n, m, k = 3, 200, 768
    g = synth.rng(int(np.log2(scale)) + 500)
    X = (synth.normal_f32(g, (n, k)).astype(np.float64) * scale).astype(np.float32)
    img = synth.draw_weights(g, BF16, m, k)
    check(oracle_mod, n, m, k, 0, X, img, what=f"X scaled by 2^{np.log2(scale):.0f}")


def test_exact_integers(oracle_mod):
    """Small integers in X and W: every product and partial sum is exact, so the
    result equals the oracle's bit for bit."""
    n, m, k = 4, 160, 512
    g = synth.rng(77)
    X = g.integers(-8, 9, size=(n, k)).astype(np.float32)
    Wf = g.integers(-8, 9, size=(m, k)).astype(np.float32)
    img = synth.bf16_pairs((Wf.view(np.uint32) >> 16).astype(np.uint16))  # exact in bf16
    Y = run(n, m, k, 0, X, img)
    Yref, _ = oracle_mod.gemm(n, m, k, BF16, 0, X, img)
    assert (Y == Yref.astype(np.float32)).all()


def test_in_place_residual_and_gelu(oracle_mod):
    n, m, k = 6, 1000, 1024
    g = synth.rng(31)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, BF16, m, k)
    bias = synth.normal_f32(g, (m,), 0.1)
    R = synth.normal_f32(g, (n, m))
    out = Guarded(n * m, R)
    st = wq.wq_gemv(n, m, k, BF16, BIAS | GELU | RES, dev(X), weights_dev(img, BF16, m, k),
                    dev(bias), out.view, out.view)
    wq.check(st, "wq_gemv")
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n, m)
    Yref, S = oracle_mod.gemm(n, m, k, BF16, BIAS | GELU | RES, X, img, bias=bias, residual=R)
    assert_within(Y, Yref, S, TAU, gelu=True, bias=bias, R=R, what="in-place residual")


def test_small_n_gemm_takes_it(oracle_mod):
    """wq_gemm with n <= 16 runs the same kernel."""
    n, m, k = 16, 700, 512
    g = synth.rng(41)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, BF16, m, k)
    bias = synth.normal_f32(g, (m,), 0.1)
    check(oracle_mod, n, m, k, BIAS, X, img, bias, fn=wq.wq_gemm, what="wq_gemm n=16")


def test_bit_identical_reruns():
    n, m, k = 5, 3000, 2048
    g = synth.rng(3)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, BF16, m, k)
    Y1 = run(n, m, k, 0, X, img)
    Y2 = run(n, m, k, 0, X, img)
    assert (Y1.view(np.int32) == Y2.view(np.int32)).all()
