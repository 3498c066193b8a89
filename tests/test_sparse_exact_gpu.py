"""Zero and sparse quantised weights through the tensor-core GEMV and MoE kernels.

A row whose codes all mean zero (Q4_0 code 8, Q8_0 code 0, under a nonzero block
scale) must give exactly 0 (or exactly the bias / residual) whatever X holds,
here X spanning 2^-40..2^40 inside each block with a zero block.  A row with a
single nonzero weight must give that one product within the per-element
tolerance, which leaves no room for error relative to any other element: X is
drawn with magnitudes 2^-40..2^40 across blocks but within a factor of two inside
a block, the range in which the tensor-core kernels keep every element to
better than 2^-20 of itself (their representation of x is relative to the
largest |x| of its 32-block).
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

Q8_0, Q4_0 = wq.WQ_Q8_0, wq.WQ_Q4_0
BIAS, RES = wq.WQ_BIAS, wq.WQ_RESIDUAL
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def sparse_weights(g, wtype, m, k):
    """Rows 0 mod 3: every weight zero (nonzero scales); rows 1 mod 3: one nonzero
    weight at a random column; the rest: random codes."""
    nb = k // 32
    d = synth.f16_bits(g.uniform(1e-3, 1e-2, size=(m, nb)))
    if wtype == Q4_0:
        q = g.integers(0, 16, size=(m, k)).astype(np.uint8)
        q[0::3] = 8
        q[1::3] = 8
        cols = g.integers(0, k, size=q[1::3].shape[0])
        q[1::3][np.arange(cols.size), cols] = g.integers(0, 16, size=cols.size).astype(np.uint8) | 1
        return synth.encode_q4_0(d, q)
    q = g.integers(-127, 128, size=(m, k)).astype(np.int8)
    q[0::3] = 0
    q[1::3] = 0
    cols = g.integers(0, k, size=q[1::3].shape[0])
    q[1::3][np.arange(cols.size), cols] = g.integers(1, 128, size=cols.size).astype(np.int8)
    return synth.encode_q8_0(d, q)


def wide_x(g, n, k):
    """Magnitudes 2^-40..2^40 element by element, and a zero block."""
    X = synth.normal_f32(g, (n, k)) * np.exp2(g.integers(-40, 41, size=(n, k))).astype(np.float32)
    X[:, 32:64] = 0.0
    return X


def blockwise_x(g, n, k):
    """|x| in [2^e, 2^(e+1)) with e drawn per 32-block from -40..40, random signs."""
    e = np.repeat(g.integers(-40, 41, size=(n, k // 32)), 32, axis=1)
    mag = g.uniform(1.0, 2.0, size=(n, k)) * np.exp2(e)
    return (np.where(g.integers(0, 2, size=(n, k)) == 1, mag, -mag)).astype(np.float32)


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("flags", [0, BIAS | RES])
def test_gemv_zero_and_single_weight_rows(oracle_mod, wtype, n, flags):
    m, k = 150, 2048
    g = synth.rng(700 + 10 * n + wtype + flags)
    img = sparse_weights(g, wtype, m, k)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & RES else None
    for X, what in ((wide_x(g, n, k), "wide"), (blockwise_x(g, n, k), "blockwise")):
        out = Guarded(n * m)
        wq.check(wq.wq_gemv(n, m, k, wtype, flags, dev(X), weights_dev(img, wtype, m, k),
                            None if bias is None else dev(bias), None if R is None else dev(R),
                            out.view), "wq_gemv")
        torch.cuda.synchronize()
        status_ok()
        Y = out.result().reshape(n, m)
        Yref, S = oracle_mod.gemm(n, m, k, wtype, flags, X, img, bias=bias, residual=R)
        zero_rows = np.arange(0, m, 3)
        assert (S[:, zero_rows] == 0).all()
        want = np.zeros((n, zero_rows.size), np.float32)
        if bias is not None:
            want = want + bias[zero_rows]
        if R is not None:
            want = want + R[:, zero_rows]
        got = Y[:, zero_rows]
        assert (got.view(np.int32) == want.astype(np.float32).view(np.int32)).all(), \
            f"{what} X: zero-weight rows are not exactly 0 / bias / residual"
        rows = np.arange(m) if what == "blockwise" else np.arange(2, m, 3)  # all, or dense rows
        assert_within(Y[:, rows], Yref[:, rows], S[:, rows], TAU,
                      bias=None if bias is None else bias[rows],
                      R=None if R is None else R[:, rows], what=f"sparse gemv {what} X n={n}")


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
def test_moe_zero_and_single_weight_rows(oracle_mod, wtype):
    n_tok, topk, E, m, k = 6, 3, 5, 90, 1024
    g = synth.rng(760 + wtype)
    bank = sparse_weights(g, wtype, E * m, k).reshape(E, m, -1)
    ids = synth.moe_ids(g, n_tok, topk, E)
    for X, what in ((wide_x(g, n_tok, k), "wide"), (blockwise_x(g, n_tok, k), "blockwise")):
        out = Guarded(n_tok * topk * m)
        wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, 0, dev(X),
                                weights_dev(bank, wtype, E * m, k), dev(ids), None, None,
                                out.view), "wq_moe_gemv")
        torch.cuda.synchronize()
        status_ok()
        Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wtype, 0, X, bank, ids)
        Y = out.result().reshape(Yref.shape)
        zero = S == 0
        assert zero.any()
        assert (Y[zero] == 0).all(), f"{what} X: zero-weight rows are not exactly 0"
        cols = np.arange(m) if what == "blockwise" else np.arange(2, m, 3)
        assert_within(Y[:, cols], Yref[:, cols], S[:, cols], TAU, what=f"sparse moe {what} X")
