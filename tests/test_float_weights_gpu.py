"""GPU parity for wavo's F16 and F32 weight types (wavo 0.3.0 src/gpu/mod.rs,
Linear, pipeline index 0 for F32 and 1 for F16) on every route that takes them: the
weight-streaming GEMV and MoE, the f32-FMA GEMM (tiled and cluster split-k),
dequantize, the embedding gather and the tensor-core workspace GEMM (elements
rounded to bf16 there, like d*q).  The f32 routes are held to 1e-5 sum|x||w|."""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

F16, F32 = wq.WQ_F16, wq.WQ_F32
BIAS, GELU, RES, TC = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL, wq.WQ_TC_BF16
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def gemm_case(oracle_mod, n, m, k, wtype, flags, seed, entry="gemm", cols=None, tau=TAU):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wtype, m, k, std=0.05)
    b = synth.normal_f32(g, (m,), 0.1)
    R = synth.normal_f32(g, (n, m))
    out = Guarded(n * m)
    args = (n, m, k, wtype, flags, dev(X), weights_dev(img, wtype, m, k), dev(b), dev(R), out.view)
    if entry == "gemv":
        st = wq.wq_gemv(*args)
    elif entry == "ws":
        need = wq.wq_gemm_workspace_bytes(n, m, k, wtype, flags)
        work = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = wq.wq_gemm_ws(*args, work, need)
    else:
        st = wq.wq_gemm(*args)
    wq.check(st, entry)
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n, m)
    j0, j1 = cols or (0, m)
    Yref, S = oracle_mod.gemm(n, m, k, wtype, flags & ~TC, X, img, bias=b, residual=R,
                              rows=(j0, j1))
    assert_within(Y[:, j0:j1], Yref[:, j0:j1], S[:, j0:j1], tau, gelu=bool(flags & GELU),
                  bias=b[j0:j1], R=R[:, j0:j1], what=f"{entry} wtype={wtype} {n}x{m}x{k}")
    if flags & TC:  # the arithmetic apart from the roundings of both operands
        Yr, Sr = oracle_mod.gemm(n, m, k, wtype, flags & ~TC, X, img, bias=b, residual=R,
                                 rows=(j0, j1), round_x=True, round_w=True)
        assert_within(Y[:, j0:j1], Yr[:, j0:j1], Sr[:, j0:j1], (k / 16 + 32) * 2.0 ** -23,
                      gelu=bool(flags & GELU), bias=b[j0:j1], R=R[:, j0:j1])


@pytest.mark.parametrize("wtype", [F16, F32])
@pytest.mark.parametrize("n", [1, 3, 8, 13])
def test_float_weights_gemv(oracle_mod, wtype, n):
    gemm_case(oracle_mod, n, 777, 1032, wtype, BIAS | GELU | RES, seed=n + wtype, entry="gemv")


@pytest.mark.parametrize("wtype", [F16, F32])
@pytest.mark.parametrize("shape", [(32, 96, 264), (48, 300, 520), (200, 130, 1000)])
def test_float_weights_fma_gemm(oracle_mod, wtype, shape):
    """n > 16 without WQ_TC_BF16: the tiled f32-FMA kernel or, under one wave, the
    cluster split-k kernel."""
    n, m, k = shape
    gemm_case(oracle_mod, n, m, k, wtype, BIAS | RES, seed=n + m + wtype)


@pytest.mark.parametrize("wtype", [F16, F32])
@pytest.mark.parametrize("shape", [(300, 520, 1032), (1500, 3000, 264)])
def test_float_weights_tensor_cores(oracle_mod, wtype, shape):
    n, m, k = shape
    gemm_case(oracle_mod, n, m, k, wtype, BIAS | GELU | TC, seed=n + wtype, entry="ws",
              cols=(0, min(m, 300)), tau=8e-3)


@pytest.mark.parametrize("wtype", [F16, F32])
def test_float_weights_moe(oracle_mod, wtype):
    n_tok, topk, E, m, k = 16, 6, 64, 140, 520
    g = synth.rng(40 + wtype)
    bank = synth.draw_weights(g, wtype, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = synth.moe_ids(g, n_tok, topk, E)
    bias = synth.normal_f32(g, (E, m), 0.1)
    R = synth.normal_f32(g, (n_tok * topk, m))
    out = Guarded(n_tok * topk * m)
    st = wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, BIAS | GELU | RES, dev(X),
                        weights_dev(bank, wtype, E * m, k), dev(ids), dev(bias), dev(R), out.view)
    wq.check(st, "wq_moe_gemv")
    torch.cuda.synchronize()
    status_ok()
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wtype, BIAS | GELU | RES, X, bank, ids,
                             bias=bias, residual=R)
    Y = out.result().reshape(n_tok * topk, m)
    assert_within(Y, Yref, S, TAU, gelu=True, R=R, what=f"moe wtype={wtype}")


@pytest.mark.parametrize("wtype", [F16, F32])
def test_float_weights_dequantize_and_embed_bit_exact(oracle_mod, wtype):
    rows, k = 333, 136
    g = synth.rng(50 + wtype)
    img = synth.draw_weights(g, wtype, rows, k, std=4.0)
    Wd = weights_dev(img, wtype, rows, k)
    out = torch.empty(rows * k, device="cuda")
    wq.check(wq.wq_dequantize(wtype, rows, k, Wd, out), "wq_dequantize")
    want = oracle_mod.dequant(wtype, rows, k, img)
    assert (out.cpu().numpy().reshape(rows, k).astype(np.float64) == want).all()
    ids = np.array([0, 332, 17, 17], np.int32)
    emb = torch.empty(len(ids) * k, device="cuda")
    wq.check(wq.wq_embed(len(ids), rows, k, wtype, Wd, dev(ids), None, None, emb), "wq_embed")
    torch.cuda.synchronize()
    status_ok()
    assert (emb.cpu().numpy().reshape(len(ids), k).astype(np.float64) == want[ids]).all()
