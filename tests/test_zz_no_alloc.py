"""wq_gemm_noalloc (the tensor-core GEMM with its bf16 X in a fixed device array)
against wq_gemm_ws (the same kernels with a caller workspace), through the C ABI.

Two calls in a row on different inputs, each compared with wq_gemm_ws on the same
inputs, so that a second call reading anything left over from the first fails.
Collected last on purpose: it must also pass after every other test has run.
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16, TC = wq.WQ_BF16, wq.WQ_TC_BF16
TAU_TC = 8e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def inputs(seed, n, m, k, flags):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_bf16_weights(g, m, k, 0.03)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & wq.WQ_BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & wq.WQ_RESIDUAL else None
    return X, img, bias, R


def call(fn, n, m, k, flags, X, img, bias, R):
    out = Guarded(n * m)
    args = (n, m, k, BF16, flags, dev(X), weights_dev(img, BF16, m, k),
            None if bias is None else dev(bias), None if R is None else dev(R), out.view)
    if fn is wq.wq_gemm_ws:
        need = wq.wq_gemm_workspace_bytes(n, m, k, BF16, flags)
        work = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        st = fn(*args, work, need)
    else:
        st = fn(*args)
    wq.check(st, fn.__name__)
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def bound(X, img, m, k):
    """sum_k |x||w| per output; the weights are the bf16 values of the pairs image
    (element 2c in the low half of word c, so the u16 view is in element order)."""
    bits = np.ascontiguousarray(img).view(np.uint16).reshape(m, k).astype(np.uint32) << 16
    w = bits.view(np.float32)
    return np.abs(X.astype(np.float64)) @ np.abs(w.astype(np.float64)).T


@pytest.mark.parametrize("shape,flags", [
    ((300, 520, 1032), wq.WQ_BIAS | wq.WQ_GELU),
    ((1500, 1024, 4096), wq.WQ_BIAS | wq.WQ_RESIDUAL),
    ((2048, 256, 4096), 0),  # 2*n*k = the whole 16 MiB array
], ids=["ragged", "encoder-down", "full-scratch"])
def test_noalloc_matches_workspace_entry_point_twice(shape, flags):
    n, m, k = shape
    flags |= TC
    assert 0 < wq.wq_gemm_workspace_bytes(n, m, k, BF16, flags) <= wq.WQ_GEMM_NOALLOC_SCRATCH_BYTES
    for seed in (11, 12):  # two calls in a row, different X and W
        X, img, bias, R = inputs(seed + n, n, m, k, flags)
        Yna = call(wq.wq_gemm_noalloc, n, m, k, flags, X, img, bias, R)
        Yws = call(wq.wq_gemm_ws, n, m, k, flags, X, img, bias, R)
        S = bound(X, img, m, k)
        assert_within(Yna, Yws.astype(np.float64), S, TAU_TC, gelu=bool(flags & wq.WQ_GELU),
                      bias=bias, R=R, what=f"noalloc vs ws {shape} seed {seed}")


def test_noalloc_small_n_routes_like_wq_gemm():
    """n <= WQ_GEMV_MAX_N needs no scratch: the call is wq_gemm's GEMV route."""
    n, m, k = 4, 512, 1024
    X, img, bias, _ = inputs(5, n, m, k, wq.WQ_BIAS)
    flags = wq.WQ_BIAS | TC
    Yna = call(wq.wq_gemm_noalloc, n, m, k, flags, X, img, bias, None)
    Yg = call(wq.wq_gemm, n, m, k, flags, X, img, bias, None)
    assert (Yna.view(np.int32) == Yg.view(np.int32)).all()
