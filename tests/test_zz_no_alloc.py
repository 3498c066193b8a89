"""wq_gemm_noalloc (the tensor-core GEMM with its bf16 X in a fixed device array)
against wq_gemm_ws (the same kernels with a caller workspace), through the C ABI.

Both entry points run the same kernels on the same inputs, so their outputs must
be bit-identical.  Two calls in a row on different inputs, each compared with
wq_gemm_ws on the same inputs, so that a second call reading anything left over
from the first (or a misplaced or stale part of the array) fails.  A Q4_0 case
puts the bf16 copy of W in the array after X's.  Collected last on purpose: it
must also pass after every other test has run.
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16, Q4_0, TC = wq.WQ_BF16, wq.WQ_Q4_0, wq.WQ_TC_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def inputs(seed, n, m, k, flags, wtype=BF16):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    if wtype == BF16:
        img = synth.draw_bf16_weights(g, m, k, 0.03)
    else:
        img = synth.draw_q4_0_weights(g, m, k)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & wq.WQ_BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & wq.WQ_RESIDUAL else None
    return X, img, bias, R


def call(fn, n, m, k, flags, X, img, bias, R, wtype=BF16):
    out = Guarded(n * m)
    args = (n, m, k, wtype, flags, dev(X), weights_dev(img, wtype, m, k),
            None if bias is None else dev(bias), None if R is None else dev(R), out.view)
    if fn is wq.wq_gemm_ws:
        need = wq.wq_gemm_workspace_bytes(n, m, k, wtype, flags)
        work = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        st = fn(*args, work, need)
    else:
        st = fn(*args)
    wq.check(st, fn.__name__)
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def same_bits(a, b, what):
    ia, ib = a.view(np.int32), b.view(np.int32)
    bad = np.flatnonzero(ia != ib)
    assert bad.size == 0, f"{what}: {bad.size} elements differ, first at {bad[0]}"


@pytest.mark.parametrize("shape,flags,wtype", [
    ((300, 520, 1032), wq.WQ_BIAS | wq.WQ_GELU, BF16),
    ((1500, 1024, 4096), wq.WQ_BIAS | wq.WQ_RESIDUAL, BF16),
    ((2048, 256, 4096), 0, BF16),  # 2*n*k = the whole 16 MiB array
    ((200, 1408, 2048), wq.WQ_BIAS, Q4_0),  # bf16 X, then bf16 W, in the array
], ids=["ragged", "encoder-down", "full-scratch", "q4_0-w-in-array"])
def test_noalloc_matches_workspace_entry_point_twice(shape, flags, wtype):
    n, m, k = shape
    flags |= TC
    need = wq.wq_gemm_workspace_bytes(n, m, k, wtype, flags)
    assert 0 < need <= wq.WQ_GEMM_NOALLOC_SCRATCH_BYTES
    if wtype != BF16:
        assert need > 2 * n * k  # the W copy is in the array too
    for seed in (11, 12):  # two calls in a row, different X and W
        X, img, bias, R = inputs(seed + n, n, m, k, flags, wtype)
        Yna = call(wq.wq_gemm_noalloc, n, m, k, flags, X, img, bias, R, wtype)
        Yws = call(wq.wq_gemm_ws, n, m, k, flags, X, img, bias, R, wtype)
        assert np.isfinite(Yws).all()
        same_bits(Yna, Yws, f"noalloc vs ws {shape} seed {seed}")


def test_noalloc_rejects_oversize():
    """A request whose scratch exceeds the array is refused before any launch."""
    n, m, k = 4096, 256, 4096  # 2*n*k = 32 MiB
    flags = TC
    assert wq.wq_gemm_workspace_bytes(n, m, k, BF16, flags) > wq.WQ_GEMM_NOALLOC_SCRATCH_BYTES
    X = torch.zeros(n * k, device="cuda")
    W = torch.zeros(wq.wq_weight_bytes(BF16, m, k), dtype=torch.uint8, device="cuda")
    Y = torch.full((n * m,), 7.0, device="cuda")
    st = wq.wq_gemm_noalloc(n, m, k, BF16, flags, X, W, None, None, Y)
    assert st == wq.WQ_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert (Y == 7.0).all()


def test_noalloc_small_n_routes_like_wq_gemm():
    """n <= WQ_GEMV_MAX_N needs no scratch: the call is wq_gemm's GEMV route."""
    n, m, k = 4, 512, 1024
    X, img, bias, _ = inputs(5, n, m, k, wq.WQ_BIAS)
    flags = wq.WQ_BIAS | TC
    Yna = call(wq.wq_gemm_noalloc, n, m, k, flags, X, img, bias, None)
    Yg = call(wq.wq_gemm, n, m, k, flags, X, img, bias, None)
    same_bits(Yna, Yg, "noalloc small n vs wq_gemm")
