"""wq_gemm_ln_ws: Y = epi(LayerNorm(X) . W^T) through the C ABI, against the f64
oracle's LayerNorm (cortiq-engine ae_ln) followed by its contraction.

The reference feeds the oracle's normalised rows, rounded to f32, to the oracle's
GEMM; the library normalises in f32 (fixed-order warp reductions), so the two
differ by a few f32 ulps per normalised value -- far inside the tolerances (1e-5
sum|x||w| on the exact paths, 8e-3 on the tensor-core route).
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu
BF16, Q8_0, Q4_0 = wq.WQ_BF16, wq.WQ_Q8_0, wq.WQ_Q4_0
BIAS, GELU, RES, TC = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL, wq.WQ_TC_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run_ln(oracle_mod, n, m, k, wtype, flags, seed, tau):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k), 3.0) + np.float32(1.5)   # rows with a mean and a scale
    gb = np.concatenate([synth.normal_f32(g, (k,), 0.1) + np.float32(1.0),
                         synth.normal_f32(g, (k,), 0.1)])
    img = synth.draw_weights(g, wtype, m, k)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & RES else None
    need = wq.wq_gemm_ln_workspace_bytes(n, m, k, wtype, flags)
    work = torch.empty(need, dtype=torch.uint8, device="cuda")
    Y = Guarded(n * m)
    st = wq.wq_gemm_ln_ws(n, m, k, wtype, flags, dev(X), dev(gb), weights_dev(img, wtype, m, k),
                          dev(bias) if bias is not None else None,
                          dev(R) if R is not None else None, Y.view, work, need)
    wq.check(st, "wq_gemm_ln_ws")
    torch.cuda.synchronize()
    status_ok()
    Xln = oracle_mod.layer_norm(X, gb).astype(np.float32)
    Yref, S = oracle_mod.gemm(n, m, k, wtype, flags & ~TC, Xln, img, bias=bias, residual=R)
    assert_within(Y.result(), Yref, S, tau, gelu=bool(flags & GELU), bias=bias, R=R,
                  what=f"ln wtype={wtype} n={n} m={m} k={k} flags={flags}")


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("n,m,k,flags", [(1, 130, 512, BIAS), (5, 64, 1056, GELU | RES),
                                         (16, 300, 256, BIAS | RES), (40, 200, 320, BIAS | GELU)])
def test_layernorm_exact_paths(oracle_mod, wtype, n, m, k, flags):
    run_ln(oracle_mod, n, m, k, wtype, flags, seed=n + m + wtype, tau=1e-5)


@pytest.mark.parametrize("wtype", [BF16, Q4_0])
@pytest.mark.parametrize("n,m,k,flags", [(100, 256, 1024, BIAS), (300, 520, 1024, BIAS | GELU),
                                         (1500, 512, 1024, BIAS | RES)])
def test_layernorm_tensor_cores(oracle_mod, wtype, n, m, k, flags):
    run_ln(oracle_mod, n, m, k, wtype, flags | TC, seed=7 * n + wtype, tau=8e-3)
