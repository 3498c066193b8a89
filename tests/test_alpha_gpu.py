"""GPU parity of wq_gemm_alpha: wavo's Epilogue::Residual(a), c += alpha (a W^T + b),
Y = R + alpha * act(X.W^T + bias), on every route (GEMV, f32-FMA GEMM, tensor-core
GEMM with and without a workspace), against the oracle with the same alpha; alpha =
1 must reproduce wq_gemm / wq_gemm_ws bit for bit."""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BIAS, GELU, RES, TC = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL, wq.WQ_TC_BF16


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def draw(n, m, k, wtype, seed):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wtype, m, k)
    b = synth.normal_f32(g, (m,), 0.1)
    R = synth.normal_f32(g, (n, m))
    return X, img, b, R


def run(n, m, k, wtype, flags, alpha, X, img, b, R, ws):
    """One call with a separate residual buffer (so that every schedule, including
    the helper schedule that parks partial sums in Y, can run); alpha None: the
    plain entry point."""
    out = Guarded(n * m)
    Wd, Rd = weights_dev(img, wtype, m, k), dev(R)
    work, need = None, 0
    if ws:
        need = wq.wq_gemm_workspace_bytes(n, m, k, wtype, flags)
        work = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    if alpha is None:
        if ws:
            st = wq.wq_gemm_ws(n, m, k, wtype, flags, dev(X), Wd, dev(b), Rd, out.view, work, need)
        else:
            st = wq.wq_gemm(n, m, k, wtype, flags, dev(X), Wd, dev(b), Rd, out.view)
    else:
        st = wq.wq_gemm_alpha(n, m, k, wtype, flags, alpha, dev(X), Wd, dev(b), Rd, out.view,
                              work, need)
    wq.check(st, "wq_gemm_alpha")
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


ROUTES = [  # (n, m, k, wtype, flags, workspace, tau)
    ((3, 640, 1024, wq.WQ_Q4_0), BIAS | GELU | RES, False, 1e-5),     # GEMV, tensor-core mma
    ((5, 300, 520, wq.WQ_BF16), BIAS | RES, False, 1e-5),             # GEMV, f32 stream kernel
    ((48, 200, 256, wq.WQ_Q8_0), BIAS | GELU | RES, False, 1e-5),     # f32-FMA GEMM
    ((300, 520, 1032, wq.WQ_BF16), BIAS | GELU | RES | TC, False, 8e-3),  # tcgen05, X inside
    ((1400, 3000, 264, wq.WQ_BF16), BIAS | RES | TC, True, 8e-3),     # SM-pair schedule
    ((700, 1000, 2048, wq.WQ_Q4_0), BIAS | RES | TC, True, 8e-3),     # helper schedule, quantised W
]


@pytest.mark.parametrize("alpha", [0.5, -2.0, 0.0])
@pytest.mark.parametrize("route", range(len(ROUTES)))
def test_alpha_matches_oracle(oracle_mod, route, alpha):
    (n, m, k, wtype), flags, ws, tau = ROUTES[route]
    X, img, b, R = draw(n, m, k, wtype, seed=route * 13 + 1)
    Y = run(n, m, k, wtype, flags, alpha, X, img, b, R, ws)
    cols = (0, min(m, 256))
    Yref, S = oracle_mod.gemm(n, m, k, wtype, flags & ~TC, X, img, bias=b, residual=R,
                              alpha=alpha, rows=cols)
    j0, j1 = cols
    assert_within(Y[:, j0:j1], Yref[:, j0:j1], S[:, j0:j1], tau, gelu=bool(flags & GELU),
                  bias=abs(alpha) * b[j0:j1], R=R[:, j0:j1],
                  what=f"alpha={alpha} route={ROUTES[route]}")


@pytest.mark.parametrize("route", range(len(ROUTES)))
def test_alpha_one_is_the_plain_call(route):
    (n, m, k, wtype), flags, ws, _ = ROUTES[route]
    X, img, b, R = draw(n, m, k, wtype, seed=route * 13 + 2)
    Y1 = run(n, m, k, wtype, flags, 1.0, X, img, b, R, ws)
    Y0 = run(n, m, k, wtype, flags, None, X, img, b, R, ws)
    assert (Y1.view(np.int32) == Y0.view(np.int32)).all()
