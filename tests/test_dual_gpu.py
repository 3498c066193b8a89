"""GPU parity of wq_gemm_dual: wavo's dual outputs (wavo 0.3.0 src/gpu/mod.rs,
Gpu::linear with a bias of `dual` more values, and its gemm test).  Columns
j < m of each row of Y take the usual epilogue; columns m + j, j < dual, take
the same sum of output j plus bias2[j], with no activation, alpha or residual.
Every route is checked against the oracle on both bands, at windows that span
the end of the second band; with bias2 = 0 and no epilogue both bands must agree
bit for bit (one accumulation feeds both)."""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import CANARY, Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BIAS, GELU, RES, TC = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL, wq.WQ_TC_BF16
ACTS = wq.WQ_GELU | wq.WQ_SILU | wq.WQ_RELU | wq.WQ_TANH


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def draw(n, m, k, wtype, dual, seed):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wtype, m, k)
    b = synth.normal_f32(g, (m,), 0.1)
    b2 = synth.normal_f32(g, (max(dual, 1),), 0.5)[:dual]
    R = synth.normal_f32(g, (n, m + dual))
    R[:, m:] = np.nan  # the residual's second band is never read
    return X, img, b, b2, R


def workspace(n, m, k, wtype, flags, ws):
    if not ws:
        return None, 0
    need = wq.wq_gemm_workspace_bytes(n, m, k, wtype, flags)
    return torch.empty(max(need, 256), dtype=torch.uint8, device="cuda"), need


def run(n, m, k, dual, wtype, flags, alpha, X, img, b, b2, R, ws, out=None):
    out = out if out is not None else Guarded(n * (m + dual))
    work, need = workspace(n, m, k, wtype, flags, ws)
    st = wq.wq_gemm_dual(n, m, k, dual, wtype, flags, alpha, dev(X), weights_dev(img, wtype, m, k),
                         dev(b), None if dual == 0 else dev(b2),
                         None if R is None else dev(R), out.view, work, need)
    wq.check(st, "wq_gemm_dual")
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m + dual)


def check_bands(oracle_mod, Y, n, m, k, dual, wtype, flags, alpha, X, img, b, b2, R, tau,
                windows, what):
    acts = bool(flags & ACTS)
    for j0, j1 in windows:
        Yref, S = oracle_mod.gemm(n, m, k, wtype, flags & ~TC, X, img, bias=b, residual=R,
                                  alpha=alpha, dual=dual, bias2=b2, rows=(j0, j1))
        assert_within(Y[:, j0:j1], Yref[:, j0:j1], S[:, j0:j1], tau, gelu=acts,
                      bias=abs(alpha) * b[j0:j1], R=None if R is None else R[:, j0:j1],
                      what=f"{what} band 1 [{j0}, {j1})")
        d1 = min(j1, dual)
        if j0 < d1:
            c0, c1 = m + j0, m + d1
            assert_within(Y[:, c0:c1], Yref[:, c0:c1], S[:, c0:c1], tau, bias=b2[j0:d1],
                          what=f"{what} band 2 [{j0}, {d1})")


def windows_of(m, dual, w=96):
    """The first outputs, and outputs either side of the end of the second band."""
    wins = [(0, min(m, w))]
    if dual > 0:
        lo = max(0, dual - w // 2)
        wins.append((lo, min(m, lo + w)))
    return wins


ROUTES = [  # ((n, m, k, wtype), flags, workspace, tau, dual)
    ((3, 640, 1024, wq.WQ_Q4_0), BIAS | GELU | RES, False, 1e-5, 100),    # GEMV, mma
    ((5, 300, 520, wq.WQ_BF16), BIAS | RES, False, 1e-5, 37),              # GEMV, stream kernel
    ((5, 300, 512, wq.WQ_BF16), BIAS | GELU | RES, False, 1e-5, 37),       # GEMV, bf16 mma
    ((9, 200, 96, wq.WQ_F16), BIAS | wq.WQ_SILU, False, 1e-5, 200),        # GEMV, dual = m
    ((48, 200, 256, wq.WQ_Q8_0), BIAS | GELU | RES, False, 1e-5, 77),      # f32-FMA split-k
    ((700, 900, 64, wq.WQ_Q8_0), BIAS | RES, False, 1e-5, 130),            # f32-FMA tiles
    ((300, 520, 1032, wq.WQ_BF16), BIAS | GELU | RES | TC, False, 8e-3, 260),  # tcgen05 per tile
    ((64, 2048, 256, wq.WQ_BF16), BIAS | RES | TC, True, 8e-3, 300),       # one-SM 128 tiles
    ((20, 38400, 1024, wq.WQ_BF16), BIAS | TC, True, 8e-3, 1000),          # one-SM 256 tiles
    ((1400, 3000, 264, wq.WQ_BF16), BIAS | RES | TC, True, 8e-3, 1000),    # SM pairs, 256 wide
    ((1500, 4000, 520, wq.WQ_BF16), BIAS | GELU | TC, True, 8e-3, 1024),   # SM pairs, 192 wide
    ((700, 1000, 2048, wq.WQ_Q4_0), BIAS | RES | TC, True, 8e-3, 500),     # helper clusters
    ((300, 522, 256, wq.WQ_BF16), BIAS | RES | TC, True, 8e-3, 10),        # m % 4: per tile
    ((300, 512, 256, wq.WQ_BF16), BIAS | RES | TC, True, 8e-3, 3),         # row stride % 4
]


@pytest.mark.parametrize("route", range(len(ROUTES)), ids=lambda r: str(ROUTES[r][0]))
def test_dual_matches_oracle(oracle_mod, route):
    (n, m, k, wtype), flags, ws, tau, dual = ROUTES[route]
    X, img, b, b2, R = draw(n, m, k, wtype, dual, seed=route * 7 + 3)
    Rr = R if flags & RES else None
    Y = run(n, m, k, dual, wtype, flags, -0.75, X, img, b, b2, Rr, ws)
    assert np.isfinite(Y).all(), "an output of either band was not written"
    check_bands(oracle_mod, Y, n, m, k, dual, wtype, flags, -0.75, X, img, b, b2, Rr, tau,
                windows_of(m, dual), what=f"route {ROUTES[route][0]}")


@pytest.mark.parametrize("route", range(len(ROUTES)), ids=lambda r: str(ROUTES[r][0]))
def test_dual_bands_bit_identical(route):
    """bias2 = 0, no epilogue, alpha = 1: the second band repeats the first dual
    columns exactly, on every route and schedule."""
    (n, m, k, wtype), flags, ws, _, dual = ROUTES[route]
    X, img, b, _, _ = draw(n, m, k, wtype, dual, seed=route * 7 + 4)
    Y = run(n, m, k, dual, wtype, flags & TC, 1.0, X, img, b, np.zeros(dual, np.float32), None,
            ws)
    assert (Y[:, m:] == Y[:, :dual]).all()


@pytest.mark.parametrize("route", [0, 1, 4, 5, 8], ids=lambda r: str(ROUTES[r][0]))
def test_dual_residual_in_place(oracle_mod, route):
    """residual == Y: the first band adds the old Y; the second band's old values
    (here 1e30) are overwritten, not read."""
    (n, m, k, wtype), flags, ws, tau, dual = ROUTES[route]
    X, img, b, b2, R = draw(n, m, k, wtype, dual, seed=route * 7 + 5)
    R[:, m:] = 1e30
    out = Guarded(n * (m + dual), init=R)
    work, need = workspace(n, m, k, wtype, flags | RES, ws)
    st = wq.wq_gemm_dual(n, m, k, dual, wtype, flags | RES, 0.5, dev(X),
                         weights_dev(img, wtype, m, k), dev(b), dev(b2), out.view, out.view,
                         work, need)
    wq.check(st, "wq_gemm_dual in place")
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n, m + dual)
    check_bands(oracle_mod, Y, n, m, k, dual, wtype, flags | RES, 0.5, X, img, b, b2, R, tau,
                windows_of(m, dual), what=f"in place {ROUTES[route][0]}")


def test_dual_tensor_core_misaligned_y(oracle_mod):
    """Y 4 bytes past a 16-byte boundary (m and the row stride multiples of 4): the
    tensor-core route must fall back to element stores, and write both bands."""
    n, m, k, dual, wtype, flags = 300, 512, 256, 64, wq.WQ_BF16, BIAS | RES | TC
    X, img, b, b2, R = draw(n, m, k, wtype, dual, seed=91)
    count = n * (m + dual)
    buf = torch.full((count + 2 * CANARY + 1,), -1, dtype=torch.int32, device="cuda")
    buf = buf.view(torch.float32)
    Yv = buf[CANARY + 1:CANARY + 1 + count]
    assert Yv.data_ptr() % 16 == 4
    work, need = workspace(n, m, k, wtype, flags, True)
    st = wq.wq_gemm_dual(n, m, k, dual, wtype, flags, 1.0, dev(X), weights_dev(img, wtype, m, k),
                         dev(b), dev(b2), dev(R), Yv, work, need)
    wq.check(st, "wq_gemm_dual misaligned")
    torch.cuda.synchronize()
    status_ok()
    host = buf.view(torch.int32).cpu().numpy()
    assert (host[:CANARY + 1] == -1).all() and (host[CANARY + 1 + count:] == -1).all()
    Y = Yv.cpu().numpy().reshape(n, m + dual)
    check_bands(oracle_mod, Y, n, m, k, dual, wtype, flags, 1.0, X, img, b, b2, R, 8e-3,
                windows_of(m, dual), what="misaligned Y")


WAVO_EPILOGUES = [  # wavo's Epilogue variants as (flags, alpha)
    (BIAS, 1.0), (BIAS | wq.WQ_SILU, 1.0), (BIAS | wq.WQ_RELU, 1.0), (BIAS | RES, 0.5),
    (BIAS | GELU, 1.0), (BIAS | GELU | RES, 1.0), (BIAS | wq.WQ_TANH, 1.0),
]


@pytest.mark.parametrize("wtype", [wq.WQ_F32, wq.WQ_F16, wq.WQ_Q8_0])
@pytest.mark.parametrize("rows", [164, 288])
def test_dual_wavo_gemm_shapes(oracle_mod, rows, wtype):
    """The shapes of wavo's gemm test: 164 or 288 weight rows, k = 96, 64 dual
    outputs, 1, 37, 70 and 2100 activation rows, every epilogue variant, the
    page's three weight types; n > 16 also on the tensor cores (workspace)."""
    k, dual = 96, 64
    for n in (1, 37, 70, 2100):
        X, img, b, b2, R = draw(n, rows, k, wtype, dual, seed=rows + n + 10 * wtype)
        for flags, alpha in WAVO_EPILOGUES:
            tries = [(0, False, 1e-5)] + ([(TC, True, 8e-3)] if n > wq.WQ_GEMV_MAX_N else [])
            for tc, ws, tau in tries:
                Rr = R if flags & RES else None
                Y = run(n, rows, k, dual, wtype, flags | tc, alpha, X, img, b, b2, Rr, ws)
                check_bands(oracle_mod, Y, n, rows, k, dual, wtype, flags, alpha, X, img, b,
                            b2, Rr, tau, [(0, rows)],
                            what=f"wavo rows={rows} n={n} flags={flags | tc}")
