"""GPU parity of the tcgen05 GEMM (WQ_TC_BF16): X is rounded to bf16 in the kernel.

Two checks per case:
  * against the oracle on the UNROUNDED X, tau = 8e-3 (the contract of the path);
  * against the oracle fed bf16(X) (round to nearest even, the oracle's own
    rounding), tau_k = (k/16 + 32) * 2^-23: the tensor core's f32 accumulation
    over k/16 MMA steps plus the rounding inside each step.  This pins the
    kernel's arithmetic apart from the input rounding.
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16 = wq.WQ_BF16
BIAS, GELU, RES, TC = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL, wq.WQ_TC_BF16
TAU_TC = 8e-3


def tau_exact(k):
    return (k / 16 + 32) * 2.0 ** -23


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run_tc(n, m, k, flags, X, img, bias=None, R=None, inplace=False, ws=False):
    """wq_gemm (X rounded inside the GEMM) or, with ws=True, wq_gemm_ws (X rounded
    into a workspace by a separate pass, then both operands by TMA)."""
    if inplace:
        out = Guarded(n * m, R)
        Rd = out.view
    else:
        out = Guarded(n * m)
        Rd = dev(R) if R is not None else None
    args = (n, m, k, BF16, flags | TC, dev(X), weights_dev(img, BF16, m, k),
            dev(bias) if bias is not None else None, Rd, out.view)
    if ws:
        need = wq.wq_gemm_workspace_bytes(n, m, k, BF16, flags | TC)
        assert need >= 2 * n * k
        work = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = wq.wq_gemm_ws(*args, work, need)
    else:
        st = wq.wq_gemm(*args)
    wq.check(st, "wq_gemm(TC)")
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def check_tc(oracle_mod, n, m, k, flags, seed, rows=None, inplace=False, std=0.03, ws=False):
    g = synth.rng(seed)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_bf16_weights(g, m, k, std)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & RES else None
    Y = run_tc(n, m, k, flags, X, img, bias, R, inplace=inplace, ws=ws)
    j0, j1 = rows if rows else (0, m)
    gelu = bool(flags & (GELU | wq.WQ_SILU | wq.WQ_RELU | wq.WQ_TANH))
    for round_x, tau in ((False, TAU_TC), (True, tau_exact(k))):
        Yref, S = oracle_mod.gemm(n, m, k, BF16, flags, X, img, bias=bias, residual=R,
                                  round_x=round_x, rows=(j0, j1))
        assert_within(Y[:, j0:j1], Yref[:, j0:j1], S[:, j0:j1], tau, gelu=gelu,
                      bias=None if bias is None else bias[j0:j1],
                      R=None if R is None else R[:, j0:j1],
                      what=f"tc n={n} m={m} k={k} flags={flags} round_x={round_x}")
    return Y


@pytest.mark.parametrize("ws", [False, True], ids=["fused", "workspace"])
@pytest.mark.parametrize("shape", [(17, 16, 8), (128, 128, 64), (130, 256, 128), (300, 520, 1032),
                                   (257, 300, 200), (1000, 1000, 512), (64, 2048, 256),
                                   (1400, 3000, 264)])
def test_tc_shapes(oracle_mod, shape, ws):
    n, m, k = shape
    check_tc(oracle_mod, n, m, k, BIAS, seed=n + m + k, ws=ws)


@pytest.mark.parametrize("ws", [False, True], ids=["fused", "workspace"])
@pytest.mark.parametrize("flags", [0, BIAS, GELU, BIAS | GELU, RES, BIAS | RES, BIAS | GELU | RES,
                                   BIAS | wq.WQ_SILU, BIAS | wq.WQ_RELU | RES, wq.WQ_TANH | RES])
def test_tc_epilogues(oracle_mod, flags, ws):
    check_tc(oracle_mod, 200, 384, 320, flags, seed=flags, ws=ws)


@pytest.mark.parametrize("ws", [False, True], ids=["fused", "workspace"])
def test_tc_residual_in_place_ragged_m(oracle_mod, ws):
    check_tc(oracle_mod, 150, 203, 264, BIAS | RES, seed=3, inplace=True, ws=ws)


@pytest.mark.parametrize("cols", [(0, 300), (3700, 4000)])
def test_tc_pair_schedule_192_wide_ragged(oracle_mod, cols):
    """256 x 192 SM-pair tiles (chosen when 256-wide tiles would need as many
    rounds): ragged rows (1500), columns (4000 = 20 x 192 + 160) and k (520)."""
    check_tc(oracle_mod, 1500, 4000, 520, BIAS | RES, seed=19, ws=True, rows=cols)


@pytest.mark.parametrize("inplace", [False, True], ids=["separate", "in-place"])
def test_tc_helper_schedule_residual(oracle_mod, inplace):
    """A shape with fewer 128 x 128 tiles than SMs and a long k (the helper-cluster
    schedule, which parks partial sums in Y): with a separate residual it runs
    that schedule; with Y as the residual it must take another (Y holds old
    values the epilogue still reads), and both are correct."""
    check_tc(oracle_mod, 700, 1000, 2048, BIAS | RES, seed=11, inplace=inplace, ws=True,
             rows=(0, 300))


@pytest.mark.parametrize("shape,flags", [((600, 1100, 2048), BIAS | GELU), ((1280, 1280, 2056), BIAS)])
def test_tc_helper_schedule_odd_tiles(oracle_mod, shape, flags):
    """Helper clusters whose last cluster has fewer tiles than owners (45 tiles for
    two owners per cluster, 100 for three: idle owners and a helper with fewer
    segments), with ragged rows and columns and, in the second, a ragged k."""
    n, m, k = shape
    check_tc(oracle_mod, n, m, k, flags, seed=n + 5, ws=True, rows=(0, 260))


@pytest.mark.parametrize("shape", [(1000, 1000, 512), (257, 300, 200), (1400, 3000, 264)])
def test_tc_workspace_path_bit_identical(shape):
    """Both tensor-core paths round X the same way and accumulate in the same
    order, so their outputs agree bit for bit.  (Shapes whose workspace path
    takes the helper schedule add two k ranges instead and are checked against
    the oracle, e.g. (300, 520, 1032) in test_tc_shapes.)"""
    n, m, k = shape
    g = synth.rng(17)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_bf16_weights(g, m, k, 0.03)
    b = synth.normal_f32(g, (m,), 0.1)
    Y1 = run_tc(n, m, k, BIAS | GELU, X, img, b)
    Y2 = run_tc(n, m, k, BIAS | GELU, X, img, b, ws=True)
    assert (Y1.view(np.int32) == Y2.view(np.int32)).all()


def test_tc_integer_exact():
    """bf16-exact small integers: every partial sum is an integer below 2^24, so the
    tensor core must produce the exact result."""
    n, m, k = 256, 256, 512
    g = synth.rng(99)
    X = g.integers(-4, 5, size=(n, k)).astype(np.float32)
    Wv = g.integers(-4, 5, size=(m, k)).astype(np.float32)
    img = synth.bf16_pairs(synth.bf16_bits_rne(Wv))
    Y = run_tc(n, m, k, 0, X, img)
    want = X.astype(np.float64) @ Wv.astype(np.float64).T
    assert (Y == want).all()


def test_tc_deterministic():
    n, m, k = 300, 512, 1024
    g = synth.rng(4)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_bf16_weights(g, m, k, 0.03)
    b = synth.normal_f32(g, (m,), 0.1)
    Y1 = run_tc(n, m, k, BIAS | GELU, X, img, b)
    Y2 = run_tc(n, m, k, BIAS | GELU, X, img, b)
    assert (Y1.view(np.int32) == Y2.view(np.int32)).all()


@pytest.mark.parametrize("ws,shape", [(False, (512, 1024, 4096)), (True, (512, 1024, 4096)),
                                      (True, (1400, 3000, 256))],
                         ids=["fused", "workspace", "workspace-pair"])
def test_tc_wait_limit_expires_without_hang(oracle_mod, ws, shape):
    """A one-poll wait limit aborts the tensor-core kernel's CTAs at their first
    unfilled stage: they record WQ_ERR_DEVICE_TIMEOUT, drain their TMA copies and
    MMAs, free TMEM and return; the next call with the default limit is correct.
    The last case runs the SM-pair schedule (256-row tiles over two CTAs)."""
    n, m, k = shape
    g = synth.rng(6)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_bf16_weights(g, m, k, 0.03)
    Xd, Wd = dev(X), weights_dev(img, BF16, m, k)
    Y = torch.zeros(n * m, device="cuda")
    need = wq.wq_gemm_workspace_bytes(n, m, k, BF16, TC)
    work = torch.empty(need, dtype=torch.uint8, device="cuda")

    def call():
        if ws:
            return wq.wq_gemm_ws(n, m, k, BF16, TC, Xd, Wd, None, None, Y, work, need)
        return wq.wq_gemm(n, m, k, BF16, TC, Xd, Wd, None, None, Y)

    seen = []
    wq.wq_set_wait_limit(1)
    try:
        for _ in range(5):
            wq.check(call())
            seen.append(wq.wq_get_device_status())
            if seen[-1] == wq.WQ_ERR_DEVICE_TIMEOUT:
                break
    finally:
        wq.wq_set_wait_limit(0)
    assert wq.WQ_ERR_DEVICE_TIMEOUT in seen, seen
    wq.check(call())
    status_ok()
    Yref, S = oracle_mod.gemm(n, m, k, BF16, 0, X, img, round_x=True, rows=(0, 64))
    assert_within(Y.cpu().numpy().reshape(n, m)[:, :64], Yref[:, :64], S[:, :64], tau_exact(k))


# ----------------------------------------------- quantised W on the tensor cores --

def run_tcq(n, m, k, wtype, flags, X, img, bias=None, R=None):
    Y = Guarded(n * m)
    need = wq.wq_gemm_workspace_bytes(n, m, k, wtype, flags | TC)
    assert need >= 2 * n * k + 2 * m * k
    work = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = wq.wq_gemm_ws(n, m, k, wtype, flags | TC, dev(X), weights_dev(img, wtype, m, k),
                       dev(bias) if bias is not None else None,
                       dev(R) if R is not None else None, Y.view, work, need)
    wq.check(st, "wq_gemm_ws(TC, quantised)")
    torch.cuda.synchronize()
    status_ok()
    return Y.result().reshape(n, m)


@pytest.mark.parametrize("wtype", [wq.WQ_Q8_0, wq.WQ_Q4_0])
@pytest.mark.parametrize("shape,flags", [((17, 32, 32), 0), ((130, 256, 128), BIAS),
                                         ((300, 520, 1056), BIAS | GELU), ((257, 300, 224), RES),
                                         ((1500, 1024, 1024), BIAS | RES)])
def test_tc_quantised_weights(oracle_mod, wtype, shape, flags):
    """X and the dequantised W both rounded to bf16: within 8e-3 sum|x||w| of the exact
    result, and within the accumulation bound of the oracle fed the same roundings."""
    n, m, k = shape
    g = synth.rng(n * 7 + m + wtype)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wtype, m, k)
    bias = synth.normal_f32(g, (m,), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n, m)) if flags & RES else None
    Y = run_tcq(n, m, k, wtype, flags, X, img, bias, R)
    rows = (0, m) if m <= 520 else (m // 2 - 32, m // 2 + 32)
    j0, j1 = rows
    for rnd, tau in ((False, TAU_TC), (True, tau_exact(k))):
        Yref, S = oracle_mod.gemm(n, m, k, wtype, flags, X, img, bias=bias, residual=R,
                                  round_x=rnd, round_w=rnd, rows=rows)
        assert_within(Y[:, j0:j1], Yref[:, j0:j1], S[:, j0:j1], tau, gelu=bool(flags & GELU),
                      bias=None if bias is None else bias[j0:j1],
                      R=None if R is None else R[:, j0:j1],
                      what=f"tc quantised wtype={wtype} {shape} flags={flags} rounded={rnd}")


def test_tc_quantised_needs_workspace_entry_point():
    n, m, k = 64, 64, 64
    Xd = torch.zeros(n * k, device="cuda")
    Wd = torch.zeros(wq.wq_weight_bytes(wq.WQ_Q8_0, m, k), dtype=torch.uint8, device="cuda")
    Y = torch.zeros(n * m, device="cuda")
    assert wq.wq_gemm(n, m, k, wq.WQ_Q8_0, TC, Xd, Wd, None, None, Y) == wq.WQ_ERR_UNSUPPORTED
