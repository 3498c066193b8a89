"""GPU parity of the tensor-core GEMV for bf16-pair and F16 weights (gemv_half.cu),
which wq_gemv and the small-n wq_gemm take for those weights when k % 256 == 0
(cortiq-engine 0.8.49 AudioEncoder::gemm: W as bf16 pairs; wavo's F16 weights).
X is scaled by a power of two per token and 64-element slice and split into
three bf16 or two f16 terms; every check is against the f64 oracle at tau = 1e-5.
The group sizes of the kernel (2, 4, 6 or 8 tiles of 16 rows per CTA, one or two
halves of eight tokens) follow m and n, so the shapes below reach each of them.
For F16 weights with X near 2^-120 the f16 terms reach f16's subnormal floor for
elements 2^-17 below their slice's largest |x|, an absolute 2^-39 of it."""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16, F16 = wq.WQ_BF16, wq.WQ_F16
HALF = pytest.mark.parametrize("wt", [BF16, F16], ids=["bf16", "f16"])
BIAS, GELU, RES = wq.WQ_BIAS, wq.WQ_GELU, wq.WQ_RESIDUAL
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run(n, m, k, flags, X, img, bias=None, R=None, fn=None, wt=BF16):
    fn = fn or wq.wq_gemv
    out = Guarded(n * m)
    st = fn(n, m, k, wt, flags, dev(X), weights_dev(img, wt, m, k),
            dev(bias) if bias is not None else None, dev(R) if R is not None else None, out.view)
    wq.check(st, fn.__name__)
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def check(oracle_mod, n, m, k, flags, X, img, bias=None, R=None, rows=None, what="", fn=None,
          wt=BF16):
    Y = run(n, m, k, flags, X, img, bias, R, fn, wt)
    assert np.isfinite(Y).all()
    Yref, S = oracle_mod.gemm(n, m, k, wt, flags, X, img, bias=bias, residual=R, rows=rows)
    sl = slice(*rows) if rows else slice(None)
    assert_within(Y[:, sl], Yref[:, sl], S[:, sl], TAU, gelu=bool(flags & GELU),
                  bias=None if bias is None else bias[sl], R=None if R is None else R[:, sl],
                  what=what)


# m and n that select each group size: tiles per SM <= 2, 4, 6 and more (8), with
# one half of tokens (n <= 8) or two (n <= 16); ragged m and n in each.
GROUPS = [(1, 4000, 1024), (3, 9000, 512), (8, 14336, 256), (2, 20000, 768),
          (9, 3000, 512), (16, 9000, 256), (12, 515, 1280)]


@HALF
@pytest.mark.parametrize("n,m,k", GROUPS)
def test_group_sizes(oracle_mod, wt, n, m, k):
    g = synth.rng(n * 7 + m)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wt, m, k)
    bias = synth.normal_f32(g, (m,), 0.1)
    R = synth.normal_f32(g, (n, m))
    check(oracle_mod, n, m, k, BIAS | RES, X, img, bias, R, wt=wt,
          what=f"wtype {wt} mma n={n} m={m} k={k}")


@HALF
@pytest.mark.parametrize("n", [1, 5, 12])
def test_wide_range_x(oracle_mod, wt, n):
    """X spanning 2^-60 .. 2^60, a zero slice, a slice near 2^100 and an f32
    subnormal: the power-of-two scaling per 64-element slice keeps the three terms
    normal and every product exact to the tolerance."""
    m, k = 300, 1024
    g = synth.rng(190 + n)
    X = synth.normal_f32(g, (n, k)) * np.exp2(g.integers(-60, 61, size=(n, k))).astype(np.float32)
    X[:, 64:128] = 0.0                                                         # a zero slice
    X[:, 256:320] = synth.normal_f32(g, (n, 64)) * np.float32(2.0 ** 100)    # a huge slice
    X[:, 400] = np.float32(1e-40)                                              # f32 subnormal
    img = synth.draw_weights(g, wt, m, k)
    check(oracle_mod, n, m, k, 0, X, img, wt=wt, what=f"wide-range X wtype {wt} n={n}")


@HALF
@pytest.mark.parametrize("scale", [2.0 ** -120, 2.0 ** -100, 2.0 ** 110])
def test_tiny_and_huge_x(oracle_mod, wt, scale):
    """X entirely near the bottom (below where an unscaled third bf16 term would be
    subnormal) or near the top of the f32 range."""
    n, m, k = 3, 200, 768
    g = synth.rng(int(np.log2(scale)) + 500)
    X = (synth.normal_f32(g, (n, k)).astype(np.float64) * scale).astype(np.float32)
    img = synth.draw_weights(g, wt, m, k)
    check(oracle_mod, n, m, k, 0, X, img, wt=wt, what=f"wtype {wt} X scaled by 2^{np.log2(scale):.0f}")


@HALF
def test_exact_integers(oracle_mod, wt):
    """Small integers in X and W: every product and partial sum is exact, so the
    result equals the oracle's bit for bit."""
    n, m, k = 4, 160, 512
    g = synth.rng(77)
    X = g.integers(-8, 9, size=(n, k)).astype(np.float32)
    Wf = g.integers(-8, 9, size=(m, k)).astype(np.float32)
    if wt == BF16:
        img = synth.bf16_pairs((Wf.view(np.uint32) >> 16).astype(np.uint16))  # exact in bf16
    else:
        img = Wf.astype(np.float16).view(np.uint8).reshape(m, 2 * k)       # exact in f16
    Y = run(n, m, k, 0, X, img, wt=wt)
    Yref, _ = oracle_mod.gemm(n, m, k, wt, 0, X, img)
    assert (Y == Yref.astype(np.float32)).all()


@HALF
def test_in_place_residual_and_gelu(oracle_mod, wt):
    n, m, k = 6, 1000, 1024
    g = synth.rng(31)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wt, m, k)
    bias = synth.normal_f32(g, (m,), 0.1)
    R = synth.normal_f32(g, (n, m))
    out = Guarded(n * m, R)
    st = wq.wq_gemv(n, m, k, wt, BIAS | GELU | RES, dev(X), weights_dev(img, wt, m, k),
                    dev(bias), out.view, out.view)
    wq.check(st, "wq_gemv")
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n, m)
    Yref, S = oracle_mod.gemm(n, m, k, wt, BIAS | GELU | RES, X, img, bias=bias, residual=R)
    assert_within(Y, Yref, S, TAU, gelu=True, bias=bias, R=R, what="in-place residual")


@HALF
def test_small_n_gemm_takes_it(oracle_mod, wt):
    """wq_gemm with n <= 16 runs the same kernel."""
    n, m, k = 16, 700, 512
    g = synth.rng(41)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wt, m, k)
    bias = synth.normal_f32(g, (m,), 0.1)
    check(oracle_mod, n, m, k, BIAS, X, img, bias, fn=wq.wq_gemm, wt=wt, what="wq_gemm n=16")


@HALF
def test_bit_identical_reruns(wt):
    n, m, k = 5, 3000, 2048
    g = synth.rng(3)
    X = synth.normal_f32(g, (n, k))
    img = synth.draw_weights(g, wt, m, k)
    Y1 = run(n, m, k, 0, X, img, wt=wt)
    Y2 = run(n, m, k, 0, X, img, wt=wt)
    assert (Y1.view(np.int32) == Y2.view(np.int32)).all()


# -------------------------------------------------------------------- MoE --
# wq_moe_gemv with bf16 or F16 banks and k % 256 == 0 runs the same arithmetic per
# chunk (hanzo-ml 0.11.13 moe_matvec_gpu: y[s] = W[ids[s]] . x[s / topk]), with the
# window's slots sorted by expert in shared memory and groups of four 16-row tiles
# that never cross an expert; short groups (m / 16 not a multiple of 4) load only
# their own rows.

def run_moe(oracle_mod, wt, n_tok, topk, E, m, k, flags, ids, seed, slots=None):
    g = synth.rng(seed)
    bank = synth.draw_weights(g, wt, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    bias = synth.normal_f32(g, (E, m), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n_tok * topk, m)) if flags & RES else None
    out = Guarded(n_tok * topk * m)
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wt, flags, dev(X),
                            weights_dev(bank, wt, E * m, k), dev(ids),
                            None if bias is None else dev(bias),
                            None if R is None else dev(R), out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n_tok * topk, m)
    q0, q1 = slots or (0, n_tok * topk)
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wt, flags, X, bank, ids, bias=bias,
                             residual=R, slots=(q0, q1))
    extra = np.zeros((n_tok * topk, m))
    if bias is not None:
        extra += np.abs(bias[ids.reshape(-1)])
    if R is not None:
        extra += np.abs(R)
    sl = slice(q0, q1)
    assert_within(Y[sl], Yref[sl], S[sl], TAU, gelu=bool(flags & GELU), R=extra[sl],
                  what=f"moe wtype {wt} slots={n_tok * topk} E={E} m={m} k={k}")
    return Y


MOE_CFGS = [(1, 1, 1, 33, 256),        # one slot; three tiles: a 2 + 1 short group
            (3, 2, 5, 70, 512),        # five tiles: a full group and a 1-tile group
            (16, 6, 64, 140, 2048),    # the decode routing of a 64-expert layer
            (8, 3, 4, 257, 4096),      # a ragged last tile
            (32, 8, 4, 72, 512)]       # ~64 slots per expert: eight passes of 8 slots


@HALF
@pytest.mark.parametrize("cfg", MOE_CFGS)
def test_moe(oracle_mod, wt, cfg):
    n_tok, topk, E, m, k = cfg
    g = synth.rng(sum(cfg) + 60 * wt)
    ids = synth.moe_ids(g, n_tok, topk, E) if topk <= E else \
        g.integers(0, E, size=(n_tok, topk)).astype(np.int32)
    run_moe(oracle_mod, wt, n_tok, topk, E, m, k, BIAS | GELU | RES, ids, sum(cfg) + wt)


@HALF
def test_moe_windows(oracle_mod, wt):
    """512 tokens at top-6: 3,072 slots, twelve routing windows."""
    n_tok, topk, E, m, k = 512, 6, 64, 72, 512
    ids = synth.moe_ids(synth.rng(910 + wt), n_tok, topk, E)
    run_moe(oracle_mod, wt, n_tok, topk, E, m, k, BIAS | RES, ids, 911 + wt)


@HALF
def test_moe_one_expert_takes_every_slot(oracle_mod, wt):
    n_tok, topk, E, m, k = 1024, 3, 8, 40, 256
    ids = np.full((n_tok, topk), 5, np.int32)
    run_moe(oracle_mod, wt, n_tok, topk, E, m, k, 0, ids, 960 + wt)


@HALF
def test_moe_window_edge(oracle_mod, wt):
    """257 slots: one full window and a window of one slot."""
    n_tok, topk, E, m, k = 257, 1, 7, 33, 512
    ids = synth.rng(987).integers(0, E, size=(n_tok, topk)).astype(np.int32)
    run_moe(oracle_mod, wt, n_tok, topk, E, m, k, BIAS, ids, 988 + wt)


@HALF
def test_moe_repeated_expert_and_bad_id(oracle_mod, wt):
    """A token may route twice to one expert; a bad id sets the device status and
    leaves only its own slot's row unwritten."""
    n_tok, topk, E, m, k = 4, 3, 6, 50, 256
    g = synth.rng(12 + wt)
    bank = synth.draw_weights(g, wt, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = np.array([[1, 1, 2], [5, 0, 1], [3, 9, 3], [2, 2, 2]], np.int32)  # 9 is out of range
    out = Guarded(n_tok * topk * m)
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wt, 0, dev(X), weights_dev(bank, wt, E * m, k),
                            dev(ids), None, None, out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    assert wq.wq_get_device_status() == wq.WQ_ERR_BAD_EXPERT
    status_ok()  # cleared by the read
    Y = out.result().reshape(n_tok * topk, m)
    bad = 2 * topk + 1
    assert (Y[bad].view(np.int32) == -1).all()
    good = [q for q in range(n_tok * topk) if q != bad]
    ids_ok = ids.copy()
    ids_ok[2, 1] = 0
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wt, 0, X, bank, ids_ok)
    assert_within(Y[good], Yref[good], S[good], TAU, what="moe repeated ids")


@HALF
def test_moe_exact_integers(oracle_mod, wt):
    """Small integers in X and the bank: every product and partial sum is exact, so
    each slot's row equals the oracle's bit for bit."""
    n_tok, topk, E, m, k = 6, 4, 5, 90, 768
    g = synth.rng(78 + wt)
    X = g.integers(-8, 9, size=(n_tok, k)).astype(np.float32)
    Wf = g.integers(-8, 9, size=(E * m, k)).astype(np.float32)
    if wt == BF16:
        img = synth.bf16_pairs((Wf.view(np.uint32) >> 16).astype(np.uint16))
    else:
        img = Wf.astype(np.float16).view(np.uint8).reshape(E * m, 2 * k)
    bank = img.reshape(E, m, -1)
    ids = synth.moe_ids(g, n_tok, topk, E)
    out = Guarded(n_tok * topk * m)
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wt, 0, dev(X), weights_dev(bank, wt, E * m, k),
                            dev(ids), None, None, out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n_tok * topk, m)
    Yref, _ = oracle_mod.moe(n_tok, topk, E, m, k, wt, 0, X, bank, ids)
    assert (Y == Yref.astype(np.float32)).all()


@HALF
def test_moe_bit_identical_reruns(oracle_mod, wt):
    n_tok, topk, E, m, k = 16, 6, 64, 300, 1024
    ids = synth.moe_ids(synth.rng(4), n_tok, topk, E)
    Y1 = run_moe(oracle_mod, wt, n_tok, topk, E, m, k, BIAS, ids, 5, slots=(0, 8))
    Y2 = run_moe(oracle_mod, wt, n_tok, topk, E, m, k, BIAS, ids, 5, slots=(0, 8))
    assert (Y1.view(np.int32) == Y2.view(np.int32)).all()


@HALF
def test_moe_window_of_bad_ids_only(oracle_mod, wt):
    """A first window whose 256 ids are all out of range (no segment to run) and a
    second window of valid ids: the device status says WQ_ERR_BAD_EXPERT, the bad
    slots' rows stay unwritten and the second window's rows are correct."""
    n_tok, topk, E, m, k = 300, 1, 5, 40, 256
    g = synth.rng(70 + wt)
    bank = synth.draw_weights(g, wt, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = g.integers(0, E, size=(n_tok, topk)).astype(np.int32)
    ids[:256] = -3
    out = Guarded(n_tok * topk * m)
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wt, 0, dev(X), weights_dev(bank, wt, E * m, k),
                            dev(ids), None, None, out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    assert wq.wq_get_device_status() == wq.WQ_ERR_BAD_EXPERT
    status_ok()
    Y = out.result().reshape(n_tok * topk, m)
    assert (Y[:256].view(np.int32) == -1).all()
    ids_ok = ids.copy()
    ids_ok[:256] = 0
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wt, 0, X, bank, ids_ok, slots=(256, 300))
    assert_within(Y[256:], Yref[256:], S[256:], TAU, what="moe after a bad window")


@HALF
def test_moe_in_place_residual(oracle_mod, wt):
    """residual == Y: each slot's row is read and rewritten by the same thread."""
    n_tok, topk, E, m, k = 16, 6, 64, 140, 512
    g = synth.rng(80 + wt)
    bank = synth.draw_weights(g, wt, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    ids = synth.moe_ids(g, n_tok, topk, E)
    bias = synth.normal_f32(g, (E, m), 0.1)
    R = synth.normal_f32(g, (n_tok * topk, m))
    out = Guarded(n_tok * topk * m, R)
    flags = BIAS | GELU | RES
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wt, flags, dev(X),
                            weights_dev(bank, wt, E * m, k), dev(ids), dev(bias), out.view,
                            out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(n_tok * topk, m)
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wt, flags, X, bank, ids, bias=bias, residual=R)
    assert_within(Y, Yref, S, TAU, gelu=True, R=np.abs(R) + np.abs(bias[ids.reshape(-1)]),
                  what="moe in-place residual")
