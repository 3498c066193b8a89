"""Pins of the f64 oracle against facts fixed outside it (CPU only).

Each test pins one part of the oracle to something other than the oracle:
hand-worked format blocks, exhaustive comparison with numpy/torch format
conversions, identity and one-hot weights, the closed-form probe printed in
wavo's ``probe_tensor``, exact integer brute force, textbook erf-GELU values,
and closed forms of the MoE routing.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from conftest import golden_lines

BF16, Q8_0, Q4_0 = synth.WTYPE_BF16, synth.WTYPE_Q8_0, synth.WTYPE_Q4_0
BIAS, GELU, RESIDUAL = synth.FLAG_BIAS, synth.FLAG_GELU, synth.FLAG_RESIDUAL


# ----------------------------------------------------------------- formats --

def test_half_hand_values(oracle_mod):
    o = oracle_mod
    assert o.half_to_f64(0x3C00) == 1.0
    assert o.half_to_f64(0xC000) == -2.0
    assert o.half_to_f64(0x2000) == 2.0 ** -7
    assert o.half_to_f64(0x0001) == 2.0 ** -24
    assert o.half_to_f64(0x03FF) == 1023 * 2.0 ** -24
    assert o.half_to_f64(0x0400) == 2.0 ** -14
    assert o.half_to_f64(0x7BFF) == 65504.0
    assert o.half_to_f64(0x3555) == 0.333251953125
    z = o.half_to_f64(0x8000)
    assert z == 0.0 and np.signbit(z)
    assert o.half_to_f64(0x7C00) == np.inf and o.half_to_f64(0xFC00) == -np.inf
    assert np.isnan(o.half_to_f64(0x7E00))


def test_half_exhaustive_vs_numpy(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_f64(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()
    assert (np.signbit(got) == np.signbit(want)).all()


def test_bf16_exhaustive_vs_torch(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.int32)
    t = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16)
    want = t.to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_to_f64(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_bf16_pair_words(oracle_mod):
    """Hand-decoded pair words: low half = even k, high half = odd k."""
    for line in golden_lines("bf16_pairs.txt"):
        word_hex, lo, hi = line.split()
        word = int(word_hex, 16)
        img = np.frombuffer(np.array([word], dtype="<u4").tobytes(), dtype=np.uint8)
        w = oracle_mod.dequant(BF16, 1, 2, img.reshape(1, 4))
        assert w[0, 0] == float(lo) and w[0, 1] == float(hi), line
        assert np.signbit(w[0, 0]) == np.signbit(float(lo))
        assert np.signbit(w[0, 1]) == np.signbit(float(hi))


def test_q4_0_hand_blocks(oracle_mod):
    lines = golden_lines("q4_0_block.txt")
    pairs = [(lines[i], lines[i + 1]) for i in range(0, len(lines), 2)]
    assert len(pairs) == 2
    for b_line, v_line in pairs:
        blk = np.array([int(x, 16) for x in b_line.split(":")[1].split()], dtype=np.uint8)
        want = np.array([float(x) for x in v_line.split(":")[1].split()])
        assert blk.size == 18 and want.size == 32
        got = oracle_mod.dequant(Q4_0, 1, 32, blk.reshape(1, 18))[0]
        assert (got == want).all(), (got, want)


def test_q8_0_hand_blocks(oracle_mod):
    lines = golden_lines("q8_0_block.txt")
    codes = [int(x) for x in lines[0].split(":")[1].split()]
    assert len(codes) == 32
    scales = [ln.split(":")[1].split() for ln in lines[1:]]
    assert len(scales) == 4
    for bits_hex, unit in scales:
        bits = int(bits_hex, 16)
        blk = np.array([bits & 0xFF, bits >> 8] + [c & 0xFF for c in codes], dtype=np.uint8)
        got = oracle_mod.dequant(Q8_0, 1, 32, blk.reshape(1, 34))[0]
        want = np.array([float(unit) * c for c in codes])
        assert (got == want).all(), bits_hex


def test_q8_0_exhaustive_codes(oracle_mod):
    """All 256 codes under a power-of-two scale, across 8 blocks of two rows."""
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(2, 128)
    d = np.full((2, 4), 0x3400, dtype=np.uint16)  # 0.25
    img = synth.encode_q8_0(d, codes)
    got = oracle_mod.dequant(Q8_0, 2, 128, img)
    assert (got == codes.astype(np.float64) * 0.25).all()


def test_q4_0_all_nibbles_every_position(oracle_mod):
    """Every code at every in-block position; a swapped nibble order fails."""
    q4 = (np.arange(32)[None, :] + np.arange(16)[:, None]) % 16
    d = np.full((16, 1), 0x4000, dtype=np.uint16)  # 2.0
    img = synth.encode_q4_0(d, q4.astype(np.uint8))
    got = oracle_mod.dequant(Q4_0, 16, 32, img)
    assert (got == 2.0 * (q4 - 8)).all()


def test_round_bf16(oracle_mod):
    r = oracle_mod.round_bf16
    assert r(1.0 + 2.0 ** -8) == 1.0                      # tie -> even (down)
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6      # tie -> even (up)
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert r(-(1.0 + 2.0 ** -8)) == -1.0
    assert r(3.4e38) == np.inf
    assert r(2.0 ** -140) == 0.0 or r(2.0 ** -140) == 2.0 ** -133 * round(2.0 ** -7)
    g = np.random.default_rng(7)
    x = np.concatenate([g.standard_normal(20000).astype(np.float32),
                        (g.standard_normal(2000) * 1e-39).astype(np.float32),
                        (g.standard_normal(2000) * 1e30).astype(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([r(float(v)) for v in x])
    assert (got == want).all()


# ------------------------------------------------------------- contraction --

def _identity_image(wtype, k, one_code=None):
    """W = I (k x k) in the given format; exact value 1.0 on the diagonal."""
    if wtype == BF16:
        bits = np.zeros((k, k), dtype=np.uint16)
        np.fill_diagonal(bits, 0x3F80)
        return synth.bf16_pairs(bits)
    d = np.full((k, k // 32), 0x3C00, dtype=np.uint16)
    if wtype == Q8_0:
        q = np.zeros((k, k), dtype=np.int8)
        np.fill_diagonal(q, 1)
        return synth.encode_q8_0(d, q)
    q = np.full((k, k), 8, dtype=np.uint8)
    np.fill_diagonal(q, 9)
    return synth.encode_q4_0(d, q)


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_identity_weights(oracle_mod, wtype):
    k, n = 96, 5
    X = synth.normal_f32(synth.rng(11), (n, k))
    Y, S = oracle_mod.gemm(n, k, k, wtype, 0, X, _identity_image(wtype, k))
    assert (Y == X.astype(np.float64)).all()
    assert (S == np.abs(X).astype(np.float64)).all()


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_wavo_probe_closed_form(oracle_mod, wtype):
    """The printed probe of wavo's tensor GEMM: c[r][j] = j % 32 + r % 32."""
    cfg = dict(ln.split(":") for ln in golden_lines("wavo_probe.txt"))
    n, m, k = int(cfg["n"]), int(cfg["m"]), int(cfg["k"])
    a = np.array([[x + r % 32 for x in range(k)] for r in range(n)], dtype=np.float32)
    onehot = np.array([[1 if x == j % 32 else 0 for x in range(k)] for j in range(m)])
    if wtype == BF16:
        img = synth.bf16_pairs(np.where(onehot == 1, 0x3F80, 0).astype(np.uint16))
    elif wtype == Q8_0:
        img = synth.encode_q8_0(np.full((m, 1), 0x3C00, np.uint16), onehot.astype(np.int8))
    else:
        img = synth.encode_q4_0(np.full((m, 1), 0x3C00, np.uint16), (onehot + 8).astype(np.uint8))
    Y, _ = oracle_mod.gemm(n, m, k, wtype, BIAS, a, img, bias=np.zeros(m, np.float32))
    want = np.array([[j % 32 + r % 32 for j in range(m)] for r in range(n)], dtype=np.float64)
    assert (Y == want).all()


def _exact_case(g, wtype, n, m, k):
    """Random small-integer inputs whose every product and sum is exact in f64."""
    X = g.integers(-3, 4, size=(n, k)).astype(np.float32)
    nb = k // 32
    if wtype == BF16:
        wv = g.integers(-8, 9, size=(m, k)) * 0.5  # exact in bf16
        img = synth.bf16_pairs(synth.bf16_bits_rne(wv.astype(np.float32)))
        Wf = [[Fraction(v) for v in row] for row in wv]
    else:
        exps = g.integers(-3, 3, size=(m, nb))
        sign = g.choice([-1, 1], size=(m, nb))
        dval = sign * np.ldexp(1.0, exps)
        dbits = synth.f16_bits(dval)
        if wtype == Q8_0:
            q = g.integers(-128, 128, size=(m, k)).astype(np.int8)
            img = synth.encode_q8_0(dbits, q)
            Wf = [[Fraction(dval[j, t // 32]) * int(q[j, t]) for t in range(k)] for j in range(m)]
        else:
            q4 = g.integers(0, 16, size=(m, k)).astype(np.uint8)
            img = synth.encode_q4_0(dbits, q4)
            Wf = [[Fraction(dval[j, t // 32]) * (int(q4[j, t]) - 8) for t in range(k)]
                  for j in range(m)]
    return X, img, Wf


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("shape", [(1, 3, 32), (3, 5, 64), (7, 2, 96), (4, 33, 32)])
def test_exact_integer_brute_force(oracle_mod, wtype, shape):
    """Exact rational arithmetic on the intended values (not on the byte image)."""
    n, m, k = shape
    g = np.random.default_rng(1000 * wtype + 10 * n + m)
    X, img, Wf = _exact_case(g, wtype, n, m, k)
    bias = g.integers(-4, 5, size=m).astype(np.float32)
    R = g.integers(-4, 5, size=(n, m)).astype(np.float32)
    for flags in (0, BIAS, RESIDUAL, BIAS | RESIDUAL):
        Y, S = oracle_mod.gemm(n, m, k, wtype, flags, X, img, bias=bias, residual=R)
        for i in range(n):
            for j in range(m):
                acc = sum(Fraction(float(X[i, t])) * Wf[j][t] for t in range(k))
                s = sum(abs(Fraction(float(X[i, t])) * Wf[j][t]) for t in range(k))
                if flags & BIAS:
                    acc += Fraction(float(bias[j]))
                if flags & RESIDUAL:
                    acc += Fraction(float(R[i, j]))
                assert Y[i, j] == float(acc), (flags, i, j)
                assert S[i, j] == float(s)


def test_gelu_closed_forms(oracle_mod):
    pts = [tuple(float(v) for v in ln.split()) for ln in golden_lines("gelu_points.txt")]
    for v, want in pts:
        got = oracle_mod.gelu(v)
        assert abs(got - want) <= 2e-16 * max(1.0, abs(want)), (v, got, want)
    for v in np.linspace(-6, 6, 241):
        assert abs((oracle_mod.gelu(v) - oracle_mod.gelu(-v)) - v) <= 4e-16 * max(1, abs(v))


def test_gelu_through_gemm_and_scipy(oracle_mod):
    from scipy.special import erf
    k = 32
    v = np.linspace(-5, 5, 64).astype(np.float32).reshape(2, k)
    Y, _ = oracle_mod.gemm(2, k, k, Q8_0, GELU, v, _identity_image(Q8_0, k))
    want = 0.5 * v.astype(np.float64) * (1 + erf(v.astype(np.float64) / np.sqrt(2.0)))
    # 1 + erf(.) cancels in the left tail: compare on the scale of |v|.
    assert (np.abs(Y - want) <= 1e-15 * np.maximum(1.0, np.abs(v))).all()


def test_epilogue_order(oracle_mod):
    """bias -> GELU -> residual, as cortiq-engine's ae_put orders them."""
    k = 32
    X = np.ones((1, k), np.float32)
    Y, _ = oracle_mod.gemm(1, k, k, Q4_0, BIAS | GELU | RESIDUAL, X, _identity_image(Q4_0, k),
                           bias=np.ones(k, np.float32), residual=np.ones((1, k), np.float32))
    want = 1.9544997361036416 + 1.0  # gelu(1 + 1) + 1
    assert np.allclose(Y, want, rtol=1e-15)


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("alpha", [1.0, 0.5, -2.0, 0.0])
def test_residual_alpha_closed_form(oracle_mod, wtype, alpha):
    """wavo's Residual(a): c += alpha (a W^T + b).  With W = I every product is one x, so
    Y = R + alpha (x + b) exactly for small integers and halves; the bound scales."""
    n, k = 3, 64
    g = np.random.default_rng(4)
    X = g.integers(-20, 21, size=(n, k)).astype(np.float32)
    b = g.integers(-5, 6, size=k).astype(np.float32)
    R = g.integers(-9, 10, size=(n, k)).astype(np.float32)
    Y, S = oracle_mod.gemm(n, k, k, wtype, BIAS | RESIDUAL, X, _identity_image(wtype, k), bias=b,
                           residual=R, alpha=alpha)
    assert (Y == R + alpha * (X.astype(np.float64) + b)).all()
    assert (S == abs(alpha) * np.abs(X).astype(np.float64)).all()


def test_residual_alpha_scales_the_activation(oracle_mod):
    """The scale applies to the activation's output, before the residual."""
    k = 32
    X = np.ones((1, k), np.float32)
    Y, _ = oracle_mod.gemm(1, k, k, Q4_0, BIAS | GELU | RESIDUAL, X, _identity_image(Q4_0, k),
                           bias=np.ones(k, np.float32), residual=np.ones((1, k), np.float32),
                           alpha=-0.25)
    assert np.allclose(Y, 1.0 - 0.25 * 1.9544997361036416, rtol=1e-15)  # 1 - gelu(2) / 4


# ------------------------------------------- wavo's dual outputs (Gpu::linear) --

@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_dual_outputs_identity_closed_form(oracle_mod, wtype):
    """A bias with `dual` extra values: with W = I the first m columns are
    R + alpha * relu(x + b), and columns m + j (j < dual) are x_j + b2_j, with no
    activation, scale or residual (the residual's own columns m.. are not read)."""
    n, k, dual = 3, 64, 24
    g = np.random.default_rng(7)
    X = g.integers(-6, 7, size=(n, k)).astype(np.float32)
    b = g.integers(-3, 4, size=k).astype(np.float32)
    b2 = g.integers(-9, 10, size=dual).astype(np.float32)
    R = g.integers(-5, 6, size=(n, k + dual)).astype(np.float32)
    R[:, k:] = np.nan
    relu = 16
    Y, S = oracle_mod.gemm(n, k, k, wtype, BIAS | relu | RESIDUAL, X, _identity_image(wtype, k),
                           bias=b, residual=R, alpha=-0.5, dual=dual, bias2=b2)
    Xd = X.astype(np.float64)
    assert Y.shape == (n, k + dual)
    assert (Y[:, :k] == R[:, :k] - 0.5 * np.maximum(Xd + b, 0.0)).all()
    assert (Y[:, k:] == Xd[:, :dual] + b2).all()
    assert (S[:, :k] == 0.5 * np.abs(Xd)).all()
    assert (S[:, k:] == np.abs(Xd[:, :dual])).all()


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
@pytest.mark.parametrize("dual", [1, 5, 7])
def test_dual_outputs_exact_integer_brute_force(oracle_mod, wtype, dual):
    """Exact rational arithmetic: columns m + j hold output j's plain sum + b2_j
    whatever the first band's epilogue (GELU here)."""
    n, m, k = 3, 7, 64
    g = np.random.default_rng(300 + 10 * wtype + dual)
    X, img, Wf = _exact_case(g, wtype, n, m, k)
    b = g.integers(-4, 5, size=m).astype(np.float32)
    b2 = g.integers(-4, 5, size=dual).astype(np.float32)
    Y, S = oracle_mod.gemm(n, m, k, wtype, BIAS | GELU, X, img, bias=b, dual=dual, bias2=b2)
    for i in range(n):
        for j in range(dual):
            acc = sum(Fraction(float(X[i, t])) * Wf[j][t] for t in range(k))
            s = sum(abs(Fraction(float(X[i, t])) * Wf[j][t]) for t in range(k))
            assert Y[i, m + j] == float(acc + Fraction(float(b2[j]))), (i, j)
            assert S[i, m + j] == float(s)
            v = float(acc + Fraction(float(b[j])))
            assert Y[i, j] == oracle_mod.gelu(v)


def test_dual_outputs_rows_and_arguments(oracle_mod):
    """rows=(j0, j1) computes both bands of those outputs only; dual = 0 is the
    plain call; dual outside [0, m] or a missing bias2 is refused."""
    n, m, k = 2, 40, 32
    g = np.random.default_rng(12)
    X, img, _ = _exact_case(g, Q8_0, n, m, k)
    b2 = np.arange(m, dtype=np.float32)
    Y, _ = oracle_mod.gemm(n, m, k, Q8_0, 0, X, img, dual=m, bias2=b2, rows=(3, 9))
    done = np.zeros(2 * m, bool)
    done[3:9] = True
    done[m + 3:m + 9] = True
    assert np.isfinite(Y[:, done]).all() and np.isnan(Y[:, ~done]).all()
    Y0, _ = oracle_mod.gemm(n, m, k, Q8_0, 0, X, img, dual=0)
    Yp, _ = oracle_mod.gemm(n, m, k, Q8_0, 0, X, img)
    assert (Y0 == Yp).all()
    for dual, bias2 in ((m + 1, np.zeros(m + 1, np.float32)), (-1, b2), (3, None)):
        with pytest.raises(ValueError):
            oracle_mod.gemm(n, m, k, Q8_0, 0, X, img, dual=dual, bias2=bias2)


@pytest.mark.parametrize("wtype", [Q8_0, Q4_0])
def test_zero_weights_residual(oracle_mod, wtype):
    n, m, k = 3, 7, 64
    d = np.full((m, k // 32), 0x3C00, np.uint16)
    img = (synth.encode_q8_0(d, np.zeros((m, k), np.int8)) if wtype == Q8_0
           else synth.encode_q4_0(d, np.full((m, k), 8, np.uint8)))
    g = synth.rng(3)
    X, R, b = synth.normal_f32(g, (n, k)), synth.normal_f32(g, (n, m)), synth.normal_f32(g, (m,))
    Y, S = oracle_mod.gemm(n, m, k, wtype, BIAS | RESIDUAL, X, img, bias=b, residual=R)
    assert (Y == (b[None, :].astype(np.float64) + R.astype(np.float64))).all()
    assert (S == 0).all()


def test_row_range_and_threads(oracle_mod):
    w = synth.workload_q8_0_gemv(n=2, m=96, k=128)
    Y1, S1 = oracle_mod.gemm(2, 96, 128, Q8_0, 0, w["X"], w["W"], threads=1)
    Y2, S2 = oracle_mod.gemm(2, 96, 128, Q8_0, 0, w["X"], w["W"], threads=4)
    assert (Y1 == Y2).all() and (S1 == S2).all()
    Y3, _ = oracle_mod.gemm(2, 96, 128, Q8_0, 0, w["X"], w["W"], rows=(10, 20))
    assert (Y3[:, 10:20] == Y1[:, 10:20]).all() and np.isnan(Y3[:, :10]).all()


def test_round_x_feeds_bf16_rounded_inputs(oracle_mod):
    """round_x=True equals feeding torch-rounded X (library RNE) with round_x=False."""
    w = synth.workload_bf16_gemm(n=4, m=40, k=64)
    Xr = torch.from_numpy(w["X"]).to(torch.bfloat16).to(torch.float32).numpy()
    Ya, _ = oracle_mod.gemm(4, 40, 64, BF16, 3, w["X"], w["W"], bias=w["bias"], round_x=True)
    Yb, _ = oracle_mod.gemm(4, 40, 64, BF16, 3, Xr, w["W"], bias=w["bias"])
    assert (Ya == Yb).all()


@pytest.mark.parametrize("d_bits,q,exact,rounded", [
    (0x3C01, 3, 3.0029296875, 3.0),            # (1 + 2^-10) * 3: below half a bf16 step
    (0x3C01, 5, 5.0048828125, 5.0),
    (0x3C0C, 1, 1.01171875, 1.015625),         # 1 + 1.5 * 2^-7: a tie, to the even neighbour
    (0x3C00, -7, -7.0, -7.0),                  # exact in bf16: unchanged
    (0x5BFF, 127, 32496.125, 32512.0),         # 255.875 * 127; bf16 step 128 there
])
def test_round_w_rounds_each_dequantised_weight(oracle_mod, d_bits, q, exact, rounded):
    """round_w=True feeds W = bf16_rne(d*q): a one-hot X picks the weight out."""
    k = 32
    d = np.full((1, 1), d_bits, np.uint16)
    qs = np.zeros((1, k), np.int8)
    qs[0, 5] = q
    img = synth.encode_q8_0(d, qs)
    X = np.zeros((1, k), np.float32)
    X[0, 5] = 1.0
    Ye, _ = oracle_mod.gemm(1, 1, k, Q8_0, 0, X, img)
    Yr, Sr = oracle_mod.gemm(1, 1, k, Q8_0, 0, X, img, round_w=True)
    assert Ye[0, 0] == exact and Yr[0, 0] == rounded and Sr[0, 0] == abs(rounded)


def test_round_w_equals_bf16_rounded_dequantised_image(oracle_mod):
    """round_w on a Q4_0 image equals round_w-free use of the torch-rounded (RNE)
    dequantised weights written as bf16 pairs."""
    g = synth.rng(31)
    m, k = 24, 96
    img = synth.draw_q4_0_weights(g, m, k)
    X = synth.normal_f32(g, (3, k))
    Wd = oracle_mod.dequant(Q4_0, m, k, img).astype(np.float32)
    bits = torch.from_numpy(Wd).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    pairs = synth.bf16_pairs(bits)
    Ya, _ = oracle_mod.gemm(3, m, k, Q4_0, 0, X, img, round_w=True)
    Yb, _ = oracle_mod.gemm(3, m, k, BF16, 0, X, pairs)
    assert (Ya == Yb).all()


SILU, RELU, TANH = 8, 16, 32


@pytest.mark.parametrize("flag,x,want", [
    (SILU, 0.0, 0.0),
    (SILU, float(np.float32(np.log(3.0))), None),   # sigma(ln 3) = 3/4: checked below
    (RELU, -3.0, 0.0), (RELU, 2.5, 2.5), (RELU, 0.0, 0.0),
    (TANH, 0.0, 0.0),
    (TANH, float(np.float32(np.log(2.0))), None),   # tanh(ln 2) = 3/5: checked below
])
def test_activation_closed_forms(oracle_mod, flag, x, want):
    """wavo's Silu / Relu / Tanh epilogues through a one-hot GEMM (Y = act(x))."""
    k = 32
    img = synth.bf16_pairs(np.where(np.arange(k) == 0, 0x3F80, 0).astype(np.uint16)[None, :])
    X = np.zeros((1, k), np.float32)
    X[0, 0] = x
    Y, _ = oracle_mod.gemm(1, 1, k, BF16, flag, X, img)
    if want is not None:
        assert Y[0, 0] == want
    elif flag == SILU:  # x = f32(ln 3): x * 3/4 up to the f32 rounding of ln 3
        assert abs(Y[0, 0] - 0.75 * np.log(3.0)) < 1e-7
    else:               # tanh(f32(ln 2)) = 0.6 up to that rounding
        assert abs(Y[0, 0] - 0.6) < 1e-7


@pytest.mark.parametrize("flag", [SILU, TANH])
def test_activation_symmetries(oracle_mod, flag):
    """silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1); tanh is odd."""
    k = 32
    img = synth.bf16_pairs(np.where(np.arange(k) == 0, 0x3F80, 0).astype(np.uint16)[None, :])
    for x in (0.3, 1.7, 6.0):
        X = np.zeros((2, k), np.float32)
        X[0, 0], X[1, 0] = x, -x
        Y, _ = oracle_mod.gemm(2, 1, k, BF16, flag, X, img)
        if flag == SILU:
            assert abs((Y[0, 0] - Y[1, 0]) - np.float32(x)) < 1e-15
        else:
            assert Y[0, 0] == -Y[1, 0]


def test_one_activation_per_call(oracle_mod):
    img = np.zeros((1, 64), np.uint8)
    X = np.zeros((1, 32), np.float32)
    for flags in (2 | 8, 8 | 16, 16 | 32, 2 | 32):
        with pytest.raises(ValueError):
            oracle_mod.gemm(1, 1, 32, BF16, flags, X, img)


def test_layer_norm_closed_forms(oracle_mod):
    """cortiq-engine ae_ln: (x - mean) / sqrt(var + 1e-5) * g + b, biased variance."""
    k = 4
    gb = np.array([1, 1, 1, 1, 0, 0, 0, 0], np.float32)
    X = np.array([[1, 3, 1, 3],          # mean 2, var 1
                  [5, 5, 5, 5],          # constant row: var 0 -> 0 (then + b)
                  [0, 0, 0, 8]], np.float32)  # mean 2, var (3*4 + 36)/4 = 12
    Y = oracle_mod.layer_norm(X, gb)
    r1 = 1.0 / np.sqrt(1.0 + 1e-5)
    assert np.array_equal(Y[0], np.array([-r1, r1, -r1, r1]))
    assert np.array_equal(Y[1], np.zeros(4))
    r3 = 1.0 / np.sqrt(12.0 + 1e-5)
    assert np.allclose(Y[2], np.array([-2, -2, -2, 6]) * r3, rtol=1e-15, atol=0)
    # gamma scales, beta shifts, per column
    gb2 = np.array([2, -1, 0.5, 1, 10, 20, 30, 40], np.float32)
    Y2 = oracle_mod.layer_norm(X[:1], gb2)
    assert np.array_equal(Y2[0], np.array([-2 * r1 + 10, -r1 + 20, -0.5 * r1 + 30, r1 + 40]))


def test_layer_norm_invariants(oracle_mod):
    """Unit gamma, zero beta: every row has mean 0 and variance var/(var + eps)."""
    g = synth.rng(8)
    X = synth.normal_f32(g, (5, 1000), 3.0) + np.float32(7.0)
    gb = np.concatenate([np.ones(1000, np.float32), np.zeros(1000, np.float32)])
    Y = oracle_mod.layer_norm(X, gb)
    x = X.astype(np.float64)
    var = x.var(axis=1)
    assert np.allclose(Y.mean(axis=1), 0.0, atol=1e-12)
    assert np.allclose((Y ** 2).mean(axis=1), var / (var + 1e-5), rtol=1e-12)


def test_bad_arguments(oracle_mod):
    img = np.zeros((2, 34), np.uint8)
    with pytest.raises(ValueError):
        oracle_mod.gemm(1, 2, 40, Q8_0, 0, np.zeros((1, 40), np.float32), img)
    with pytest.raises(ValueError):
        oracle_mod.gemm(1, 2, 32, Q8_0, BIAS, np.zeros((1, 32), np.float32), img)


# ------------------------------------------------------------------- MoE --

def test_moe_scaled_identity_routing(oracle_mod):
    """Expert e = (e+1)*2^-6 * I, so Y[t][s] = (ids[t][s]+1)*2^-6 * X[t] exactly."""
    E, k, n_tok, topk = 8, 64, 5, 3
    imgs = []
    for e in range(E):
        d = np.full((k, k // 32), synth.f16_bits((e + 1) * 2.0 ** -6)[()], np.uint16)
        q = np.zeros((k, k), np.int8)
        np.fill_diagonal(q, 1)
        imgs.append(synth.encode_q8_0(d, q))
    bank = np.stack(imgs)
    g = synth.rng(5)
    X = synth.normal_f32(g, (n_tok, k))
    ids = synth.moe_ids(g, n_tok, topk, E)
    Y, _ = oracle_mod.moe(n_tok, topk, E, k, k, Q8_0, 0, X, bank, ids)
    for t in range(n_tok):
        for s in range(topk):
            want = (ids[t, s] + 1) * 2.0 ** -6 * X[t].astype(np.float64)
            assert (Y[t * topk + s] == want).all()


def test_moe_bias_per_expert_and_bad_id(oracle_mod):
    E, m, k = 3, 4, 32
    d = np.full((E * m, 1), 0x3C00, np.uint16)
    bank = synth.encode_q4_0(d, np.full((E * m, k), 8, np.uint8)).reshape(E, m, -1)  # W = 0
    bias = np.arange(E * m, dtype=np.float32).reshape(E, m)
    ids = np.array([[2, 0], [1, 2]], np.int32)
    X = np.ones((2, k), np.float32)
    Y, _ = oracle_mod.moe(2, 2, E, m, k, Q4_0, BIAS, X, bank, ids, bias=bias)
    for q, e in enumerate(ids.reshape(-1)):
        assert (Y[q] == bias[e]).all()
    with pytest.raises(ValueError):
        oracle_mod.moe(2, 2, E, m, k, Q4_0, 0, X, bank, np.array([[0, 3], [1, 2]], np.int32))


def test_synth_ids_distinct_and_in_range():
    ids = synth.moe_ids(synth.rng(5), 16, 6, 64)
    assert ids.shape == (16, 6) and ids.min() >= 0 and ids.max() < 64
    assert all(len(set(row)) == 6 for row in ids.tolist())


# ------------------------------------------------------- embedding row gather --
# wavo 0.3.0 src/gpu/mod.rs, Recorder::embed: out = W[id] + pos + bias.  Closed
# forms: tables whose row r holds a value that depends only on r (and on the
# column), so the gathered rows, and their sums with pos and bias, are known
# without dequantising anything.

def _embed_tables(rows, k):
    """One table per format whose element (r, j) is known in closed form."""
    r = np.arange(rows)[:, None] * np.ones((1, k))
    j = np.ones((rows, 1)) * (np.arange(k)[None, :] % 4)
    v_bf16 = r + j                                  # small integers: exact in bf16
    bf = synth.bf16_pairs(synth.bf16_bits_rne(v_bf16.astype(np.float32)))
    # Q8_0: d = 1, q = (r % 100) - 50 + j  ->  value q
    q8 = ((r % 100) - 50 + j).astype(np.int8)
    img8 = synth.encode_q8_0(np.full((rows, k // 32), synth.f16_bits(1.0)[()], np.uint16), q8)
    # Q4_0: d = 0.5, code = 8 + (r % 8) - j  ->  value 0.5 * ((r % 8) - j)
    c4 = (8 + (r % 8) - j).astype(np.uint8)
    img4 = synth.encode_q4_0(np.full((rows, k // 32), synth.f16_bits(0.5)[()], np.uint16), c4)
    return {BF16: (bf, v_bf16), Q8_0: (img8, q8.astype(np.float64)),
            Q4_0: (img4, 0.5 * ((r % 8) - j))}


@pytest.mark.parametrize("wtype", [BF16, Q8_0, Q4_0])
def test_embed_gathers_rows_in_closed_form(oracle_mod, wtype):
    rows, k = 120, 96
    img, value = _embed_tables(rows, k)[wtype]
    ids = np.array([7, 0, 119, 7, 63], np.int32)
    out, valid = oracle_mod.embed(len(ids), rows, k, wtype, img, ids)
    assert valid.all()
    assert (out == value[ids]).all()


def test_embed_adds_pos_then_bias(oracle_mod):
    """The page's test picks id 1 of [5, 7] with the second position row of pos and
    the first k bias values; here with integers, so every sum is exact."""
    rows, k = 100, 64
    img, value = _embed_tables(rows, k)[BF16]
    pos_tab = np.arange(2 * k, dtype=np.float32) * 3.0      # two position rows
    bias = -np.arange(rows, dtype=np.float32)              # the table's bias (rows values)
    ids = np.array([5, 7], np.int32)
    out, valid = oracle_mod.embed(1, rows, k, BF16, img, ids[1:], pos=pos_tab[k:2 * k],
                                  bias=bias[:k])
    want = value[7] + 3.0 * np.arange(k, 2 * k) - np.arange(k)
    assert valid.all() and (out[0] == want).all()


def test_embed_leaves_rows_of_bad_ids(oracle_mod):
    rows, k = 10, 32
    img, value = _embed_tables(rows, k)[Q4_0]
    ids = np.array([3, -1, 10, 9], np.int32)
    init = np.full((4, k), 42.0)
    out, valid = oracle_mod.embed(4, rows, k, Q4_0, img, ids, init=init)
    assert valid.tolist() == [True, False, False, True]
    assert (out[1] == 42.0).all() and (out[2] == 42.0).all()
    assert (out[0] == value[3]).all() and (out[3] == value[9]).all()


# ----------------------------------------------- F16 / F32 weights (wavo ty 1 / 0) --

@pytest.mark.parametrize("wtype", [synth.WTYPE_F16, synth.WTYPE_F32])
def test_plain_float_weights_dequantise_like_numpy(oracle_mod, wtype):
    """wavo's F16 and F32 weight types are IEEE elements row after row: the oracle's
    decode equals numpy's own conversions, specials included."""
    g = synth.rng(31)
    m, k = 9, 40
    img = synth.draw_weights(g, wtype, m, k, std=3.0)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, 65504.0, 2.0 ** -24, -(2.0 ** -14)])
    if wtype == synth.WTYPE_F16:
        img[0, :2 * len(specials)] = specials.astype(np.float16).view(np.uint8)
        want = img.view(np.float16).astype(np.float64)
    else:
        img[0, :4 * len(specials)] = specials.astype(np.float32).view(np.uint8)
        want = img.view(np.float32).astype(np.float64)
    got = oracle_mod.dequant(wtype, m, k, img)
    assert np.array_equal(got, want.reshape(m, k))


@pytest.mark.parametrize("wtype", [synth.WTYPE_F16, synth.WTYPE_F32])
def test_plain_float_weights_exact_integer_gemm(oracle_mod, wtype):
    """Small integers are exact in f16 and f32: the oracle's GEMM equals integer
    brute force."""
    g = synth.rng(32)
    n, m, k = 3, 5, 24
    Wv = g.integers(-9, 10, size=(m, k))
    X = g.integers(-9, 10, size=(n, k)).astype(np.float32)
    img = (Wv.astype(np.float16) if wtype == synth.WTYPE_F16 else Wv.astype(np.float32))
    img = img.view(np.uint8).reshape(m, -1)
    Y, _ = oracle_mod.gemm(n, m, k, wtype, 0, X, img)
    assert (Y == X.astype(np.int64) @ Wv.T).all()
