"""The five workloads at their full sizes, through the C ABI, in the launch
configuration the benchmark times, against the f64 oracle.

The oracle computes every output of every workload, the encoder GEMMs
(1500 x 3072/4096/1024, k up to 4096) included: each of their outputs is
compared against the oracle on unrounded X at tau = 8e-3 and against the oracle
fed bf16(X) at tau = (k/16 + 32) * 2^-23 (the kernel's own arithmetic).  The
oracle's results for an encoder GEMM are computed once and shared by the two
routes that run it.
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run(fn, w, flags_extra=0):
    n, m, k = w["n"], w["m"], w["k"]
    out = Guarded(n * m)
    b = dev(w["bias"]) if w["bias"] is not None else None
    R = dev(w["residual"]) if w["residual"] is not None else None
    args = (n, m, k, w["wtype"], w["flags"] | flags_extra, dev(w["X"]),
            weights_dev(w["W"], w["wtype"], m, k), b, R, out.view)
    if fn is wq.wq_gemm_ws:
        need = wq.wq_gemm_workspace_bytes(n, m, k, w["wtype"], w["flags"] | flags_extra)
        work = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        st = fn(*args, work, need)
    else:
        st = fn(*args)
    wq.check(st, w["name"])
    torch.cuda.synchronize()
    status_ok()
    return out.result().reshape(n, m)


def check_full(oracle_mod, w, fn):
    Y = run(fn, w)
    Yref, S = oracle_mod.gemm(w["n"], w["m"], w["k"], w["wtype"], w["flags"], w["X"], w["W"],
                              bias=w["bias"], residual=w["residual"])
    return assert_within(Y, Yref, S, TAU, gelu=bool(w["flags"] & wq.WQ_GELU), bias=w["bias"],
                         R=w["residual"], what=w["name"])


def test_bf16_gemm_bias_gelu(oracle_mod):
    check_full(oracle_mod, synth.workload_bf16_gemm(), wq.wq_gemm)


def test_q8_0_gemv(oracle_mod):
    check_full(oracle_mod, synth.workload_q8_0_gemv(), wq.wq_gemv)


@pytest.mark.parametrize("n", [1, 4, 8])
def test_q4_0_gemv_residual(oracle_mod, n):
    check_full(oracle_mod, synth.workload_q4_0_gemv(n=n), wq.wq_gemv)


_ORACLE_CACHE = {}


def encoder_oracle(oracle_mod, which, w, round_x):
    key = (which, round_x)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle_mod.gemm(w["n"], w["m"], w["k"], w["wtype"], w["flags"],
                                             w["X"], w["W"], bias=w["bias"],
                                             residual=w["residual"], round_x=round_x)
    return _ORACLE_CACHE[key]


@pytest.mark.parametrize("fn", [wq.wq_gemm, wq.wq_gemm_ws], ids=["fused", "workspace"])
@pytest.mark.parametrize("which", [0, 1, 2])
def test_encoder_gemm_tc(oracle_mod, which, fn):
    w = synth.workload_encoder_gemms()[which]
    k = w["k"]
    Y = run(fn, w, flags_extra=wq.WQ_TC_BF16)
    assert np.isfinite(Y).all()
    for round_x, tau in ((False, 8e-3), (True, (k / 16 + 32) * 2.0 ** -23)):
        Yref, S = encoder_oracle(oracle_mod, which, w, round_x)
        assert_within(Y, Yref, S, tau, gelu=bool(w["flags"] & wq.WQ_GELU), bias=w["bias"],
                      R=w["residual"], what=f"{w['name']} round_x={round_x}")


def test_moe_q4_0(oracle_mod):
    w = synth.workload_moe()
    E, m, k, nt, tk = w["n_experts"], w["m"], w["k"], w["n_tok"], w["topk"]
    out = Guarded(nt * tk * m)
    st = wq.wq_moe_gemv(nt, tk, E, m, k, w["wtype"], w["flags"], dev(w["X"]),
                        weights_dev(w["W"], w["wtype"], E * m, k), dev(w["ids"]), None, None,
                        out.view)
    wq.check(st, w["name"])
    torch.cuda.synchronize()
    status_ok()
    Y = out.result().reshape(nt * tk, m)
    Yref, S = oracle_mod.moe(nt, tk, E, m, k, w["wtype"], w["flags"], w["X"], w["W"], w["ids"])
    assert_within(Y, Yref, S, TAU, what=w["name"])
