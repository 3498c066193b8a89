"""wq_moe_gemv beyond one routing window of WQ_MOE_WINDOW_SLOTS slots: a prompt
of 512 tokens at top-6 (3,072 slots, twelve windows) and the degenerate routing
where one expert takes every slot, on the tensor-core kernel (Q8_0/Q4_0 with
k % 256 == 0) and on the weight-streaming kernel (bf16, and Q4_0 with
k % 256 != 0), element by element against the oracle.
"""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, assert_within, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu

BF16, Q8_0, Q4_0 = wq.WQ_BF16, wq.WQ_Q8_0, wq.WQ_Q4_0
BIAS, RES = wq.WQ_BIAS, wq.WQ_RESIDUAL
TAU = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run(oracle_mod, n_tok, topk, E, m, k, wtype, flags, ids, seed):
    g = synth.rng(seed)
    bank = synth.draw_weights(g, wtype, E * m, k).reshape(E, m, -1)
    X = synth.normal_f32(g, (n_tok, k))
    bias = synth.normal_f32(g, (E, m), 0.1) if flags & BIAS else None
    R = synth.normal_f32(g, (n_tok * topk, m)) if flags & RES else None
    out = Guarded(n_tok * topk * m)
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, flags, dev(X),
                            weights_dev(bank, wtype, E * m, k), dev(ids),
                            None if bias is None else dev(bias),
                            None if R is None else dev(R), out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    status_ok()
    Yref, S = oracle_mod.moe(n_tok, topk, E, m, k, wtype, flags, X, bank, ids, bias=bias,
                             residual=R)
    Y = out.result().reshape(Yref.shape)
    # the epilogue's rounding allowance sees |bias| of each slot's expert and |R|
    extra = np.zeros(Yref.shape)
    if bias is not None:
        extra += np.abs(bias[ids.reshape(-1)])
    if R is not None:
        extra += np.abs(R)
    assert_within(Y, Yref, S, TAU, R=extra, what=f"moe windows wtype={wtype} slots={n_tok * topk}")


@pytest.mark.parametrize("wtype,k", [(Q4_0, 2048), (Q8_0, 1024), (BF16, 520), (Q4_0, 1056)])
def test_moe_512_tokens_top6(oracle_mod, wtype, k):
    n_tok, topk, E, m = 512, 6, 64, 72
    g = synth.rng(900 + wtype)
    ids = synth.moe_ids(g, n_tok, topk, E)
    run(oracle_mod, n_tok, topk, E, m, k, wtype, BIAS | RES, ids, 901 + wtype + k)


@pytest.mark.parametrize("wtype,k", [(Q4_0, 1024), (Q8_0, 512), (BF16, 264)])
def test_moe_one_expert_takes_every_slot(oracle_mod, wtype, k):
    n_tok, topk, E, m = 1024, 3, 8, 40
    ids = np.full((n_tok, topk), 5, np.int32)
    run(oracle_mod, n_tok, topk, E, m, k, wtype, 0, ids, 950 + wtype + k)


def test_moe_window_edge(oracle_mod):
    """257 slots: one full window and a window of one slot."""
    n_tok, topk, E, m, k = 257, 1, 7, 33, 512
    g = synth.rng(977)
    ids = g.integers(0, E, size=(n_tok, topk)).astype(np.int32)
    run(oracle_mod, n_tok, topk, E, m, k, Q4_0, BIAS, ids, 978)


@pytest.mark.parametrize("wtype,k", [(Q4_0, 256),   # tensor-core MoE (quantised)
                                     (BF16, 256),   # tensor-core MoE (bf16)
                                     (Q4_0, 32)])   # weight-streaming MoE
def test_moe_bank_of_2_24_experts(oracle_mod, wtype, k):
    """A bank of 2^24 + 5 one-row experts: expert ids no longer fit the 24 bits of
    the compact routing key, so the window is sorted with 64-bit keys.  The bank is
    zero but for the rows the ids select (ids near both ends of the range); the
    oracle runs on those rows alone, with the ids renumbered."""
    E, m, n_tok, topk = (1 << 24) + 5, 1, 5, 3
    g = synth.rng(4242 + wtype + k)
    ids = np.array([[0, E - 1, 7], [E - 1, 3, 1 << 23], [E - 2, 0, 5],
                    [1 << 24, 9, E - 3], [2, (1 << 24) - 1, 11]], np.int32)
    used = np.unique(ids)
    small = synth.draw_weights(g, wtype, len(used) * m, k).reshape(len(used), m, -1)
    sb = np.ascontiguousarray(small).view(np.uint8).reshape(len(used), -1)  # bytes per expert
    bank = torch.zeros(wq.wq_weight_bytes(wtype, E * m, k), dtype=torch.uint8, device="cuda")
    rows = bank[:E * sb.shape[1]].view(E, sb.shape[1])
    rows[torch.from_numpy(used.astype(np.int64)).cuda()] = dev(sb)
    X = synth.normal_f32(g, (n_tok, k))
    out = Guarded(n_tok * topk * m)
    wq.check(wq.wq_moe_gemv(n_tok, topk, E, m, k, wtype, 0, dev(X), bank, dev(ids), None, None,
                            out.view), "wq_moe_gemv")
    torch.cuda.synchronize()
    status_ok()
    remap = {int(e): i for i, e in enumerate(used)}
    ids_small = np.vectorize(remap.get)(ids).astype(np.int32)
    Yref, S = oracle_mod.moe(n_tok, topk, len(used), m, k, wtype, 0, X, small, ids_small)
    Y = out.result().reshape(Yref.shape)
    assert_within(Y, Yref, S, TAU, what=f"moe 2^24 experts wtype={wtype} k={k}")
    del bank, rows
    torch.cuda.empty_cache()
