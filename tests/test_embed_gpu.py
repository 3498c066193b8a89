"""GPU parity of wq_embed, the embedding row gather (wavo 0.3.0 src/gpu/mod.rs,
Recorder::embed: row ids[t] of the weight table + pos[t] + bias), against the
f64 oracle: every value is a dequantised weight (exact in f32) plus at most two
f32 additions, so the tolerance is a few ulps of |w| + |pos| + |bias|."""
import numpy as np
import pytest
import torch

import gemv_transformer_gb300 as wq
import synth
from helpers import Guarded, dev, status_ok, weights_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_transformer_gb300 import build
    build.build()
    wq.load()
    yield
    status_ok()


def run_embed(rows, k, wtype, img, ids, pos=None, bias=None, init=None):
    n_ids = len(ids)
    out = Guarded(n_ids * k, init)
    st = wq.wq_embed(n_ids, rows, k, wtype, weights_dev(img, wtype, rows, k),
                     dev(np.asarray(ids, np.int32)),
                     dev(pos) if pos is not None else None,
                     dev(bias) if bias is not None else None, out.view)
    wq.check(st, "wq_embed")
    torch.cuda.synchronize()
    return out


def check(oracle_mod, rows, k, wtype, ids, with_pos, with_bias, seed):
    g = synth.rng(seed)
    img = synth.draw_weights(g, wtype, rows, k)
    pos = synth.normal_f32(g, (len(ids), k)) if with_pos else None
    bias = synth.normal_f32(g, (k,), 0.1) if with_bias else None
    out = run_embed(rows, k, wtype, img, ids, pos, bias)
    status_ok()
    want, valid = oracle_mod.embed(len(ids), rows, k, wtype, img, ids, pos=pos, bias=bias)
    assert valid.all()
    got = out.result().reshape(len(ids), k).astype(np.float64)
    mag = np.abs(oracle_mod.embed(len(ids), rows, k, wtype, img, ids)[0])
    if pos is not None:
        mag = mag + np.abs(pos.astype(np.float64))
    if bias is not None:
        mag = mag + np.abs(bias.astype(np.float64))[None, :]
    assert (np.abs(got - want) <= 2.0 ** -22 * mag).all()
    if pos is None and bias is None:  # the gathered weight alone is exact
        assert (got == want).all()


@pytest.mark.parametrize("wtype", [wq.WQ_BF16, wq.WQ_Q8_0, wq.WQ_Q4_0])
@pytest.mark.parametrize("with_pos,with_bias", [(False, False), (True, False), (False, True),
                                                (True, True)])
def test_embed_matches_oracle(oracle_mod, wtype, with_pos, with_bias):
    rows, k = 300, 96
    ids = np.array([5, 7, 0, 299, 7, 150, 31], np.int32)
    check(oracle_mod, rows, k, wtype, ids, with_pos, with_bias, seed=wtype * 10 + with_pos)


@pytest.mark.parametrize("wtype", [wq.WQ_BF16, wq.WQ_Q4_0])
def test_embed_large_table_many_ids(oracle_mod, wtype):
    """A vocabulary-sized table (151,936 rows of 1024) and 512 ids drawn over it."""
    rows, k = 151936, 1024
    g = synth.rng(77)
    ids = g.integers(0, rows, size=512).astype(np.int32)
    check(oracle_mod, rows, k, wtype, ids, True, True, seed=78)


def test_embed_bad_ids_leave_their_rows(oracle_mod):
    rows, k = 64, 64
    g = synth.rng(5)
    img = synth.draw_weights(g, wq.WQ_Q8_0, rows, k)
    ids = np.array([3, -1, 64, 63, 1 << 30], np.int32)
    init = np.full(len(ids) * k, 7.5, np.float32)
    out = run_embed(rows, k, wq.WQ_Q8_0, img, ids, init=init)
    assert wq.wq_get_device_status() == wq.WQ_ERR_BAD_INDEX
    got = out.result().reshape(len(ids), k)
    want, valid = oracle_mod.embed(len(ids), rows, k, wq.WQ_Q8_0, img, ids,
                                   init=init.reshape(len(ids), k))
    assert valid.tolist() == [True, False, False, True, False]
    assert (got.astype(np.float64) == want).all()


def test_embed_unaligned_outputs_take_the_scalar_path(oracle_mod):
    """pos, bias and out one float past a 16-byte boundary: the same values."""
    rows, k, wtype = 200, 64, wq.WQ_BF16
    g = synth.rng(9)
    img = synth.draw_weights(g, wtype, rows, k)
    ids = np.array([1, 199, 42], np.int32)
    pos = synth.normal_f32(g, (3, k))
    bias = synth.normal_f32(g, (k,), 0.1)
    pos_d = torch.zeros(3 * k + 1, device="cuda")
    pos_d[1:] = dev(pos.reshape(-1))
    bias_d = torch.zeros(k + 1, device="cuda")
    bias_d[1:] = dev(bias)
    out_d = torch.full((3 * k + 2,), -1.0, device="cuda")
    st = wq.wq_embed(3, rows, k, wtype, weights_dev(img, wtype, rows, k), dev(ids), pos_d[1:],
                     bias_d[1:], out_d[1:3 * k + 1])
    wq.check(st, "wq_embed")
    torch.cuda.synchronize()
    status_ok()
    got = out_d.cpu().numpy()
    assert got[0] == -1.0 and got[-1] == -1.0
    want, _ = oracle_mod.embed(3, rows, k, wtype, img, ids, pos=pos, bias=bias)
    mag = np.abs(want) + np.abs(pos) + np.abs(bias)[None, :]
    assert (np.abs(got[1:-1].reshape(3, k) - want) <= 2.0 ** -21 * mag).all()

