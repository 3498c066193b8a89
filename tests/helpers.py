"""Shared helpers of the parity tests: device buffers, canaries, the tolerance.

Tolerance (per output element, f32-FMA paths tau = 1e-5, tensor-core path
tau = 8e-3 against unrounded X):

    |Y - Y_ref| <= tau * L * S + 2^-21 * (|Y_ref| + |bias_j| + |R_ij|)

S = sum_k |x||w| (the oracle's bound), L = 1.13 (the largest slope of erf-GELU)
when GELU is applied, else 1.  The second term covers the f32 rounding of the
epilogue's adds and of the GELU evaluation, which sum|x||w| does not see
(bias and residual are not part of the contraction).
"""
from __future__ import annotations

import numpy as np
import torch

import gemv_transformer_gb300 as wq

CANARY = 64  # guard floats on each side of an output


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def weights_dev(img: np.ndarray, wtype: int, m: int, k: int) -> torch.Tensor:
    """Device copy of a weight byte image, padded to wq_weight_bytes."""
    need = wq.wq_weight_bytes(wtype, m, k)
    flat = np.ascontiguousarray(img, dtype=np.uint8).reshape(-1)
    assert flat.size <= need
    buf = np.zeros(need, np.uint8)
    buf[:flat.size] = flat
    return dev(buf)


class Guarded:
    """An f32 output of `count` elements between two NaN-pattern guard zones."""

    def __init__(self, count: int, init: np.ndarray | None = None):
        self.count = count
        self.buf = torch.full((count + 2 * CANARY,), -1, dtype=torch.int32, device="cuda")
        self.buf = self.buf.view(torch.float32)  # 0xFFFFFFFF: a NaN bit pattern
        if init is not None:
            self.view.copy_(torch.from_numpy(np.ascontiguousarray(init, np.float32).reshape(-1)))

    @property
    def view(self) -> torch.Tensor:
        return self.buf[CANARY:CANARY + self.count]

    def result(self) -> np.ndarray:
        host = self.buf.view(torch.int32).cpu().numpy()
        assert (host[:CANARY] == -1).all(), "guard before the output was written"
        assert (host[CANARY + self.count:] == -1).all(), "guard after the output was written"
        return self.buf[CANARY:CANARY + self.count].cpu().numpy()


def assert_within(Y, Yref, S, tau, gelu=False, bias=None, R=None, what=""):
    Y = np.asarray(Y, np.float64).reshape(Yref.shape)
    L = 1.13 if gelu else 1.0
    extra = np.abs(Yref)
    if bias is not None:
        extra = extra + np.abs(np.asarray(bias, np.float64)).reshape(1, -1)
    if R is not None:
        extra = extra + np.abs(np.asarray(R, np.float64)).reshape(Yref.shape)
    tol = tau * L * S + 2.0 ** -21 * extra
    err = np.abs(Y - Yref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first "
            + ", ".join(f"{tuple(i)} got {Y[tuple(i)]!r} want {Yref[tuple(i)]!r} "
                        f"tol {tol[tuple(i)]:.3g}" for i in idx))
    return float((err / np.maximum(S, 1e-300)).max())


def status_ok():
    s = wq.wq_get_device_status()
    assert s == wq.WQ_OK, wq.wq_status_string(s)
