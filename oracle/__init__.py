"""f64 CPU oracle for the weight-format contraction (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package.  The C source ``wq_oracle.c`` is
compiled with gcc into ``oracle/_build/liboracle.so`` on first use and loaded
with ctypes.  It shares no code with the CUDA library.

Every function here is a thin ctypes marshaller; the arithmetic is in the C
file, which cites the definition each step follows.

Parity pins: every function is pinned by the ``not gpu`` tests in
``tests/test_oracle.py`` (hand-worked blocks, exhaustive comparisons against
numpy/torch format conversions, identity and one-hot weights, the wavo probe's
closed form, exact integer brute force, erf-GELU closed forms, MoE routing
closed forms, embedding gathers from tables with closed-form rows).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, Q8_0, Q4_0, F16, F32 = 0, 1, 2, 3, 4
BIAS, GELU, RESIDUAL = 1, 2, 4


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, OpenMP, no fast-math, no FP contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f64, u16 = ctypes.c_double, ctypes.c_uint16
            vp, ci, cu = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
            lib.oracle_half_to_f64.argtypes = [u16]
            lib.oracle_half_to_f64.restype = f64
            lib.oracle_bf16_to_f64.argtypes = [u16]
            lib.oracle_bf16_to_f64.restype = f64
            lib.oracle_round_bf16.argtypes = [f64]
            lib.oracle_round_bf16.restype = f64
            lib.oracle_gelu.argtypes = [f64]
            lib.oracle_gelu.restype = f64
            lib.oracle_dequant.argtypes = [ci, ci, ci, vp, vp]
            lib.oracle_dequant.restype = ci
            lib.oracle_gemm.argtypes = [ci, ci, ci, ci, cu, ci, vp, vp, vp, vp, vp, vp, ci, ci, ci]
            lib.oracle_gemm.restype = ci
            lib.oracle_gemm_alpha.argtypes = [ci, ci, ci, ci, cu, ci, f64, vp, vp, vp, vp, vp, vp,
                                              ci, ci, ci]
            lib.oracle_gemm_alpha.restype = ci
            lib.oracle_gemm_dual.argtypes = [ci, ci, ci, ci, ci, cu, ci, f64, vp, vp, vp, vp, vp,
                                             vp, vp, ci, ci, ci]
            lib.oracle_gemm_dual.restype = ci
            lib.oracle_moe.argtypes = [ci, ci, ci, ci, ci, ci, cu, vp, vp, vp, vp, vp, vp, vp,
                                       ci, ci, ci]
            lib.oracle_moe.restype = ci
            lib.oracle_layer_norm.argtypes = [ci, ci, vp, vp, vp]
            lib.oracle_layer_norm.restype = ci
            lib.oracle_embed.argtypes = [ci, ci, ci, ci, vp, vp, vp, vp, vp, vp]
            lib.oracle_embed.restype = ci
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def half_to_f64(bits: int) -> float:
    return float(_load().oracle_half_to_f64(int(bits) & 0xFFFF))


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits) & 0xFFFF))


def round_bf16(x: float) -> float:
    return float(_load().oracle_round_bf16(float(x)))


def gelu(v: float) -> float:
    return float(_load().oracle_gelu(float(v)))


def layer_norm(X: np.ndarray, gb: np.ndarray) -> np.ndarray:
    """f64 row LayerNorm of f32 X [n][k] with gb = [gamma (k) | beta (k)], eps 1e-5."""
    Xc, gc = _c(X, np.float32), _c(gb, np.float32)
    n, k = Xc.shape
    assert gc.size == 2 * k
    Y = np.empty((n, k), dtype=np.float64)
    if _load().oracle_layer_norm(n, k, _ptr(Xc), _ptr(gc), _ptr(Y)) != 0:
        raise ValueError("oracle_layer_norm: bad arguments")
    return Y


def dequant(wtype: int, m: int, k: int, W: np.ndarray) -> np.ndarray:
    """f64 ``[m][k]`` weights from the byte image ``W``."""
    Wb = _c(W, np.uint8)
    out = np.empty((m, k), dtype=np.float64)
    rc = _load().oracle_dequant(wtype, m, k, _ptr(Wb), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_dequant: bad arguments (wtype={wtype}, m={m}, k={k})")
    return out


def gemm(n, m, k, wtype, flags, X, W, bias=None, residual=None, round_x=False,
         rows=None, threads=0, bound=True, round_w=False, alpha=1.0, dual=0, bias2=None):
    """f64 ``(Y, S)`` of ``epi(X . W^T)``, each ``[n][m + dual]``.

    ``alpha`` scales the contribution before the residual is added (wavo's
    ``Residual(alpha)``: ``Y = R + alpha * act(X . W^T + bias)``); S scales with it.

    ``dual`` (wavo's dual outputs): columns ``m + j`` for ``j < dual`` hold the
    plain sum of output ``j`` plus ``bias2[j]``, with no activation, alpha or
    residual; ``residual`` then has rows of ``m + dual`` values too.

    ``round_x`` / ``round_w`` feed X / the dequantised W rounded to the nearest
    bf16 (ties to even): the operands of the tensor-core path.

    ``rows=(j0, j1)`` restricts the computed outputs to those of W rows
    ``[j0, j1)`` (with their dual columns); the rest of Y and S stays NaN.
    """
    Xc, Wc = _c(X, np.float32), _c(W, np.uint8)
    bc, Rc, b2c = _c(bias, np.float32), _c(residual, np.float32), _c(bias2, np.float32)
    ld = m + dual
    Y = np.full((n, ld), np.nan, dtype=np.float64)
    S = np.full((n, ld), np.nan, dtype=np.float64) if bound else None
    j0, j1 = (0, m) if rows is None else rows
    rnd = int(bool(round_x)) | (int(bool(round_w)) << 1)
    rc = _load().oracle_gemm_dual(n, m, k, int(dual), wtype, flags, rnd, float(alpha), _ptr(Xc),
                                  _ptr(Wc), _ptr(bc), _ptr(b2c), _ptr(Rc), _ptr(Y), _ptr(S), j0,
                                  j1, int(threads))
    if rc != 0:
        raise ValueError("oracle_gemm: bad arguments")
    return Y, S


def moe(n_tok, topk, n_experts, m, k, wtype, flags, X, Wbank, ids, bias=None, residual=None,
        slots=None, threads=0, bound=True):
    """f64 ``(Y [n_tok*topk][m], S)`` of the routed matvec; ``slots=(q0, q1)`` restricts."""
    Xc, Wc = _c(X, np.float32), _c(Wbank, np.uint8)
    ic = _c(ids, np.int32)
    bc, Rc = _c(bias, np.float32), _c(residual, np.float32)
    nq = n_tok * topk
    Y = np.full((nq, m), np.nan, dtype=np.float64)
    S = np.full((nq, m), np.nan, dtype=np.float64) if bound else None
    q0, q1 = (0, nq) if slots is None else slots
    rc = _load().oracle_moe(n_tok, topk, n_experts, m, k, wtype, flags, _ptr(Xc), _ptr(Wc),
                            _ptr(ic), _ptr(bc), _ptr(Rc), _ptr(Y), _ptr(S), q0, q1, int(threads))
    if rc == -2:
        raise ValueError("oracle_moe: expert id out of range")
    if rc != 0:
        raise ValueError("oracle_moe: bad arguments")
    return Y, S


def embed(n_ids, rows, k, wtype, W, ids, pos=None, bias=None, init=None):
    """f64 ``(out [n_ids][k], valid [n_ids])``: row ``ids[t]`` of the table ``W``
    (``rows`` x ``k``) + ``pos[t]`` + ``bias``.  Rows of invalid ids keep ``init``
    (NaN when not given)."""
    Wc, ic = _c(W, np.uint8), _c(ids, np.int32)
    pc, bc = _c(pos, np.float32), _c(bias, np.float32)
    out = (np.full((n_ids, k), np.nan, dtype=np.float64) if init is None
           else np.array(init, dtype=np.float64).reshape(n_ids, k).copy())
    valid = np.zeros(n_ids, dtype=np.int32)
    rc = _load().oracle_embed(n_ids, rows, k, wtype, _ptr(Wc), _ptr(ic), _ptr(pc), _ptr(bc),
                              _ptr(out), _ptr(valid))
    if rc != 0:
        raise ValueError("oracle_embed: bad arguments")
    return out, valid.astype(bool)
