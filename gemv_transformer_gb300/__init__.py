"""Python binding of libwq (the weight-format GEMM/GEMV library for sm_103a).

Argument marshalling only: every function forwards to the C entry point of the
same name in ``_build/libwq.so`` (declared in ``include/wq.h``); all the work runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is not
built, or no CUDA device is present, the calls raise.

Tensor arguments may be ``torch.Tensor`` (device memory) or raw integer device
pointers; ``stream`` may be a ``torch.cuda.Stream``, a raw ``cudaStream_t``
integer, or ``None`` for torch's current stream on the current device.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libwq.so")

WQ_BF16, WQ_Q8_0, WQ_Q4_0, WQ_F16, WQ_F32 = 0, 1, 2, 3, 4
WQ_BIAS, WQ_GELU, WQ_RESIDUAL, WQ_TC_BF16 = 1, 2, 4, 256
WQ_SILU, WQ_RELU, WQ_TANH = 8, 16, 32
WQ_OK, WQ_ERR_INVALID_ARG, WQ_ERR_UNSUPPORTED, WQ_ERR_CUDA = 0, 1, 2, 3
WQ_ERR_DEVICE_TIMEOUT, WQ_ERR_BAD_EXPERT, WQ_ERR_TOO_LARGE, WQ_ERR_BAD_INDEX = 4, 5, 6, 7
WQ_GEMM_NOALLOC_SCRATCH_BYTES = 16 << 20
WQ_GEMV_MAX_N = 16
WQ_MOE_WINDOW_SLOTS = 256

EXPORTS = ("wq_gemm", "wq_gemm_ws", "wq_gemm_alpha", "wq_gemm_dual", "wq_gemm_workspace_bytes",
           "wq_gemm_noalloc",
           "wq_gemm_ln_ws", "wq_gemm_ln_workspace_bytes", "wq_gemv",
           "wq_moe_gemv", "wq_weight_bytes", "wq_dequantize", "wq_embed", "wq_get_device_status",
           "wq_status_string", "wq_set_wait_limit")

_lock = threading.Lock()
_lib = None


class WqError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {wq_status_string(status)} ({status})" if what
                         else f"{wq_status_string(status)} ({status})")


def _open(path: str):
    """Open a libwq build and declare its signatures (raises if the file is missing)."""
    if not os.path.exists(path):
        raise RuntimeError(f"libwq is not built ({path} missing): run "
                           "gemv_transformer_gb300.build.build()")
    lib = ctypes.CDLL(path)
    ci, cu, vp, sz = ctypes.c_int, ctypes.c_uint, ctypes.c_void_p, ctypes.c_size_t
    gemm_args = [ci, ci, ci, ci, cu, vp, vp, vp, vp, vp, vp]
    lib.wq_gemm.argtypes = gemm_args
    lib.wq_gemm.restype = ci
    lib.wq_gemv.argtypes = gemm_args
    lib.wq_gemv.restype = ci
    lib.wq_gemm_ln_ws.argtypes = gemm_args[:6] + [vp] + gemm_args[6:-1] + [vp, sz, vp]
    lib.wq_gemm_ln_ws.restype = ci
    lib.wq_gemm_ln_workspace_bytes.argtypes = [ci, ci, ci, ci, cu]
    lib.wq_gemm_ln_workspace_bytes.restype = sz
    lib.wq_gemm_noalloc.argtypes = gemm_args
    lib.wq_gemm_noalloc.restype = ci
    lib.wq_gemm_ws.argtypes = gemm_args[:-1] + [vp, sz, vp]
    lib.wq_gemm_ws.restype = ci
    lib.wq_gemm_workspace_bytes.argtypes = [ci, ci, ci, ci, cu]
    lib.wq_gemm_workspace_bytes.restype = sz
    lib.wq_moe_gemv.argtypes = [ci, ci, ci, ci, ci, ci, cu, vp, vp, vp, vp, vp, vp, vp]
    lib.wq_moe_gemv.restype = ci
    lib.wq_weight_bytes.argtypes = [ci, ci, ci]
    lib.wq_weight_bytes.restype = sz
    lib.wq_dequantize.argtypes = [ci, ci, ci, vp, vp, vp]
    lib.wq_dequantize.restype = ci
    lib.wq_gemm_alpha.argtypes = [ci, ci, ci, ci, ctypes.c_uint, ctypes.c_float, vp, vp, vp, vp,
                                  vp, vp, sz, vp]
    lib.wq_gemm_alpha.restype = ci
    lib.wq_gemm_dual.argtypes = [ci, ci, ci, ci, ci, ctypes.c_uint, ctypes.c_float, vp, vp, vp, vp,
                                 vp, vp, vp, sz, vp]
    lib.wq_gemm_dual.restype = ci
    lib.wq_embed.argtypes = [ci, ci, ci, ci, vp, vp, vp, vp, vp, vp]
    lib.wq_embed.restype = ci
    lib.wq_get_device_status.argtypes = [vp]
    lib.wq_get_device_status.restype = ci
    lib.wq_status_string.argtypes = [ci]
    lib.wq_status_string.restype = ctypes.c_char_p
    lib.wq_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.wq_set_wait_limit.restype = None
    return lib


def load():
    """The process-wide libwq handle (raises if the library has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIB_PATH)
        return _lib


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def wq_gemm(n, m, k, wtype, flags, X, W, bias=None, residual=None, Y=None, stream=None) -> int:
    return load().wq_gemm(n, m, k, wtype, flags, _p(X), _p(W), _p(bias), _p(residual), _p(Y),
                          _s(stream))


def wq_gemm_ws(n, m, k, wtype, flags, X, W, bias=None, residual=None, Y=None, workspace=None,
               workspace_bytes=0, stream=None) -> int:
    return load().wq_gemm_ws(n, m, k, wtype, flags, _p(X), _p(W), _p(bias), _p(residual), _p(Y),
                             _p(workspace), int(workspace_bytes), _s(stream))


def wq_gemm_noalloc(n, m, k, wtype, flags, X, W, bias=None, residual=None, Y=None,
                    stream=None) -> int:
    return load().wq_gemm_noalloc(n, m, k, wtype, flags, _p(X), _p(W), _p(bias), _p(residual),
                                  _p(Y), _s(stream))


def wq_gemm_ln_ws(n, m, k, wtype, flags, X, ln_gb, W, bias=None, residual=None, Y=None,
                  workspace=None, workspace_bytes=0, stream=None) -> int:
    return load().wq_gemm_ln_ws(n, m, k, wtype, flags, _p(X), _p(ln_gb), _p(W), _p(bias),
                                _p(residual), _p(Y), _p(workspace), int(workspace_bytes),
                                _s(stream))


def wq_gemm_ln_workspace_bytes(n, m, k, wtype, flags) -> int:
    return int(load().wq_gemm_ln_workspace_bytes(n, m, k, wtype, flags))


def wq_gemm_workspace_bytes(n, m, k, wtype, flags) -> int:
    return int(load().wq_gemm_workspace_bytes(n, m, k, wtype, flags))


def wq_gemv(n, m, k, wtype, flags, X, W, bias=None, residual=None, Y=None, stream=None) -> int:
    return load().wq_gemv(n, m, k, wtype, flags, _p(X), _p(W), _p(bias), _p(residual), _p(Y),
                          _s(stream))


def wq_moe_gemv(n_tok, topk, n_experts, m, k, wtype, flags, X, Wbank, ids, bias=None,
                residual=None, Y=None, stream=None) -> int:
    return load().wq_moe_gemv(n_tok, topk, n_experts, m, k, wtype, flags, _p(X), _p(Wbank),
                              _p(ids), _p(bias), _p(residual), _p(Y), _s(stream))


def wq_weight_bytes(wtype, m, k) -> int:
    return int(load().wq_weight_bytes(wtype, m, k))


def wq_dequantize(wtype, m, k, W, out, stream=None) -> int:
    return load().wq_dequantize(wtype, m, k, _p(W), _p(out), _s(stream))


def wq_gemm_alpha(n, m, k, wtype, flags, alpha, X, W, bias=None, residual=None, Y=None,
                  workspace=None, workspace_bytes=0, stream=None) -> int:
    return load().wq_gemm_alpha(n, m, k, wtype, flags, float(alpha), _p(X), _p(W), _p(bias),
                                _p(residual), _p(Y), _p(workspace), int(workspace_bytes),
                                _s(stream))


def wq_gemm_dual(n, m, k, dual, wtype, flags, alpha, X, W, bias=None, bias2=None, residual=None,
                 Y=None, workspace=None, workspace_bytes=0, stream=None) -> int:
    return load().wq_gemm_dual(n, m, k, dual, wtype, flags, float(alpha), _p(X), _p(W), _p(bias),
                               _p(bias2), _p(residual), _p(Y), _p(workspace), int(workspace_bytes),
                               _s(stream))


def wq_embed(n_ids, rows, k, wtype, W, ids, pos=None, bias=None, out=None, stream=None) -> int:
    return load().wq_embed(n_ids, rows, k, wtype, _p(W), _p(ids), _p(pos), _p(bias), _p(out),
                           _s(stream))


def wq_get_device_status(stream=None) -> int:
    return load().wq_get_device_status(_s(stream))


def wq_status_string(status) -> str:
    return load().wq_status_string(int(status)).decode()


def wq_set_wait_limit(polls: int) -> None:
    load().wq_set_wait_limit(int(polls))


def check(status: int, what: str = "") -> None:
    """Raise WqError unless ``status`` is WQ_OK."""
    if status != WQ_OK:
        raise WqError(status, what)
