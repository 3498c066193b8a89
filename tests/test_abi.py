"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks reject bad calls before touching a device (CPU only)."""
import os
import re

import pytest

import gemv_transformer_gb300 as wq
from gemv_transformer_gb300 import build as wqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    wqbuild.build()
    return wq.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "wq.h")) as f:
        text = f.read()
    return re.findall(r"WQ_API\s+[\w\s\*]+?\b(wq_\w+)\s*\(", text)


def test_header_declares_the_binding_names():
    assert sorted(declared_functions()) == sorted(wq.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_weight_bytes():
    assert wq.wq_weight_bytes(wq.WQ_BF16, 512, 256) == 2 * 512 * 256
    assert wq.wq_weight_bytes(wq.WQ_Q8_0, 4096, 4096) == 17_825_792
    assert wq.wq_weight_bytes(wq.WQ_Q4_0, 14336, 4096) == 33_030_144
    assert wq.wq_weight_bytes(wq.WQ_Q8_0, 1, 32) == 48      # 34 rounded up to 16
    assert wq.wq_weight_bytes(wq.WQ_Q4_0, 3, 64) == 112     # 108 rounded up
    assert wq.wq_weight_bytes(wq.WQ_Q4_0, 1, 40) == 0       # k % 32
    assert wq.wq_weight_bytes(wq.WQ_BF16, 1, 12) == 0       # k % 8
    assert wq.wq_weight_bytes(7, 1, 32) == 0
    assert wq.wq_weight_bytes(wq.WQ_F16, 3, 40) == 240
    assert wq.wq_weight_bytes(wq.WQ_F32, 3, 40) == 480
    assert wq.wq_weight_bytes(wq.WQ_F16, 3, 36) == 0       # k % 8
    assert wq.wq_weight_bytes(wq.WQ_F32, 1, 12) == 0


def test_status_strings():
    for code in range(8):
        assert wq.wq_status_string(code) != "unknown status"
    assert wq.wq_status_string(99) == "unknown status"


A = 0x10000  # a 16-byte aligned fake device address: never dereferenced below


@pytest.mark.parametrize("call", [
    lambda: wq.wq_gemm(0, 8, 32, wq.WQ_Q8_0, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 0, 32, wq.WQ_Q8_0, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 40, wq.WQ_Q8_0, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 36, wq.WQ_Q4_0, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 12, wq.WQ_BF16, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 12, wq.WQ_F16, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 20, wq.WQ_F32, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, 7, 0, A, A, None, None, A, 0),      # unknown wtype
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, 64, A, A, None, None, A, 0),      # unknown flag
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, wq.WQ_GELU | wq.WQ_SILU, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, wq.WQ_RELU | wq.WQ_TANH, A, A, None, None, A, 0),
    lambda: wq.wq_gemv(1, 8, 32, wq.WQ_Q8_0, wq.WQ_SILU | wq.WQ_TANH, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, 0, None, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, 0, A, None, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, 0, A, A, None, None, None, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, wq.WQ_BIAS, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, wq.WQ_RESIDUAL, A, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, 0, A + 4, A, None, None, A, 0),
    lambda: wq.wq_gemm(1, 8, 32, wq.WQ_Q8_0, 0, A, A + 2, None, None, A, 0),
    lambda: wq.wq_gemv(17, 8, 32, wq.WQ_Q8_0, 0, A, A, None, None, A, 0),
    lambda: wq.wq_gemv(1, 8, 32, wq.WQ_BF16, wq.WQ_TC_BF16, A, A, None, None, A, 0),
    lambda: wq.wq_moe_gemv(2, 0, 4, 8, 32, wq.WQ_Q4_0, 0, A, A, A, None, None, A, 0),
    lambda: wq.wq_moe_gemv(2, 2, 0, 8, 32, wq.WQ_Q4_0, 0, A, A, A, None, None, A, 0),
    lambda: wq.wq_moe_gemv(2, 2, 4, 8, 32, wq.WQ_Q4_0, 0, A, A, None, None, None, A, 0),
    lambda: wq.wq_moe_gemv(2, 2, 4, 8, 32, wq.WQ_Q4_0, wq.WQ_TC_BF16, A, A, A, None, None, A, 0),
    lambda: wq.wq_dequantize(wq.WQ_Q8_0, 4, 40, A, A, 0),
    lambda: wq.wq_gemm_alpha(1, 8, 32, wq.WQ_Q8_0, 0, float("nan"), A, A, None, None, A, None, 0, 0),
    lambda: wq.wq_gemm_alpha(1, 8, 32, wq.WQ_Q8_0, 0, float("inf"), A, A, None, None, A, None, 0, 0),
    lambda: wq.wq_gemm_alpha(1, 8, 40, wq.WQ_Q8_0, 0, 0.5, A, A, None, None, A, None, 0, 0),
    lambda: wq.wq_gemm_alpha(1, 8, 32, wq.WQ_Q8_0, wq.WQ_RESIDUAL, 0.5, A, A, None, None, A, None,
                             0, 0),
    lambda: wq.wq_gemm_dual(1, 8, 32, 9, wq.WQ_Q8_0, 0, 1.0, A, A, None, A, None, A, None, 0, 0),
    lambda: wq.wq_gemm_dual(1, 8, 32, -1, wq.WQ_Q8_0, 0, 1.0, A, A, None, A, None, A, None, 0, 0),
    lambda: wq.wq_gemm_dual(1, 8, 32, 4, wq.WQ_Q8_0, 0, 1.0, A, A, None, None, None, A, None, 0,
                            0),
    lambda: wq.wq_gemm_dual(1, 8, 32, 4, wq.WQ_Q8_0, 0, float("nan"), A, A, None, A, None, A, None,
                            0, 0),
    lambda: wq.wq_gemm_dual(1, 8, 32, 4, wq.WQ_Q8_0, wq.WQ_BIAS, 1.0, A, A, None, A, None, A, None,
                            0, 0),
    lambda: wq.wq_gemm_dual(1, 8, 32, 4, wq.WQ_Q8_0, 0, 1.0, A, A, None, A, None, None, None, 0, 0),
    lambda: wq.wq_gemm_dual(1, 0x7FFFFFE0, 32, 0x40, wq.WQ_Q8_0, 0, 1.0, A, A, None, A, None, A,
                            None, 0, 0),
    lambda: wq.wq_embed(0, 8, 32, wq.WQ_Q8_0, A, A, None, None, A, 0),
    lambda: wq.wq_embed(2, 0, 32, wq.WQ_Q8_0, A, A, None, None, A, 0),
    lambda: wq.wq_embed(2, 8, 40, wq.WQ_Q4_0, A, A, None, None, A, 0),
    lambda: wq.wq_embed(2, 8, 12, wq.WQ_BF16, A, A, None, None, A, 0),
    lambda: wq.wq_embed(2, 8, 32, 7, A, A, None, None, A, 0),
    lambda: wq.wq_embed(2, 8, 32, wq.WQ_Q8_0, None, A, None, None, A, 0),
    lambda: wq.wq_embed(2, 8, 32, wq.WQ_Q8_0, A, None, None, None, A, 0),
    lambda: wq.wq_embed(2, 8, 32, wq.WQ_Q8_0, A, A, None, None, None, 0),
    lambda: wq.wq_embed(2, 8, 32, wq.WQ_Q8_0, A + 2, A, None, None, A, 0),
    lambda: wq.wq_dequantize(wq.WQ_Q8_0, 4, 32, None, A, 0),
])
def test_invalid_arguments_rejected_on_host(lib, call):
    assert call() == wq.WQ_ERR_INVALID_ARG


@pytest.mark.parametrize("wtype", [wq.WQ_Q8_0, wq.WQ_Q4_0, wq.WQ_F16, wq.WQ_F32])
def test_tensor_core_gemm_of_other_formats_needs_a_workspace(lib, wtype):
    assert wq.wq_gemm(20, 8, 32, wtype, wq.WQ_TC_BF16, A, A, None, None, A, 0) == \
        wq.WQ_ERR_UNSUPPORTED


def test_workspace_sizes_and_errors(lib):
    TC = wq.WQ_TC_BF16
    assert wq.wq_gemm_workspace_bytes(1500, 3072, 1024, wq.WQ_BF16, TC) == 1500 * 1024 * 2
    assert wq.wq_gemm_workspace_bytes(1500, 3072, 1000, wq.WQ_BF16, TC) == 3_000_064  # -> 256
    assert wq.wq_gemm_workspace_bytes(16, 3072, 1024, wq.WQ_BF16, TC) == 0   # GEMV route
    assert wq.wq_gemm_workspace_bytes(1500, 3072, 1024, wq.WQ_BF16, 0) == 0  # f32-FMA route
    # quantised W on the tensor cores: bf16 X, then bf16 W, each rounded up to 256 bytes
    assert wq.wq_gemm_workspace_bytes(1500, 3072, 1024, wq.WQ_Q8_0, TC) == 3_072_000 + 6_291_456
    assert wq.wq_gemm_workspace_bytes(1500, 100, 1024, wq.WQ_Q4_0, TC) == 3_072_000 + 204_800
    assert wq.wq_gemm_workspace_bytes(16, 3072, 1024, wq.WQ_Q4_0, TC) == 0   # GEMV route
    need = wq.wq_gemm_workspace_bytes(32, 64, 64, wq.WQ_BF16, TC)
    call = lambda ws, nb: wq.wq_gemm_ws(32, 64, 64, wq.WQ_BF16, TC, A, A, None, None, A, ws, nb, 0)
    assert call(None, need) == wq.WQ_ERR_INVALID_ARG          # missing
    assert call(A + 16, need) == wq.WQ_ERR_INVALID_ARG        # not 256-byte aligned
    assert call(A, need - 1) == wq.WQ_ERR_INVALID_ARG         # too small


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    """2*n*k above the fixed 16 MiB array is refused on the host, before any device
    work; one element less than the limit is not refused for its size."""
    TC = wq.WQ_TC_BF16
    assert wq.wq_gemm_noalloc(2049, 64, 4096, wq.WQ_BF16, TC, A, A, None, None, A, 0) == \
        wq.WQ_ERR_TOO_LARGE
    assert wq.wq_gemm_noalloc(2048, 64, 4096, wq.WQ_BF16, TC, None, A, None, None, A, 0) == \
        wq.WQ_ERR_INVALID_ARG
    assert wq.wq_gemm_noalloc(0, 64, 4096, wq.WQ_BF16, TC, A, A, None, None, A, 0) == \
        wq.WQ_ERR_INVALID_ARG


def test_layernorm_workspace_sizes_and_errors(lib):
    TC = wq.WQ_TC_BF16
    # tensor-core route: as wq_gemm_workspace_bytes; else the f32 normalised rows
    assert wq.wq_gemm_ln_workspace_bytes(1500, 3072, 1024, wq.WQ_BF16, TC) == 1500 * 1024 * 2
    assert wq.wq_gemm_ln_workspace_bytes(1500, 3072, 1024, wq.WQ_BF16, 0) == 1500 * 1024 * 4
    assert wq.wq_gemm_ln_workspace_bytes(3, 64, 96, wq.WQ_Q8_0, 0) == 1280   # 1152 -> 256
    assert wq.wq_gemm_ln_workspace_bytes(0, 64, 96, wq.WQ_Q8_0, 0) == 0
    need = wq.wq_gemm_ln_workspace_bytes(4, 64, 64, wq.WQ_BF16, 0)
    call = lambda gb, ws, nb: wq.wq_gemm_ln_ws(4, 64, 64, wq.WQ_BF16, 0, A, gb, A, None, None,
                                               A + 4096, ws, nb, 0)
    assert call(None, A + 65536, need) == wq.WQ_ERR_INVALID_ARG      # no gamma/beta
    assert call(A, None, need) == wq.WQ_ERR_INVALID_ARG              # no workspace
    assert call(A, A + 65536 + 16, need) == wq.WQ_ERR_INVALID_ARG    # not 256-byte aligned
    assert call(A, A + 65536, need - 1) == wq.WQ_ERR_INVALID_ARG     # too small


def test_unsupported_requests(lib):
    assert wq.wq_gemm(32, 8, 32, wq.WQ_Q8_0, wq.WQ_TC_BF16, A, A, None, None, A, 0) == \
        wq.WQ_ERR_UNSUPPORTED


def test_moe_slot_count_limit(lib):
    """Any n_tok * topk up to 2^31 - 1 is accepted (routed in windows); beyond the
    int range the call is refused before touching the device."""
    assert wq.wq_moe_gemv(1 << 16, (1 << 15) + 1, 8, 8, 32, wq.WQ_Q4_0, 0, A, A, A, None, None,
                          A, 0) == wq.WQ_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        wq._open(str(tmp_path / "missing.so"))
