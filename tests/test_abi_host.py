"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from ternary_weight_linear_06_b300 import _lib
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "bitlinear.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"BL_API\s+[\w\s\*]+?\b(bitlinear_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 9
    lib = _lib.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(_lib.SIGNATURES), "binding misses a declared entry point"


def _prototypes():
    """name -> parameter count, from the BL_API declarations of the header."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"BL_API\s+[\w\s\*]+?\b(bitlinear_\w+)\s*\(([^)]*)\)\s*;", src):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_lists_match_the_header():
    protos = _prototypes()
    assert set(protos) == set(_declared())
    for name, n in protos.items():
        assert len(_lib.SIGNATURES[name][1]) == n, (name, n, len(_lib.SIGNATURES[name][1]))


def test_version_and_status_strings():
    lib = _lib.lib()
    assert lib.bitlinear_version() == 102
    for s in range(8):
        assert lib.bitlinear_status_str(s)
    assert b"unknown" in lib.bitlinear_status_str(99)


def test_workspace_bytes_rules():
    f = _lib.lib().bitlinear_workspace_bytes
    assert f(_lib.BL_OP_FORWARD, 4, 256, 256) >= 256 + 4 * 256 * 2
    assert f(_lib.BL_OP_FORWARD, 4, 256, 100) == 0          # K % 64 != 0
    assert f(_lib.BL_OP_FORWARD, -1, 256, 256) == 0
    assert f(_lib.BL_OP_FORWARD, 1, 256, 65536 + 64) == 0   # K above the exactness bound
    assert f(_lib.BL_OP_FORWARD, 1, 1 << 16, 1 << 15) == 0  # N*K >= 2^31
    assert f(_lib.BL_OP_PACK, 0, 0, 256) == 0
    assert f(_lib.BL_OP_PACK, 0, 256, 256) > 256
    assert f(_lib.BL_OP_FFN, 8, 6912, 2560) > 8 * 6912 * 4
    assert f(99, 1, 1, 64) == 0


def test_host_argument_checks_fail_before_launch():
    lib = _lib.lib()
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) // 16 * 16        # a 16-byte aligned host address, never dereferenced
    # null pointers
    assert lib.bitlinear_pack(None, 4, 64, 1e-5, p, p, p, 4096, None) == _lib.BL_ERR_ARG
    # bad eps
    assert lib.bitlinear_pack(p, 4, 64, 0.0, p, p, p, 4096, None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_pack(p, 4, 64, float("nan"), p, p, p, 4096, None) == _lib.BL_ERR_ARG
    # shapes
    assert lib.bitlinear_pack(p, 4, 100, 1e-5, p, p, p, 4096, None) == _lib.BL_ERR_SHAPE
    assert lib.bitlinear_pack(p, 0, 64, 1e-5, p, p, p, 4096, None) == _lib.BL_ERR_SHAPE
    assert lib.bitlinear_forward(p, 0, 1, 96, p, p, 4, 1e-5, p, None, p, 4096, None) == _lib.BL_ERR_SHAPE
    assert lib.bitlinear_forward(p, 0, -1, 64, p, p, 4, 1e-5, p, None, p, 4096, None) == _lib.BL_ERR_SHAPE
    # bad dtype
    assert lib.bitlinear_forward(p, 7, 1, 64, p, p, 4, 1e-5, p, None, p, 4096, None) == _lib.BL_ERR_ARG
    # misaligned pointers
    assert lib.bitlinear_forward(p + 4, 0, 1, 64, p, p, 4, 1e-5, p, None, p, 4096, None) == _lib.BL_ERR_ALIGN
    assert lib.bitlinear_pack(p, 4, 64, 1e-5, p + 8, p, p, 4096, None) == _lib.BL_ERR_ALIGN
    # workspace too small
    assert lib.bitlinear_forward(p, 0, 1, 64, p, p, 4, 1e-5, p, None, p, 16, None) == _lib.BL_ERR_WORKSPACE
    assert lib.bitlinear_ffn(p, 0, 2, 64, p, p, p, p, 128, 1e-5, p, p, 16, None) == _lib.BL_ERR_WORKSPACE
    # empty problems are a no-op that touches nothing
    assert lib.bitlinear_forward(None, 0, 0, 64, None, None, 4, 1e-5, None, None, None, 0, None) == _lib.BL_OK
    assert lib.bitlinear_forward(None, 0, 3, 64, None, None, 0, 1e-5, None, None, None, 0, None) == _lib.BL_OK
    assert lib.bitlinear_quant_act(None, 0, 0, 64, 1e-5, None, None, None) == _lib.BL_OK
    assert lib.bitlinear_workspace_status(None, None) == _lib.BL_ERR_ARG
    # gated FFN: the gate is required; workspace sized for the gate buffer
    assert lib.bitlinear_ffn_gated(p, 0, 2, 64, p, p, None, p, p, p, 128, 1e-5, p, p, 1 << 20, None) == _lib.BL_ERR_ARG
    need = lib.bitlinear_workspace_bytes(_lib.BL_OP_FFN_GATED, 2, 128, 64)
    assert need > lib.bitlinear_workspace_bytes(_lib.BL_OP_FFN, 2, 128, 64)
    assert lib.bitlinear_ffn_gated(p, 0, 2, 64, p, p, p, p, p, p, 128, 1e-5, p, p, need - 256, None) == \
        _lib.BL_ERR_WORKSPACE
    assert lib.bitlinear_ffn_gated(p, 0, 2, 64, p, p, p + 4, p, p, p, 128, 1e-5, p, p, need, None) == _lib.BL_ERR_ALIGN
    # RMSNorm fused into the quantization: eps_norm must be positive and finite,
    # the gain 16-byte aligned (or NULL)
    nan = float("nan")
    assert lib.bitlinear_rmsnorm_quant(p, 0, 2, 64, p, 0.0, 1e-5, p, p, None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_rmsnorm_quant(p, 0, 2, 64, p, nan, 1e-5, p, p, None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_rmsnorm_quant(p, 0, 2, 96, p, 1e-5, 1e-5, p, p, None) == _lib.BL_ERR_SHAPE
    assert lib.bitlinear_rmsnorm_quant(p, 0, 2, 64, p + 4, 1e-5, 1e-5, p, p, None) == _lib.BL_ERR_ALIGN
    assert lib.bitlinear_rmsnorm_quant(None, 0, 0, 64, None, 1e-5, 1e-5, None, None, None) == _lib.BL_OK
    assert lib.bitlinear_forward_rmsnorm(p, 0, 1, 64, p, -1.0, p, p, 4, 1e-5, p, None, p, 4096, None) == \
        _lib.BL_ERR_ARG
    assert lib.bitlinear_forward_rmsnorm(p, 0, 1, 64, p + 8, 1e-5, p, p, 4, 1e-5, p, None, p, 4096, None) == \
        _lib.BL_ERR_ALIGN
    assert lib.bitlinear_forward_rmsnorm(p, 0, 1, 64, None, 1e-5, p, p, 4, 1e-5, p, None, p, 16, None) == \
        _lib.BL_ERR_WORKSPACE
    assert lib.bitlinear_forward_rmsnorm(p, 0, 1, 96, None, 1e-5, p, p, 4, 1e-5, p, None, p, 4096, None) == \
        _lib.BL_ERR_SHAPE
    assert lib.bitlinear_forward_rmsnorm(None, 0, 0, 64, None, 1e-5, None, None, 4, 1e-5, None, None, None, 0,
                                         None) == _lib.BL_OK
    # SubLN FFN: gate and s_gate together; the gated form needs the gated workspace
    assert lib.bitlinear_ffn_subln(p, 0, 2, 64, None, p, p, p, None, None, p, p, 128, 1e-5, 1e-5, p, p, 1 << 20,
                                   None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_ffn_subln(p, 0, 2, 64, None, p, p, None, None, None, p, p, 128, 0.0, 1e-5, p, p, 1 << 20,
                                   None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_ffn_subln(p, 0, 2, 64, None, p, p, None, None, p + 4, p, p, 128, 1e-5, 1e-5, p, p,
                                   1 << 20, None) == _lib.BL_ERR_ALIGN
    plain = lib.bitlinear_workspace_bytes(_lib.BL_OP_FFN, 2, 128, 64)
    assert lib.bitlinear_ffn_subln(p, 0, 2, 64, None, p, p, p, p, None, p, p, 128, 1e-5, 1e-5, p, p, plain,
                                   None) == _lib.BL_ERR_WORKSPACE
    # tensor-core operand form
    assert lib.bitlinear_quant_act_tc(p, 0, 2, 96, 1e-5, p, p, None) == _lib.BL_ERR_SHAPE
    assert lib.bitlinear_quant_act_tc(p, 0, 2, 64, 1e-5, p + 8, p, None) == _lib.BL_ERR_ALIGN
    assert lib.bitlinear_forward_tc(p, p, 2, 64, p, p, 4, p, None, p, 16, None) == _lib.BL_ERR_WORKSPACE
    assert lib.bitlinear_forward_tc(p + 8, p, 2, 64, p, p, 4, p, None, p, 4096, None) == _lib.BL_ERR_ALIGN
    assert lib.bitlinear_forward_tc(None, None, 0, 64, None, None, 4, None, None, None, 0, None) == _lib.BL_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_batch_argument_checks():
    lib = _lib.lib()
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    D = _lib.ForwardDesc
    good = D(p, 0, 1, 64, 4, p, p, p, None)
    arr = (D * 2)(good, good)
    assert lib.bitlinear_forward_batch(arr, 129, 1e-5, p, 4096, None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_forward_batch(arr, -1, 1e-5, p, 4096, None) == _lib.BL_ERR_ARG
    assert lib.bitlinear_forward_batch(arr, 0, 1e-5, p, 4096, None) == _lib.BL_OK
    assert lib.bitlinear_forward_batch(arr, 2, 1e-5, p, 16, None) == _lib.BL_ERR_WORKSPACE
    arr[1].K = 96
    assert lib.bitlinear_forward_batch(arr, 2, 1e-5, p, 4096, None) == _lib.BL_ERR_SHAPE
    arr[1].K = 64
    arr[1].Y = p + 4
    assert lib.bitlinear_forward_batch(arr, 2, 1e-5, p, 4096, None) == _lib.BL_ERR_ALIGN
    arr[1].Y = p
    arr[1].x_dtype = 5
    assert lib.bitlinear_forward_batch(arr, 2, 1e-5, p, 4096, None) == _lib.BL_ERR_ARG
    # an already-quantized input needs its per-token scales
    arr[1].x_dtype = _lib.BL_DTYPE_I8
    assert lib.bitlinear_forward_batch(arr, 2, 1e-5, p, 4096, None) == _lib.BL_ERR_ARG
    arr[1].m = p + 2
    assert lib.bitlinear_forward_batch(arr, 2, 1e-5, p, 4096, None) == _lib.BL_ERR_ALIGN
    assert lib.bitlinear_workspace_bytes(_lib.BL_OP_FORWARD_BATCH, 0, 0, 0) == 256
