"""ctypes loader for libbitlinear.so (the C ABI declared in include/bitlinear.h).

Loading fails loudly: there is no fallback path. Build the library with
``python -m ternary_weight_linear_06_b300.build`` (or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbitlinear.so")

BL_OK = 0
BL_ERR_ARG = 1
BL_ERR_SHAPE = 2
BL_ERR_ALIGN = 3
BL_ERR_CUDA = 4
BL_ERR_TIMEOUT = 5
BL_ERR_UNSUPPORTED = 6
BL_ERR_WORKSPACE = 7

BL_DTYPE_F32 = 0
BL_DTYPE_BF16 = 1
BL_DTYPE_I8 = 2

BL_STATIC_SCRATCH_BYTES = 8 << 20

BL_OP_PACK = 0
BL_OP_FORWARD = 1
BL_OP_FFN = 2
BL_OP_FORWARD_BATCH = 3
BL_OP_FFN_GATED = 4
BL_MAX_BATCH = 128


class ForwardDesc(ctypes.Structure):
    """Mirror of bl_forward_desc in include/bitlinear.h."""
    _fields_ = [("X", ctypes.c_void_p), ("x_dtype", ctypes.c_int), ("M", ctypes.c_int), ("K", ctypes.c_int),
                ("N", ctypes.c_int), ("packed", ctypes.c_void_p), ("s_w", ctypes.c_void_p),
                ("Y", ctypes.c_void_p), ("acc", ctypes.c_void_p), ("m", ctypes.c_void_p)]

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes); the order matches include/bitlinear.h
SIGNATURES = {
    "bitlinear_version": (_i, []),
    "bitlinear_status_str": (ctypes.c_char_p, [_i]),
    "bitlinear_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "bitlinear_pack": (_i, [_vp, _i, _i, _f, _vp, _vp, _vp, _sz, _vp]),
    "bitlinear_quant_act": (_i, [_vp, _i, _i, _i, _f, _vp, _vp, _vp]),
    "bitlinear_forward": (_i, [_vp, _i, _i, _i, _vp, _vp, _i, _f, _vp, _vp, _vp, _sz, _vp]),
    "bitlinear_forward_batch": (_i, [ctypes.POINTER(ForwardDesc), _i, _f, _vp, _sz, _vp]),
    "bitlinear_forward_q8": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "bitlinear_quant_act_tc": (_i, [_vp, _i, _i, _i, _f, _vp, _vp, _vp]),
    "bitlinear_forward_tc": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp]),
    "bitlinear_forward_noalloc": (_i, [_vp, _i, _i, _i, _vp, _vp, _i, _f, _vp, _vp, _vp]),
    "bitlinear_ffn": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _f, _vp, _vp, _sz, _vp]),
    "bitlinear_ffn_gated": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _f, _vp, _vp, _sz, _vp]),
    "bitlinear_rmsnorm_quant": (_i, [_vp, _i, _i, _i, _vp, _f, _f, _vp, _vp, _vp]),
    "bitlinear_forward_rmsnorm": (_i, [_vp, _i, _i, _i, _vp, _f, _vp, _vp, _i, _f, _vp, _vp, _vp, _sz, _vp]),
    "bitlinear_ffn_subln": (_i, [_vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _f, _f, _vp, _vp,
                                 _sz, _vp]),
    "bitlinear_unpack": (_i, [_vp, _i, _i, _vp, _vp]),
    "bitlinear_workspace_status": (_i, [_vp, _vp]),
}


class BitLinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"BitLinear CUDA library not built ({LIB_PATH} missing); run "
                "`python -m ternary_weight_linear_06_b300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def status_str(status: int) -> str:
    return lib().bitlinear_status_str(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != BL_OK:
        raise BitLinearError(status, where)
