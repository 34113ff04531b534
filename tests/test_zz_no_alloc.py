"""bitlinear_forward_noalloc: the forward for callers that cannot allocate
device memory (a runtime with a fixed memory plan, a plugin whose host
framework owns all device memory). It must give what bitlinear_forward gives,
call after call, while using the library's own fixed device scratch array.

Collected last on purpose, and written to pass both alone in a fresh process
and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import ternary_weight_linear_06_b300 as BL
from ternary_weight_linear_06_b300 import _lib
from ternary_weight_linear_06_b300 import workloads as WL

pytestmark = pytest.mark.gpu
RTOL = 1e-5


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_forward_noalloc_matches_forward_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    lib = _lib.lib()
    stream = torch.cuda.current_stream().cuda_stream
    W = torch.from_numpy(WL.decode_weights("kv", 7)).cuda()
    packed, s_w = BL.pack(W)
    K, N = 2560, 640
    # two calls in a row with different inputs and sizes; the second one sees
    # the first one's leftovers in the shared scratch
    for call, (M, seed) in enumerate([(3, 11), (2, 12)]):
        X = torch.from_numpy(WL.student_t(M, K, seed=seed)).cuda()
        Y_ref, acc_ref = BL.forward(X, packed, s_w, return_acc=True)
        Y = torch.full((M, N), float("nan"), device="cuda")
        acc = torch.zeros((M, N), dtype=torch.int32, device="cuda")
        st = lib.bitlinear_forward_noalloc(_p(X), _lib.BL_DTYPE_F32, M, K, _p(packed), _p(s_w), N, 1e-5, _p(Y),
                                           _p(acc), ctypes.c_void_p(stream))
        assert st == _lib.BL_OK, _lib.status_str(st)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref.cpu().numpy())
        y, y_ref = Y.cpu().numpy().astype(np.float64), Y_ref.cpu().numpy().astype(np.float64)
        rel = np.abs(y - y_ref) / np.maximum(np.abs(y_ref), 1e-30)
        assert rel.max() <= RTOL, (call, rel.max())


def test_forward_noalloc_rejects_sizes_beyond_the_scratch():
    lib = _lib.lib()
    M, K, N = 4096, 4096, 64          # q alone needs 4096*4096*2 bytes > 8 MiB
    assert lib.bitlinear_workspace_bytes(_lib.BL_OP_FORWARD, M, N, K) > _lib.BL_STATIC_SCRATCH_BYTES
    st = lib.bitlinear_forward_noalloc(ctypes.c_void_p(16), 0, M, K, ctypes.c_void_p(16), ctypes.c_void_p(16), N,
                                       1e-5, ctypes.c_void_p(16), None, None)
    assert st == _lib.BL_ERR_WORKSPACE
