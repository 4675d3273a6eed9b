"""The bounded-wait error path: a wait that runs out sets the device error
word, w4q_device_error reports it once and clears it, and the context stays
usable.  The wait is made to run out by a barrier phase that nothing
completes (w4q_selftest_wait_expiry, a limit of a few milliseconds); nothing
faults, traps or hangs."""
import ctypes

import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close, quantized

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_once_and_cleared(cuda):
    assert w4q.device_error() == 0
    lib = w4q.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.w4q_selftest_wait_expiry(2000, stream) == 0
    code = ctypes.c_uint32(0)
    assert lib.w4q_device_error(ctypes.byref(code)) == 6     # W4Q_ERR_DEVICE
    assert code.value == 1                                   # the full-stage wait bit
    assert lib.w4q_device_error(ctypes.byref(code)) == 0     # read once, then cleared
    assert code.value == 0
    # the context is still usable: an ordinary call afterwards is correct
    N, K, M = 384, 1024, 2
    W, q, s, z = quantized(N, K, seed=3)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(M, K, seed=4)
    assert_close(w4q.w4a16_gemm(x.to(cuda), packed, N, K), oracle.w4a16(x, q, s, z), "after")
    assert w4q.device_error() == 0


def test_selftest_rejects_bad_limits():
    lib = w4q.lib()
    assert lib.w4q_selftest_wait_expiry(0, None) == 1
    assert lib.w4q_selftest_wait_expiry(100001, None) == 1
