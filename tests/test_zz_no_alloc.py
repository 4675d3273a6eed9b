"""w4a16_gemm_noalloc: the W4A16 call for callers that cannot allocate.

Some callers may not allocate device memory on the path that runs a layer
(code running during CUDA-graph stream capture, hosts that plan all device
memory up front, plug-ins inside a framework that owns the device memory),
so this entry point takes no workspace and uses a fixed scratch array the
library keeps in device memory.  These tests call it through the C ABI on
two calls in a row (the second call finds the array holding the first
call's contents) and compare each call with the CPU oracle and with
w4a16_gemm, which takes a caller workspace.  One shape needs nearly all of
the array, so its top end is written and read.

The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close, quantized

FAKE = 1 << 20   # a 16-byte aligned non-null address for host-side rejections
LIMIT = 16 << 20  # W4Q_NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_invalid_arguments_on_the_host():
    lib = w4q.lib()
    assert lib.w4a16_gemm_noalloc(None, FAKE, FAKE, 1, 256, 256, 32, None) == 1
    assert lib.w4a16_gemm_noalloc(FAKE, FAKE, FAKE, 1, 256, 300, 32, None) == 2
    assert lib.w4a16_gemm_noalloc(FAKE, FAKE, FAKE, 65, 256, 256, 32, None) == 2
    assert lib.w4a16_gemm_noalloc(FAKE + 2, FAKE, FAKE, 1, 256, 256, 32, None) == 3


@pytest.mark.gpu
def test_noalloc_rejects_calls_beyond_its_scratch(cuda):
    # M = 64 with K = 2^18 needs about 35 MB of prepared activations, more
    # than the 16 MiB array: refused before anything is launched.
    lib = w4q.lib()
    assert w4q.workspace_bytes(64, 16, 1 << 18) > LIMIT
    st = lib.w4a16_gemm_noalloc(FAKE, FAKE, FAKE, 64, 16, 1 << 18, 32,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2


def _two_calls(cuda, N, K, M):
    lib = w4q.lib()
    W, q, s, z = quantized(N, K, seed=N + K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    stream = torch.cuda.current_stream()
    for call in range(2):
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M) + call)
        xd = x.to(cuda)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        st = lib.w4a16_gemm_noalloc(xd.data_ptr(), packed.data_ptr(), out.data_ptr(), M, N, K,
                                    32, ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, w4q.status_string(st)
        torch.cuda.synchronize()
        what = "noalloc call %d N=%d K=%d M=%d" % (call, N, K, M)
        assert_close(out, oracle.w4a16(x, q, s, z), what)
        ref = w4q.w4a16_gemm(xd, packed, N, K)
        assert torch.equal(out, ref), what   # same kernels, same partition: same bits
    assert w4q.device_error() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,M", [(8448, 6656, 4), (257, 512, 1), (6656, 4096, 16),
                                   (1536, 512, 64), (256, 6656, 3)])
def test_noalloc_matches_the_oracle_twice(cuda, N, K, M):
    _two_calls(cuda, N, K, M)


@pytest.mark.gpu
def test_noalloc_near_the_top_of_its_scratch(cuda):
    # the tensor-core path's split-K partials at M = 44 on 6656 x 19968 fill
    # most of the array (on a 152-SM GB300: about 15.6 of 16.8 MB)
    N, K, M = 6656, 19968, 44
    need = w4q.workspace_bytes(M, N, K)
    assert 0.85 * LIMIT <= need <= LIMIT, need
    _two_calls(cuda, N, K, M)
