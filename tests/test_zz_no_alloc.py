"""w4a16_gemm_noalloc: the W4A16 call for callers that cannot allocate.

Some callers may not allocate device memory on the path that runs a layer
(code running during CUDA-graph stream capture, hosts that plan all device
memory up front, plug-ins inside a framework that owns the device memory),
so this entry point takes no workspace and uses a fixed scratch array the
library keeps in device memory.  These tests call it through the C ABI and
compare it with w4a16_gemm, which takes a caller workspace, on two calls in
a row (the second call finds the array holding the first call's contents).

The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close, to_f64

FAKE = 1 << 20   # a 16-byte aligned non-null address for host-side rejections


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
    st = lib.w4a16_gemm_noalloc(FAKE, FAKE, FAKE, 64, 16, 1 << 18, 32,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,M", [(8448, 6656, 4), (257, 512, 1), (6656, 4096, 16),
                                   (1536, 512, 64), (256, 6656, 3)])
def test_noalloc_matches_the_workspace_entry_point_twice(cuda, N, K, M):
    lib = w4q.lib()
    packed = w4q.w4_pack_weights(workloads.w4_weight(N, K, seed=N + K).to(cuda))
    stream = torch.cuda.current_stream()
    for call in range(2):
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M) + call).to(cuda)
        ref = w4q.w4a16_gemm(x, packed, N, K)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        st = lib.w4a16_gemm_noalloc(x.data_ptr(), packed.data_ptr(), out.data_ptr(), M, N, K,
                                    32, ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, w4q.status_string(st)
        torch.cuda.synchronize()
        assert_close(out, to_f64(ref), "noalloc call %d N=%d K=%d M=%d" % (call, N, K, M))
        assert torch.equal(out, ref)   # same kernels, same partition: same bits
    assert w4q.device_error() == 0
