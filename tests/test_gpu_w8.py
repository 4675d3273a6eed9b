"""W8 GEMV on the GPU vs the oracle ("gpt-fast issue #114":
WeightOnlyInt8Linear.forward and its fused int8 -> fp32 reduction)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close

pytestmark = pytest.mark.gpu


def _check(cuda, N, K, M, seed):
    W, sc, x = workloads.w8_inputs(N=N, K=K, M=M, seed=seed)
    out = w4q.w8_gemv(x.to(cuda), W.to(cuda), sc.to(cuda))
    assert out.shape == (M, N) and out.dtype == torch.bfloat16
    assert_close(out, oracle.w8(x, W.numpy(), sc), "W8 N=%d K=%d M=%d" % (N, K, M))


def test_w8_workload_8192(cuda):
    N, K = workloads.W8_GEMV["N"], workloads.W8_GEMV["K"]
    _check(cuda, N, K, 1, workloads.W8_GEMV["seed"])


@pytest.mark.parametrize("N,K,M", [(1, 16, 1), (7, 48, 2), (257, 4096, 3), (1000, 8192, 4),
                                   (64, 16384, 1), (300, 12288, 2), (8192, 8192, 2),
                                   (33, 8208, 1)])
def test_w8_shapes(cuda, N, K, M):
    _check(cuda, N, K, M, seed=N + K + M)


def test_w8_extremes(cuda):
    # every weight -128 or 127 with all-ones activations: exact integer sums
    N, K = 64, 8192
    W = torch.where(torch.arange(N * K).view(N, K) % 3 == 0, -128, 127).to(torch.int8)
    sc = torch.ones(N, dtype=torch.bfloat16)
    x = torch.ones(1, K, dtype=torch.bfloat16)
    out = w4q.w8_gemv(x.to(cuda), W.to(cuda), sc.to(cuda))
    ref = oracle.w8(x, W.numpy(), sc)
    assert_close(out, ref, "extremes")
    assert np.array_equal(out.float().cpu().numpy(),
                          torch.tensor(ref).to(torch.bfloat16).float().numpy())
