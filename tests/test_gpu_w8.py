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


# ------------------------------------------------ w8_gemm: 1 <= M <= 64
def _check_gemm(cuda, N, K, M, seed, x=None):
    W, sc, x0 = workloads.w8_inputs(N=N, K=K, M=M, seed=seed)
    x = x0 if x is None else x
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
    w4q.w8_gemm(x.to(cuda), W.to(cuda), sc.to(cuda), out=out)
    assert_close(out, oracle.w8(x, W.numpy(), sc), "W8 gemm N=%d K=%d M=%d" % (N, K, M))
    return out


@pytest.mark.parametrize("M", (1, 2, 3, 4, 5, 8, 9, 16, 17, 32, 33, 48, 64))
def test_w8_gemm_8192(cuda, M):
    # the 8192 x 8192 workload at every bucket of M (every output compared;
    # the output starts as NaN)
    N, K = workloads.W8_GEMV["N"], workloads.W8_GEMV["K"]
    _check_gemm(cuda, N, K, M, seed=workloads.W8_GEMV["seed"] + M)


@pytest.mark.parametrize("N,K,M", [(1, 16, 5), (7, 48, 6), (257, 4096, 9), (300, 528, 12),
                                   (1000, 8208, 16), (383, 12288, 24), (129, 256, 40),
                                   (64, 32768, 3), (1024, 40960, 48), (4096, 1024, 20)])
def test_w8_gemm_shapes(cuda, N, K, M):
    # ragged N (not a multiple of 128 or 256), K not a multiple of 256, K
    # beyond the CUDA-core kernel (32768 at M = 3), whole-K and split CTAs
    _check_gemm(cuda, N, K, M, seed=N + K + M)


def test_w8_gemm_every_m(cuda):
    N, K = 520, 2304
    W, sc, _ = workloads.w8_inputs(N=N, K=K, M=1, seed=11)
    Wd, scd = W.to(cuda), sc.to(cuda)
    for M in range(1, 65):
        x = workloads.activation(M, K, seed=200 + M)
        assert_close(w4q.w8_gemm(x.to(cuda), Wd, scd), oracle.w8(x, W.numpy(), sc), "M=%d" % M)


def test_w8_gemm_activation_magnitudes(cuda):
    # each row of x at its own scale (the per-row power of two): huge, tiny,
    # subnormal-only, zero, and a row whose max dwarfs the rest
    N, K, M = 384, 4096, 8
    W, sc, x = workloads.w8_inputs(N=N, K=K, M=M, seed=12)
    x = x.float()
    x[0] *= 2.0 ** 100
    x[1] *= 2.0 ** -100
    x[2] = torch.where(torch.arange(K) % 7 == 0, 2.0 ** -130, 0.0)
    x[3] = 0.0
    x[4, 5] = 3.0e4
    x = x.to(torch.bfloat16)
    out = _check_gemm(cuda, N, K, M, seed=12, x=x)
    assert torch.all(out[3] == 0)


def test_w8_gemm_extremes_exact(cuda):
    # weights -128 / 127, all-ones x: integer sums, exact through fp16/fp32
    N, K, M = 256, 8192, 16
    W = torch.where(torch.arange(N * K).view(N, K) % 3 == 0, -128, 127).to(torch.int8)
    sc = torch.ones(N, dtype=torch.bfloat16)
    x = torch.ones(M, K, dtype=torch.bfloat16)
    out = w4q.w8_gemm(x.to(cuda), W.to(cuda), sc.to(cuda))
    ref = oracle.w8(x, W.numpy(), sc)
    assert np.array_equal(out.float().cpu().numpy(),
                          torch.tensor(ref).to(torch.bfloat16).float().numpy())


def test_w8_gemm_repeatable_and_workspace_checked(cuda):
    N, K, M = 8192, 8192, 16
    W, sc, x = workloads.w8_inputs(N=N, K=K, M=M, seed=13)
    Wd, scd, xd = W.to(cuda), sc.to(cuda), x.to(cuda)
    need = w4q.w8_workspace_bytes(M, N, K)
    assert need > 0 and w4q.w8_workspace_bytes(1, N, K) == 0
    assert w4q.w8_kernel_launches(1, N, K) == 1 and w4q.w8_kernel_launches(M, N, K) in (2, 3)
    # M = 2 stays on the CUDA cores while its rows fit one wave (64 per SM)
    sms = torch.cuda.get_device_properties(cuda).multi_processor_count
    assert (w4q.w8_kernel_launches(2, N, K) == 1) == (N <= 64 * sms)
    assert w4q.w8_kernel_launches(2, 64 * sms + 128, K) in (2, 3)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda)
    a = w4q.w8_gemm(xd, Wd, scd, workspace=ws)
    for _ in range(3):
        assert torch.equal(w4q.w8_gemm(xd, Wd, scd, workspace=ws), a)
    out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(w4q.W4QError) as e:
        w4q.w8_gemm(xd, Wd, scd, out=out, workspace=ws[:need - 256])
    assert e.value.status == 4 and torch.all(out == 7.0)
    with pytest.raises(w4q.W4QError) as e:
        w4q.w8_gemm(torch.zeros(65, K, dtype=torch.bfloat16, device=cuda), Wd, scd)
    assert e.value.status == 2
    assert w4q.device_error() == 0
