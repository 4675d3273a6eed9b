"""W4A8 on the GPU vs the oracle ("test_int4_quantized_gemm.py": the W4A8
bucket kernels and Int4QuantizedGemmPrecisionTest).  The integer parts (the
int8 activations, their scales and the per-group dot products) must match
bit-exactly; the float output within the float tolerance of the W4A8 oracle
and within the pages' precision class of the W4A16 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close, quantized

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1, 256), (4, 6656), (3, 19968), (64, 512)])
def test_activation_quantizer_bit_exact(cuda, M, K):
    x = workloads.activation(M, K, seed=M * 7 + K)
    x[0, 5] = 0.0
    if M > 1:
        x[1] = 0.0                       # an all-zero row: sx = 0, xq = 0
    xq, sx = w4q.w4a8_quantize_act(x.to(cuda))
    oxq, osx = oracle.act_quant(x, K)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oxq)


def test_activation_quantizer_ties(cuda):
    K = 256
    vals = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.0, -127.0]
    x = torch.tensor(vals * (K // 8), dtype=torch.float32).to(torch.bfloat16).view(1, K)
    xq, sx = w4q.w4a8_quantize_act(x.to(cuda))
    assert sx.item() == 1.0
    assert xq[0, :8].tolist() == [127, 0, 2, 2, 0, -2, 3, -127]


@pytest.mark.parametrize("N,K,M", [(257, 512, 1), (256, 768, 4), (1536, 512, 3), (768, 256, 2),
                                   (300, 6656, 4), (96, 512, 64)])
def test_group_dots_bit_exact(cuda, N, K, M):
    W, q, s, z = quantized(N, K, seed=N ^ K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(M, K, seed=M + 17)
    D = w4q.w4a8_group_dots(x.to(cuda), packed, N, K).cpu().numpy()
    xq, sx = oracle.act_quant(x, K)
    ref = oracle.w4a8_group_dots(xq, q, z)
    assert np.array_equal(D, ref), np.argwhere(D != ref)[:5]
    assert np.abs(D).max() <= 32 * 15 * 127


def _check(cuda, N, K, Ms, split_k=None, seed_w=None, window=None):
    W, q, s, z = quantized(N, K, seed_w)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in Ms:
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        out = w4q.w4a8_gemm(x.to(cuda), packed, N, K, split_k=split_k)
        xq, sx = oracle.act_quant(x, K)
        a, b = window if window else (0, N)
        ref8 = oracle.w4a8(xq, sx, q, s, z, a, b)
        assert_close(out[:, a:b], ref8, "W4A8 N=%d K=%d M=%d split=%s" % (N, K, M, split_k))
        ref16 = oracle.w4a16(x, q, s, z, a, b)
        o = out[:, a:b].float().cpu().numpy()
        rel = np.abs(o - ref16).mean() / np.abs(ref16).mean()
        assert rel < 0.02, ("precision class vs W4A16", M, rel)


@pytest.mark.parametrize("N,K", workloads.SMALL_SHAPES + ((257, 256),))
def test_small_shapes(cuda, N, K):
    _check(cuda, N, K, (1, 2, 3, 4, 8, 16, 64), seed_w=N + K)


def test_w4a8_workload_full_size(cuda):
    N, K = workloads.W4A8_SHAPE
    _check(cuda, N, K, workloads.W4A8_MS)


def test_every_legal_split_matches(cuda):
    N, K = 256, 4096
    for split in (0, 1, 2, 4, 16):
        _check(cuda, N, K, (1, 4), split_k=split, seed_w=91)


def test_zero_rows_and_zero_input(cuda):
    N, K = 128, 512
    W, q, s, z = quantized(N, K, seed=4)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(3, K, seed=9)
    x[1] = 0
    out = w4q.w4a8_gemm(x.to(cuda), packed, N, K)
    assert torch.all(out[1] == 0)
    xq, sx = oracle.act_quant(x, K)
    assert_close(out, oracle.w4a8(xq, sx, q, s, z), "zero row")
