"""W4A8 on the GPU vs the oracle ("test_int4_quantized_gemm.py": the W4A8
bucket kernels and Int4QuantizedGemmPrecisionTest).  The integer parts (the
int8 activations, their per-(row, group of 32) scales and the per-group dot
products) must match bit-exactly; the float output within the float
tolerance of the W4A8 oracle and within the pages' precision criteria
against the W4A16 oracle and the dense product, with and without the
pages' outlier channels."""
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
    x[0, 64:96] = 0.0                    # an all-zero group: sx = 0, xq = 0
    x[0, 200] = 300.0                    # an outlier: only its own group's scale grows
    if M > 1:
        x[1] = 0.0                       # an all-zero row
    xq, sx = w4q.w4a8_quantize_act(x.to(cuda))
    oxq, osx = oracle.act_quant(x, K)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oxq)


def test_activation_quantizer_every_bf16_value(cuda):
    # every positive bf16 magnitude, in groups of 32 whose maxima vary: the
    # int8 codes and per-group scales bit for bit
    K = 32768
    bits = np.arange(1, K + 1, dtype=np.uint32)
    v = (bits << 16).view(np.float32)
    v = np.where(np.isfinite(v), v, np.float32(1.0))
    v = np.where(np.arange(K) % 3 == 0, -v, v)
    rows = [v, v[::-1].copy(), np.roll(v, 7)]
    x = torch.from_numpy(np.stack(rows)).to(torch.bfloat16)
    xq, sx = w4q.w4a8_quantize_act(x.to(cuda))
    oxq, osx = oracle.act_quant(x, K)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oxq), np.argwhere(xq.cpu().numpy() != oxq)[:5]


def test_activation_quantizer_ties(cuda):
    K = 256
    vals = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.0, -127.0]
    x = torch.tensor(vals * (K // 8), dtype=torch.float32).to(torch.bfloat16).view(1, K)
    xq, sx = w4q.w4a8_quantize_act(x.to(cuda))
    assert sx.shape == (1, K // 32) and bool(torch.all(sx == 1.0))
    assert xq[0, :8].tolist() == [127, 0, 2, 2, 0, -2, 3, -127]


@pytest.mark.parametrize("N,K,M", [(257, 512, 1), (256, 768, 4), (1536, 512, 3), (768, 256, 2),
                                   (300, 6656, 4), (96, 512, 8), (40, 256, 6)])
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
    _check(cuda, N, K, (1, 2, 3, 4, 5, 8), seed_w=N + K)


def test_more_than_eight_rows_is_rejected(cuda):
    N, K = 64, 256
    packed = w4q.w4_pack_weights(workloads.w4_weight(N, K, seed=2).to(cuda))
    x = torch.randn(9, K, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a8_gemm(x, packed, N, K)
    assert e.value.status == 2


def test_w4a8_workload_full_size(cuda):
    N, K = workloads.W4A8_SHAPE
    _check(cuda, N, K, workloads.W4A8_MS)


def test_every_legal_split_matches(cuda):
    N, K = 256, 4096
    for split in (0, 1, 2, 4, 16):
        _check(cuda, N, K, (1, 4), split_k=split, seed_w=91)


def test_stream_k(cuda):
    # explicit stream-K on 8448 x 6656 (groups split between CTAs): every
    # output against the oracle
    _check(cuda, 8448, 6656, (1, 2, 4, 7), split_k=0, seed_w=98)
    assert w4q.device_error() == 0


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


def _precision_case(cuda, N, K, M, outliers, seed_w, seed_x):
    W = workloads.w4_weight(N, K, seed=seed_w)
    q, s, z = oracle.quantize_w4(W, N, K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = (workloads.outlier_activation if outliers else workloads.activation)(M, K, seed=seed_x)
    a8 = w4q.w4a8_gemm(x.to(cuda), packed, N, K).double().cpu().numpy()
    a16 = oracle.w4a16(x, q, s, z)
    dense = (x.double() @ W.double().T).numpy()
    return a8, a16, dense


@pytest.mark.parametrize("N,K", workloads.MODEL_SHAPES + workloads.SMALL_SHAPES)
def test_precision_gaussian_and_outliers(cuda, N, K):
    # "test_int4_quantized_gemm.py", Int4QuantizedGemmPrecisionTest,
    # test_precision_gaussian_and_outliers / _check_precision_case: finite;
    # mean |a8 - dense| within 1.10x of W4A16's; mean |a8 - a16| / mean |a16|
    # <= 0.02; max |a8 - dense| within max(2, 0.02 max |dense|) of W4A16's.
    for M in workloads.W4A8_BUCKETS:
        for outliers in (False, True):
            a8, a16, dense = _precision_case(cuda, N, K, M, outliers, seed_w=1200 + N % 97,
                                             seed_x=9100 + M)
            label = "M=%d N=%d K=%d %s" % (M, N, K, "outliers" if outliers else "gaussian")
            assert np.isfinite(a8).all(), label
            e8, e16 = np.abs(a8 - dense), np.abs(a16 - dense)
            assert e8.mean() / max(e16.mean(), 1e-6) <= 1.10, label
            assert np.abs(a8 - a16).mean() / max(np.abs(a16).mean(), 1e-6) <= 0.02, label
            assert e8.max() <= e16.max() + max(2.0, 0.02 * np.abs(dense).max()), label


def test_logits_top1_and_cosine(cuda):
    # "test_int4_quantized_gemm.py", test_logits_top1_and_cosine: N = 32768,
    # K = 6656, outlier activations: argmax of every row agrees with W4A16
    # (>= 99%), cosine similarity >= 0.999.
    N, K = 32768, 6656
    for M in workloads.W4A8_BUCKETS:
        a8, a16, _ = _precision_case(cuda, N, K, M, True, seed_w=4242, seed_x=4300 + M)
        agree = (a8.argmax(axis=1) == a16.argmax(axis=1)).mean()
        cos = (a8 * a16).sum(1) / (np.linalg.norm(a8, axis=1) * np.linalg.norm(a16, axis=1))
        assert agree >= 0.99 and cos.min() >= 0.999, (M, agree, cos.min())
