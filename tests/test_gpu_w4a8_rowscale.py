"""W4A8 with one int8 activation scale per whole row on the GPU vs the oracle
(the 39936 x 6656 W4A8 workload's scheme; "test_int4_quantized_gemm.py": the
W4A8 bucket kernels and Int4QuantizedGemmPrecisionTest, gaussian case).  The
integer parts (int8 activations, the row scales, the per-group dot products)
must match bit-exactly; the float output within the float tolerance of the
per-row W4A8 oracle and within the pages' 0.02 precision class against the
W4A16 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close, quantized

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1, 256), (4, 6656), (3, 19968), (8, 512), (2, 2048)])
def test_activation_quantizer_bit_exact(cuda, M, K):
    x = workloads.activation(M, K, seed=M * 11 + K)
    x[0, 5] = 0.0
    x[0, 64:96] = 0.0                    # an all-zero group: still the row's scale
    x[0, 200] = 300.0                    # an outlier sets the whole row's scale
    if M > 1:
        x[1] = 0.0                       # an all-zero row: sx = 0, xq = 0
    xq, sx = w4q.w4a8_quantize_act_rowscale(x.to(cuda))
    oxq, osx = oracle.act_quant_row(x, K)
    assert sx.shape == (M,)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oxq)


def _all_bf16_rows(maxima):
    """One row per maximum a: a, then every positive finite bf16 number up to
    a (each larger one replaced by a, the row padded with a), signs
    alternating.  K = 32768."""
    K = 32768
    bits = np.arange(1, 0x7F80, dtype=np.uint32)      # the positive finite bf16 numbers
    vals = (bits << 16).view(np.float32)
    vals = np.concatenate([vals, np.full(K - 1 - vals.size, np.inf, np.float32)])
    rows = []
    for a in maxima:
        a = float(torch.tensor(a, dtype=torch.bfloat16))
        v = np.minimum(vals, np.float32(a))
        v = np.where(np.arange(v.size) % 2 == 0, v, -v)
        rows.append(np.concatenate([[np.float32(a)], v]))
    return torch.from_numpy(np.stack(rows).astype(np.float32)).to(torch.bfloat16), K


def test_activation_quantizer_every_bf16_value(cuda):
    # every positive bf16 magnitude under several row maxima (quotients near
    # every half-integer included): the int8 codes and scales bit for bit
    x, K = _all_bf16_rows((127.0, 1.0, 3.7e-3, 300.0, 1e30, 2.0 ** -120, 0.4375, 6.02e4))
    xq, sx = w4q.w4a8_quantize_act_rowscale(x.to(cuda))
    oxq, osx = oracle.act_quant_row(x, K)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), osx.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), oxq), np.argwhere(xq.cpu().numpy() != oxq)[:5]


def test_activation_quantizer_ties(cuda):
    # max |x| = 127 -> sx = 1 exactly; .5 ties round to even
    K = 512
    vals = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 3.0, -126.0]
    x = torch.tensor(vals * (K // 8), dtype=torch.float32).to(torch.bfloat16).view(1, K)
    xq, sx = w4q.w4a8_quantize_act_rowscale(x.to(cuda))
    assert float(sx[0]) == 1.0
    assert xq[0, :8].tolist() == [127, 0, 2, 2, 0, -2, 3, -126]


@pytest.mark.parametrize("N,K,M", [(257, 512, 1), (256, 768, 4), (1536, 512, 3), (768, 256, 2),
                                   (300, 6656, 4), (96, 512, 8), (40, 256, 6)])
def test_group_dots_bit_exact(cuda, N, K, M):
    W, q, s, z = quantized(N, K, seed=N ^ K ^ 5)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(M, K, seed=M + 23)
    x[0, K - 3] = 40.0   # row 0's max sits in the last K slice (the last CTA of a cluster)
    D = w4q.w4a8_group_dots_rowscale(x.to(cuda), packed, N, K).cpu().numpy()
    xq, sx = oracle.act_quant_row(x, K)
    ref = oracle.w4a8_group_dots(xq, q, z)
    assert np.array_equal(D, ref), np.argwhere(D != ref)[:5]


def _check(cuda, N, K, Ms, split_k=None, seed_w=None):
    W, q, s, z = quantized(N, K, seed_w)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in Ms:
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        w4q.w4a8_gemm_rowscale(x.to(cuda), packed, N, K, split_k=split_k, out=out)
        xq, sx = oracle.act_quant_row(x, K)
        ref8 = oracle.w4a8_row(xq, sx, q, s, z)
        assert_close(out, ref8, "W4A8 row N=%d K=%d M=%d split=%s" % (N, K, M, split_k))
        ref16 = oracle.w4a16(x, q, s, z)
        o = out.double().cpu().numpy()
        rel = np.abs(o - ref16).mean() / np.abs(ref16).mean()
        assert rel < 0.02, ("precision class vs W4A16", M, rel)


@pytest.mark.parametrize("N,K", workloads.SMALL_SHAPES + ((257, 256), (16, 256)))
def test_small_shapes(cuda, N, K):
    _check(cuda, N, K, (1, 2, 3, 4, 5, 8), seed_w=N + K)


def test_w4a8_rowscale_workload_full_size(cuda):
    # N = 39936, K = 6656, M = 1..4: every output against the oracle
    N, K = workloads.W4A8_SHAPE
    _check(cuda, N, K, workloads.W4A8_MS)


@pytest.mark.parametrize("N,K", ((8448, 6656), (6656, 4096), (6656, 19968), (256, 6656)))
def test_model_shapes(cuda, N, K):
    _check(cuda, N, K, (1, 4))


def test_every_legal_split_matches(cuda):
    N, K = 256, 4096
    for split in (0, 1, 2, 3, 4, 5, 7, 8, 16):
        _check(cuda, N, K, (1, 4), split_k=split, seed_w=93)


def test_stream_k(cuda):
    # explicit stream-K on 8448 x 6656 (groups split between CTAs): every
    # output against the oracle, repeated calls bitwise equal
    N, K = 8448, 6656
    _check(cuda, N, K, (1, 2, 3, 4, 8), split_k=0, seed_w=96)
    W = workloads.w4_weight(N, K, 96)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(3, K, seed=97).to(cuda)
    ref = w4q.w4a8_gemm_rowscale(x, packed, N, K, split_k=0)
    for _ in range(3):
        assert torch.equal(w4q.w4a8_gemm_rowscale(x, packed, N, K, split_k=0), ref)
    assert w4q.device_error() == 0


def test_row_max_in_another_slice_of_the_cluster(cuda):
    # per-row scale with the row's max in a different K slice for each row,
    # under every cluster split: the slices' maxima must be combined
    N, K = 384, 2048
    W, q, s, z = quantized(N, K, seed=94)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(4, K, seed=95)
    for m, k in enumerate((5, 700, 1300, K - 1)):
        x[m, k] = 60.0 * (1 if m % 2 else -1)
    xq, sx = oracle.act_quant_row(x, K)
    ref8 = oracle.w4a8_row(xq, sx, q, s, z)
    for split in (1, 2, 3, 5, 8):
        out = w4q.w4a8_gemm_rowscale(x.to(cuda), packed, N, K, split_k=split)
        assert_close(out, ref8, "split %d" % split)


def test_zero_rows_and_more_than_eight_rows(cuda):
    N, K = 128, 512
    W, q, s, z = quantized(N, K, seed=8)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = workloads.activation(3, K, seed=10)
    x[1] = 0
    out = w4q.w4a8_gemm_rowscale(x.to(cuda), packed, N, K)
    assert torch.all(out[1] == 0)
    xq, sx = oracle.act_quant_row(x, K)
    assert_close(out, oracle.w4a8_row(xq, sx, q, s, z), "zero row")
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a8_gemm_rowscale(torch.zeros(9, K, dtype=torch.bfloat16, device=cuda), packed, N, K)
    assert e.value.status == 2
    assert w4q.device_error() == 0
