"""The compact W4 metadata on the GPU vs the oracle ("test_int4_quantized_gemm.py":
CudaCoalescedInt4Tensor's uint8 scale / zero_point codes with float16
scale_step / zero_point_step, read as code x step).  The packer's bytes must
equal the oracle's bit for bit; the W4A16 output must match the compact
oracle within the float tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close

pytestmark = pytest.mark.gpu


def _quantized_c(N, K, seed=None):
    W = workloads.w4_weight(N, K, seed)
    return (W,) + tuple(oracle.quantize_w4c(W, N, K))


@pytest.mark.parametrize("N,K", [(16, 256), (257, 512), (768, 256), (1536, 512), (300, 6656)])
def test_pack_bit_exact(cuda, N, K):
    W, q, sc, zc, st = _quantized_c(N, K, seed=N + K)
    packed = w4q.w4_pack_weights_compact(W.to(cuda))
    assert packed.numel() == oracle.packed_bytes_c(N, K)
    assert np.array_equal(packed.cpu().numpy(), oracle.pack_w4c(q, sc, zc, st))
    gq, gsc, gzc, gst = w4q.w4_unpack_weights_compact(packed, N, K)
    assert np.array_equal(gq.cpu().numpy(), q) and np.array_equal(gsc.cpu().numpy(), sc)
    assert np.array_equal(gzc.cpu().numpy(), zc)
    assert np.array_equal(gst.cpu().view(torch.int16).numpy().view(np.uint16), st)


def test_pack_bit_exact_adversarial_groups(cuda):
    # constant, all-zero, same-sign, tiny and large groups in one weight
    N, K = 64, 512
    g = torch.Generator().manual_seed(9)
    W = torch.randn(N, K, generator=g)
    W[0, :32] = 3.0
    W[1, :64] = 0.0
    W[2, :32] = W[2, :32].abs() + 1.0
    W[3, 32:64] = -W[3, 32:64].abs() - 2.0
    W[4] *= 1e-4
    W[5] *= 500.0
    W = W.to(torch.bfloat16)
    q, sc, zc, st = oracle.quantize_w4c(W, N, K)
    packed = w4q.w4_pack_weights_compact(W.to(cuda))
    assert np.array_equal(packed.cpu().numpy(), oracle.pack_w4c(q, sc, zc, st))


def test_pack_bit_exact_full_size(cuda):
    N, K = workloads.W4A8_SHAPE
    W, q, sc, zc, st = _quantized_c(N, K)
    packed = w4q.w4_pack_weights_compact(W.to(cuda))
    assert np.array_equal(packed.cpu().numpy(), oracle.pack_w4c(q, sc, zc, st))


@pytest.mark.parametrize("N,K", workloads.SMALL_SHAPES + ((257, 256), (8448, 6656), (6656, 4096),
                                                          (256, 6656)))
def test_gemm_matches_oracle(cuda, N, K):
    W, q, sc, zc, st = _quantized_c(N, K, seed=N ^ K)
    packed = w4q.w4_pack_weights_compact(W.to(cuda))
    for M in (1, 2, 3, 4, 5, 8):
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        w4q.w4a16_gemm_compact(x.to(cuda), packed, N, K, out=out)
        assert_close(out, oracle.w4a16c(x, q, sc, zc, st), "compact N=%d K=%d M=%d" % (N, K, M))
    assert w4q.device_error() == 0


def test_gemm_full_size(cuda):
    N, K = workloads.W4A8_SHAPE
    W, q, sc, zc, st = _quantized_c(N, K)
    packed = w4q.w4_pack_weights_compact(W.to(cuda))
    for M in (1, 4):
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        out = w4q.w4a16_gemm_compact(x.to(cuda), packed, N, K)
        assert_close(out, oracle.w4a16c(x, q, sc, zc, st), "compact full M=%d" % M)


def test_compact_rejects_more_than_eight_rows(cuda):
    N, K = 64, 256
    packed = w4q.w4_pack_weights_compact(workloads.w4_weight(N, K, seed=1).to(cuda))
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a16_gemm_compact(torch.zeros(9, K, dtype=torch.bfloat16, device=cuda), packed, N, K)
    assert e.value.status == 2


def test_compact_is_within_the_precision_class_of_the_standard_format(cuda):
    # the compact metadata adds little error to the dense product: mean
    # |out_c - dense| / mean |dense| within 1.2x of the standard format's
    N, K, M = 4096, 4096, 4
    W = workloads.w4_weight(N, K, seed=12)
    x = workloads.activation(M, K, seed=13)
    dense = (x.double() @ W.double().T).numpy()
    Wd = W.to(cuda)
    oc = w4q.w4a16_gemm_compact(x.to(cuda), w4q.w4_pack_weights_compact(Wd), N, K)
    os_ = w4q.w4a16_gemm(x.to(cuda), w4q.w4_pack_weights(Wd), N, K)
    ec = np.abs(oc.double().cpu().numpy() - dense).mean()
    es = np.abs(os_.double().cpu().numpy() - dense).mean()
    assert ec <= 1.2 * es, (ec, es)
