"""GPU quantizer/packer vs the oracle: the packed bytes must match bit-exactly
("test_int4_quantized_gemm.py", _packed_with_dense: INT4, group 32,
asymmetric min-max; layout of include/w4q.h)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("N,K", [(16, 256), (257, 256), (256, 768), (768, 256), (1536, 512),
                                 (40, 1024), (1, 256), (300, 6656)])
def test_pack_is_bit_exact(cuda, N, K):
    W = workloads.w4_weight(N, K, seed=N + K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    q, s, z = oracle.quantize_w4(W, N, K)
    ref = oracle.pack_w4(q, s, z)
    got = packed.cpu().numpy()
    assert got.shape == ref.shape
    mism = np.flatnonzero(got != ref)
    assert mism.size == 0, "first mismatching bytes: %s" % mism[:10]


def test_unpack_roundtrip(cuda):
    N, K = 257, 512
    W = workloads.w4_weight(N, K, seed=3)
    packed = w4q.w4_pack_weights(W.to(cuda))
    q, s, z = w4q.w4_unpack_weights(packed, N, K)
    oq, os_, oz = oracle.quantize_w4(W, N, K)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(_bits(s.cpu()), os_)
    assert np.array_equal(z.cpu().numpy(), oz)


def test_pack_adversarial_groups(cuda):
    # ties with odd and even zero points, constant and same-sign groups,
    # signed zeros, subnormal and huge ranges: one group per row
    def grp(vals):
        vals = list(vals) + [vals[-1]] * (32 - len(vals))
        return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    tiny = torch.tensor([1], dtype=torch.int16).view(torch.bfloat16).float().item()
    rows = [
        [-1.0, 14.0, 0.5, 1.5, 2.5, -0.5, 3.5, 12.5],
        [-2.0, 13.0, 0.5, 1.5, 2.5, -1.5, 4.5],
        [0.0], [-0.0, 0.0, -0.0], [3.0], [-3.0],
        [1.0, 1.25, 1.5, 2.0], [-1.0, -1.25, -1.5, -2.0],
        [-2.0, 5.5, -1.5, 0.0, 0.5, 3.0, 4.5],
        [tiny, 3 * tiny],
        [-3.3e38, 3.3e38, 1.0e38],
    ]
    N, K = 16, 256
    W = torch.zeros(N, K, dtype=torch.bfloat16)
    for i, r in enumerate(rows):
        W[i, 32:64] = grp(r)       # group 1 of row i
        W[i, 0:32] = grp(r[::-1])  # group 0 reversed
    packed = w4q.w4_pack_weights(W.to(cuda))
    q, s, z = oracle.quantize_w4(W, N, K)
    assert np.array_equal(packed.cpu().numpy(), oracle.pack_w4(q, s, z))


def test_pack_full_size_largest_shape(cuda):
    # the largest shape of the workloads, 39936 x 6656 (158 MB packed)
    N, K = workloads.W4A8_SHAPE
    W = workloads.w4_weight(N, K)
    packed = w4q.w4_pack_weights(W.to(cuda)).cpu().numpy()
    q, s, z = oracle.quantize_w4(W, N, K)
    ref = oracle.pack_w4(q, s, z)
    assert np.array_equal(packed, ref)
