"""W4A16 on the GPU vs the fp64 oracle ("test_int4_quantized_gemm.py": the
dequant + F.linear reference, every bucket on small and model shapes, the
tail shape N = 257, every legal split, dynamic M)."""
import pytest
import torch

import oracle
import workloads
from gemv_w4a16_gemm_gb300 import w4q
from helpers import assert_close, quantized

pytestmark = pytest.mark.gpu

BUCKETS = (1, 2, 3, 4, 8, 16, 32, 64)


def _run(cuda, N, K, Ms, seed_w=None, split_k=None):
    W, q, s, z = quantized(N, K, seed_w)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in Ms:
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        out = w4q.w4a16_gemm(x.to(cuda), packed, N, K, split_k=split_k)
        assert out.shape == (M, N) and out.dtype == torch.bfloat16
        assert_close(out, oracle.w4a16(x, q, s, z), "N=%d K=%d M=%d split=%s" % (N, K, M, split_k))


@pytest.mark.parametrize("N,K", workloads.SMALL_SHAPES + ((257, 256), (257, 512), (16, 256), (1, 256)))
def test_small_shapes_every_bucket(cuda, N, K):
    _run(cuda, N, K, BUCKETS, seed_w=N + K)


def test_tiny_workload(cuda):
    W, x = workloads.tiny_w4a16()
    N, K = W.shape
    q, s, z = oracle.quantize_w4(W, N, K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    assert_close(w4q.w4a16_gemm(x.to(cuda), packed, N, K), oracle.w4a16(x, q, s, z), "tiny")


@pytest.mark.parametrize("N,K", workloads.W4A16_GEMV_SHAPES)
def test_gemv_model_shapes_full(cuda, N, K):
    _run(cuda, N, K, workloads.W4A16_GEMV_MS)


@pytest.mark.parametrize("N,K", workloads.TC_SHAPES)
def test_skinny_gemm_shapes(cuda, N, K):
    # M = 16 / 64 on the full shapes, every output against the oracle (the
    # 39936 x 6656 M = 64 case is about 17 G multiply-adds on the host).  The
    # output starts as NaN, so a row the kernels never write fails.
    W, q, s, z = quantized(N, K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in workloads.TC_MS:
        x = workloads.activation(M, K, seed=workloads.x_seed(N, K, M))
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        w4q.w4a16_gemm(x.to(cuda), packed, N, K, out=out)
        assert_close(out, oracle.w4a16(x, q, s, z), "N=%d K=%d M=%d" % (N, K, M))


def test_tensor_core_split_pairs(cuda):
    # Stream-K on the tensor core with each 256-row pair's K spread over up
    # to 17 CTAs (2560 x 19968: 780 units over 152 CTAs), so the partial-sum
    # launch loads its contributors in several batches.  Every output is
    # compared (the output starts as NaN), and repeated calls agree bitwise.
    N, K = 2560, 19968
    W, q, s, z = quantized(N, K, seed=55)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in (9, 17, 40, 64):
        x = workloads.activation(M, K, seed=500 + M)
        xd = x.to(cuda)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        w4q.w4a16_gemm(xd, packed, N, K, out=out)
        assert_close(out, oracle.w4a16(x, q, s, z), "split pairs M=%d" % M)
        for _ in range(3):
            assert torch.equal(w4q.w4a16_gemm(xd, packed, N, K), out), M
    assert w4q.device_error() == 0


def test_every_legal_split_matches(cuda):
    # "test_int4_quantized_gemm.py", test_every_split_matches_dequant_matmul
    N, K = 256, 4096
    W, q, s, z = quantized(N, K, seed=91)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in (1, 2, 3, 4, 16, 17, 40, 64):
        x = workloads.activation(M, K, seed=100 + M)
        ref = oracle.w4a16(x, q, s, z)
        for split in (0, 1, 2, 3, 4, 5, 7, 8, 16):
            assert_close(w4q.w4a16_gemm(x.to(cuda), packed, N, K, split_k=split), ref,
                         "M=%d split=%d" % (M, split))


def test_stream_k_every_m(cuda):
    # 8448 x 6656 under explicit stream-K: 1716 units over two CTA slots per
    # SM, so most tile groups are split between CTAs and summed through the
    # split-K partials.  Every output is compared (the output starts as NaN),
    # and repeated calls must agree bitwise (the parts are summed in a fixed
    # order, whichever CTA arrives last).
    N, K = 8448, 6656
    W, q, s, z = quantized(N, K, seed=77)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in range(1, 9):
        x = workloads.activation(M, K, seed=300 + M)
        xd = x.to(cuda)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda)
        w4q.w4a16_gemm(xd, packed, N, K, split_k=0, out=out)
        assert_close(out, oracle.w4a16(x, q, s, z), "stream-K M=%d" % M)
        for _ in range(3):
            assert torch.equal(w4q.w4a16_gemm(xd, packed, N, K, split_k=0), out), M
    assert w4q.device_error() == 0


def test_illegal_split_is_rejected(cuda):
    N, K = 256, 768
    W = workloads.w4_weight(N, K, seed=0)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = torch.randn(1, K, dtype=torch.bfloat16, device=cuda)
    out = torch.full((1, N), 7.0, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a16_gemm(x, packed, N, K, split_k=4, out=out)
    assert e.value.status == 2
    assert torch.all(out == 7.0)   # nothing launched, output untouched


def test_every_runtime_m_up_to_64(cuda):
    # one compiled kernel per n8 width serves every M below it (rows masked)
    N, K = 300, 512
    W, q, s, z = quantized(N, K, seed=5)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in range(1, 65):
        x = workloads.activation(M, K, seed=M)
        assert_close(w4q.w4a16_gemm(x.to(cuda), packed, N, K), oracle.w4a16(x, q, s, z), "M=%d" % M)


def test_workspace_too_small_is_rejected(cuda):
    # The stream-K partition (split 0) needs a workspace: w4_workspace_bytes
    # covers both W4A16 and W4A8 (the larger, with the int8 activation
    # buffers); a buffer 16 bytes short fails W4A8, and a 16-byte buffer
    # fails W4A16 (its split-K counters and partials do not fit).
    N, K, M = 8448, 6656, 4
    need = w4q.workspace_bytes(M, N, K, split_k=0)
    assert need > 0
    W = workloads.w4_weight(N, K)
    packed = w4q.w4_pack_weights(W.to(cuda))
    x = torch.randn(M, K, dtype=torch.bfloat16, device=cuda)
    out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device=cuda)
    small = torch.empty(need - 16, dtype=torch.uint8, device=cuda)
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a8_gemm(x, packed, N, K, split_k=0, workspace=small, out=out)
    assert e.value.status == 4
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a16_gemm(x, packed, N, K, split_k=0, workspace=small[:16], out=out)
    assert e.value.status == 4
    assert torch.all(out == 3.0)


def test_misaligned_pointer_is_rejected(cuda):
    N, K = 64, 256
    W = workloads.w4_weight(N, K, seed=1)
    packed = w4q.w4_pack_weights(W.to(cuda))
    xbuf = torch.zeros(2 * K + 8, dtype=torch.bfloat16, device=cuda)
    x = xbuf[1:1 + K].view(1, K)      # 2-byte offset
    with pytest.raises(w4q.W4QError) as e:
        w4q.w4a16_gemm(x, packed, N, K)
    assert e.value.status == 3


def test_zero_activation_gives_zero(cuda):
    N, K = 257, 512
    W = workloads.w4_weight(N, K, seed=2)
    packed = w4q.w4_pack_weights(W.to(cuda))
    for M in (1, 4, 64):
        out = w4q.w4a16_gemm(torch.zeros(M, K, dtype=torch.bfloat16, device=cuda), packed, N, K)
        assert torch.all(out == 0)
    assert w4q.device_error() == 0


def _magnitude_rows(K, seed=11):
    """Nine bf16 activation rows of very different magnitudes (K = 8 super-blocks
    of 256): ordinary, near the bf16 normal limit, 2^100, 2^-100, one lone tiny
    super-block, alternating zero / 2^40 super-blocks, 2^-60 .. 2^80 across the
    row, subnormals only, and zero.  Every value stays below 2^122."""
    g = torch.Generator().manual_seed(seed)
    r = lambda: torch.randn(K, generator=g)  # noqa: E731
    rows = [r(), r() * 2.0 ** -126, r() * 2.0 ** 100, r() * 2.0 ** -100]
    lone = torch.zeros(K)
    lone[768:1024] = r()[768:1024] * 2.0 ** -60
    alt = r() * 2.0 ** 40
    for b in range(0, K // 256, 2):
        alt[256 * b:256 * (b + 1)] = 0
    wide = r()
    for b in range(K // 256):
        wide[256 * b:256 * (b + 1)] *= 2.0 ** (-60 + 20 * b)
    rows += [lone, alt, wide, r() * 2.0 ** -131, torch.zeros(K)]
    return torch.stack(rows).to(torch.bfloat16)


def test_activation_magnitudes_per_row(cuda):
    # The power-of-two prescale of x is chosen per row and 256-column
    # super-block (in the main kernel at M <= 2, in the prologue above), so
    # every row must come out right relative to its own size.  Per row:
    # |out - ref| <= 1e-2 * max |ref| + 2^-133 (one bf16 subnormal step, the
    # output format's own resolution); zero rows give exact zeros.
    N, K = 384, 2048
    W, q, s, z = quantized(N, K, seed=7)
    packed = w4q.w4_pack_weights(W.to(cuda))
    X = _magnitude_rows(K)
    for M in (1, 2, 3, 4, 8):
        for start in range(0, X.shape[0], M):
            idx = [(start + j) % X.shape[0] for j in range(M)]
            x = X[idx]
            out = w4q.w4a16_gemm(x.to(cuda), packed, N, K).double().cpu().numpy()
            ref = oracle.w4a16(x, q, s, z)
            for j, row in enumerate(idx):
                what = "M=%d row regime %d" % (M, row)
                assert (abs(out[j]) < float("inf")).all(), what
                if not x[j].any():
                    assert (out[j] == 0).all(), what
                    continue
                err = abs(out[j] - ref[j]).max()
                assert err <= 1e-2 * abs(ref[j]).max() + 2.0 ** -133, (what, err, abs(ref[j]).max())
    assert w4q.device_error() == 0


def test_partition_choice_and_launch_count(cuda):
    # Tensor-core path (M >= 9) with at most 4 super-blocks and no more
    # 256-row pairs than SMs: each CTA takes a pair's whole K (split 1), so
    # the call is two launches, with no partial-sum launch.
    for M in (9, 16, 64):
        assert w4q.split_choice(M, 1536, 512) == 1, M
        assert w4q.kernel_launches(M, 1536, 512) == 2, M
    # Longer K keeps the balanced stream-K partition, and its partial-sum
    # launch where row-group pairs are split over CTAs.
    assert w4q.split_choice(16, 39936, 6656) == 0
    assert w4q.kernel_launches(16, 39936, 6656) == 3
    # M <= 8: a cluster split (1..8 CTAs per 128-row group) is one launch
    # with no workspace; stream-K (0) is a prologue and the main kernel.
    for (N, K) in ((1536, 512), (256, 6656), (8448, 6656), (6656, 4096), (6656, 19968),
                   (39936, 6656), (300, 512)):
        for M in (1, 2, 3, 4, 8):
            for kind in (False, "group", "row"):
                if kind and M > 8:
                    continue
                c = w4q.split_choice(M, N, K)
                assert 0 <= c <= 8, (N, K, M, c)
                n = w4q.kernel_launches(M, N, K, kind)
                if kind is False:
                    assert n == (1 if c >= 1 else 2), (N, K, M, c, n)
                    if c >= 1:
                        assert w4q.workspace_bytes(M, N, K, split_k=c) == 0
                else:
                    assert n in (1, 2), (N, K, M, kind, n)
