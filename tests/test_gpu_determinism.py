"""Bitwise reproducibility: repeated calls and CUDA-graph replay equal eager
("test_int4_quantized_gemm.py": test_cuda_graph_replay_matches_eager and the
repeated-launch equality of the split-K tests)."""
import pytest
import torch

import workloads
from gemv_w4a16_gemm_gb300 import w4q

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16, 32, 64])
def test_graph_replay_matches_eager(cuda, M):
    N, K = 256, 768
    packed = w4q.w4_pack_weights(workloads.w4_weight(N, K, seed=88).to(cuda))
    x = workloads.activation(M, K, seed=M).to(cuda)
    W8, sc, _ = workloads.w8_inputs(N=N, K=K, M=1, seed=5)
    W8, sc = W8.to(cuda), sc.to(cuda)
    x8 = x[: min(M, 4)].contiguous()
    xa8 = x[: min(M, 8)].contiguous()          # W4A8 serves up to 8 rows
    eager = (w4q.w4a16_gemm(x, packed, N, K), w4q.w4a8_gemm(xa8, packed, N, K),
             w4q.w8_gemv(x8, W8, sc))
    # one workspace for the W4A16 call (M rows) and the W4A8 call (min(M, 8) rows)
    need = max(w4q.workspace_bytes(M, N, K), w4q.workspace_bytes(min(M, 8), N, K), 16)
    ws = torch.empty(need, dtype=torch.uint8, device=cuda)
    outs = (torch.empty_like(eager[0]), torch.empty_like(eager[1]), torch.empty_like(eager[2]))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            w4q.w4a16_gemm(x, packed, N, K, out=outs[0], workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4q.w4a16_gemm(x, packed, N, K, out=outs[0], workspace=ws)
        w4q.w4a8_gemm(xa8, packed, N, K, out=outs[1], workspace=ws)
        w4q.w8_gemv(x8, W8, sc, out=outs[2])
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)


def test_repeated_calls_are_bitwise_equal(cuda):
    N, K = 8448, 6656
    packed = w4q.w4_pack_weights(workloads.w4_weight(N, K).to(cuda))
    for M in (1, 4, 16, 64):
        x = workloads.activation(M, K, seed=M).to(cuda)
        for split in (None, 1, 4):
            a = w4q.w4a16_gemm(x, packed, N, K, split_k=split)
            b = w4q.w4a16_gemm(x, packed, N, K, split_k=split)
            assert torch.equal(a, b)
        if M <= 8:
            assert torch.equal(w4q.w4a8_gemm(x, packed, N, K), w4q.w4a8_gemm(x, packed, N, K))
    assert w4q.device_error() == 0
