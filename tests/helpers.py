"""Shared test helpers: the float acceptance rule and oracle-side preparation."""
import numpy as np
import torch

import oracle
import workloads

# Float acceptance against the fp64 oracle (per output tensor):
#   max |out - ref| <= 1e-2 * max |ref| + 1e-2   and
#   mean |out - ref| / mean |ref| <= 5e-3  (ratio of means, the form of the
#   precision checks in "test_int4_quantized_gemm.py", _check_close).
MAX_REL, MAX_ABS, MEAN_REL = 1e-2, 1e-2, 5e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(out, ref, what=""):
    o = to_f64(out) if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    assert o.shape == ref.shape, (what, o.shape, ref.shape)
    assert np.isfinite(o).all(), what
    err = np.abs(o - ref)
    bound = MAX_REL * np.abs(ref).max() + MAX_ABS
    assert err.max() <= bound, "%s: max err %g > %g" % (what, err.max(), bound)
    mean_rel = err.mean() / max(np.abs(ref).mean(), 1e-30)
    assert mean_rel <= MEAN_REL, "%s: mean rel err %g > %g" % (what, mean_rel, MEAN_REL)
    return err.max(), mean_rel


def quantized(N, K, seed=None):
    """(dense bf16 CPU weight, q, s, z) from the oracle quantizer."""
    W = workloads.w4_weight(N, K, seed)
    q, s, z = oracle.quantize_w4(W, N, K)
    return W, q, s, z
