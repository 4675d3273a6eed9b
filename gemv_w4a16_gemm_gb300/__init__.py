"""GB300 (sm_103a) weight-only quantized linear layer: W4A16, W4A8 and W8.

The compute lives in libw4q.so (CUDA kernels behind the C ABI of
include/w4q.h); ``w4q`` is its thin Python binding.
"""
from . import w4q  # noqa: F401
from .w4q import (W4QError, device_error, packed_bytes, split_choice,  # noqa: F401
                  w4_pack_weights, w4_unpack_weights, w4a8_gemm, w4a8_gemm_rowscale,
                  w4a8_group_dots, w4a8_group_dots_rowscale, w4a8_quantize_act,
                  w4a8_quantize_act_rowscale, w4a16_gemm, w8_gemv, workspace_bytes)
