"""CPU oracle (test infrastructure): plain C fp64 reference of the quantized
linear layer, wrapped with numpy.  Only tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the product library never does."""
from .oracle import (GROUP, act_quant, act_quant_row, bf16_bits_to_f64, build,  # noqa: F401
                     dequant_w4, pack_w4, packed_bytes, quantize_w4, set_threads,
                     unpack_w4, w4a8, w4a8_group_dots, w4a8_row, w4a16, w8)
from .oracle import (dequant_w4c, pack_w4c, packed_bytes_c, quantize_w4c,  # noqa: F401
                     unpack_w4c, w4a16c)
