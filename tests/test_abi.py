"""CPU-only checks of the C ABI: the library loads, exports every entry point
declared in include/w4q.h, and rejects invalid arguments on the host before
touching the GPU."""
import ctypes
import os
import re

import pytest

from gemv_w4a16_gemm_gb300 import w4q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4q.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_expected_api():
    names = declared_functions()
    for required in ("w4_pack_weights", "w4a16_gemm", "w4a8_gemm", "w8_gemv"):
        assert required in names
    assert set(names) == set(w4q.SIGNATURES), set(names) ^ set(w4q.SIGNATURES)


def test_library_exports_every_declared_symbol():
    lib = w4q.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings():
    for code in range(7):
        assert w4q.status_string(code).startswith(w4q.STATUS[code])
    assert w4q.status_string(99) == "W4Q_ERR_UNKNOWN"


def test_packed_bytes():
    assert w4q.packed_bytes(256, 768) == 116736
    assert w4q.packed_bytes(257, 256) == 3 * 8 * 2432
    assert w4q.packed_bytes(39936, 6656) == 157827072
    assert w4q.packed_bytes(64, 288) == 0          # K % 256 != 0
    assert w4q.packed_bytes(64, 256, 64) == 0      # group != 32
    assert w4q.packed_bytes(0, 256) == 0


FAKE = 1 << 20   # a 16-byte aligned non-null "device" address, never dereferenced


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, 1, 256, 288, 32, None, 0, None), 2),   # K % 256 != 0
    ((FAKE, FAKE, FAKE, 1, 256, 256, 64, None, 0, None), 2),   # group != 32
    ((FAKE, FAKE, FAKE, 65, 256, 256, 32, None, 0, None), 2),  # M above 64
    ((FAKE, FAKE, FAKE, 0, 256, 256, 32, None, 0, None), 1),   # M = 0
    ((FAKE, FAKE, FAKE, 1, -3, 256, 32, None, 0, None), 1),    # negative N
    ((None, FAKE, FAKE, 1, 256, 256, 32, None, 0, None), 1),   # null x
    ((FAKE + 2, FAKE, FAKE, 1, 256, 256, 32, None, 0, None), 3),  # misaligned x
    ((FAKE, FAKE + 8, FAKE, 1, 256, 256, 32, None, 0, None), 3),  # misaligned packed
])
def test_gemm_rejects_invalid_arguments_on_the_host(args, status):
    lib = w4q.lib()
    assert lib.w4a16_gemm(*args) == status
    assert lib.w4a8_gemm(*args) == status


def test_split_rules_on_the_host():
    lib = w4q.lib()
    # "test_int4_quantized_gemm.py", test_an_illegal_split_is_rejected:
    # K = 768 has 3 super-blocks of 256, so split 4 is illegal.
    assert lib.w4a16_gemm_split(FAKE, FAKE, FAKE, 1, 256, 768, 32, 4, None, 0, None) == 2
    assert lib.w4a16_gemm_split(FAKE, FAKE, FAKE, 1, 256, 768, 32, -1, None, 0, None) == 1
    assert lib.w4_workspace_bytes_split(1, 256, 768, 32, 4) == 0


def test_other_entry_points_reject_on_the_host():
    lib = w4q.lib()
    assert lib.w4_pack_weights(None, 16, 256, 32, FAKE, None) == 1
    assert lib.w4_pack_weights(FAKE, 16, 300, 32, FAKE, None) == 2
    assert lib.w4_pack_weights(FAKE + 4, 16, 256, 32, FAKE, None) == 3
    assert lib.w4_unpack_weights(FAKE, 16, 256, 32, None, FAKE, FAKE, None) == 1
    assert lib.w4a8_quantize_act(FAKE, 1, 100, FAKE, FAKE, None) == 2
    assert lib.w4a8_group_dots(FAKE, FAKE, 1, 16, 256, 32, None, None, 0, None) == 1
    assert lib.w8_gemv(FAKE, FAKE, FAKE, FAKE, 5, 16, 256, None) == 2    # M > 4
    assert lib.w8_gemv(FAKE, FAKE, FAKE, FAKE, 1, 16, 250, None) == 2    # K % 16
    assert lib.w8_gemv(FAKE, FAKE, FAKE, FAKE, 1, 16, 32768, None) == 2  # K too large
    assert lib.w8_gemv(None, FAKE, FAKE, FAKE, 1, 16, 256, None) == 1
    assert lib.w8_gemv(FAKE, FAKE + 1, FAKE, FAKE, 1, 16, 256, None) == 3
    assert lib.w4q_device_error(None) == 1


def test_split_k_legality_fixture():
    # tests/golden/split_k_legality.txt: the pages' rule split <= K // 256.
    path = os.path.join(ROOT, "tests", "golden", "split_k_legality.txt")
    lib = w4q.lib()
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        k, split, legal = line.split()
        st = lib.w4a16_gemm_split(FAKE, FAKE, FAKE, 1, 256, int(k), 32, int(split), None, 0, None)
        if legal == "illegal":
            assert st == 2, (k, split)
        n += 1
    assert n >= 10
