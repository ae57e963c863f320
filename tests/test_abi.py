"""CPU checks of the C ABI: the library builds, loads without a GPU and
exports every function include/moefp8.h declares; host-side argument checks
reject bad calls before touching the device."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moefp8.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from fp8_quantized_moe_gb300 import _native
    return _native.load()


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("moe_quantize_rows", "moe_ragged_sort", "gmm_fp8", "tgmm_fp8", "ragged_gather_reduce",
              "moe_swiglu_quant", "moe_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from fp8_quantized_moe_gb300 import _native
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), n
        assert n in _native.SIGNATURES, f"{n} has no ctypes signature"
    out = subprocess.run(["nm", "-D", "--defined-only", _native.library_path()], capture_output=True, text=True)
    exported = set(re.findall(r" T (\w+)$", out.stdout, flags=re.M))
    assert set(names) <= exported


def test_host_side_argument_checks(lib):
    # null pointers and bad sizes are rejected on the host: no device call
    assert lib.moe_quantize_rows(None, 4, 16, 0, None, None, None, None) == 1
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    assert lib.moe_quantize_rows(p, 1, 17, 0, None, p, p, None) == 1        # cols % 16 != 0
    assert lib.moe_quantize_rows(p, 1, 16, 7, None, p, p, None) == 1        # bad mode
    assert lib.gmm_fp8(p, p, 0, p, p, 0, p, 0, 0, 1, 1, 128, 256, p, None) == 1      # E = 0
    assert lib.gmm_fp8(p, p, 0, p, p, 0, p, 2, 1, 2, 1, 128, 256, p, None) == 1      # shard past E
    assert lib.gmm_fp8(p, p, 0, p, p, 0, p, 1, 0, 1, 1, 120, 256, p, None) == 1      # K % 16
    assert lib.gmm_fp8(p, p, 1, p, p, 0, p, 1, 0, 1, 1, 144, 256, p, None) == 1      # blockwise K % 128
    assert lib.ragged_gather_reduce(p, p, None, 1, 33, 16, p, None) == 1             # k > 32
    assert lib.tgmm_fp8(p, p, 0, p, p, 2, p, 1, 0, 1, 1, 16, 16, p, p, 1 << 20, None) == 1  # lhs per-row
    assert lib.moe_ragged_sort_workspace_bytes(1000, 8, 256) >= 4 * 256
    assert lib.tgmm_fp8_workspace_bytes(1000, 256, 512, 8) >= (1000 + 8 * 128) * (256 + 512)
    assert lib.moe_status_string(0) == b"ok"
