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


def test_host_side_argument_checks_of_the_fused_and_backward_entries(lib):
    # one violated condition each; all are caught before any CUDA call
    raw = ctypes.create_string_buffer(512)
    p = ctypes.c_void_p((ctypes.addressof(raw) + 15) & ~15)  # a 16-byte aligned host address
    # router: null input, k above 8, E above 256, D not a multiple of 8 (16 for the backward), short workspace
    assert lib.moe_router_topk(None, p, 4, 128, 8, 2, p, p, p, None) == 1
    assert lib.moe_router_topk(p, p, 4, 128, 16, 9, p, p, p, None) == 1
    assert lib.moe_router_topk(p, p, 4, 128, 300, 2, p, p, p, None) == 1
    assert lib.moe_router_topk(p, p, 4, 12, 8, 2, p, p, p, None) == 1
    assert lib.moe_router_topk(p, p, 4, 128, 8, 9, p, p, p, None) == 1
    ws = lib.moe_router_backward_workspace_bytes(4, 128, 8)
    assert ws > 0
    assert lib.moe_router_backward(p, p, p, p, p, p, p, 4, 24, 8, 2, p, p, p, p, p, 1 << 30, None) == 1
    assert lib.moe_router_backward(p, p, p, p, p, p, p, 4, 128, 8, 2, p, p, p, p, p, ws - 1, None) == 1
    # gmm_fp8_swiglu: null lhs; F not a multiple of 128; blockwise lhs scales with K % 128 != 0;
    # an unknown scale mode
    assert lib.gmm_fp8_swiglu(None, p, 0, p, p, 0, p, 1, 0, 1, 1, 128, 128, 0, None, None, p, p, p, None) == 1
    assert lib.gmm_fp8_swiglu(p, p, 0, p, p, 0, p, 1, 0, 1, 1, 128, 64, 0, None, None, p, p, p, None) == 1
    assert lib.gmm_fp8_swiglu(p, p, 1, p, p, 0, p, 1, 0, 1, 1, 144, 128, 0, None, None, p, p, p, None) == 1
    assert lib.gmm_fp8_swiglu(p, p, 0, p, p, 1, p, 1, 0, 1, 1, 144, 128, 0, None, None, p, p, p, None) == 1
    assert lib.gmm_fp8_swiglu(p, p, 3, p, p, 0, p, 1, 0, 1, 1, 128, 128, 0, None, None, p, p, p, None) == 1
    # gmm_fp8_ksplit: K_split not a multiple of 128; K_split past K
    assert lib.gmm_fp8_ksplit(p, p, 0, p, p, 100, p, 1, 0, 1, 1, 256, 256, p, None) == 1
    assert lib.gmm_fp8_ksplit(p, p, 0, p, p, 384, p, 1, 0, 1, 1, 256, 256, p, None) == 1
    # tgmm_fp8_gcq: workspace too small; null gradient
    assert lib.tgmm_fp8_gcq(p, p, 2, p, p, p, 1, 0, 1, 1, 16, 16, p, p, 0, None) == 1
    assert lib.tgmm_fp8_gcq(p, p, 2, None, p, p, 1, 0, 1, 1, 16, 16, p, p, 1 << 20, None) == 1
    # moe_quantize_sort: D not a multiple of 16; k > 32
    assert lib.moe_quantize_sort(p, p, 1, 1, 1, 24, 0, None, p, p, p, p, p, p, p, 1 << 20, None) == 1
    assert lib.moe_quantize_sort(p, p, 1, 33, 1, 16, 0, None, p, p, p, p, p, p, p, 1 << 20, None) == 1
    # the backward's requantisers and the weight layout
    assert lib.moe_gather_scale_quant(p, None, p, 1, 1, 24, p, p, p, None) == 1       # D % 16
    assert lib.moe_swiglu_bwd_quant(p, p, 1, 24, p, p, p, None) == 1                  # F % 16
    assert lib.moe_quantize_group_cols(p, 1, 24, p, 1, 0, 1, p, p, None) == 1         # N % 16
    assert lib.moe_quantize_group_cols(p, 1, 16, p, 1, 1, 1, p, p, None) == 1         # shard past E
    assert lib.moe_swiglu_quant(p, 1, 24, 0, None, p, p, None) == 1                   # F % 16
    assert lib.moe_swiglu_quant(p, 1, 16, 2, None, p, p, None) == 1                   # static mode, no scale
    assert lib.moe_transpose_u8(p, 1, 24, 16, p, None) == 1                           # R % 16


def test_host_side_argument_checks_of_the_mxfp8_entries(lib):
    p = ctypes.c_void_p(256)  # a 16-byte aligned dummy address (never dereferenced)
    # quantiser: cols not a multiple of 32; null scale output
    assert lib.moe_quantize_rows_mx(p, 4, 48, p, p, None) == 1
    assert lib.moe_quantize_rows_mx(p, 4, 64, p, None, None) == 1
    # quantise + sort: D not a multiple of 32; short workspace
    assert lib.moe_quantize_sort_mx(p, p, 4, 2, 4, 48, p, p, p, p, p, p, p, 1 << 20, None) == 1
    assert lib.moe_quantize_sort_mx(p, p, 4, 2, 4, 64, p, p, p, p, p, p, p, 0, None) == 1
    # gmm: K not a multiple of 128; N not a multiple of 16; null rhs scales; shard past E
    assert lib.gmm_fp8_mx(p, p, p, p, p, 1, 0, 1, 8, 96, 256, p, None) == 1
    assert lib.gmm_fp8_mx(p, p, p, p, p, 1, 0, 1, 8, 128, 24, p, None) == 1
    assert lib.gmm_fp8_mx(p, p, p, None, p, 1, 0, 1, 8, 128, 256, p, None) == 1
    assert lib.gmm_fp8_mx(p, p, p, p, p, 2, 1, 2, 8, 128, 256, p, None) == 1
    # fused SwiGLU: F not a multiple of 128; null h scales
    assert lib.gmm_fp8_mx_swiglu(p, p, p, p, p, 1, 0, 1, 8, 128, 96, None, p, p, None) == 1
    assert lib.gmm_fp8_mx_swiglu(p, p, p, p, p, 1, 0, 1, 8, 128, 128, None, p, None, None) == 1
    # unfused SwiGLU requantisation: F not a multiple of 32
    assert lib.moe_swiglu_quant_mx(p, 4, 48, p, p, None) == 1


def test_host_side_argument_checks_of_the_int8_weight_entries(lib):
    p = ctypes.c_void_p(256)  # a 16-byte aligned dummy address (never dereferenced)
    # quantiser: K not a multiple of 16; blockwise K not a multiple of 128; null scales; static without scale
    assert lib.moe_quantize_weights_int8(p, 1, 4, 24, 0, None, p, p, None) == 1
    assert lib.moe_quantize_weights_int8(p, 1, 4, 144, 1, None, p, p, None) == 1
    assert lib.moe_quantize_weights_int8(p, 1, 4, 128, 0, None, p, None, None) == 1
    assert lib.moe_quantize_weights_int8(p, 1, 4, 128, 2, None, p, None, None) == 1
    # gmm: per-128 activation scales (not taken); K % 16; blockwise K % 128; N % 16;
    # shard past E; null weight scales
    assert lib.gmm_fp8_w8(p, p, 1, p, p, 0, p, 1, 0, 1, 8, 128, 256, p, None, 0, None) == 1
    assert lib.gmm_fp8_w8(p, p, 0, p, p, 0, p, 1, 0, 1, 8, 120, 256, p, None, 0, None) == 1
    assert lib.gmm_fp8_w8(p, p, 0, p, p, 1, p, 1, 0, 1, 8, 144, 256, p, None, 0, None) == 1
    assert lib.gmm_fp8_w8(p, p, 0, p, p, 0, p, 1, 0, 1, 8, 128, 24, p, None, 0, None) == 1
    assert lib.gmm_fp8_w8(p, p, 0, p, p, 0, p, 2, 1, 2, 8, 128, 256, p, None, 0, None) == 1
    assert lib.gmm_fp8_w8(p, p, 0, p, None, 0, p, 1, 0, 1, 8, 128, 256, p, None, 0, None) == 1
    # a workspace smaller than 2 M K bytes, or misaligned
    assert lib.gmm_fp8_w8_workspace_bytes(8, 128) == 2 * 8 * 128
    assert lib.gmm_fp8_w8(p, p, 0, p, p, 0, p, 1, 0, 1, 8, 128, 256, p, p, 2 * 8 * 128 - 1, None) == 1
    assert lib.gmm_fp8_w8(p, p, 0, p, p, 0, p, 1, 0, 1, 8, 128, 256, p, ctypes.c_void_p(264), 1 << 20, None) == 1
