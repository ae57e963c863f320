"""GB300 (sm_103a) FP8-quantized MoE expert FFN.

Python binding of libmoefp8.so (C ABI in include/moefp8.h).  Every function
here only marshals arguments: it allocates outputs with PyTorch, passes raw
device pointers and the current CUDA stream, and checks the status.  All
arithmetic runs in the library's CUDA kernels; there is no fallback.

Forward path (the order of "Quantize activations before EP all gather"):
quantize_rows -> ragged_sort -> gmm (wi_0 | wi_1) -> swiglu_quant ->
gmm (wo) -> ragged_gather_reduce.  With int8 expert weights ("Keep qwix out
of tpu-inference's fused MoE kernel and pre-quantize weights": float8_e4m3fn
or int8 weights) both contractions run gmm_w8.  The backward pass of the static scheme
("Support quantization for tokamax gmm v2": fp8_static_wa) adds
gather_scale_quant, swiglu_bwd_quant, quantize_group_cols and tgmm.

The MXFP8 variant (MX32: OCP MX v1.0 blocks of 32 e4m3 values sharing one
E8M0 power-of-two scale along the contracted dimension) runs the same
forward path on the block-scaled tensor-core MMA: quantize_sort_mx ->
gmm_mx_swiglu (or gmm_mx + swiglu_quant_mx) -> gmm_mx -> ragged_gather_reduce.
"""

from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import torch

from . import _native
from ._native import MoEError, check

PER_ROW = 0
PER_ROW_BLOCK128 = 1
PER_TENSOR = 2
PER_GROUP_COL = 3
MX32 = 4  # MXFP8: uint8 E8M0 codes, K-block-major [cols/128, rows, 4]

__all__ = [
    "PER_ROW", "PER_ROW_BLOCK128", "PER_TENSOR", "PER_GROUP_COL", "MoEError", "lib", "device_error",
    "quantize_rows", "quantize_weights", "ragged_sort", "gmm", "gmm_swiglu", "swiglu_fusable", "swiglu_fuse_pays", "swiglu_quant", "ragged_gather_reduce",
    "gather_scale_quant", "swiglu_bwd_quant", "quantize_group_cols", "tgmm", "transpose_u8",
    "router_topk", "router_backward", "MX32", "quantize_rows_mx", "quantize_weights_mx", "quantize_sort_mx",
    "gmm_mx", "gmm_mx_swiglu", "swiglu_quant_mx", "quantize_weights_int8", "gmm_w8", "gmm_w8_workspace_bytes",
    "prepare_weights_w8",
    "ExpertWeights", "prepare_weights", "FFNBuffers", "ffn_forward", "ffn_backward",
]


def lib():
    return _native.load()


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise MoEError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise MoEError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _nb(cols: int) -> int:
    return (cols + 127) // 128


def device_error() -> int:
    """Synchronise the current stream and return (and clear) the device error word."""
    code = ctypes.c_int(0)
    st = lib().moe_get_device_error(_s(), ctypes.byref(code))
    if st not in (0, 4):
        check(st, "moe_get_device_error")
    return code.value


def _scale_buf(mode: int, rows: int, cols: int, device, out=None):
    if out is not None:
        return out
    if mode == PER_ROW:
        return torch.empty(rows, dtype=torch.float32, device=device)
    if mode == PER_ROW_BLOCK128:
        return torch.empty(rows, _nb(cols), dtype=torch.float32, device=device)
    if mode == MX32:
        return torch.empty(cols // 128, rows, 4, dtype=torch.uint8, device=device)
    return None


def quantize_rows(x: torch.Tensor, mode: int, static_scale: Optional[torch.Tensor] = None, q=None, scale=None):
    """bf16 [rows, cols] -> (e4m3 codes uint8 [rows, cols], fp32 scales or None)."""
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device) if q is None else q
    scale = _scale_buf(mode, rows, cols, x.device, scale)
    check(lib().moe_quantize_rows(_p(x), rows, cols, mode, _p(static_scale), _p(q), _p(scale), _s()),
          "moe_quantize_rows")
    return q, scale


def quantize_weights(w: torch.Tensor, mode: int, static_scale: Optional[torch.Tensor] = None):
    """bf16 [E, N, K] -> (codes [E, N, K], scales [E, N] | [E, K/128, N] | None)."""
    E, N, K = w.shape
    q = torch.empty(E, N, K, dtype=torch.uint8, device=w.device)
    if mode == PER_ROW:
        s = torch.empty(E, N, dtype=torch.float32, device=w.device)
    elif mode == PER_ROW_BLOCK128:
        s = torch.empty(E, _nb(K), N, dtype=torch.float32, device=w.device)
    else:
        s = None
    check(lib().moe_quantize_weights(_p(w), E, N, K, mode, _p(static_scale), _p(q), _p(s), _s()),
          "moe_quantize_weights")
    return q, s


def quantize_weights_int8(w: torch.Tensor, mode: int, static_scale: Optional[torch.Tensor] = None):
    """bf16 [E, N, K] -> (int8 codes [E, N, K], scales [E, N] | [E, K/128, N] | None)."""
    E, N, K = w.shape
    q = torch.empty(E, N, K, dtype=torch.int8, device=w.device)
    if mode == PER_ROW:
        s = torch.empty(E, N, dtype=torch.float32, device=w.device)
    elif mode == PER_ROW_BLOCK128:
        s = torch.empty(E, _nb(K), N, dtype=torch.float32, device=w.device)
    else:
        s = None
    check(lib().moe_quantize_weights_int8(_p(w), E, N, K, mode, _p(static_scale), _p(q), _p(s), _s()),
          "moe_quantize_weights_int8")
    return q, s


def quantize_rows_mx(x: torch.Tensor, q=None, sf=None):
    """MXFP8: bf16 [rows, cols] -> (e4m3 codes [rows, cols], E8M0 codes uint8 [cols/128, rows, 4])."""
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device=x.device) if q is None else q
    sf = _scale_buf(MX32, rows, cols, x.device, sf)
    check(lib().moe_quantize_rows_mx(_p(x), rows, cols, _p(q), _p(sf), _s()), "moe_quantize_rows_mx")
    return q, sf


def quantize_weights_mx(w: torch.Tensor):
    """MXFP8 weights: bf16 [E, N, K] -> (codes [E, N, K], E8M0 codes [K/128, E*N, 4])."""
    E, N, K = w.shape
    q, sf = quantize_rows_mx(w.reshape(E * N, K))
    return q.view(E, N, K), sf


def ragged_sort(topk_ids: torch.Tensor, E: int, x_q: torch.Tensor, x_scale: Optional[torch.Tensor], mode: int,
                out: Optional[dict] = None):
    """Returns dict(sorted_src, pos, group_sizes, group_offsets, xs_q, xs_scale)."""
    T, k = topk_ids.shape
    D = x_q.shape[1]
    R = T * k
    dev = x_q.device
    o = out if out is not None else {}
    if "sorted_src" not in o:
        o["sorted_src"] = torch.empty(R, dtype=torch.int32, device=dev)
        o["pos"] = torch.empty(R, dtype=torch.int32, device=dev)
        o["group_sizes"] = torch.empty(E, dtype=torch.int32, device=dev)
        o["group_offsets"] = torch.empty(E + 1, dtype=torch.int32, device=dev)
        o["xs_q"] = torch.empty(R, D, dtype=torch.uint8, device=dev)
        o["xs_scale"] = _scale_buf(mode, R, D, dev)
    nws = lib().moe_ragged_sort_workspace_bytes(T, k, E)
    if "sort_ws" not in o or o["sort_ws"].numel() < nws:
        o["sort_ws"] = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    xs_scale = o["xs_scale"]
    check(lib().moe_ragged_sort(_p(topk_ids), T, k, E, _p(x_q), _p(x_scale), D, mode, _p(o["sorted_src"]),
                                _p(o["pos"]), _p(o["group_sizes"]), _p(o["group_offsets"]), _p(o["xs_q"]),
                                _p(xs_scale), _p(o["sort_ws"]), o["sort_ws"].numel(), _s()), "moe_ragged_sort")
    return o


def quantize_sort(x: torch.Tensor, topk_ids: torch.Tensor, E: int, mode: int,
                  static_scale: Optional[torch.Tensor] = None, out: Optional[dict] = None):
    """Steps 1 + 2 fused: sort indices and the gathered codes/scales of x.
    Returns the same dict as ragged_sort (bit-identical xs_q / xs_scale)."""
    T, k = topk_ids.shape
    D = x.shape[1]
    R = T * k
    dev = x.device
    o = out if out is not None else {}
    if "sorted_src" not in o:
        o["sorted_src"] = torch.empty(R, dtype=torch.int32, device=dev)
        o["pos"] = torch.empty(R, dtype=torch.int32, device=dev)
        o["group_sizes"] = torch.empty(E, dtype=torch.int32, device=dev)
        o["group_offsets"] = torch.empty(E + 1, dtype=torch.int32, device=dev)
        o["xs_q"] = torch.empty(R, D, dtype=torch.uint8, device=dev)
        o["xs_scale"] = _scale_buf(mode, R, D, dev)
    nws = lib().moe_ragged_sort_workspace_bytes(T, k, E)
    if "sort_ws" not in o or o["sort_ws"].numel() < nws:
        o["sort_ws"] = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    xs_scale = o["xs_scale"] if mode != PER_TENSOR else None
    check(lib().moe_quantize_sort(_p(x), _p(topk_ids), T, k, E, D, mode, _p(static_scale), _p(o["sorted_src"]),
                                  _p(o["pos"]), _p(o["group_sizes"]), _p(o["group_offsets"]), _p(o["xs_q"]),
                                  _p(xs_scale), _p(o["sort_ws"]), o["sort_ws"].numel(), _s()), "moe_quantize_sort")
    return o


def quantize_sort_mx(x: torch.Tensor, topk_ids: torch.Tensor, E: int, out: Optional[dict] = None):
    """MXFP8 steps 1 + 2: the dict of quantize_sort with xs_scale = E8M0 codes [D/128, T*k, 4]."""
    T, k = topk_ids.shape
    D = x.shape[1]
    R = T * k
    dev = x.device
    o = out if out is not None else {}
    if "sorted_src" not in o:
        o["sorted_src"] = torch.empty(R, dtype=torch.int32, device=dev)
        o["pos"] = torch.empty(R, dtype=torch.int32, device=dev)
        o["group_sizes"] = torch.empty(E, dtype=torch.int32, device=dev)
        o["group_offsets"] = torch.empty(E + 1, dtype=torch.int32, device=dev)
        o["xs_q"] = torch.empty(R, D, dtype=torch.uint8, device=dev)
        o["xs_scale"] = _scale_buf(MX32, R, D, dev)
    nws = lib().moe_ragged_sort_workspace_bytes(T, k, E)
    if "sort_ws" not in o or o["sort_ws"].numel() < nws:
        o["sort_ws"] = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    check(lib().moe_quantize_sort_mx(_p(x), _p(topk_ids), T, k, E, D, _p(o["sorted_src"]), _p(o["pos"]),
                                     _p(o["group_sizes"]), _p(o["group_offsets"]), _p(o["xs_q"]), _p(o["xs_scale"]),
                                     _p(o["sort_ws"]), o["sort_ws"].numel(), _s()), "moe_quantize_sort_mx")
    return o


def gmm_mx(lhs_q, lhs_sf, rhs_q, rhs_sf, group_sizes, group_offset: int = 0, E_local: Optional[int] = None,
           out=None):
    """MXFP8 grouped matmul -> bf16 [M, N]; lhs_sf [K/128, M, 4], rhs_sf [K/128, E_local*N, 4]."""
    M, K = lhs_q.shape
    El, N, K2 = rhs_q.shape
    if K2 != K:
        raise MoEError("lhs/rhs K mismatch")
    E = group_sizes.numel()
    E_local = El if E_local is None else E_local
    out = torch.empty(M, N, dtype=torch.bfloat16, device=lhs_q.device) if out is None else out
    check(lib().gmm_fp8_mx(_p(lhs_q), _p(lhs_sf), _p(rhs_q), _p(rhs_sf), _p(group_sizes), E, group_offset, E_local,
                           M, K, N, _p(out), _s()), "gmm_fp8_mx")
    return out


def gmm_mx_swiglu(lhs_q, lhs_sf, rhs_q, rhs_sf, group_sizes, group_offset: int = 0, E_local: Optional[int] = None,
                  keep_a: bool = False, a_out=None, h_q=None, h_sf=None):
    """MXFP8 gmm with [wi_0 | wi_1] fused with SwiGLU and the MXFP8
    requantisation of h.  Returns (h_q [M, F], h_sf [F/128, M, 4], a [M, 2F] bf16 or None)."""
    M, K = lhs_q.shape
    El, F2, K2 = rhs_q.shape
    if K2 != K:
        raise MoEError("lhs/rhs K mismatch")
    F = F2 // 2
    dev = lhs_q.device
    E = group_sizes.numel()
    E_local = El if E_local is None else E_local
    h_q = torch.empty(M, F, dtype=torch.uint8, device=dev) if h_q is None else h_q
    h_sf = _scale_buf(MX32, M, F, dev, h_sf)
    if keep_a and a_out is None:
        a_out = torch.empty(M, F2, dtype=torch.bfloat16, device=dev)
    check(lib().gmm_fp8_mx_swiglu(_p(lhs_q), _p(lhs_sf), _p(rhs_q), _p(rhs_sf), _p(group_sizes), E, group_offset,
                                  E_local, M, K, F, _p(a_out), _p(h_q), _p(h_sf), _s()), "gmm_fp8_mx_swiglu")
    return h_q, h_sf, a_out


def swiglu_quant_mx(a: torch.Tensor, h_q=None, h_sf=None):
    """MXFP8 step 4: a = [a0 | a1] bf16 [R, 2F] -> (h codes [R, F], h E8M0 codes [F/128, R, 4])."""
    R, F2 = a.shape
    F = F2 // 2
    h_q = torch.empty(R, F, dtype=torch.uint8, device=a.device) if h_q is None else h_q
    h_sf = _scale_buf(MX32, R, F, a.device, h_sf)
    check(lib().moe_swiglu_quant_mx(_p(a), R, F, _p(h_q), _p(h_sf), _s()), "moe_swiglu_quant_mx")
    return h_q, h_sf


def gmm(lhs_q, lhs_scale, lhs_mode, rhs_q, rhs_scale, rhs_mode, group_sizes, group_offset: int = 0,
        E_local: Optional[int] = None, out=None):
    """Grouped matmul -> bf16 [M, N]."""
    M, K = lhs_q.shape
    El, N, K2 = rhs_q.shape
    if K2 != K:
        raise MoEError("lhs/rhs K mismatch")
    E = group_sizes.numel()
    E_local = El if E_local is None else E_local
    out = torch.empty(M, N, dtype=torch.bfloat16, device=lhs_q.device) if out is None else out
    check(lib().gmm_fp8(_p(lhs_q), _p(lhs_scale), lhs_mode, _p(rhs_q), _p(rhs_scale), rhs_mode, _p(group_sizes),
                        E, group_offset, E_local, M, K, N, _p(out), _s()), "gmm_fp8")
    return out


def gmm_w8(lhs_q, lhs_scale, lhs_mode, rhs_q, rhs_scale, rhs_mode, group_sizes, group_offset: int = 0,
           E_local: Optional[int] = None, out=None, workspace=None):
    """Grouped matmul with int8 weights rhs_q [E_local, N, K] -> bf16 [M, N].

    workspace: optional uint8 device buffer of gmm_w8_workspace_bytes(M, K)
    bytes or more; with it the activations are decoded to f16 there first
    (the same result, faster where the tensor pipe binds)."""
    M, K = lhs_q.shape
    El, N, K2 = rhs_q.shape
    if K2 != K:
        raise MoEError("lhs/rhs K mismatch")
    if rhs_q.dtype != torch.int8:
        raise MoEError("gmm_w8 takes int8 weight codes")
    E = group_sizes.numel()
    E_local = El if E_local is None else E_local
    out = torch.empty(M, N, dtype=torch.bfloat16, device=lhs_q.device) if out is None else out
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(lib().gmm_fp8_w8(_p(lhs_q), _p(lhs_scale), lhs_mode, _p(rhs_q), _p(rhs_scale), rhs_mode,
                           _p(group_sizes), E, group_offset, E_local, M, K, N, _p(out), _p(workspace), ws_bytes,
                           _s()), "gmm_fp8_w8")
    return out


def gmm_w8_workspace_bytes(M: int, K: int) -> int:
    return int(lib().gmm_fp8_w8_workspace_bytes(M, K))


def gmm_ksplit(lhs_q, lhs_scale, lhs_mode, rhs_q, rhs_scale2, K_split: int, group_sizes, group_offset: int = 0,
               E_local: Optional[int] = None, out=None):
    """Grouped matmul over two K segments with one static weight scale each
    (rhs_scale2 = [s0, s1]) -> bf16 [M, N]."""
    M, K = lhs_q.shape
    El, N, K2 = rhs_q.shape
    if K2 != K:
        raise MoEError("lhs/rhs K mismatch")
    E = group_sizes.numel()
    E_local = El if E_local is None else E_local
    out = torch.empty(M, N, dtype=torch.bfloat16, device=lhs_q.device) if out is None else out
    check(lib().gmm_fp8_ksplit(_p(lhs_q), _p(lhs_scale), lhs_mode, _p(rhs_q), _p(rhs_scale2), K_split,
                               _p(group_sizes), E, group_offset, E_local, M, K, N, _p(out), _s()), "gmm_fp8_ksplit")
    return out


def gmm_swiglu(lhs_q, lhs_scale, lhs_mode, rhs_q, rhs_scale, rhs_mode, group_sizes, h_mode: int,
               h_static: Optional[torch.Tensor] = None, group_offset: int = 0, E_local: Optional[int] = None,
               keep_a: bool = False, a_out=None, h=None, h_q=None, h_scale=None):
    """gmm with [wi_0 | wi_1] fused with SwiGLU and the requantisation of h.

    Returns (h_q uint8 [M, F], h_scale or None, a [M, 2F] bf16 or None)."""
    M, K = lhs_q.shape
    El, F2, K2 = rhs_q.shape
    if K2 != K:
        raise MoEError("lhs/rhs K mismatch")
    F = F2 // 2
    dev = lhs_q.device
    E = group_sizes.numel()
    E_local = El if E_local is None else E_local
    h_q = torch.empty(M, F, dtype=torch.uint8, device=dev) if h_q is None else h_q
    h_scale = _scale_buf(h_mode, M, F, dev, h_scale)
    if h_mode == PER_ROW and h is None:
        h = torch.empty(M, F, dtype=torch.bfloat16, device=dev)
    if keep_a and a_out is None:
        a_out = torch.empty(M, F2, dtype=torch.bfloat16, device=dev)
    check(lib().gmm_fp8_swiglu(_p(lhs_q), _p(lhs_scale), lhs_mode, _p(rhs_q), _p(rhs_scale), rhs_mode,
                               _p(group_sizes), E, group_offset, E_local, M, K, F, h_mode, _p(h_static), _p(a_out),
                               _p(h), _p(h_q), _p(h_scale), _s()), "gmm_fp8_swiglu")
    return h_q, h_scale, a_out


def swiglu_fusable(act_mode: int, w_mode: int, F: int) -> bool:
    """gmm_fp8_swiglu covers every operand scale mode (per row, per row and
    128 columns, per tensor) when F % 128 == 0."""
    modes = (PER_ROW, PER_ROW_BLOCK128, PER_TENSOR)
    return act_mode in modes and w_mode in modes and F % 128 == 0


def swiglu_fuse_pays(act_mode: int, w_mode: int, F: int) -> bool:
    """Whether the forward runs steps 3 and 4 as one gmm_fp8_swiglu call.

    With a blockwise operand scale the contraction's epilogue is already the
    bound (it folds every 128-wide K block into fp32 registers), and the
    SwiGLU tail cannot overlap the next tile there, so gmm_fp8 followed by
    moe_swiglu_quant is faster (measured on the DeepSeek-V3-shaped layer:
    5.1 + 0.5 ms against 6.5 ms); the two are bit-identical."""
    blockwise = act_mode == PER_ROW_BLOCK128 or w_mode == PER_ROW_BLOCK128
    return swiglu_fusable(act_mode, w_mode, F) and not blockwise


def swiglu_quant(a: torch.Tensor, mode: int, static_scale: Optional[torch.Tensor] = None, h_q=None, h_scale=None):
    R, F2 = a.shape
    F = F2 // 2
    h_q = torch.empty(R, F, dtype=torch.uint8, device=a.device) if h_q is None else h_q
    h_scale = _scale_buf(mode, R, F, a.device, h_scale)
    check(lib().moe_swiglu_quant(_p(a), R, F, mode, _p(static_scale), _p(h_q), _p(h_scale), _s()),
          "moe_swiglu_quant")
    return h_q, h_scale


def ragged_gather_reduce(rows: torch.Tensor, pos: torch.Tensor, weights: Optional[torch.Tensor], k: int,
                         out=None):
    R, D = rows.shape
    T = R // k
    out = torch.empty(T, D, dtype=torch.bfloat16, device=rows.device) if out is None else out
    check(lib().ragged_gather_reduce(_p(rows), _p(pos), _p(weights), T, k, D, _p(out), _s()),
          "ragged_gather_reduce")
    return out


def gather_scale_quant(G: torch.Tensor, w: Optional[torch.Tensor], sorted_src: torch.Tensor, k: int):
    T, D = G.shape
    R = T * k
    dev = G.device
    dO = torch.empty(R, D, dtype=torch.bfloat16, device=dev)
    dO_q = torch.empty(R, D, dtype=torch.uint8, device=dev)
    dO_s = torch.empty(R, dtype=torch.float32, device=dev)
    check(lib().moe_gather_scale_quant(_p(G), _p(w), _p(sorted_src), T, k, D, _p(dO), _p(dO_q), _p(dO_s), _s()),
          "moe_gather_scale_quant")
    return dO, dO_q, dO_s


def swiglu_bwd_quant(dH: torch.Tensor, a: torch.Tensor):
    R, F = dH.shape
    dev = dH.device
    dA = torch.empty(R, 2 * F, dtype=torch.bfloat16, device=dev)
    dA_q = torch.empty(R, 2 * F, dtype=torch.uint8, device=dev)
    dA_s = torch.empty(R, dtype=torch.float32, device=dev)
    check(lib().moe_swiglu_bwd_quant(_p(dH), _p(a), R, F, _p(dA), _p(dA_q), _p(dA_s), _s()), "moe_swiglu_bwd_quant")
    return dA, dA_q, dA_s


def quantize_group_cols(g: torch.Tensor, group_sizes: torch.Tensor, group_offset: int = 0,
                        E_local: Optional[int] = None, scales_only: bool = False):
    """Per-(expert, column) e4m3 codes and scales of g; (None, scales) with scales_only."""
    M, N = g.shape
    E = group_sizes.numel()
    E_local = E - group_offset if E_local is None else E_local
    # rows of other experts stay unwritten
    q = None if scales_only else torch.empty(M, N, dtype=torch.uint8, device=g.device)
    s = torch.empty(E_local, N, dtype=torch.float32, device=g.device)
    check(lib().moe_quantize_group_cols(_p(g), M, N, _p(group_sizes), E, group_offset, E_local, _p(q), _p(s), _s()),
          "moe_quantize_group_cols")
    return q, s


def tgmm(lhs_q, lhs_scale, lhs_mode, rhs_q, rhs_scale, rhs_mode, group_sizes, group_offset: int = 0,
         E_local: Optional[int] = None, out=None, workspace=None):
    """Transposed grouped matmul -> fp32 [E_local, K, N]."""
    M, K = lhs_q.shape
    M2, N = rhs_q.shape
    if M2 != M:
        raise MoEError("lhs/rhs M mismatch")
    E = group_sizes.numel()
    E_local = E - group_offset if E_local is None else E_local
    out = torch.empty(E_local, K, N, dtype=torch.float32, device=lhs_q.device) if out is None else out
    nws = lib().tgmm_fp8_workspace_bytes(M, K, N, E_local)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=lhs_q.device)
    check(lib().tgmm_fp8(_p(lhs_q), _p(lhs_scale), lhs_mode, _p(rhs_q), _p(rhs_scale), rhs_mode, _p(group_sizes), E,
                         group_offset, E_local, M, K, N, _p(out), _p(workspace), workspace.numel(), _s()), "tgmm_fp8")
    return out


def tgmm_gcq(lhs_q, lhs_scale, lhs_mode, rhs_g, rhs_scale, group_sizes, group_offset: int = 0,
             E_local: Optional[int] = None, out=None, workspace=None):
    """tgmm with the rhs as a bf16 gradient and its per-(expert, column) scales
    -> fp32 [E_local, K, N] (the codes are made in the contraction's layout)."""
    M, K = lhs_q.shape
    M2, N = rhs_g.shape
    if M2 != M:
        raise MoEError("lhs/rhs M mismatch")
    E = group_sizes.numel()
    E_local = E - group_offset if E_local is None else E_local
    out = torch.empty(E_local, K, N, dtype=torch.float32, device=lhs_q.device) if out is None else out
    nws = lib().tgmm_fp8_workspace_bytes(M, K, N, E_local)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(nws, dtype=torch.uint8, device=lhs_q.device)
    check(lib().tgmm_fp8_gcq(_p(lhs_q), _p(lhs_scale), lhs_mode, _p(rhs_g), _p(rhs_scale), _p(group_sizes), E,
                             group_offset, E_local, M, K, N, _p(out), _p(workspace), workspace.numel(), _s()),
          "tgmm_fp8_gcq")
    return out


def router_topk(x: torch.Tensor, w_gate: torch.Tensor, k: int):
    """Gate layer + softmax top-k: (logits fp32 [T, E], ids int32 [T, k], w fp32 [T, k])."""
    T, D = x.shape
    E = w_gate.shape[0]
    dev = x.device
    logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    check(lib().moe_router_topk(_p(x), _p(w_gate), T, D, E, k, _p(logits), _p(ids), _p(w), _s()), "moe_router_topk")
    return logits, ids, w


def router_backward(G: torch.Tensor, o: torch.Tensor, pos: torch.Tensor, x: torch.Tensor, w_gate: torch.Tensor,
                    logits: torch.Tensor, ids: torch.Tensor, workspace: Optional[torch.Tensor] = None):
    """Router gradient: (dw fp32 [T, k], dlogits bf16 [T, E], grad_gate fp32 [E, D], state_grad bf16 [T, D])."""
    T, D = x.shape
    E = w_gate.shape[0]
    k = ids.shape[1]
    dev = x.device
    dw = torch.empty(T, k, dtype=torch.float32, device=dev)
    dl = torch.empty(T, E, dtype=torch.bfloat16, device=dev)
    gg = torch.empty(E, D, dtype=torch.float32, device=dev)
    sg = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    nws = lib().moe_router_backward_workspace_bytes(T, D, E)
    if workspace is None or workspace.numel() < nws:
        workspace = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    check(lib().moe_router_backward(_p(G), _p(o), _p(pos), _p(x), _p(w_gate), _p(logits), _p(ids), T, D, E, k,
                                    _p(dw), _p(dl), _p(gg), _p(sg), _p(workspace), workspace.numel(), _s()),
          "moe_router_backward")
    return dw, dl, gg, sg


def transpose_u8(x: torch.Tensor) -> torch.Tensor:
    """Batched byte transpose [B, R, C] -> [B, C, R] (weight layout preparation)."""
    B, R, C = x.shape
    out = torch.empty(B, C, R, dtype=torch.uint8, device=x.device)
    check(lib().moe_transpose_u8(_p(x), B, R, C, _p(out), _s()), "moe_transpose_u8")
    return out


# ---------------------------------------------------------------------------
# The expert FFN
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class ExpertWeights:
    """Pre-quantised expert weights in the device layout.

    w_in  [E, 2F, D] codes (wi_0 rows, then wi_1 rows), scales per in_mode;
    w_out [E, D, F] codes, scales per out_mode.  For the backward pass the
    transposed codes w_in_t [E, D, 2F] and w_out_t [E, F, D] are kept too."""
    w_in: torch.Tensor
    s_in: torch.Tensor
    in_mode: int
    w_out: torch.Tensor
    s_out: torch.Tensor
    out_mode: int
    w_in_t: Optional[torch.Tensor] = None
    s_in_t: Optional[torch.Tensor] = None
    w_out_t: Optional[torch.Tensor] = None
    s_in_split: Optional[torch.Tensor] = None  # [s_w0, s_w1]: the two K halves of w_in_t


def prepare_weights(w_in: torch.Tensor, w_out: torch.Tensor, w_mode: int, static: Optional[dict] = None,
                    for_backward: bool = False) -> ExpertWeights:
    """Quantise the bf16 expert weights once (outside the timed FFN).

    Static scheme: wi_0, wi_1 and wo each carry one fixed scale; the wi_0 |
    wi_1 concatenation then has a per-channel scale vector."""
    dev = w_in.device
    E, F2, D = w_in.shape
    F = F2 // 2
    if w_mode == MX32:
        qin, sin = quantize_weights_mx(w_in)
        qo, so = quantize_weights_mx(w_out)
        return ExpertWeights(qin, sin, MX32, qo, so, MX32)
    if w_mode == PER_TENSOR:
        s0 = torch.tensor([static["w0"]], dtype=torch.float32, device=dev)
        s1 = torch.tensor([static["w1"]], dtype=torch.float32, device=dev)
        so = torch.tensor([static["wo"]], dtype=torch.float32, device=dev)
        q0, _ = quantize_weights(w_in[:, :F].contiguous(), PER_TENSOR, s0)
        q1, _ = quantize_weights(w_in[:, F:].contiguous(), PER_TENSOR, s1)
        qin = torch.cat([q0, q1], dim=1).contiguous()
        sin = torch.empty(E, F2, dtype=torch.float32, device=dev)
        sin[:, :F] = static["w0"]
        sin[:, F:] = static["w1"]
        qo, _ = quantize_weights(w_out, PER_TENSOR, so)
        W = ExpertWeights(qin, sin, PER_ROW, qo, so, PER_TENSOR)
        if for_backward:
            if F2 % 128 != 0 or F % 128 != 0:
                raise MoEError("the backward pass needs F % 128 == 0")
            W.w_in_t = transpose_u8(qin)
            nb = F2 // 128
            st = torch.empty(E, nb, D, dtype=torch.float32, device=dev)
            st[:, : F // 128] = static["w0"]
            st[:, F // 128:] = static["w1"]
            W.s_in_t = st
            W.s_in_split = torch.tensor([static["w0"], static["w1"]], dtype=torch.float32, device=dev)
            W.w_out_t = transpose_u8(qo)
        return W
    qin, sin = quantize_weights(w_in, w_mode)
    qo, so = quantize_weights(w_out, w_mode)
    return ExpertWeights(qin, sin, w_mode, qo, so, w_mode)


def prepare_weights_w8(w_in: torch.Tensor, w_out: torch.Tensor, w_mode: int) -> ExpertWeights:
    """int8 expert weights (per channel or blockwise), quantised once outside
    the timed FFN; ffn_forward then runs both contractions with gmm_w8."""
    if w_mode not in (PER_ROW, PER_ROW_BLOCK128):
        raise MoEError("int8 weights take per-channel or blockwise scales")
    qin, sin = quantize_weights_int8(w_in, w_mode)
    qo, so = quantize_weights_int8(w_out, w_mode)
    return ExpertWeights(qin, sin, w_mode, qo, so, w_mode)


class FFNBuffers:
    """Every intermediate of one forward (and backward) pass, allocated once."""

    def __init__(self, T, D, E, k, F, act_mode, device, backward=False):
        R = T * k
        f = lambda *s, dt=torch.uint8: torch.empty(*s, dtype=dt, device=device)
        self.T, self.D, self.E, self.k, self.F, self.act_mode = T, D, E, k, F, act_mode
        self.x_q = f(T, D)
        self.x_s = _scale_buf(act_mode, T, D, device)
        self.sort = {}
        self.a = f(R, 2 * F, dt=torch.bfloat16)
        self.h = f(R, F, dt=torch.bfloat16)  # scratch of the fused per-row path
        self.keep_a = backward
        self.h_q = f(R, F)
        self.h_s = _scale_buf(act_mode, R, F, device)
        self.o = f(R, D, dt=torch.bfloat16)
        self.y = f(T, D, dt=torch.bfloat16)
        self._w8_ws = None
        if backward:
            self.dH = f(R, F, dt=torch.bfloat16)
            self.dXs = f(R, D, dt=torch.bfloat16)
            self.dX = f(T, D, dt=torch.bfloat16)

    def w8_workspace(self) -> torch.Tensor:
        """The int8-weight contractions' f16 activation workspace, allocated on
        first use: 2 bytes per element of the larger of their two lhs,
        [T*k, D] and [T*k, F]."""
        if self._w8_ws is None:
            n = gmm_w8_workspace_bytes(self.T * self.k, max(self.D, self.F))
            self._w8_ws = torch.empty(n, dtype=torch.uint8, device=self.y.device)
        return self._w8_ws


def ffn_forward(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, W: ExpertWeights, act_mode: int,
                buf: FFNBuffers, static_x: Optional[torch.Tensor] = None,
                static_h: Optional[torch.Tensor] = None, fuse_swiglu: bool = True,
                fuse_quant_sort: bool = True) -> torch.Tensor:
    """One forward pass of the expert FFN; returns buf.y (bf16 [T, D]).

    Steps 1 and 2 run as one call (moe_quantize_sort; buf.x_q / buf.x_s are
    then not written), and where the scale modes allow it steps 3 and 4 run as
    one fused kernel (gmm_fp8_swiglu, bit-identical to gmm_fp8 +
    moe_swiglu_quant); buf.a then holds a only when the buffers were made for
    a backward pass."""
    E = W.w_in.shape[0]
    k = topk_ids.shape[1]
    if act_mode == MX32:
        if W.in_mode != MX32:
            raise MoEError("the MXFP8 forward needs MXFP8 weights")
        s = quantize_sort_mx(x, topk_ids, E, out=buf.sort)
        if fuse_swiglu and buf.F % 128 == 0:
            gmm_mx_swiglu(s["xs_q"], s["xs_scale"], W.w_in, W.s_in, s["group_sizes"],
                          a_out=buf.a if buf.keep_a else None, h_q=buf.h_q, h_sf=buf.h_s)
        else:
            gmm_mx(s["xs_q"], s["xs_scale"], W.w_in, W.s_in, s["group_sizes"], out=buf.a)
            swiglu_quant_mx(buf.a, h_q=buf.h_q, h_sf=buf.h_s)
        gmm_mx(buf.h_q, buf.h_s, W.w_out, W.s_out, s["group_sizes"], out=buf.o)
        ragged_gather_reduce(buf.o, s["pos"], topk_w, k, out=buf.y)
        return buf.y
    w8 = W.w_in.dtype == torch.int8
    if w8 and act_mode not in (PER_ROW, PER_TENSOR):
        raise MoEError("int8 weights take per-token or static activation scales")
    if fuse_quant_sort:
        s = quantize_sort(x, topk_ids, E, act_mode, static_x, out=buf.sort)
    else:
        quantize_rows(x, act_mode, static_x, q=buf.x_q, scale=buf.x_s)
        s = ragged_sort(topk_ids, E, buf.x_q, buf.x_s if act_mode != PER_TENSOR else static_x, act_mode,
                        out=buf.sort)
    xs_s = s["xs_scale"] if act_mode != PER_TENSOR else static_x
    if w8:
        ws = buf.w8_workspace()
        gmm_w8(s["xs_q"], xs_s, act_mode, W.w_in, W.s_in, W.in_mode, s["group_sizes"], out=buf.a, workspace=ws)
        swiglu_quant(buf.a, act_mode, static_h, h_q=buf.h_q, h_scale=buf.h_s)
    elif fuse_swiglu and swiglu_fuse_pays(act_mode, W.in_mode, buf.F):
        gmm_swiglu(s["xs_q"], xs_s, act_mode, W.w_in, W.s_in, W.in_mode, s["group_sizes"], act_mode, static_h,
                   a_out=buf.a if buf.keep_a else None, h=buf.h, h_q=buf.h_q, h_scale=buf.h_s)
    else:
        gmm(s["xs_q"], xs_s, act_mode, W.w_in, W.s_in, W.in_mode, s["group_sizes"], out=buf.a)
        swiglu_quant(buf.a, act_mode, static_h, h_q=buf.h_q, h_scale=buf.h_s)
    h_s = buf.h_s if act_mode != PER_TENSOR else static_h
    if w8:
        gmm_w8(buf.h_q, h_s, act_mode, W.w_out, W.s_out, W.out_mode, s["group_sizes"], out=buf.o, workspace=ws)
    else:
        gmm(buf.h_q, h_s, act_mode, W.w_out, W.s_out, W.out_mode, s["group_sizes"], out=buf.o)
    ragged_gather_reduce(buf.o, s["pos"], topk_w, k, out=buf.y)
    return buf.y


def ffn_backward(dY: torch.Tensor, topk_w: torch.Tensor, W: ExpertWeights, buf: FFNBuffers,
                 static_x: torch.Tensor, static_h: torch.Tensor, keep: Optional[dict] = None):
    """Backward pass of the static scheme after ffn_forward on `buf`.

    Returns (dX bf16 [T, D], dW_in fp32 [E, D, 2F], dW_out fp32 [E, F, D]):
    dW_in holds grad_wi_0 | grad_wi_1 and dW_out grad_wo, in the pages'
    [E, in, out] layouts.  With `keep` (a dict), the intermediate gradients
    (dO, dO_q, dO_s, dA, dA_q, dA_s, dAg_s, dOg_s) are stored in it."""
    s = buf.sort
    k = buf.k
    dO, dO_q, dO_s = gather_scale_quant(dY, topk_w, s["sorted_src"], k)
    gmm(dO_q, dO_s, PER_ROW, W.w_out_t, W.s_out, PER_TENSOR, s["group_sizes"], out=buf.dH)
    dA, dA_q, dA_s = swiglu_bwd_quant(buf.dH, buf.a)
    # dXs = dA0 W0^T + dA1 W1^T: one contraction over [dA0 | dA1], one static scale per K half
    gmm_ksplit(dA_q, dA_s, PER_ROW, W.w_in_t, W.s_in_split, buf.F, s["group_sizes"], out=buf.dXs)
    ragged_gather_reduce(buf.dXs, s["pos"], None, k, out=buf.dX)
    # per-(expert, column) gradient scales; their codes are made inside the weight-gradient contractions
    _, dAg_s = quantize_group_cols(dA, s["group_sizes"], scales_only=True)
    _, dOg_s = quantize_group_cols(dO, s["group_sizes"], scales_only=True)
    dW_in = tgmm_gcq(s["xs_q"], static_x, PER_TENSOR, dA, dAg_s, s["group_sizes"])
    dW_out = tgmm_gcq(buf.h_q, static_h, PER_TENSOR, dO, dOg_s, s["group_sizes"])
    if keep is not None:
        keep.update(dO=dO, dO_q=dO_q, dO_s=dO_s, dA=dA, dA_q=dA_q, dA_s=dA_s, dAg_s=dAg_s, dOg_s=dOg_s)
    return buf.dX, dW_in, dW_out
