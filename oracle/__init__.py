"""Oracle for the FP8-quantized MoE expert FFN (test infrastructure only).

A plain, slow, obviously correct CPU statement of what the expert-FFN path
computes, written in C (``moe_oracle.c``, fp64 accumulation) with thin numpy
wrappers here.  Only the tests, the package smoke check and the benchmark's
CPU-baseline leg may import it; the product path never does.  It shares no
code with the CUDA path.

Every function cites the page passage it follows (see the C file's header for
the three MaxText pull-request pages: "Quantize activations before EP all
gather", "Support quantization for tokamax gmm v2" and "Keep qwix out of
tpu-inference's fused MoE kernel and pre-quantize weights").

Parity status: every function below is pinned by the CPU tests in
``tests/test_oracle_*.py`` (closed forms, invariants, brute force, adjoint
and finite-difference identities) except the end-to-end accuracy against a
bf16 dense layer, which is parity unpinned: the pages print no worked
example, only error figures of unknown shapes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PER_ROW = 0
PER_ROW_BLOCK128 = 1
PER_TENSOR = 2
PER_GROUP_COL = 3
MX32 = 4  # MXFP8 variant: E8M0 codes (uint8), one per 32 values along the contracted dimension

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmoe_oracle.so")
_SRC = os.path.join(_HERE, "moe_oracle.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-frounding-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            sig = {
                "or_bf16_to_f64": ([ctypes.c_uint16], ctypes.c_double),
                "or_f64_to_bf16": ([ctypes.c_double], ctypes.c_uint16),
                "or_e4m3_to_f64": ([ctypes.c_uint8], ctypes.c_double),
                "or_f32_to_e4m3": ([f32], ctypes.c_uint8),
                "or_exp_f32": ([f32], f32),
                "or_silu_f32": ([f32], f32),
                "or_quantize_rows": ([P, i64, i64, i32, f32, P, P], None),
                "or_quantize_weights": ([P, i64, i64, i64, i32, f32, P, P], None),
                "or_ragged_sort": ([P, i64, i32, i32, P, P, P, P], i32),
                "or_gather_rows": ([P, P, i32, i64, P, i64, i32, P, P], None),
                "or_gmm": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, P, i64, P, P], None),
                "or_gmm_f64": ([P, P, P, i32, i32, i32, i64, i64, i64, P], None),
                "or_swiglu_quant": ([P, i64, i64, i32, f32, P, P, P], None),
                "or_combine": ([P, P, P, i64, i32, i64, P, i64, P, P], None),
                "or_combine_f64": ([P, P, P, i64, i32, i64, P], None),
                "or_gather_scale": ([P, P, P, i64, i32, i64, P], None),
                "or_gather_scale_f64": ([P, P, P, i64, i32, i64, P], None),
                "or_swiglu_bwd": ([P, P, i64, i64, P], None),
                "or_swiglu_f64": ([P, i64, i64, P], None),
                "or_swiglu_bwd_f64": ([P, P, i64, i64, P], None),
                "or_quantize_group_cols": ([P, P, i32, i32, i32, i64, i64, P, P], None),
                "or_tgmm": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, P, i64, P, P], None),
                "or_tgmm_f64": ([P, P, P, i32, i32, i32, i64, i64, i64, P], None),
                "or_router_logits": ([P, P, i64, i64, i64, P], None),
                "or_router_topk": ([P, i64, i64, i32, P, P, P], None),
                "or_router_dw": ([P, P, P, i64, i32, i64, P], None),
                "or_router_dlogits": ([P, P, P, i64, i64, i32, P], None),
                "or_router_grads": ([P, P, P, i64, i64, i64, P, P], None),
                "or_quantize_rows_mx": ([P, i64, i64, P, P], None),
                "or_gmm_mx": ([P, P, P, P, P, i32, i32, i32, i64, i64, i64, P, i64, P, P], None),
                "or_swiglu_quant_mx": ([P, i64, i64, P, P, P], None),
                "or_quantize_weights_int8": ([P, i64, i64, i64, i32, f32, P, P], None),
                "or_gmm_w8": ([P, P, i32, P, P, i32, P, i32, i32, i32, i64, i64, i64, P, i64, P, P], None),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def bf16_bits(t) -> np.ndarray:
    """uint16 view of a bf16 torch tensor (or pass through a uint16 array)."""
    if isinstance(t, np.ndarray):
        return _c(t, np.uint16)
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns."""
    u = (_c(bits, np.uint16).astype(np.uint32) << 16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    L = lib()
    flat = np.asarray(v, dtype=np.float64).ravel()
    return np.array([L.or_f64_to_bf16(float(x)) for x in flat], dtype=np.uint16).reshape(np.shape(v))


_E4M3_TABLE = None


def e4m3_table() -> np.ndarray:
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        L = lib()
        _E4M3_TABLE = np.array([L.or_e4m3_to_f64(c) for c in range(256)], dtype=np.float64)
    return _E4M3_TABLE


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    return e4m3_table()[_c(codes, np.uint8)]


def f32_to_e4m3(v) -> int:
    return int(lib().or_f32_to_e4m3(float(np.float32(v))))


def exp_f32(x) -> float:
    return float(np.float32(lib().or_exp_f32(float(np.float32(x)))))


def silu_f32(x) -> float:
    return float(np.float32(lib().or_silu_f32(float(np.float32(x)))))


# --------------------------------------------------------------------------
# Path steps
# --------------------------------------------------------------------------

def nblocks(cols: int) -> int:
    return (cols + 127) // 128


def quantize_rows(x_bits, mode: int, static_scale: float = 1.0):
    """bf16 [rows, cols] -> (codes uint8 [rows, cols], scales float32)."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    if mode == PER_ROW:
        s = np.empty(rows, np.float32)
    elif mode == PER_ROW_BLOCK128:
        s = np.empty((rows, nblocks(cols)), np.float32)
    else:
        s = np.array([static_scale], np.float32)
    lib().or_quantize_rows(_p(x), rows, cols, mode, float(static_scale), _p(q),
                           _p(s) if mode != PER_TENSOR else None)
    return q, s


def quantize_weights(w_bits, mode: int, static_scale: float = 1.0):
    """bf16 [E, N, K] -> (codes [E, N, K], scales [E, N] | [E, K/128, N] | [1])."""
    w = _c(w_bits, np.uint16)
    E, N, K = w.shape
    q = np.empty((E, N, K), np.uint8)
    if mode == PER_ROW:
        s = np.empty((E, N), np.float32)
    elif mode == PER_ROW_BLOCK128:
        s = np.empty((E, nblocks(K), N), np.float32)
    else:
        s = np.array([static_scale], np.float32)
    lib().or_quantize_weights(_p(w), E, N, K, mode, float(static_scale), _p(q),
                              _p(s) if mode != PER_TENSOR else None)
    return q, s


def quantize_weights_int8(w_bits, mode: int, static_scale: float = 1.0):
    """int8 expert weights ("Keep qwix out of tpu-inference's fused MoE kernel
    and pre-quantize weights": float8_e4m3fn or int8 weights with [E, blocks,
    1, N] scales): bf16 [E, N, K] -> (int8 codes [E, N, K], scales [E, N] |
    [E, K/128, N] | [1]).  s = fp32(amax / 127), q = rint(fp32(x / s))."""
    w = _c(w_bits, np.uint16)
    E, N, K = w.shape
    q = np.empty((E, N, K), np.int8)
    if mode == PER_ROW:
        s = np.empty((E, N), np.float32)
    elif mode == PER_ROW_BLOCK128:
        s = np.empty((E, nblocks(K), N), np.float32)
    else:
        s = np.array([static_scale], np.float32)
    lib().or_quantize_weights_int8(_p(w), E, N, K, mode, float(static_scale), _p(q),
                                   _p(s) if mode != PER_TENSOR else None)
    return q, s


def quantize_rows_mx(x_bits):
    """MXFP8 (OCP MX v1.0): bf16 [rows, cols], cols a multiple of 32 ->
    (codes uint8 [rows, cols], E8M0 codes uint8 [rows, cols/32])."""
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    assert cols % 32 == 0
    q = np.empty((rows, cols), np.uint8)
    sf = np.empty((rows, cols // 32), np.uint8)
    lib().or_quantize_rows_mx(_p(x), rows, cols, _p(q), _p(sf))
    return q, sf


def quantize_weights_mx(w_bits):
    """MXFP8 weights: bf16 [E, N, K] -> (codes [E, N, K], E8M0 codes [E, N, K/32])."""
    w = _c(w_bits, np.uint16)
    E, N, K = w.shape
    q, sf = quantize_rows_mx(w.reshape(E * N, K))
    return q.reshape(E, N, K), sf.reshape(E, N, K // 32)


def ragged_sort(topk_ids: np.ndarray, E: int):
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    R = T * k
    sorted_src = np.empty(R, np.int32)
    pos = np.empty(R, np.int32)
    sizes = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    rc = lib().or_ragged_sort(_p(ids), T, k, E, _p(sorted_src), _p(pos), _p(sizes), _p(offsets))
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    return sorted_src, pos, sizes, offsets


def gather_rows(x_q, x_scale, mode: int, sorted_src, k: int):
    x_q = _c(x_q, np.uint8)
    T, D = x_q.shape
    R = len(sorted_src)
    xs = np.empty((R, D), np.uint8)
    if mode == PER_ROW:
        xss = np.empty(R, np.float32)
    elif mode == PER_ROW_BLOCK128:
        xss = np.empty((R, nblocks(D)), np.float32)
    else:
        xss = np.array(x_scale, np.float32).reshape(-1)[:1].copy()
    src = _c(sorted_src, np.int32)
    lib().or_gather_rows(_p(x_q), _p(_c(x_scale, np.float32)), mode, D, _p(src), R, k, _p(xs),
                         _p(xss) if mode != PER_TENSOR else None)
    return xs, xss


def gmm(lhs, lhs_scale, lhs_mode, rhs, rhs_scale, rhs_mode, group_sizes, group_offset=0, E_local=None,
        rows=None, want="bf16"):
    """Grouped matmul; returns bf16 bits [rows, N] (want='bf16') or float64."""
    lhs = _c(lhs, np.uint8)
    rhs = _c(rhs, np.uint8)
    M, K = lhs.shape
    El, N, K2 = rhs.shape
    assert K2 == K
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    assert El == E_local
    r = None if rows is None else _c(rows, np.int64)
    nrows = M if r is None else len(r)
    ob = np.empty((nrows, N), np.uint16) if want == "bf16" else None
    of = np.empty((nrows, N), np.float64) if want != "bf16" else None
    lib().or_gmm(_p(lhs), _p(_c(lhs_scale, np.float32)), lhs_mode, _p(rhs), _p(_c(rhs_scale, np.float32)),
                 rhs_mode, _p(sizes), E, group_offset, E_local, M, K, N, _p(r), nrows, _p(ob), _p(of))
    return ob if want == "bf16" else of


def gmm_w8(lhs, lhs_scale, lhs_mode, rhs, rhs_scale, rhs_mode, group_sizes, group_offset=0, E_local=None,
           rows=None, want="bf16"):
    """Grouped matmul with int8 weights rhs [E_local, N, K] (each code the
    integer it holds); otherwise as gmm."""
    lhs = _c(lhs, np.uint8)
    rhs = _c(rhs, np.int8)
    M, K = lhs.shape
    El, N, K2 = rhs.shape
    assert K2 == K
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    assert El == E_local
    r = None if rows is None else _c(rows, np.int64)
    nrows = M if r is None else len(r)
    ob = np.empty((nrows, N), np.uint16) if want == "bf16" else None
    of = np.empty((nrows, N), np.float64) if want != "bf16" else None
    lib().or_gmm_w8(_p(lhs), _p(_c(lhs_scale, np.float32)), lhs_mode, _p(rhs), _p(_c(rhs_scale, np.float32)),
                    rhs_mode, _p(sizes), E, group_offset, E_local, M, K, N, _p(r), nrows, _p(ob), _p(of))
    return ob if want == "bf16" else of


def gather_rows_mx(x_q, x_sf, sorted_src, k: int):
    """MXFP8 rows follow their token: sorted row r takes token sorted_src[r] // k's
    codes and its E8M0 codes (the scales are per token and block, so they are
    gathered with the rows)."""
    t = _c(sorted_src, np.int64) // k
    return _c(x_q, np.uint8)[t], _c(x_sf, np.uint8)[t]


def gmm_mx(lhs, lhs_sf, rhs, rhs_sf, group_sizes, group_offset=0, E_local=None, rows=None, want="bf16"):
    """MXFP8 grouped matmul: lhs [M, K] with E8M0 codes [M, K/32], rhs
    [E_local, N, K] with [E_local, N, K/32]; bf16 bits or float64 out."""
    lhs = _c(lhs, np.uint8)
    rhs = _c(rhs, np.uint8)
    M, K = lhs.shape
    El, N, K2 = rhs.shape
    assert K2 == K and K % 32 == 0
    lsf = _c(lhs_sf, np.uint8)
    rsf = _c(rhs_sf, np.uint8)
    assert lsf.shape == (M, K // 32) and rsf.shape == (El, N, K // 32)
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    assert El == E_local
    r = None if rows is None else _c(rows, np.int64)
    nrows = M if r is None else len(r)
    ob = np.empty((nrows, N), np.uint16) if want == "bf16" else None
    of = np.empty((nrows, N), np.float64) if want != "bf16" else None
    lib().or_gmm_mx(_p(lhs), _p(lsf), _p(rhs), _p(rsf), _p(sizes), E, group_offset, E_local, M, K, N, _p(r), nrows,
                    _p(ob), _p(of))
    return ob if want == "bf16" else of


def gmm_f64(lhs, rhs, group_sizes, group_offset=0, E_local=None):
    lhs = _c(lhs, np.float64)
    rhs = _c(rhs, np.float64)
    M, K = lhs.shape
    El, N, _ = rhs.shape
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    out = np.empty((M, N), np.float64)
    lib().or_gmm_f64(_p(lhs), _p(rhs), _p(sizes), E, group_offset, E_local, M, K, N, _p(out))
    return out


def swiglu_quant(a_bits, mode: int, static_scale: float = 1.0):
    """a = [a0 | a1] bf16 [R, 2F] -> (h codes [R, F], h scales, h bf16 bits)."""
    a = _c(a_bits, np.uint16)
    R, F2 = a.shape
    F = F2 // 2
    hq = np.empty((R, F), np.uint8)
    hb = np.empty((R, F), np.uint16)
    if mode == PER_ROW:
        hs = np.empty(R, np.float32)
    elif mode == PER_ROW_BLOCK128:
        hs = np.empty((R, nblocks(F)), np.float32)
    else:
        hs = np.array([static_scale], np.float32)
    lib().or_swiglu_quant(_p(a), R, F, mode, float(static_scale), _p(hq),
                          _p(hs) if mode != PER_TENSOR else None, _p(hb))
    return hq, hs, hb


def swiglu_quant_mx(a_bits):
    """a = [a0 | a1] bf16 [R, 2F] -> (h codes [R, F], h E8M0 codes [R, F/32], h bf16 bits)."""
    a = _c(a_bits, np.uint16)
    R, F2 = a.shape
    F = F2 // 2
    assert F % 32 == 0
    hq = np.empty((R, F), np.uint8)
    hsf = np.empty((R, F // 32), np.uint8)
    hb = np.empty((R, F), np.uint16)
    lib().or_swiglu_quant_mx(_p(a), R, F, _p(hq), _p(hsf), _p(hb))
    return hq, hsf, hb


def combine(o_bits, pos, w, k: int, tokens=None, want="bf16"):
    o = _c(o_bits, np.uint16)
    R, D = o.shape
    T = R // k
    t = None if tokens is None else _c(tokens, np.int64)
    n = T if t is None else len(t)
    yb = np.empty((n, D), np.uint16) if want == "bf16" else None
    yf = np.empty((n, D), np.float64) if want != "bf16" else None
    wp = None if w is None else _c(w, np.float32)
    lib().or_combine(_p(o), _p(_c(pos, np.int32)), _p(wp), T, k, D, _p(t), n, _p(yb), _p(yf))
    return yb if want == "bf16" else yf


def combine_f64(o, pos, w, k: int):
    o = _c(o, np.float64)
    R, D = o.shape
    T = R // k
    y = np.empty((T, D), np.float64)
    wp = None if w is None else _c(w, np.float32)
    lib().or_combine_f64(_p(o), _p(_c(pos, np.int32)), _p(wp), T, k, D, _p(y))
    return y


def gather_scale(G_bits, w, sorted_src, k: int):
    G = _c(G_bits, np.uint16)
    T, D = G.shape
    R = len(sorted_src)
    dO = np.empty((R, D), np.uint16)
    wp = None if w is None else _c(w, np.float32)
    lib().or_gather_scale(_p(G), _p(wp), _p(_c(sorted_src, np.int32)), R, k, D, _p(dO))
    return dO


def gather_scale_f64(G, w, sorted_src, k: int):
    G = _c(G, np.float64)
    T, D = G.shape
    R = len(sorted_src)
    dO = np.empty((R, D), np.float64)
    wp = None if w is None else _c(w, np.float32)
    lib().or_gather_scale_f64(_p(G), _p(wp), _p(_c(sorted_src, np.int32)), R, k, D, _p(dO))
    return dO


def swiglu_bwd(dH_bits, a_bits):
    dH = _c(dH_bits, np.uint16)
    a = _c(a_bits, np.uint16)
    R, F = dH.shape
    dA = np.empty((R, 2 * F), np.uint16)
    lib().or_swiglu_bwd(_p(dH), _p(a), R, F, _p(dA))
    return dA


def swiglu_f64(a):
    a = _c(a, np.float64)
    R, F2 = a.shape
    h = np.empty((R, F2 // 2), np.float64)
    lib().or_swiglu_f64(_p(a), R, F2 // 2, _p(h))
    return h


def swiglu_bwd_f64(dH, a):
    dH = _c(dH, np.float64)
    a = _c(a, np.float64)
    R, F = dH.shape
    dA = np.empty((R, 2 * F), np.float64)
    lib().or_swiglu_bwd_f64(_p(dH), _p(a), R, F, _p(dA))
    return dA


def quantize_group_cols(g_bits, group_sizes, group_offset=0, E_local=None):
    g = _c(g_bits, np.uint16)
    M, N = g.shape
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    q = np.zeros((M, N), np.uint8)
    s = np.empty((E_local, N), np.float32)
    lib().or_quantize_group_cols(_p(g), _p(sizes), E, group_offset, E_local, M, N, _p(q), _p(s))
    return q, s


def tgmm(lhs, lhs_scale, lhs_mode, rhs, rhs_scale, rhs_mode, group_sizes, group_offset=0, E_local=None,
         samples=None, want="f32"):
    lhs = _c(lhs, np.uint8)
    rhs = _c(rhs, np.uint8)
    M, K = lhs.shape
    M2, N = rhs.shape
    assert M == M2
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    s = None if samples is None else _c(samples, np.int64)
    n = E_local * K * N if s is None else len(s)
    of = np.empty(n, np.float32) if want == "f32" else None
    od = np.empty(n, np.float64) if want != "f32" else None
    lib().or_tgmm(_p(lhs), _p(_c(lhs_scale, np.float32)), lhs_mode, _p(rhs), _p(_c(rhs_scale, np.float32)),
                  rhs_mode, _p(sizes), E, group_offset, E_local, M, K, N, _p(s), n, _p(of), _p(od))
    out = of if want == "f32" else od
    return out.reshape(E_local, K, N) if s is None else out


def tgmm_f64(lhs, rhs, group_sizes, group_offset=0, E_local=None):
    lhs = _c(lhs, np.float64)
    rhs = _c(rhs, np.float64)
    M, K = lhs.shape
    _, N = rhs.shape
    sizes = _c(group_sizes, np.int32)
    E = len(sizes)
    if E_local is None:
        E_local = E - group_offset
    out = np.empty((E_local, K, N), np.float64)
    lib().or_tgmm_f64(_p(lhs), _p(rhs), _p(sizes), E, group_offset, E_local, M, K, N, _p(out))
    return out


# --------------------------------------------------------------------------
# The whole expert FFN (forward S1..S6 and backward), composed in the pages'
# order: quantise -> sort/gather -> gmm(wi_0|wi_1) -> SwiGLU + requantise ->
# gmm(wo) -> gather-reduce.
# --------------------------------------------------------------------------

def prepare_weights(w_in_bits, w_out_bits, w_mode, static=None):
    """Quantise expert weights (outside the timed FFN: pre-quantised weights).

    w_in [E, 2F, D] (wi_0 rows then wi_1 rows), w_out [E, D, F].  For the
    static scheme each of wi_0, wi_1 and wo has one fixed scale; the wi_0 |
    wi_1 concatenation then carries a per-channel scale vector."""
    if w_mode == PER_TENSOR:
        E, F2, D = w_in_bits.shape
        F = F2 // 2
        q0, _ = quantize_weights(w_in_bits[:, :F], PER_TENSOR, static["w0"])
        q1, _ = quantize_weights(w_in_bits[:, F:], PER_TENSOR, static["w1"])
        qin = np.concatenate([q0, q1], axis=1)
        sin = np.empty((E, F2), np.float32)
        sin[:, :F] = np.float32(static["w0"])
        sin[:, F:] = np.float32(static["w1"])
        qo, so = quantize_weights(w_out_bits, PER_TENSOR, static["wo"])
        return qin, sin, PER_ROW, qo, so, PER_TENSOR
    qin, sin = quantize_weights(w_in_bits, w_mode)
    qo, so = quantize_weights(w_out_bits, w_mode)
    return qin, sin, w_mode, qo, so, w_mode


def prepare_weights_w8(w_in_bits, w_out_bits, w_mode):
    """int8 expert weights (per channel or blockwise), in prepare_weights' tuple."""
    qin, sin = quantize_weights_int8(w_in_bits, w_mode)
    qo, so = quantize_weights_int8(w_out_bits, w_mode)
    return qin, sin, w_mode, qo, so, w_mode


def ffn_forward(x_bits, topk_ids, topk_w, wq, E: int, act_mode: int, static=None, tokens=None):
    """Forward pass; returns a dict of every stage's outputs.

    wq = prepare_weights(...) or prepare_weights_w8(...) (int8 weight codes:
    both contractions then take gmm_w8).  With `tokens`, the
    gmm/SwiGLU/combine stages are evaluated only on the rows those tokens
    route to (y[t] depends only on x[t]), and the per-row stage outputs are
    returned for those rows."""
    qin, sin, min_, qo, so, mo = wq
    mm = gmm_w8 if np.asarray(qin).dtype == np.int8 else gmm
    T, D = x_bits.shape
    k = topk_ids.shape[1]
    sx = static["x"] if act_mode == PER_TENSOR else 1.0
    x_q, x_s = quantize_rows(x_bits, act_mode, sx)
    sorted_src, pos, sizes, offsets = ragged_sort(topk_ids, E)
    xs_q, xs_s = gather_rows(x_q, x_s, act_mode, sorted_src, k)
    rows = None
    if tokens is not None:
        tokens = np.asarray(tokens, np.int64)
        rows = np.sort(pos.reshape(T, k)[tokens].reshape(-1)).astype(np.int64)
    a = mm(xs_q, xs_s, act_mode, qin, sin, min_, sizes, rows=rows)
    sh = static["h"] if act_mode == PER_TENSOR else 1.0
    h_q, h_s, h_b = swiglu_quant(a, act_mode, sh)
    if rows is None:
        o = mm(h_q, h_s, act_mode, qo, so, mo, sizes)
        y = combine(o, pos, topk_w, k)
    else:
        # place the computed rows in a full-size o (other rows unused)
        R = T * k
        hq_full = np.zeros((R, h_q.shape[1]), np.uint8)
        hq_full[rows] = h_q
        hs_full = h_s
        if act_mode == PER_ROW:
            hs_full = np.ones(R, np.float32)
            hs_full[rows] = h_s
        elif act_mode == PER_ROW_BLOCK128:
            hs_full = np.ones((R, h_s.shape[1]), np.float32)
            hs_full[rows] = h_s
        o_rows = mm(hq_full, hs_full, act_mode, qo, so, mo, sizes, rows=rows)
        o = np.zeros((R, D), np.uint16)
        o[rows] = o_rows
        y = combine(o, pos, topk_w, k, tokens=tokens)
        o = o_rows
    return dict(x_q=x_q, x_s=x_s, sorted_src=sorted_src, pos=pos, sizes=sizes, offsets=offsets,
                xs_q=xs_q, xs_s=xs_s, rows=rows, a=a, h_q=h_q, h_s=h_s, h_b=h_b, o=o, y=y)


def prepare_weights_mx(w_in_bits, w_out_bits):
    """MXFP8 expert weights: (w_in codes, w_in E8M0 codes, w_out codes, w_out E8M0 codes)."""
    qin, sin = quantize_weights_mx(w_in_bits)
    qo, so = quantize_weights_mx(w_out_bits)
    return qin, sin, qo, so


def ffn_forward_mx(x_bits, topk_ids, topk_w, wq, E: int, tokens=None):
    """The forward pass in the pages' order on MXFP8 operands: quantise ->
    sort/gather -> gmm(wi_0|wi_1) -> SwiGLU + MX requantise -> gmm(wo) ->
    gather-reduce.  wq = prepare_weights_mx(...); `tokens` as in ffn_forward."""
    qin, sin, qo, so = wq
    T, D = x_bits.shape
    k = topk_ids.shape[1]
    x_q, x_sf = quantize_rows_mx(x_bits)
    sorted_src, pos, sizes, offsets = ragged_sort(topk_ids, E)
    xs_q, xs_sf = gather_rows_mx(x_q, x_sf, sorted_src, k)
    rows = None
    if tokens is not None:
        tokens = np.asarray(tokens, np.int64)
        rows = np.sort(pos.reshape(T, k)[tokens].reshape(-1)).astype(np.int64)
    a = gmm_mx(xs_q, xs_sf, qin, sin, sizes, rows=rows)
    h_q, h_sf, h_b = swiglu_quant_mx(a)
    if rows is None:
        o = gmm_mx(h_q, h_sf, qo, so, sizes)
        y = combine(o, pos, topk_w, k)
    else:
        R = T * k
        hq_full = np.zeros((R, h_q.shape[1]), np.uint8)
        hq_full[rows] = h_q
        hsf_full = np.full((R, h_sf.shape[1]), 127, np.uint8)
        hsf_full[rows] = h_sf
        o_rows = gmm_mx(hq_full, hsf_full, qo, so, sizes, rows=rows)
        o = np.zeros((R, D), np.uint16)
        o[rows] = o_rows
        y = combine(o, pos, topk_w, k, tokens=tokens)
        o = o_rows
    return dict(x_q=x_q, x_sf=x_sf, sorted_src=sorted_src, pos=pos, sizes=sizes, offsets=offsets,
                xs_q=xs_q, xs_sf=xs_sf, rows=rows, a=a, h_q=h_q, h_sf=h_sf, h_b=h_b, o=o, y=y)


def ffn_backward(fwd: dict, G_bits, topk_w, wq, k: int, static: dict):
    """Backward pass of the static scheme (fp8_static_wa: fixed weight and
    activation scales, absmax-quantised gradients).

    Returns dX [T, D] bf16, dW_in [E, D, 2F] fp32 (grad of wi_0 | wi_1 in the
    pages' [E, D, F] layout) and dW_out [E, F, D] fp32 (grad of wo)."""
    qin, sin, _, qo, so, _ = wq
    sizes = fwd["sizes"]
    sorted_src, pos = fwd["sorted_src"], fwd["pos"]
    # dO = w * G[src], bf16; quantised per row for the dH gmm
    dO = gather_scale(G_bits, topk_w, sorted_src, k)
    dO_q, dO_s = quantize_rows(dO, PER_ROW)
    # dH = dO @ wo  (rhs = wo transposed to [E, F, D], K = D contracted)
    qoT = np.ascontiguousarray(np.transpose(qo, (0, 2, 1)))
    dH = gmm(dO_q, dO_s, PER_ROW, qoT, so, PER_TENSOR, sizes)
    dA = swiglu_bwd(dH, fwd["a"])
    dA_q, dA_s = quantize_rows(dA, PER_ROW)
    # dXs = dA0 @ wi_0 + dA1 @ wi_1 = [dA0 | dA1] @ w_in  (K = 2F contracted);
    # w_in^T is [E, D, 2F] with scale w0 on the first F columns of K and w1 on
    # the rest, i.e. a blockwise scale [E, 2F/128, D].
    E, F2, D = qin.shape
    qinT = np.ascontiguousarray(np.transpose(qin, (0, 2, 1)))
    sinT = np.empty((E, nblocks(F2), D), np.float32)
    blk = (np.arange(nblocks(F2)) * 128) < (F2 // 2)
    sinT[:, blk, :] = np.float32(static["w0"])
    sinT[:, ~blk, :] = np.float32(static["w1"])
    dXs = gmm(dA_q, dA_s, PER_ROW, qinT, sinT, PER_ROW_BLOCK128, sizes)
    dX = combine(dXs, pos, None, k)
    # weight gradients: per-(expert, column) requantised gradients
    dAg_q, dAg_s = quantize_group_cols(dA, sizes)
    dOg_q, dOg_s = quantize_group_cols(dO, sizes)
    dW_in = tgmm(fwd["xs_q"], np.array([static["x"]], np.float32), PER_TENSOR, dAg_q, dAg_s, PER_GROUP_COL, sizes)
    dW_out = tgmm(fwd["h_q"], np.array([static["h"]], np.float32), PER_TENSOR, dOg_q, dOg_s, PER_GROUP_COL,
                  sizes)
    return dict(dO=dO, dO_q=dO_q, dO_s=dO_s, dH=dH, dA=dA, dA_q=dA_q, dA_s=dA_s, dXs=dXs, dX=dX,
                dAg_q=dAg_q, dAg_s=dAg_s, dOg_q=dOg_q, dOg_s=dOg_s, dW_in=dW_in, dW_out=dW_out)


# --------------------------------------------------------------------------
# Router: the gate layer, softmax top-k routing and their gradients
# ("Support quantization for tokamax gmm v2", table 1: grad_gate-kernel and
# state_grad).  W_gate is [E, D] (one row per expert).
# --------------------------------------------------------------------------

def router_logits(x_bits, wg_bits):
    """bf16 x [T, D], bf16 W_gate [E, D] -> float64 logits [T, E]."""
    x = _c(x_bits, np.uint16)
    wg = _c(wg_bits, np.uint16)
    T, D = x.shape
    E = wg.shape[0]
    out = np.empty((T, E), np.float64)
    lib().or_router_logits(_p(x), _p(wg), T, D, E, _p(out))
    return out


def router_topk(logits_f32, k: int, want_p: bool = False):
    """fp32 logits [T, E] -> (ids int32 [T, k], w float32 [T, k][, p [T, E]])."""
    l = _c(logits_f32, np.float32)
    T, E = l.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    p = np.empty((T, E), np.float32) if want_p else None
    lib().or_router_topk(_p(l), T, E, k, _p(ids), _p(w), _p(p))
    return (ids, w, p) if want_p else (ids, w)


def router_dw(G_bits, o_bits, pos, k: int):
    """dL/dw [T, k] (float64) of the combine: <G[t], o[pos[t k + j]]>."""
    G = _c(G_bits, np.uint16)
    o = _c(o_bits, np.uint16)
    T, D = G.shape
    dw = np.empty((T, k), np.float64)
    lib().or_router_dw(_p(G), _p(o), _p(_c(pos, np.int32)), T, k, D, _p(dw))
    return dw


def router_dlogits(logits_f32, ids, dw_f32):
    """Softmax backward through the selected probabilities -> bf16 bits [T, E]."""
    l = _c(logits_f32, np.float32)
    T, E = l.shape
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    out = np.empty((T, E), np.uint16)
    lib().or_router_dlogits(_p(l), _p(ids), _p(_c(dw_f32, np.float32)), T, E, k, _p(out))
    return out


def router_grads(x_bits, wg_bits, dlogits_bits):
    """(grad_gate [E, D], state_grad [T, D]) in float64 from bf16 dlogits."""
    x = _c(x_bits, np.uint16)
    wg = _c(wg_bits, np.uint16)
    dl = _c(dlogits_bits, np.uint16)
    T, D = x.shape
    E = wg.shape[0]
    gg = np.empty((E, D), np.float64)
    sg = np.empty((T, D), np.float64)
    lib().or_router_grads(_p(x), _p(wg), _p(dl), T, D, E, _p(gg), _p(sg))
    return gg, sg
