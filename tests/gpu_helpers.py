"""Helpers shared by the GPU parity tests: device transfers and the
tolerance check for floating-point outputs.

Tolerance (from the statement of the path): after rounding both sides to
bf16, relative Frobenius error <= 2e-3 and elementwise |delta| <= 1e-2 *
max|ref|.  Integer, byte and index outputs must match bit for bit."""

import numpy as np
import torch

import oracle

REL_FRO = 2e-3
REL_ELT = 1e-2


def dev(a, dtype=None):
    """numpy (or torch CPU) -> CUDA tensor."""
    if isinstance(a, np.ndarray):
        if a.dtype == np.uint16:
            t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a))
    else:
        t = a
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_f64(a: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def bf16_round_f64(a: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 values (as float64), for fp32 outputs."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def close_errors(got, ref):
    """(relative Frobenius error, max |delta| / max |ref|) after bf16 rounding."""
    g = to_f64(got) if got.dtype == np.uint16 else bf16_round_f64(got)
    r = to_f64(ref) if ref.dtype == np.uint16 else bf16_round_f64(ref)
    nr = np.linalg.norm(r)
    fro = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g)
    amax = np.abs(r).max() if r.size else 0.0
    elt = np.abs(g - r).max() if r.size else 0.0
    return float(fro), float(elt / amax) if amax > 0 else float(elt)


def assert_close(got, ref, what="", rel_fro=REL_FRO, rel_elt=REL_ELT):
    g = to_f64(got) if got.dtype == np.uint16 else bf16_round_f64(got)
    r = to_f64(ref) if ref.dtype == np.uint16 else bf16_round_f64(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    nr = np.linalg.norm(r)
    fro = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g)
    amax = np.abs(r).max() if r.size else 0.0
    elt = np.abs(g - r).max() if r.size else 0.0
    assert fro <= rel_fro, f"{what}: relative Frobenius {fro:.3e} > {rel_fro}"
    assert elt <= rel_elt * amax + 1e-30, f"{what}: max |delta| {elt:.3e} > {rel_elt} * {amax:.3e}"
    return fro, elt


def rand_codes(rng, shape):
    """Random finite e4m3 codes of both signs."""
    c = rng.integers(0, 0x7F, shape).astype(np.uint8)
    return c | (rng.integers(0, 2, shape).astype(np.uint8) << 7)


def ragged_sizes(rng, E, M, zero_frac=0.25):
    """E group sizes adding up to M, some of them zero."""
    w = rng.uniform(0.2, 1.0, E)
    w[rng.uniform(0, 1, E) < zero_frac] = 0
    if w.sum() == 0:
        w[0] = 1
    raw = np.floor(w / w.sum() * M).astype(np.int64)
    raw[np.argmax(w)] += M - raw.sum()
    return raw.astype(np.int32)
