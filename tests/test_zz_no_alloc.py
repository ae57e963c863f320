"""GPU test of moe_ragged_sort_noalloc, the ragged sort for callers that may
not allocate device memory (an engine whose memory pool already owns the free
HBM, a plugin interface without an allocator, a latency-critical loop where a
device-synchronising cudaMalloc is not allowed).  It keeps its scratch in a
fixed array inside the library instead of a caller workspace.

The test calls it through the C ABI (ctypes, raw device pointers) twice in a
row, with different problems so that the second call runs over whatever the
first left in the shared array, and compares every output with the regular
moe_ragged_sort: the sort is integer and byte work, so the results must be
identical.  This file is collected last so that a run stopping at the first
failure has run every other test before it."""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("fp8_quantized_moe_gb300")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _case(seed, T, k, E, D, mode):
    rng = np.random.default_rng(seed)
    ids = torch.from_numpy(rng.integers(0, E, (T, k)).astype(np.int32)).cuda()
    x_q = torch.from_numpy(rng.integers(0, 256, (T, D)).astype(np.uint8)).cuda()
    if mode == synth.PER_ROW:
        x_s = torch.from_numpy(rng.uniform(0.1, 2, T).astype(np.float32)).cuda()
    elif mode == synth.PER_ROW_BLOCK128:
        x_s = torch.from_numpy(rng.uniform(0.1, 2, (T, (D + 127) // 128)).astype(np.float32)).cuda()
    else:
        x_s = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    return ids, x_q, x_s


def _noalloc(ids, E, x_q, x_s, mode):
    T, k = ids.shape
    D = x_q.shape[1]
    R = T * k
    out = {
        "sorted_src": torch.full((R,), -7, dtype=torch.int32, device="cuda"),
        "pos": torch.full((R,), -7, dtype=torch.int32, device="cuda"),
        "group_sizes": torch.full((E,), -7, dtype=torch.int32, device="cuda"),
        "group_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        "xs_q": torch.zeros(R, D, dtype=torch.uint8, device="cuda"),
        "xs_scale": None,
    }
    if mode == synth.PER_ROW:
        out["xs_scale"] = torch.zeros(R, dtype=torch.float32, device="cuda")
    elif mode == synth.PER_ROW_BLOCK128:
        out["xs_scale"] = torch.zeros(R, (D + 127) // 128, dtype=torch.float32, device="cuda")
    st = moe.lib().moe_ragged_sort_noalloc(
        _ptr(ids), T, k, E, _ptr(x_q), _ptr(x_s), D, mode, _ptr(out["sorted_src"]), _ptr(out["pos"]),
        _ptr(out["group_sizes"]), _ptr(out["group_offsets"]), _ptr(out["xs_q"]), _ptr(out["xs_scale"]),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, moe.lib().moe_status_string(st)
    return out


def test_noalloc_sort_matches_workspace_sort_on_two_calls_in_a_row():
    cases = [
        (1, 3000, 8, 256, 384, synth.PER_ROW_BLOCK128),  # several chunks, many experts
        (2, 700, 2, 8, 256, synth.PER_ROW),              # fewer chunks and experts: stale counts remain
    ]
    for seed, T, k, E, D, mode in cases:
        ids, x_q, x_s = _case(seed, T, k, E, D, mode)
        ref = moe.ragged_sort(ids, E, x_q, x_s, mode)
        got = _noalloc(ids, E, x_q, x_s, mode)
        torch.cuda.synchronize()
        assert moe.device_error() == 0
        for key in ("sorted_src", "pos", "group_sizes", "group_offsets", "xs_q", "xs_scale"):
            if ref[key] is None:
                continue
            assert torch.equal(got[key], ref[key]), key


def test_noalloc_sort_rejects_problems_beyond_its_scratch():
    # 2^22 (token, expert) pairs over 256 experts need 2 MiB of counts > 1 MiB
    T, k, E, D = 1 << 19, 8, 256, 16
    need = moe.lib().moe_ragged_sort_workspace_bytes(T, k, E)
    assert need > (1 << 20)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = _ptr(dummy)
    st = moe.lib().moe_ragged_sort_noalloc(p, T, k, E, p, p, D, synth.PER_ROW, p, p, p, p, p, p,
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1  # MOE_ERR_INVALID_ARG, nothing launched
