"""Pins of the oracle's quantiser and ragged sort (CPU only)."""

import numpy as np
import pytest
import torch

import oracle
import synth


def bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def nearest_code_bruteforce(v: np.ndarray) -> np.ndarray:
    """Nearest e4m3 code by exhaustive search over all finite codes, ties to
    the even code, magnitudes beyond 448 saturated."""
    t = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.int64)
    vals = t[codes]
    v = np.asarray(v, np.float64)
    out = np.empty(v.shape, np.uint8)
    for idx, x in np.ndenumerate(v):
        xs = min(max(x, -448.0), 448.0)
        d = np.abs(vals - xs)
        best = np.flatnonzero(d == d.min())
        # several candidates: +0/-0 (pick by sign), or a tie (pick even mantissa)
        cand = codes[best]
        if len(cand) > 1:
            same_sign = [c for c in cand if (c >> 7) == (1 if np.signbit(x) else 0)]
            if len(same_sign) == 1:
                cand = same_sign
            else:
                cand = [c for c in cand if (c & 1) == 0]
        out[idx] = cand[0]
    return out


# ------------------------------------------------------------ quantiser ----

def test_grid_row_with_amax_448_is_exact():
    t = oracle.e4m3_table()
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 0x7F, (4, 256)).astype(np.uint8)
    codes[:, 7] = 0x7E  # amax 448 in every row
    signs = rng.integers(0, 2, codes.shape).astype(np.uint8) << 7
    codes = codes | signs
    x = t[codes]
    q, s = oracle.quantize_rows(bf16(x), synth.PER_ROW)
    assert np.all(s == 1.0)
    assert np.array_equal(oracle.e4m3_to_f64(q), x)


def test_power_of_two_scaling_keeps_codes():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, 384)).astype(np.float32)
    xb = bf16(x)
    q0, s0 = oracle.quantize_rows(xb, synth.PER_ROW)
    for j in (-5, -1, 3, 10):
        xj = oracle.bf16_to_f64(xb) * 2.0 ** j
        qj, sj = oracle.quantize_rows(bf16(xj), synth.PER_ROW)
        assert np.array_equal(qj, q0)
        assert np.array_equal(sj, (s0 * np.float32(2.0 ** j)).astype(np.float32))


def test_zero_row_and_block():
    x = np.zeros((2, 256), np.float32)
    x[1, :] = -0.0
    x[1, 200] = 3.0  # second block of row 1 is non-zero
    xb = bf16(x)
    q, s = oracle.quantize_rows(xb, synth.PER_ROW_BLOCK128)
    assert np.array_equal(s[0], [1.0, 1.0])
    assert s[1, 0] == 1.0 and s[1, 1] == np.float32(np.float32(3.0) / np.float32(448.0))
    assert np.all(q[0] == 0x00)
    assert np.all(q[1, :128] == 0x80)  # -0 keeps its sign
    qr, sr = oracle.quantize_rows(xb[:1], synth.PER_ROW)
    assert sr[0] == 1.0 and np.all(qr == 0)


@pytest.mark.parametrize("mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128, synth.PER_TENSOR])
def test_codes_are_nearest_e4m3_of_fp32_quotient(mode):
    rng = np.random.default_rng(2 + mode)
    cols = 300  # ragged last block of 44 columns
    x = (rng.standard_normal((5, cols)) * np.exp(rng.uniform(-3, 3, (5, 1)))).astype(np.float32)
    xb = bf16(x)
    xv = oracle.bf16_to_f64(xb).astype(np.float32)
    static = 0.004
    q, s = oracle.quantize_rows(xb, mode, static)
    if mode == synth.PER_ROW:
        amax = np.abs(xv).max(axis=1)
        assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
        scale = np.repeat(s[:, None], cols, axis=1)
    elif mode == synth.PER_ROW_BLOCK128:
        assert s.shape == (5, 3)
        scale = np.empty_like(xv)
        for b in range(3):
            blk = xv[:, b * 128:(b + 1) * 128]
            sb = (np.abs(blk).max(axis=1) / np.float32(448.0)).astype(np.float32)
            assert np.array_equal(s[:, b], sb)
            scale[:, b * 128:(b + 1) * 128] = sb[:, None]
    else:
        scale = np.full_like(xv, np.float32(static))
    quot = (xv / scale).astype(np.float32)  # IEEE fp32 division
    assert np.array_equal(q, nearest_code_bruteforce(quot))


def test_static_scale_saturates():
    x = np.array([[1.0, -1.0, 0.5, 100.0]], np.float32)
    q, _ = oracle.quantize_rows(bf16(x), synth.PER_TENSOR, 0.001)
    assert list(q[0]) == [0x7E, 0xFE, 0x7E, 0x7E]


def test_weight_scale_layouts():
    rng = np.random.default_rng(3)
    w = bf16(rng.standard_normal((3, 5, 256)) * 0.02)
    q, s = oracle.quantize_weights(w, synth.PER_ROW_BLOCK128)
    assert s.shape == (3, 2, 5)  # [E, K/128, N], the pages' [E, blocks, 1, N]
    qr, sr = oracle.quantize_rows(w.reshape(15, 256), synth.PER_ROW_BLOCK128)
    assert np.array_equal(q.reshape(15, 256), qr)
    assert np.array_equal(s, sr.reshape(3, 5, 2).transpose(0, 2, 1))
    qc, sc = oracle.quantize_weights(w, synth.PER_ROW)
    assert sc.shape == (3, 5)


@pytest.mark.parametrize("mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128])
def test_quantise_before_sort_is_free(mode):
    """The reordering the first page makes: quantising the activations before
    the sort/gather gives the same bytes as quantising the gathered rows."""
    cfg = synth.scaled(synth.CONFIGS["tiny"], T=64, D=256)
    x = oracle.bf16_bits(synth.activations(cfg, 0))
    ids, _ = synth.routing(cfg, 0)
    src, pos, sizes, offs = oracle.ragged_sort(ids, cfg.E)
    q, s = oracle.quantize_rows(x, mode)
    xs_q, xs_s = oracle.gather_rows(q, s, mode, src, cfg.k)
    xg = x[src // cfg.k]
    q2, s2 = oracle.quantize_rows(xg, mode)
    assert np.array_equal(xs_q, q2) and np.array_equal(xs_s, s2)


def test_per_tensor_scale_is_not_gathered():
    x_q = np.arange(12, dtype=np.uint8).reshape(3, 4)
    xs, xss = oracle.gather_rows(x_q, np.array([0.5], np.float32), synth.PER_TENSOR,
                                 np.array([2, 0, 1], np.int32), 1)
    assert np.array_equal(xs, x_q[[2, 0, 1]]) and xss.tolist() == [0.5]


# ---------------------------------------------------------------- sort -----

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 2, 4), (64, 8, 256), (333, 6, 64), (50, 2, 3)])
def test_ragged_sort_brute_force(T, k, E):
    rng = np.random.default_rng(T * 131 + E)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    src, pos, sizes, offs = oracle.ragged_sort(ids, E)
    R = T * k
    flat = ids.reshape(-1)
    ref = sorted(range(R), key=lambda i: (flat[i], i))
    assert src.tolist() == ref
    assert np.array_equal(pos[src], np.arange(R))          # pos is the inverse
    assert sorted(src.tolist()) == list(range(R))          # bijection
    assert sizes.sum() == R and offs[0] == 0 and offs[-1] == R
    assert np.array_equal(np.diff(offs), sizes)
    assert np.array_equal(sizes, np.bincount(flat, minlength=E))
    # groups contiguous and ascending
    assert np.all(np.diff(flat[src]) >= 0)


def test_ragged_sort_zero_token_experts_and_bad_ids():
    ids = np.array([[3, 0], [3, 0]], np.int32)
    src, pos, sizes, offs = oracle.ragged_sort(ids, 6)
    assert sizes.tolist() == [2, 0, 0, 2, 0, 0]
    assert offs.tolist() == [0, 2, 2, 2, 4, 4, 4]
    with pytest.raises(ValueError):
        oracle.ragged_sort(np.array([[0, 6]], np.int32), 6)
    with pytest.raises(ValueError):
        oracle.ragged_sort(np.array([[-1, 0]], np.int32), 6)


def test_zipf_routing_has_zero_token_experts():
    cfg = synth.scaled(synth.CONFIGS["fwdbwd"], T=512)
    ids, w = synth.routing(cfg, 0)
    _, _, sizes, _ = oracle.ragged_sort(ids, cfg.E)
    assert (sizes == 0).sum() >= 8
    assert np.all(w > 0) and np.all(w <= 1)
