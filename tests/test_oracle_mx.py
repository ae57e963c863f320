"""Pins of the oracle's MXFP8 variant (CPU only).

MXFP8 follows the OCP "Microscaling Formats (MX) Specification" v1.0: every
block of 32 consecutive values along the contracted dimension holds e4m3
elements and shares one E8M0 scale, a power of two 2^X stored as the biased
exponent X + 127.  The shared exponent is floor(log2(amax)) minus 8, the
exponent of the largest power of two e4m3 can hold (256 = 2^8).

The pins do not restate the oracle's formulas:
- blocks whose codes were derived by hand from the e4m3 and E8M0 encodings;
- element codes checked against torch's float8_e4m3fn rounding (an
  independent library routine);
- the bracket 256 * 2^X <= amax < 512 * 2^X, which fixes X with no log;
- equivariance under powers of two;
- reduction of the MX matmul to the pinned per-row / per-channel gmm, block
  by block.
"""

import numpy as np
import pytest
import torch

import oracle
import synth


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def block(vals):
    row = np.zeros(32, np.float32)
    row[: len(vals)] = vals
    return row


def e8m0(code):
    return np.ldexp(1.0, np.asarray(code, np.int64) - 127)


# ------------------------------------------------------- hand-derived blocks

# (values, E8M0 code, element codes of the listed values), each derived by hand:
HAND = [
    # amax 3 = 1.5 * 2^1, so X = 1 - 8 = -7 (code 120).  x * 2^7:
    #   1 -> 128 = 2^7 (e4m3 exponent field 14: 0x70); -0.5 -> -64 (0xE8);
    #   0.25 -> 32 (0x60); 3 -> 384 = 1.5 * 2^8 (field 15, mantissa 4: 0x7C)
    ([1.0, -0.5, 0.25, 3.0], 120, [0x70, 0xE8, 0x60, 0x7C]),
    # amax 1.9375 = 1.9375 * 2^0: X = -8 (code 119).  1.9375 * 256 = 496 lies
    # above 448 and saturates (0x7E); 2^-7 * 256 = 2 (0x40); -1 -> -256 (0xF8)
    ([1.9375, 2.0 ** -7, -1.0], 119, [0x7E, 0x40, 0xF8]),
    # ties to the even mantissa at X = -8 (step 32 in [256, 512)):
    #   1.1875 -> 304, halfway between 288 (m 1) and 320 (m 2): 320 (0x7A);
    #   1.0625 -> 272, halfway between 256 (m 0) and 288: 256 (0x78).
    # subnormals (step 2^-9): 2^-17 -> 2^-9 (0x01); 3 * 2^-19 -> 0.75 * 2^-9
    # -> 2^-9 (0x01); 2^-18 -> 2^-10, halfway between 0 and 2^-9: 0 (0x00);
    # -2^-18 -> -0 (0x80)
    ([1.1875, 1.0625, 2.0 ** -17, 3 * 2.0 ** -19, 2.0 ** -18, -(2.0 ** -18)], 119,
     [0x7A, 0x78, 0x01, 0x01, 0x00, 0x80]),
    # amax 2^-126: floor(log2) - 8 = -134, clamped to E8M0's -127 (code 0);
    # 2^-126 * 2^127 = 2 (0x40)
    ([2.0 ** -126], 0, [0x40]),
    # the largest bf16 powers: amax 2^127 -> X = 119 (code 246); 2^127 / 2^119
    # = 256 (0x78); -2^120 -> -2 (0xC0)
    ([2.0 ** 127, -(2.0 ** 120)], 246, [0x78, 0xC0]),
    # a block of zeros: the smallest scale (code 0), all codes +0
    ([0.0], 0, [0x00]),
]


@pytest.mark.parametrize("vals,code,codes", HAND)
def test_hand_derived_blocks(vals, code, codes):
    q, sf = oracle.quantize_rows_mx(bf16(block(vals))[None, :])
    assert sf.shape == (1, 1) and int(sf[0, 0]) == code
    assert [int(c) for c in q[0, : len(codes)]] == codes
    assert not q[0, len(codes):].any()


def test_blocks_of_a_row_are_independent():
    # block 0: amax 1 -> X = -8 (code 119), 1 -> 256 (0x78);
    # block 1: amax 1024 = 2^10 -> X = 2 (code 129), 1024 -> 256 (0x78), 3 -> 0.75 (0x34: field 6, m 4)
    row = np.zeros(64, np.float32)
    row[0] = 1.0
    row[32] = 1024.0
    row[33] = 3.0
    q, sf = oracle.quantize_rows_mx(bf16(row)[None, :])
    assert sf.tolist() == [[119, 129]]
    assert (int(q[0, 0]), int(q[0, 32]), int(q[0, 33])) == (0x78, 0x78, 0x34)


# ------------------------------------------------------ library and bounds

def random_rows(rng, rows, cols):
    # N(0, 1) blocks, each scaled by its own power of two over a wide range
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x *= np.repeat(np.ldexp(1.0, rng.integers(-60, 60, (rows, cols // 32))), 32, axis=1).astype(np.float32)
    x[rng.random((rows, cols)) < 0.05] = 0.0
    return bf16(x)


def test_shared_exponent_brackets_amax():
    rng = np.random.default_rng(7)
    xb = random_rows(rng, 64, 256)
    q, sf = oracle.quantize_rows_mx(xb)
    x = oracle.bf16_to_f64(xb).reshape(64, 8, 32)
    amax = np.abs(x).max(axis=2)
    s = e8m0(sf)
    assert (amax > 0).all()
    assert (256 * s <= amax).all() and (amax < 512 * s).all()
    # the largest element code of every block lies in [256, 448]
    big = np.abs(oracle.e4m3_to_f64(q)).reshape(64, 8, 32).max(axis=2)
    assert (big >= 256).all() and (big <= 448).all()


def test_elements_match_torch_e4m3_rounding():
    rng = np.random.default_rng(8)
    xb = random_rows(rng, 48, 512)
    q, sf = oracle.quantize_rows_mx(xb)
    y = oracle.bf16_to_f64(xb) / np.repeat(e8m0(sf), 32, axis=1)  # exact: powers of two
    sat = np.abs(y) > 448
    ref = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q[~sat], ref[~sat])
    # only the top binade saturates, to +-448
    assert (np.abs(y[sat]) < 512).all()
    assert np.array_equal(q[sat], np.where(y[sat] > 0, 0x7E, 0xFE).astype(np.uint8))


def test_power_of_two_equivariance():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 128)).astype(np.float32)
    q0, s0 = oracle.quantize_rows_mx(bf16(x))
    for j in (-20, -3, 1, 17):
        q1, s1 = oracle.quantize_rows_mx(bf16(x * np.float32(2.0 ** j)))
        assert np.array_equal(q0, q1)
        assert np.array_equal(s1.astype(np.int64), s0.astype(np.int64) + j)


def test_weight_scale_layout():
    rng = np.random.default_rng(10)
    w = bf16(rng.standard_normal((3, 5, 96)).astype(np.float32) * 0.02)
    q, sf = oracle.quantize_weights_mx(w)
    assert q.shape == (3, 5, 96) and sf.shape == (3, 5, 3)
    for e in range(3):
        for n in range(5):
            qr, sr = oracle.quantize_rows_mx(w[e, n][None, :])
            assert np.array_equal(q[e, n], qr[0]) and np.array_equal(sf[e, n], sr[0])


# ------------------------------------------------------------------ gmm ----

def rand_mx(rng, shape, lo=100, hi=150):
    c = rng.integers(0, 0x7F, shape).astype(np.uint8) | (rng.integers(0, 2, shape).astype(np.uint8) << 7)
    sf = rng.integers(lo, hi, shape[:-1] + (shape[-1] // 32,)).astype(np.uint8)
    return c, sf


def test_gmm_mx_with_uniform_codes_is_the_per_row_per_channel_gmm():
    # one E8M0 code per row (lhs) and per channel (rhs): the MX matmul is the
    # pinned gmm with per-row scales 2^(c - 127) and per-channel scales
    rng = np.random.default_rng(11)
    M, K, N, E = 40, 160, 24, 3
    a, _ = rand_mx(rng, (M, K))
    w, _ = rand_mx(rng, (E, N, K))
    ca = rng.integers(110, 140, M)
    cw = rng.integers(110, 140, (E, N))
    asf = np.repeat(ca[:, None], K // 32, axis=1).astype(np.uint8)
    wsf = np.repeat(cw[:, :, None], K // 32, axis=2).astype(np.uint8)
    sizes = np.array([15, 0, 25], np.int32)
    out = oracle.gmm_mx(a, asf, w, wsf, sizes, want="f64")
    ref = oracle.gmm(a, e8m0(ca).astype(np.float32), synth.PER_ROW, w, e8m0(cw).astype(np.float32), synth.PER_ROW,
                     sizes, want="f64")
    assert np.array_equal(out, ref)


def test_gmm_mx_is_the_sum_of_its_32_wide_blocks():
    # block b of K alone, with its own per-row and per-channel codes, is a
    # per-row / per-channel gmm of the operands zeroed outside block b; the
    # MX matmul is the sum of these over b (a transposed or shifted scale
    # index would break the identity)
    rng = np.random.default_rng(12)
    M, K, N = 33, 192, 40
    sizes = np.array([20, 13], np.int32)
    a, asf = rand_mx(rng, (M, K))
    w, wsf = rand_mx(rng, (2, N, K))
    out = oracle.gmm_mx(a, asf, w, wsf, sizes, want="f64")
    acc = np.zeros((M, N))
    for b in range(K // 32):
        ab = np.zeros_like(a)
        wb = np.zeros_like(w)
        ab[:, 32 * b:32 * b + 32] = a[:, 32 * b:32 * b + 32]
        wb[:, :, 32 * b:32 * b + 32] = w[:, :, 32 * b:32 * b + 32]
        acc += oracle.gmm(ab, e8m0(asf[:, b]).astype(np.float32), synth.PER_ROW, wb,
                          e8m0(wsf[:, :, b]).astype(np.float32), synth.PER_ROW, sizes, want="f64")
    np.testing.assert_allclose(out, acc, rtol=1e-12, atol=1e-12 * np.abs(acc).max())


def test_gmm_mx_group_offset_and_bf16_output():
    rng = np.random.default_rng(13)
    M, K, N = 30, 64, 16
    sizes = np.array([10, 0, 12, 8], np.int32)
    a, asf = rand_mx(rng, (M, K))
    w, wsf = rand_mx(rng, (2, N, K))
    out = oracle.gmm_mx(a, asf, w, wsf, sizes, group_offset=1, E_local=2, want="f64")
    assert not out[:10].any() and not out[22:].any() and np.abs(out[10:22]).max() > 0
    ob = oracle.gmm_mx(a, asf, w, wsf, sizes, group_offset=1, E_local=2)
    assert np.array_equal(ob, oracle.f64_to_bf16(out))


# -------------------------------------------------------- SwiGLU and FFN --

def test_swiglu_quant_mx_requantises_the_pinned_h():
    rng = np.random.default_rng(14)
    a = bf16(rng.standard_normal((24, 2 * 96)).astype(np.float32) * 3)
    hq, hsf, hb = oracle.swiglu_quant_mx(a)
    _, _, hb_ref = oracle.swiglu_quant(a, synth.PER_ROW)
    assert np.array_equal(hb, hb_ref)
    q_ref, sf_ref = oracle.quantize_rows_mx(hb_ref)
    assert np.array_equal(hq, q_ref) and np.array_equal(hsf, sf_ref)


def test_ffn_forward_mx_token_subset_and_accuracy():
    cfg = synth.scaled(synth.CONFIGS["dsv3_mx"], T=96, D=256, E=8, k=2, F=128)
    x = synth.activations(cfg, seed=3)
    w_in, w_out = synth.expert_weights(cfg, seed=3)
    ids, tw = synth.routing(cfg, seed=3)
    xb, wib, wob = (oracle.bf16_bits(t) for t in (x, w_in, w_out))
    wq = oracle.prepare_weights_mx(wib, wob)
    full = oracle.ffn_forward_mx(xb, ids, tw, wq, cfg.E)
    toks = [0, 5, 77, 95]
    part = oracle.ffn_forward_mx(xb, ids, tw, wq, cfg.E, tokens=toks)
    assert np.array_equal(part["y"], full["y"][toks])
    # against the unquantised layer in double (bf16 inputs): MXFP8 error of a
    # few per cent, like the per-channel fp8 path
    y = oracle.bf16_to_f64(full["y"])
    srt, pos = full["sorted_src"], full["pos"]
    xs = oracle.bf16_to_f64(xb)[srt // cfg.k]
    a = oracle.gmm_f64(xs, oracle.bf16_to_f64(wib), full["sizes"])
    h = oracle.swiglu_f64(a)
    o = oracle.gmm_f64(h, oracle.bf16_to_f64(wob), full["sizes"])
    ref = oracle.combine_f64(o, pos, tw, cfg.k)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 0.08, rel
