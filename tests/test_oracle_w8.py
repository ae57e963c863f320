"""Pins of the oracle's int8-weight variant (CPU only).

"Keep qwix out of tpu-inference's fused MoE kernel and pre-quantize weights"
pre-quantises the expert weights to float8_e4m3fn or int8, with [E, blocks,
1, N] scales.  The int8 form is symmetric absmax: s = amax / 127 in fp32, and
every value becomes the nearest integer (ties to even) of x / s, so the
largest magnitude maps to 127.  The activations and h stay e4m3.

The pins do not restate the oracle's formulas:
- codes derived by hand where s is a power of two;
- the nearest-integer property checked by search over all 255 codes;
- the round-trip bound |q s - x| <= s / 2 and the amax element at +-127;
- equivariance under powers of two;
- the blockwise layout reduced to per-channel quantisation of each slice;
- the int8 matmul reduced to the pinned e4m3 gmm on codes both formats hold
  exactly, and to numpy's matmul of the dequantised operands.
"""

import numpy as np
import pytest
import torch

import oracle
import synth


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rows_of(vals, K=128):
    r = np.zeros((1, 1, K), np.float32)
    r[0, 0, : len(vals)] = vals
    return bf16(r)


# ------------------------------------------------------- hand-derived codes

# (values, scale, codes of the listed values), each derived by hand:
HAND = [
    # amax 127: s = 1.  Ties to even: -63.5 -> -64, 0.5 -> 0, 1.5 -> 2,
    # -2.5 -> -2, 2.5 -> 2; -0.5 -> -0 = 0
    ([127.0, -63.5, 0.5, 0.0, 1.5, -2.5, 2.5, -0.5], 1.0, [127, -64, 0, 0, 2, -2, 2, 0]),
    # amax 15.875 = 127 / 8: s = 2^-3 exactly, so q = rint(8 x):
    # 2^-4 -> 0.5 -> 0; 0.1875 -> 1.5 -> 2; -15.875 -> -127; 1 -> 8;
    # 0.3125 -> 2.5 -> 2; -0.4375 -> -3.5 -> -4
    ([2.0 ** -4, 0.1875, -15.875, 1.0, 0.3125, -0.4375], 0.125, [0, 2, -127, 8, 2, -4]),
    # amax 254: s = 2; 3 -> 1.5 -> 2; 5 -> 2.5 -> 2; -253 -> -126.5 -> -126
    ([254.0, 3.0, 5.0, -253.0], 2.0, [127, 2, 2, -126]),
]


@pytest.mark.parametrize("vals,scale,codes", HAND)
def test_hand_derived_codes(vals, scale, codes):
    q, s = oracle.quantize_weights_int8(rows_of(vals), synth.PER_ROW)
    assert s[0, 0] == np.float32(scale)
    assert q[0, 0, : len(codes)].tolist() == codes
    assert not q[0, 0, len(codes):].any()


def test_zero_row_takes_unit_scale_and_zero_codes():
    q, s = oracle.quantize_weights_int8(rows_of([]), synth.PER_ROW)
    assert s[0, 0] == 1.0 and not q.any()


# --------------------------------------------------------- random weights

def rand_w(rng, shape, std=0.02):
    return bf16(rng.standard_normal(shape).astype(np.float32) * std)


def test_codes_are_the_nearest_integers_by_search():
    rng = np.random.default_rng(21)
    w = rand_w(rng, (2, 5, 256))
    q, s = oracle.quantize_weights_int8(w, synth.PER_ROW)
    x = oracle.bf16_to_f64(w).astype(np.float32)
    v = (x / s[:, :, None].astype(np.float32)).astype(np.float64)  # the fp32 quotient
    cand = np.arange(-127, 128, dtype=np.float64)
    d = np.abs(v[..., None] - cand)
    best = d.min(axis=-1, keepdims=True)
    # among the nearest candidates (two on a tie) the code is the even one
    near = d == best
    even = (cand.astype(np.int64) % 2 == 0)
    pick = np.where(near.sum(-1) > 1, np.argmax(near & even, axis=-1), np.argmax(near, axis=-1))
    assert np.array_equal(q.astype(np.int64), cand[pick].astype(np.int64))


def test_round_trip_bound_and_amax_code():
    rng = np.random.default_rng(22)
    w = rand_w(rng, (3, 7, 384), std=1.5)
    q, s = oracle.quantize_weights_int8(w, synth.PER_ROW)
    x = oracle.bf16_to_f64(w)
    sd = s.astype(np.float64)[:, :, None]
    err = np.abs(q * sd - x)
    # the fp32 quotient carries a relative error up to 2^-24 on |x / s| <= 127
    assert np.all(err <= sd * (0.5 + 127 * 2.0 ** -23))
    assert np.all(np.abs(q).max(axis=-1) == 127)
    # the amax element carries the code +-127 with its sign
    i = np.abs(x).argmax(axis=-1)
    qa = np.take_along_axis(q, i[..., None], -1)[..., 0]
    xa = np.take_along_axis(x, i[..., None], -1)[..., 0]
    assert np.array_equal(qa, np.where(xa > 0, 127, -127))
    assert np.array_equal(s, (np.abs(x).max(-1).astype(np.float32) / np.float32(127)).astype(np.float32))


def test_power_of_two_equivariance():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((2, 4, 256)).astype(np.float32)
    w = bf16(x)
    q, s = oracle.quantize_weights_int8(w, synth.PER_ROW_BLOCK128)
    for j in (-9, 5):
        w2 = bf16(oracle.bf16_to_f64(w) * 2.0 ** j)
        q2, s2 = oracle.quantize_weights_int8(w2, synth.PER_ROW_BLOCK128)
        assert np.array_equal(q2, q)
        assert np.array_equal(s2, (s * np.float32(2.0 ** j)).astype(np.float32))


def test_blockwise_is_per_channel_on_each_slice_and_layout():
    rng = np.random.default_rng(24)
    E, N, K = 2, 6, 384
    w = rand_w(rng, (E, N, K))
    qb, sb = oracle.quantize_weights_int8(w, synth.PER_ROW_BLOCK128)
    assert sb.shape == (E, K // 128, N)
    for b in range(K // 128):
        qs, ss = oracle.quantize_weights_int8(np.ascontiguousarray(w[:, :, 128 * b:128 * b + 128]), synth.PER_ROW)
        assert np.array_equal(qb[:, :, 128 * b:128 * b + 128], qs)
        assert np.array_equal(sb[:, b, :], ss)
    # one block: the two modes agree
    q1, s1 = oracle.quantize_weights_int8(np.ascontiguousarray(w[:, :, :128]), synth.PER_ROW_BLOCK128)
    q2, s2 = oracle.quantize_weights_int8(np.ascontiguousarray(w[:, :, :128]), synth.PER_ROW)
    assert np.array_equal(q1, q2) and np.array_equal(s1[:, 0, :], s2)


def test_static_scale_codes():
    rng = np.random.default_rng(25)
    w = rand_w(rng, (1, 3, 128), std=1.0)
    q, _ = oracle.quantize_weights_int8(w, synth.PER_TENSOR, static_scale=0.25)
    x = oracle.bf16_to_f64(w)
    assert np.array_equal(q, np.clip(np.round(x * 4), -127, 127).astype(np.int8))  # x / 0.25 exact in fp32


# ------------------------------------------------------------- the matmul

def rand_lhs(rng, M, K):
    a = rng.integers(0, 256, (M, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return a


def test_gmm_w8_equals_the_e4m3_gmm_on_shared_codes():
    # the integers -16..16 are exact e4m3 values, so int8 codes in that range
    # and the e4m3 codes of the same integers must give identical products
    rng = np.random.default_rng(26)
    M, K, N = 37, 256, 24
    sizes = np.array([12, 0, 25], np.int32)
    a = rand_lhs(rng, M, K)
    sa = (rng.random(M) + 0.5).astype(np.float32)
    qi = rng.integers(-16, 17, (3, N, K)).astype(np.int8)
    table = {int(v): c for c in range(256) if (c & 0x7F) != 0x7F for v in [oracle.e4m3_to_f64(np.array([c]))[0]]
             if float(v).is_integer() and abs(v) <= 16 and not (v == 0 and c != 0)}
    qe = np.vectorize(lambda v: table[int(v)])(qi).astype(np.uint8)
    for mode, sw in ((synth.PER_ROW, (rng.random((3, N)) + 0.5).astype(np.float32)),
                     (synth.PER_ROW_BLOCK128, (rng.random((3, K // 128, N)) + 0.5).astype(np.float32)),
                     (synth.PER_TENSOR, np.array([0.75], np.float32))):
        out = oracle.gmm_w8(a, sa, synth.PER_ROW, qi, sw, mode, sizes, want="f64")
        ref = oracle.gmm(a, sa, synth.PER_ROW, qe, sw, mode, sizes, want="f64")
        assert np.array_equal(out, ref), mode


@pytest.mark.parametrize("w_mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128, synth.PER_TENSOR])
@pytest.mark.parametrize("a_mode", [synth.PER_ROW, synth.PER_TENSOR])
def test_gmm_w8_is_the_dense_product_of_the_dequantised_operands(a_mode, w_mode):
    rng = np.random.default_rng(27 + a_mode * 3 + w_mode)
    M, K, N, E = 41, 384, 20, 3
    sizes = np.array([9, 0, 32], np.int32)
    a = rand_lhs(rng, M, K)
    sa = (rng.random(M) + 0.5).astype(np.float32) if a_mode == synth.PER_ROW else np.array([0.3], np.float32)
    q = rng.integers(-127, 128, (E, N, K)).astype(np.int8)
    sw = {synth.PER_ROW: (rng.random((E, N)) + 0.5), synth.PER_ROW_BLOCK128: (rng.random((E, K // 128, N)) + 0.5),
          synth.PER_TENSOR: np.array([0.01])}[w_mode].astype(np.float32)
    out = oracle.gmm_w8(a, sa, a_mode, q, sw, w_mode, sizes, want="f64")
    ad = oracle.e4m3_to_f64(a) * (sa[:, None] if a_mode == synth.PER_ROW else sa[0])
    if w_mode == synth.PER_ROW:
        wd = q * sw.astype(np.float64)[:, :, None]
    elif w_mode == synth.PER_ROW_BLOCK128:
        wd = q * np.repeat(sw.astype(np.float64).transpose(0, 2, 1), 128, axis=2)
    else:
        wd = q * float(sw[0])
    starts = np.concatenate([[0], np.cumsum(sizes)])
    ref = np.zeros((M, N))
    for e in range(E):
        ref[starts[e]:starts[e + 1]] = ad[starts[e]:starts[e + 1]] @ wd[e].T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # group_offset: the shard's rows only, the rest zero
    sh = oracle.gmm_w8(a, sa, a_mode, q[2:], sw[2:] if w_mode != synth.PER_TENSOR else sw, w_mode, sizes,
                       group_offset=2, E_local=1, want="f64")
    assert not sh[:9].any()
    np.testing.assert_allclose(sh[9:], ref[9:], rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_gmm_w8_bf16_output_is_the_rounded_f64():
    rng = np.random.default_rng(28)
    M, K, N = 20, 128, 16
    sizes = np.array([20], np.int32)
    a = rand_lhs(rng, M, K)
    q = rng.integers(-127, 128, (1, N, K)).astype(np.int8)
    sa = np.ones(M, np.float32)
    sw = np.full((1, N), 0.01, np.float32)
    f = oracle.gmm_w8(a, sa, synth.PER_ROW, q, sw, synth.PER_ROW, sizes, want="f64")
    b = oracle.gmm_w8(a, sa, synth.PER_ROW, q, sw, synth.PER_ROW, sizes)
    assert np.array_equal(b, oracle.f64_to_bf16(f))


# ----------------------------------------------------------------- the FFN

@pytest.mark.parametrize("w_mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128])
def test_ffn_forward_w8_token_subset_and_accuracy(w_mode):
    cfg = synth.scaled(synth.CONFIGS["mixtral_w8"], T=96, D=256, E=8, k=2, F=128, w_mode=w_mode)
    x = synth.activations(cfg, seed=4)
    w_in, w_out = synth.expert_weights(cfg, seed=4)
    ids, tw = synth.routing(cfg, seed=4)
    xb, wib, wob = (oracle.bf16_bits(t) for t in (x, w_in, w_out))
    wq = oracle.prepare_weights_w8(wib, wob, w_mode)
    assert wq[0].dtype == np.int8
    full = oracle.ffn_forward(xb, ids, tw, wq, cfg.E, cfg.act_mode)
    toks = [0, 7, 50, 95]
    part = oracle.ffn_forward(xb, ids, tw, wq, cfg.E, cfg.act_mode, tokens=toks)
    assert np.array_equal(part["y"], full["y"][toks])
    # against the unquantised layer in double, and against the same layer
    # with e4m3 weights: int8 codes carry 7 significant bits to e4m3's 4, so
    # the int8 layer's error is the smaller one (the e4m3 activations and h
    # dominate both)
    srt, pos = full["sorted_src"], full["pos"]
    xs = oracle.bf16_to_f64(xb)[srt // cfg.k]
    a = oracle.gmm_f64(xs, oracle.bf16_to_f64(wib), full["sizes"])
    h = oracle.swiglu_f64(a)
    o = oracle.gmm_f64(h, oracle.bf16_to_f64(wob), full["sizes"])
    ref = oracle.combine_f64(o, pos, tw, cfg.k)
    rel8 = np.linalg.norm(oracle.bf16_to_f64(full["y"]) - ref) / np.linalg.norm(ref)
    fp8 = oracle.ffn_forward(xb, ids, tw, oracle.prepare_weights(wib, wob, w_mode), cfg.E, cfg.act_mode)
    relf = np.linalg.norm(oracle.bf16_to_f64(fp8["y"]) - ref) / np.linalg.norm(ref)
    assert rel8 < 0.06, rel8
    assert rel8 < relf, (rel8, relf)
