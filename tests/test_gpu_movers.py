"""GPU parity of the bandwidth-bound steps against the oracle: quantiser,
weight quantiser, ragged sort + gather, SwiGLU requantisation, combine and the
backward helpers.  Codes, scales and indices must match bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import assert_close, dev, host

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("fp8_quantized_moe_gb300")


def bf16_rows(rng, rows, cols, scale=1.0, specials=True):
    x = (rng.standard_normal((rows, cols)) * scale * np.exp(rng.uniform(-4, 4, (rows, 1)))).astype(np.float32)
    if specials and rows >= 4:
        x[0] = 0.0                      # all-zero row -> scale 1
        x[1, : cols // 2] = -0.0        # signed zeros
        x[2, 3] = 1e30                  # huge -> amax, the rest underflow towards 0
        x[3, :] = -x[3, :]
    return oracle.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))


@pytest.mark.parametrize("mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128, synth.PER_TENSOR])
@pytest.mark.parametrize("rows,cols", [(1, 16), (5, 128), (37, 304), (64, 2048), (9, 7168), (4, 14336),
                                       (3, 32768)])
def test_quantize_rows_bit_exact(mode, rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols + mode)
    x = bf16_rows(rng, rows, cols)
    static = 0.0123
    q_ref, s_ref = oracle.quantize_rows(x, mode, static)
    ss = torch.tensor([static], dtype=torch.float32, device="cuda")
    q, s = moe.quantize_rows(dev(x), mode, ss)
    torch.cuda.synchronize()
    assert np.array_equal(host(q), q_ref)
    if mode != synth.PER_TENSOR:
        assert np.array_equal(host(s).view(np.uint32), s_ref.view(np.uint32))


@pytest.mark.parametrize("mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128, synth.PER_TENSOR])
def test_quantize_weights_bit_exact(mode):
    rng = np.random.default_rng(7)
    E, N, K = 3, 48, 384
    w = oracle.bf16_bits(torch.from_numpy((rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)).to(torch.bfloat16))
    q_ref, s_ref = oracle.quantize_weights(w, mode, 1e-4)
    q, s = moe.quantize_weights(dev(w), mode, torch.tensor([1e-4], dtype=torch.float32, device="cuda"))
    assert np.array_equal(host(q), q_ref)
    if mode != synth.PER_TENSOR:
        assert np.array_equal(host(s), s_ref)


@pytest.mark.parametrize("T,k,E,D,mode", [
    (1, 1, 1, 16, synth.PER_ROW),
    (7, 2, 16, 128, synth.PER_ROW),           # E > T*k: zero-token experts
    (256, 2, 4, 128, synth.PER_ROW),
    (333, 6, 64, 256, synth.PER_TENSOR),
    (1000, 8, 256, 384, synth.PER_ROW_BLOCK128),
    (2500, 8, 1024, 64, synth.PER_ROW),       # several chunks, E at its limit
    (4096, 8, 64, 64, synth.PER_ROW),         # 32768 pairs, 64 experts: the one-CTA sort at its limits
    (4095, 8, 63, 32, synth.PER_TENSOR),      # the one-CTA sort, ragged last rounds
    (32769, 1, 32, 16, synth.PER_ROW),        # one pair past the one-CTA limit: the multi-CTA sort
    (300, 4, 65, 16, synth.PER_ROW),          # one expert past the one-CTA limit: the multi-CTA sort
    (16384, 8, 256, 7168, synth.PER_ROW_BLOCK128),  # DeepSeek-V3-shaped, full size
])
def test_ragged_sort_bit_exact(T, k, E, D, mode):
    rng = np.random.default_rng(T + E)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    if E > 8:
        ids[ids == 3] = 5  # expert 3 never used
    x_q = rng.integers(0, 256, (T, D)).astype(np.uint8)
    if mode == synth.PER_ROW:
        x_s = rng.uniform(0.1, 2, T).astype(np.float32)
    elif mode == synth.PER_ROW_BLOCK128:
        x_s = rng.uniform(0.1, 2, (T, oracle.nblocks(D))).astype(np.float32)
    else:
        x_s = np.array([0.5], np.float32)
    src, pos, sizes, offs = oracle.ragged_sort(ids, E)
    xs_ref, xss_ref = oracle.gather_rows(x_q, x_s, mode, src, k)
    out = moe.ragged_sort(dev(ids), E, dev(x_q), dev(x_s), mode)
    assert moe.device_error() == 0
    assert np.array_equal(host(out["sorted_src"]), src)
    assert np.array_equal(host(out["pos"]), pos)
    assert np.array_equal(host(out["group_sizes"]), sizes)
    assert np.array_equal(host(out["group_offsets"]), offs)
    assert np.array_equal(host(out["xs_q"]), xs_ref)
    if mode != synth.PER_TENSOR:
        assert np.array_equal(host(out["xs_scale"]), xss_ref)


@pytest.mark.parametrize("T,k,E,D,mode", [
    (1, 1, 1, 16, synth.PER_ROW),
    (7, 2, 16, 128, synth.PER_ROW),           # zero-token experts
    (333, 6, 64, 272, synth.PER_TENSOR),      # D not a multiple of 128
    (1000, 8, 256, 384, synth.PER_ROW_BLOCK128),
    (2500, 2, 8, 4096, synth.PER_ROW),
    (600, 8, 256, 7168, synth.PER_ROW_BLOCK128),
])
def test_quantize_sort_bit_exact(T, k, E, D, mode):
    """Steps 1 + 2 fused: sort indices, gathered codes and scales all match the
    oracle's quantise-then-sort-then-gather."""
    rng = np.random.default_rng(T * 3 + D + mode)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    x = bf16_rows(rng, T, D)
    static = 0.0211
    q_ref, s_ref = oracle.quantize_rows(x, mode, static)
    src, pos, sizes, offs = oracle.ragged_sort(ids, E)
    xs_ref, xss_ref = oracle.gather_rows(q_ref, s_ref, mode, src, k)
    ss = torch.tensor([static], dtype=torch.float32, device="cuda")
    out = moe.quantize_sort(dev(x), dev(ids), E, mode, ss)
    assert moe.device_error() == 0
    assert np.array_equal(host(out["sorted_src"]), src)
    assert np.array_equal(host(out["pos"]), pos)
    assert np.array_equal(host(out["group_sizes"]), sizes)
    assert np.array_equal(host(out["group_offsets"]), offs)
    assert np.array_equal(host(out["xs_q"]), xs_ref)
    if mode != synth.PER_TENSOR:
        assert np.array_equal(host(out["xs_scale"]).view(np.uint32), xss_ref.view(np.uint32))


def test_ragged_sort_bad_id_sets_device_error():
    ids = np.array([[0, 1], [2, 7]], np.int32)  # 7 >= E
    x_q = np.zeros((2, 16), np.uint8)
    moe.ragged_sort(dev(ids), 4, dev(x_q), dev(np.ones(2, np.float32)), synth.PER_ROW)
    assert moe.device_error() & 0x1
    assert moe.device_error() == 0  # cleared


@pytest.mark.parametrize("mode", [synth.PER_ROW, synth.PER_ROW_BLOCK128, synth.PER_TENSOR])
@pytest.mark.parametrize("R,F", [(3, 16), (64, 256), (40, 768), (8, 2048), (2, 14336)])
def test_swiglu_quant_bit_exact(mode, R, F):
    rng = np.random.default_rng(R * 7 + F + mode)
    a = (rng.standard_normal((R, 2 * F)) * np.exp(rng.uniform(-2, 2.5, (R, 1)))).astype(np.float32)
    a[0, :4] = [-95.0, 95.0, -0.0, 1e-30]  # exp overflow / underflow and tiny inputs
    a_b = oracle.bf16_bits(torch.from_numpy(a).to(torch.bfloat16))
    hq_ref, hs_ref, _ = oracle.swiglu_quant(a_b, mode, 0.05)
    hq, hs = moe.swiglu_quant(dev(a_b), mode, torch.tensor([0.05], dtype=torch.float32, device="cuda"))
    assert np.array_equal(host(hq), hq_ref)
    if mode != synth.PER_TENSOR:
        assert np.array_equal(host(hs), hs_ref)


def test_swiglu_exp_matches_cuda_expf_bound():
    """The kernel's own fp32 exponential stays within 2 ulp of CUDA's expf
    (checked through h for a1 = 1: silu values of a sweep of inputs)."""
    z = np.linspace(-30, 30, 8 * 1024).astype(np.float32)
    a = np.stack([z, np.ones_like(z)]).reshape(1, 2, -1).transpose(0, 1, 2).reshape(1, -1)
    a_b = oracle.bf16_bits(torch.from_numpy(a).to(torch.bfloat16))
    zb = torch.from_numpy(oracle.bf16_to_f64(a_b[0, : z.size]).astype(np.float32)).cuda()
    ref = (zb / (1 + torch.exp(-zb))).to(torch.bfloat16).float()
    hq, hs = moe.swiglu_quant(dev(a_b), synth.PER_ROW)
    deq = oracle.e4m3_to_f64(host(hq)[0]) * float(host(hs)[0])
    r = ref.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(deq - r)) <= 0.07 * np.abs(r).max()


@pytest.mark.parametrize("T,k,D", [(1, 1, 8), (256, 2, 128), (100, 8, 7168), (77, 6, 4096), (50, 3, 264),
                                   (40, 12, 264), (10, 32, 128), (2048, 8, 2048)])
def test_combine_matches_oracle(T, k, D):
    rng = np.random.default_rng(T * k + D)
    E = 5
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    src, pos, _, _ = oracle.ragged_sort(ids, E)
    o = oracle.bf16_bits(torch.from_numpy(rng.standard_normal((T * k, D)).astype(np.float32)).to(torch.bfloat16))
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    y_ref = oracle.combine(o, pos, w, k)
    y = moe.ragged_gather_reduce(dev(o), dev(pos), dev(w), k)
    assert_close(host(y), y_ref, "combine")
    # k = 1 with unit weights is an exact inverse permutation
    if k == 1:
        y1 = moe.ragged_gather_reduce(dev(o), dev(pos), None, 1)
        assert np.array_equal(host(y1), o[pos])


def test_combine_bad_position_raises_device_error():
    """A pos entry outside [0, T*k) (a corrupted permutation) contributes
    nothing and sets MOE_DEVERR_BAD_POSITION; the other tokens are exact and
    a following call with a valid permutation leaves the word clear."""
    rng = np.random.default_rng(7)
    T, k, D, E = 64, 2, 256, 4
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    _, pos, _, _ = oracle.ragged_sort(ids, E)
    o = oracle.bf16_bits(torch.from_numpy(rng.standard_normal((T * k, D)).astype(np.float32)).to(torch.bfloat16))
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    y_ref = oracle.combine(o, pos, w, k)
    bad = pos.copy()
    bad[5 * k + 1] = T * k + 3
    assert moe.device_error() == 0
    y = moe.ragged_gather_reduce(dev(o), dev(bad), dev(w), k)
    assert moe.device_error() == 0x10
    yh = host(y)
    others = np.arange(T) != 5
    assert_close(yh[others], y_ref[others], "combine, other tokens")
    # token 5 keeps only its valid row
    y5 = oracle.combine(o[pos[5 * k: 5 * k + 1]], np.array([0], np.int32), w[5:6, :1], 1)
    assert_close(yh[5:6], y5, "combine, token with a bad position")
    y = moe.ragged_gather_reduce(dev(o), dev(pos), dev(w), k)
    assert moe.device_error() == 0
    assert_close(host(y), y_ref, "combine after the bad call")


@pytest.mark.parametrize("T,k,D", [(1, 1, 16), (64, 6, 256), (300, 2, 4096)])
def test_gather_scale_quant_bit_exact(T, k, D):
    rng = np.random.default_rng(T + D)
    E = 7
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    src, pos, _, _ = oracle.ragged_sort(ids, E)
    G = oracle.bf16_bits(torch.from_numpy(rng.standard_normal((T, D)).astype(np.float32)).to(torch.bfloat16))
    w = rng.uniform(0, 1, T * k).astype(np.float32)
    dO_ref = oracle.gather_scale(G, w, src, k)
    q_ref, s_ref = oracle.quantize_rows(dO_ref, synth.PER_ROW)
    dO, q, s = moe.gather_scale_quant(dev(G), dev(w), dev(src), k)
    assert np.array_equal(host(dO), dO_ref)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(host(s), s_ref)


@pytest.mark.parametrize("R,F", [(1, 16), (50, 1408), (7, 4096)])
def test_swiglu_bwd_quant_bit_exact(R, F):
    rng = np.random.default_rng(R + F)
    a = oracle.bf16_bits(torch.from_numpy((rng.standard_normal((R, 2 * F)) * 3).astype(np.float32)).to(torch.bfloat16))
    dH = oracle.bf16_bits(torch.from_numpy(rng.standard_normal((R, F)).astype(np.float32)).to(torch.bfloat16))
    dA_ref = oracle.swiglu_bwd(dH, a)
    q_ref, s_ref = oracle.quantize_rows(dA_ref, synth.PER_ROW)
    dA, q, s = moe.swiglu_bwd_quant(dev(dH), dev(a))
    assert np.array_equal(host(dA), dA_ref)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(host(s), s_ref)


@pytest.mark.parametrize("M,N,E,g0,El", [(1, 16, 1, 0, 1), (300, 256, 9, 0, 9), (1000, 2816, 64, 0, 64),
                                         (500, 96, 8, 2, 4)])
def test_quantize_group_cols_bit_exact(M, N, E, g0, El):
    rng = np.random.default_rng(M + N + E)
    from tests.gpu_helpers import ragged_sizes
    sizes = ragged_sizes(rng, E, M)
    g = oracle.bf16_bits(torch.from_numpy((rng.standard_normal((M, N)) * np.exp(rng.uniform(-3, 3, (1, N)))
                                           ).astype(np.float32)).to(torch.bfloat16))
    q_ref, s_ref = oracle.quantize_group_cols(g, sizes, g0, El)
    q, s = moe.quantize_group_cols(dev(g), dev(sizes), g0, El)
    assert np.array_equal(host(s), s_ref)
    starts = np.concatenate([[0], np.cumsum(sizes)])
    lo, hi = starts[g0], starts[g0 + El]
    assert np.array_equal(host(q)[lo:hi], q_ref[lo:hi])
