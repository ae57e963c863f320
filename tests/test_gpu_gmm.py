"""GPU parity of the tcgen05 grouped matmuls (gmm_fp8, tgmm_fp8) against the
oracle: relative Frobenius <= 2e-3 and max |delta| <= 1e-2 max|ref| after
bf16 rounding, over several tiles, ragged group tails, empty groups, partial
N tiles, K tails and expert-parallel shards."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import assert_close, dev, host, rand_codes, ragged_sizes

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("fp8_quantized_moe_gb300")

R0, RB, RT, GC = synth.PER_ROW, synth.PER_ROW_BLOCK128, synth.PER_TENSOR, synth.PER_GROUP_COL


def make_case(seed, M, K, N, E, amode, wmode, zero_frac=0.25):
    rng = np.random.default_rng(seed)
    sizes = ragged_sizes(rng, E, M, zero_frac)
    a = rand_codes(rng, (M, K))
    w = rand_codes(rng, (E, N, K))
    nb = oracle.nblocks(K)
    sa = {R0: rng.uniform(0.5, 2, M), RB: rng.uniform(0.5, 2, (M, nb)), RT: [0.7]}[amode]
    sw = {R0: rng.uniform(0.5, 2, (E, N)), RB: rng.uniform(0.5, 2, (E, nb, N)), RT: [1.3]}[wmode]
    # scale the scales so that outputs are O(1): e4m3 codes reach 448
    sa = (np.asarray(sa) / 448.0).astype(np.float32)
    sw = (np.asarray(sw) / (448.0 * np.sqrt(K))).astype(np.float32)
    return sizes, a, w, sa, sw


@pytest.mark.parametrize("M,K,N,E,amode,wmode", [
    (128, 128, 256, 1, R0, R0),      # one tile
    (1, 128, 256, 1, R0, R0),        # a single row
    (200, 256, 512, 3, R0, R0),      # ragged groups, several tiles
    (300, 128, 144, 4, R0, R0),      # N not a multiple of the tile
    (257, 48, 256, 2, R0, R0),       # K tail (48 < 128)
    (640, 512, 256, 8, RT, R0),      # static lhs, per-channel rhs
    (640, 512, 256, 8, RT, RT),
    (384, 384, 256, 3, RB, RB),      # blockwise both sides (promotion)
    (384, 384, 512, 5, R0, RB),      # per-row lhs, blockwise rhs
    (256, 256, 128, 2, RB, R0),
    (1500, 1024, 768, 16, R0, R0),
    (2048, 2048, 1536, 128, R0, RB),  # prefill-chunk shaped, E = 128
    (1000, 1024, 272, 7, RB, RB),    # promotion: an N tail of 16 past the 256-column tile
    (600, 7168, 512, 3, RB, RB),     # promotion: K = 7168 (56 K blocks, the scale ring wraps)
    (130, 256, 256, 2, RB, RT),      # per-128 lhs, static rhs
    # K >= 3072 runs on CTA pairs: odd M-tile counts leave the odd CTA past its group
    (700, 4096, 512, 5, R0, R0),
    (129, 3072, 272, 2, RT, R0),     # one pair per group, N tail inside the pair's B halves
    (1, 4096, 256, 1, R0, R0),
])
def test_gmm_matches_oracle(M, K, N, E, amode, wmode):
    sizes, a, w, sa, sw = make_case(M * 31 + K + N + E, M, K, N, E, amode, wmode)
    ref = oracle.gmm(a, sa, amode, w, sw, wmode, sizes)
    out = moe.gmm(dev(a), dev(sa), amode, dev(w), dev(sw), wmode, dev(sizes))
    assert moe.device_error() == 0
    assert_close(host(out), ref, f"gmm M={M} K={K} N={N} E={E}")


def test_gmm_expert_parallel_shard_zeroes_other_rows():
    M, K, N, E = 700, 256, 256, 8
    sizes, a, w, sa, sw = make_case(5, M, K, N, E, R0, R0, zero_frac=0.0)
    g0, El = 2, 3
    ref = oracle.gmm(a, sa, R0, w[g0:g0 + El], sw[g0:g0 + El], R0, sizes, group_offset=g0, E_local=El)
    out = moe.gmm(dev(a), dev(sa), R0, dev(w[g0:g0 + El].copy()), dev(sw[g0:g0 + El].copy()), R0, dev(sizes),
                  group_offset=g0, E_local=El)
    o = host(out)
    starts = np.concatenate([[0], np.cumsum(sizes)])
    lo, hi = starts[g0], starts[g0 + El]
    assert np.all(o[:lo] == 0) and np.all(o[hi:] == 0)
    assert_close(o, ref, "gmm shard")


def test_gmm_pair_expert_parallel_shard():
    M, K, N, E = 900, 4096, 256, 6
    sizes, a, w, sa, sw = make_case(6, M, K, N, E, R0, R0, zero_frac=0.2)
    g0, El = 1, 4
    ref = oracle.gmm(a, sa, R0, w[g0:g0 + El], sw[g0:g0 + El], R0, sizes, group_offset=g0, E_local=El)
    out = moe.gmm(dev(a), dev(sa), R0, dev(w[g0:g0 + El].copy()), dev(sw[g0:g0 + El].copy()), R0, dev(sizes),
                  group_offset=g0, E_local=El)
    assert moe.device_error() == 0
    assert_close(host(out), ref, "gmm pair shard")


@pytest.mark.parametrize("M,K,N,E,K_split,amode,shard", [
    (700, 768, 512, 5, 384, R0, None),
    (640, 2816, 272, 8, 1408, R0, None),      # the backward's K = 2F, K_split = F; N tail
    (300, 512, 256, 3, 0, RT, None),          # one segment only (the second)
    (300, 512, 256, 3, 512, R0, None),        # one segment only (the first)
    (900, 1024, 256, 6, 512, R0, (1, 4)),     # expert-parallel shard
])
def test_gmm_ksplit_matches_oracle(M, K, N, E, K_split, amode, shard):
    """Two K segments with one static weight scale each equal the blockwise-scaled
    gmm whose K blocks carry s0 before K_split and s1 after."""
    sizes, a, w, sa, _ = make_case(M + K + N + K_split, M, K, N, E, amode, RT, zero_frac=0.2)
    g0, El = shard if shard else (0, E)
    w = np.ascontiguousarray(w[g0:g0 + El])
    s0, s1 = np.float32(0.7 / (448 * np.sqrt(K))), np.float32(1.9 / (448 * np.sqrt(K)))
    nb = K // 128
    sw_blk = np.empty((El, nb, N), np.float32)
    sw_blk[:, :K_split // 128] = s0
    sw_blk[:, K_split // 128:] = s1
    ref = oracle.gmm(a, sa, amode, w, sw_blk, RB, sizes, group_offset=g0, E_local=El)
    out = moe.gmm_ksplit(dev(a), dev(sa), amode, dev(w), dev(np.array([s0, s1], np.float32)), K_split, dev(sizes),
                         group_offset=g0, E_local=El)
    assert moe.device_error() == 0
    o = host(out)
    if shard:
        starts = np.concatenate([[0], np.cumsum(sizes)])
        lo, hi = starts[g0], starts[g0 + El]
        assert np.all(o[:lo] == 0) and np.all(o[hi:] == 0)
    assert_close(o, ref, f"gmm_ksplit M={M} K={K} N={N} K_split={K_split}")


def test_gmm_bad_group_sizes_sets_device_error():
    M, K, N = 64, 128, 256
    a = np.zeros((M, K), np.uint8)
    w = np.zeros((2, N, K), np.uint8)
    sizes = np.array([10, 20], np.int32)  # sums to 30 != 64
    moe.gmm(dev(a), dev(np.ones(M, np.float32)), R0, dev(w), dev(np.ones((2, N), np.float32)), R0, dev(sizes))
    assert moe.device_error() & 0x2


def test_gmm_accumulation_over_long_k():
    """K = 14336 (the wo projection of the Mixtral-shaped layer): fp32
    accumulation on the tensor cores must stay within the tolerance."""
    M, K, N, E = 256, 14336, 256, 2
    sizes, a, w, sa, sw = make_case(11, M, K, N, E, R0, R0, zero_frac=0.0)
    ref = oracle.gmm(a, sa, R0, w, sw, R0, sizes)
    out = moe.gmm(dev(a), dev(sa), R0, dev(w), dev(sw), R0, dev(sizes))
    assert_close(host(out), ref, "gmm long K")


@pytest.mark.parametrize("M,K,N,E,lmode,rmode", [
    (128, 128, 256, 1, RT, RT),
    (300, 256, 512, 4, RT, GC),
    (1000, 384, 256, 9, GC, GC),
    (2000, 128, 2816, 16, RT, GC),
])
def test_tgmm_matches_oracle(M, K, N, E, lmode, rmode):
    rng = np.random.default_rng(M + K + N)
    sizes = ragged_sizes(rng, E, M)
    x = rand_codes(rng, (M, K))
    g = rand_codes(rng, (M, N))
    sx = np.array([0.01], np.float32) if lmode == RT else rng.uniform(0.5, 2, (E, K)).astype(np.float32) / 448
    sg = np.array([0.02], np.float32) if rmode == RT else rng.uniform(0.5, 2, (E, N)).astype(np.float32) / 448
    ref = oracle.tgmm(x, sx, lmode, g, sg, rmode, sizes)
    out = moe.tgmm(dev(x), dev(sx), lmode, dev(g), dev(sg), rmode, dev(sizes))
    assert moe.device_error() == 0
    o = host(out)
    for e in np.flatnonzero(sizes == 0):
        assert np.all(o[e] == 0)
    assert_close(o, ref, f"tgmm M={M} K={K} N={N} E={E}")


@pytest.mark.parametrize("sizes,K,N,g0,El,rmode", [
    ([3000, 0, 150, 1100, 40, 900, 260], 256, 512, 0, 7, GC),  # heavy groups (>= 8 K blocks) beside light, empty ones
    ([200, 2500, 1300, 0, 90, 1200], 128, 272, 1, 4, RT),       # a shard of groups 1..4
])
def test_tgmm_heavy_and_light_groups(sizes, K, N, g0, El, rmode):
    """Groups with many 128-row blocks (long K loops of the contraction over
    rows) beside light and empty groups, in the expert-major tile order; every
    expert's result must match the oracle."""
    sizes = np.array(sizes, np.int32)
    M = int(sizes.sum())
    rng = np.random.default_rng(M + K + N)
    x = rand_codes(rng, (M, K))
    g = rand_codes(rng, (M, N))
    sx = np.array([0.01], np.float32)
    E = len(sizes)
    sg_full = rng.uniform(0.5, 2, (E, N)).astype(np.float32) / 448 if rmode == GC else np.array([0.02], np.float32)
    ref = oracle.tgmm(x, sx, RT, g, sg_full, rmode, sizes)[g0:g0 + El]
    sg = sg_full[g0:g0 + El] if rmode == GC else sg_full
    out = moe.tgmm(dev(x), dev(sx), RT, dev(g), dev(np.ascontiguousarray(sg)), rmode, dev(sizes), group_offset=g0,
                   E_local=El)
    assert moe.device_error() == 0
    o = host(out)
    for e in np.flatnonzero(sizes[g0:g0 + El] == 0):
        assert np.all(o[e] == 0)
    assert_close(o, ref, f"tgmm heavy/light {sizes.tolist()} shard {g0}+{El}")


@pytest.mark.parametrize("M,K,N,E,g0,El", [
    (1000, 384, 256, 9, 0, 9),
    (2000, 128, 2816, 16, 0, 16),
    (700, 256, 272, 6, 1, 4),          # shard, N not a multiple of 128
    (1, 128, 128, 1, 0, 1),
])
def test_tgmm_gcq_equals_quantize_then_tgmm(M, K, N, E, g0, El):
    """Codes made in the transposed layout: the same result, bit for bit, as
    moe_quantize_group_cols followed by tgmm_fp8."""
    rng = np.random.default_rng(M + K + N + El)
    sizes = ragged_sizes(rng, E, M)
    x = rand_codes(rng, (M, K))
    g = oracle.bf16_bits(torch.from_numpy((rng.standard_normal((M, N)) * np.exp(rng.uniform(-3, 3, (1, N)))
                                           ).astype(np.float32)).to(torch.bfloat16))
    sx = np.array([0.01], np.float32)
    gq, gs = moe.quantize_group_cols(dev(g), dev(sizes), g0, El)
    ref = moe.tgmm(dev(x), dev(sx), RT, gq, gs, GC, dev(sizes), group_offset=g0, E_local=El)
    _, gs2 = moe.quantize_group_cols(dev(g), dev(sizes), g0, El, scales_only=True)
    out = moe.tgmm_gcq(dev(x), dev(sx), RT, dev(g), gs2, dev(sizes), group_offset=g0, E_local=El)
    assert moe.device_error() == 0
    assert torch.equal(gs, gs2)
    assert torch.equal(out, ref)


# ---- gmm_fp8_swiglu: steps 3 + 4 fused, bit-identical to gmm_fp8 + moe_swiglu_quant

@pytest.mark.parametrize("M,K,F,E,amode,wmode,hmode,shard", [
    (300, 256, 256, 4, R0, R0, R0, None),
    (300, 256, 256, 4, R0, R0, RB, None),
    (640, 512, 384, 8, RT, RT, RT, None),
    (640, 512, 384, 8, RT, R0, RT, None),
    (1, 128, 128, 1, R0, R0, R0, None),
    (1000, 512, 384, 9, R0, R0, R0, (2, 4)),
    (1000, 512, 384, 9, R0, RT, RB, (3, 5)),
    # K >= 3072: CTA pairs
    (700, 4096, 256, 5, R0, R0, R0, None),
    (700, 4096, 256, 5, RT, RT, RT, (1, 3)),
    (450, 3072, 384, 3, R0, R0, RB, None),
    # a blockwise operand scale: the promotion kernel with the SwiGLU epilogue
    (384, 384, 256, 3, RB, RB, RB, None),      # DeepSeek-V3 style: per-128 x, h and blockwise weights
    (700, 1024, 384, 6, RB, RB, RB, (1, 4)),
    (700, 1024, 256, 5, R0, RB, R0, None),     # prefill style: per-token x and h, blockwise weights
    (300, 256, 128, 2, RB, R0, RB, None),
    (640, 512, 384, 8, RB, RB, RT, None),
    (1, 128, 128, 1, RB, RB, RB, None),
])
def test_gmm_swiglu_equals_gmm_then_swiglu(M, K, F, E, amode, wmode, hmode, shard):
    sizes, a, w, sa, sw = make_case(M + K + F + E + hmode, M, K, 2 * F, E, amode, wmode, zero_frac=0.2)
    g0, El = shard if shard else (0, E)
    w = np.ascontiguousarray(w[g0:g0 + El])
    if wmode in (R0, RB):
        sw = np.ascontiguousarray(sw[g0:g0 + El])
    # give a0/a1 a realistic O(1..5) spread so that silu and the scales are exercised
    sa = (sa * 4).astype(np.float32)
    hs = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    sz = dev(sizes)
    a_ref = moe.gmm(dev(a), dev(sa), amode, dev(w), dev(sw), wmode, sz, group_offset=g0, E_local=El)
    hq_ref, hs_ref = moe.swiglu_quant(a_ref, hmode, hs)
    hq, hsc, a_out = moe.gmm_swiglu(dev(a), dev(sa), amode, dev(w), dev(sw), wmode, sz, hmode, hs,
                                    group_offset=g0, E_local=El, keep_a=True)
    assert moe.device_error() == 0
    starts = np.concatenate([[0], np.cumsum(sizes)])
    lo, hi = starts[g0], starts[g0 + El]
    assert np.array_equal(host(a_out)[lo:hi], host(a_ref)[lo:hi])
    assert np.array_equal(host(hq), host(hq_ref))
    if hmode != RT:
        assert np.array_equal(host(hsc), host(hs_ref))
    # and against the oracle, from the oracle's own a
    a_or = oracle.gmm(a, sa, amode, w, sw, wmode, sizes, group_offset=g0, E_local=El)
    assert_close(host(a_out)[lo:hi], a_or[lo:hi], "gmm_swiglu a")


def test_bounded_wait_timeout_reports_and_recovers():
    """The failure path of the tensor-core kernels: the epilogue waits on a
    barrier that nothing arrives on (a test hook) with a 200 us limit; the
    kernel stops, drains what it issued, frees its tensor memory and sets
    MOE_DEVERR_TIMEOUT.  The context stays usable: the next call is exact.
    Also covers a kernel that had already issued loads and MMAs when the
    wait ran out (several tiles per CTA)."""
    lib = moe.lib()
    for M, K, N, E in [(256, 256, 512, 2), (8192, 512, 2048, 8)]:
        sizes, a, w, sa, sw = make_case(M + K, M, K, N, E, R0, R0)
        args = (dev(a), dev(sa), R0, dev(w), dev(sw), R0, dev(sizes))
        assert moe.device_error() == 0
        lib.moe_test_stall_epilogue(200_000)
        try:
            moe.gmm(*args)
            assert moe.device_error() == 0x4  # MOE_DEVERR_TIMEOUT
        finally:
            lib.moe_test_stall_epilogue(0)
        out = moe.gmm(*args)
        assert moe.device_error() == 0
        assert_close(host(out), oracle.gmm(a, sa, R0, w, sw, R0, sizes), "gmm after a timed-out call")
