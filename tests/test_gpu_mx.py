"""GPU parity of the MXFP8 variant against the oracle.

MXFP8 (OCP MX v1.0): blocks of 32 e4m3 values along the contracted dimension
share one E8M0 power-of-two scale.  Parity rules:
- the quantisers (plain rows, fused into the sort, SwiGLU) give bit-exact
  codes and E8M0 codes;
- the block-scaled grouped matmuls are within relative Frobenius 2e-3 and
  max |delta| <= 1e-2 max|ref| after bf16 rounding;
- the fused SwiGLU epilogue's codes are bit-exact against the oracle fed the
  GPU's own a.
Cases cover several tiles, ragged groups, empty groups, N tails, long K and
expert-parallel shards."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import assert_close, dev, host, rand_codes, ragged_sizes

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("fp8_quantized_moe_gb300")


def sf_rows(sf) -> np.ndarray:
    """The library's K-block-major E8M0 codes [K/128, rows, 4] -> the
    oracle's row-major [rows, K/32] (pure data movement)."""
    a = host(sf) if isinstance(sf, torch.Tensor) else np.asarray(sf)
    kb, rows, _ = a.shape
    return np.ascontiguousarray(a.transpose(1, 0, 2).reshape(rows, 4 * kb))


def sf_kmajor(sf) -> np.ndarray:
    """Row-major E8M0 codes [rows, K/32] -> the library's [K/128, rows, 4]."""
    rows, nb = sf.shape
    return np.ascontiguousarray(sf.reshape(rows, nb // 4, 4).transpose(1, 0, 2))


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def mx_rows(rng, rows, cols):
    """bf16 rows whose 32-column blocks span many binades, with the special
    blocks of the format: zeros, values that saturate (amax mantissa above
    1.75), ties of e4m3 rounding, tiny amax that clamps the scale."""
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x *= np.repeat(np.ldexp(1.0, rng.integers(-40, 40, (rows, cols // 32))), 32, axis=1).astype(np.float32)
    nb = cols // 32
    for r in range(rows):
        b = rng.integers(0, nb)
        kind = r % 5
        blk = x[r, 32 * b:32 * b + 32]
        if kind == 0:
            blk[:] = 0.0
        elif kind == 1:
            blk[0] = 1.9375 * 2.0 ** int(rng.integers(-10, 10))  # saturates to 448
        elif kind == 2:
            blk[:] = [1.0625, 1.1875, 0.53125, -0.59375] * 8  # ties at X = -8
        elif kind == 3:
            blk[:] *= np.float32(2.0 ** -100)  # amax far below 2^-119: X clamps to -127
    x[rng.random((rows, cols)) < 0.02] = 0.0
    return bf16(x)


# ------------------------------------------------------------ quantisers ----

@pytest.mark.parametrize("rows,cols", [(1, 128), (37, 4096), (64, 7168), (9, 14336), (300, 384)])
def test_quantize_rows_mx_bit_exact(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    xb = mx_rows(rng, rows, cols)
    q_ref, sf_ref = oracle.quantize_rows_mx(xb)
    q, sf = moe.quantize_rows_mx(dev(xb))
    assert tuple(sf.shape) == (cols // 128, rows, 4)
    assert np.array_equal(host(q), q_ref)
    assert np.array_equal(sf_rows(sf), sf_ref)


def test_quantize_weights_mx_layout():
    rng = np.random.default_rng(3)
    w = bf16(rng.standard_normal((5, 48, 256)).astype(np.float32) * 0.02)
    q_ref, sf_ref = oracle.quantize_weights_mx(w)
    q, sf = moe.quantize_weights_mx(dev(w))
    assert tuple(sf.shape) == (2, 5 * 48, 4)
    assert np.array_equal(host(q), q_ref) and np.array_equal(sf_rows(sf).reshape(5, 48, 8), sf_ref)


@pytest.mark.parametrize("T,k,E,D", [(1, 1, 1, 128), (256, 2, 4, 128), (333, 8, 64, 7168), (1024, 6, 24, 4096)])
def test_quantize_sort_mx_bit_exact(T, k, E, D):
    rng = np.random.default_rng(T + k + E + D)
    xb = mx_rows(rng, T, D)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    src, pos, sizes, offsets = oracle.ragged_sort(ids, E)
    xq, xsf = oracle.quantize_rows_mx(xb)
    xs_q, xs_sf = oracle.gather_rows_mx(xq, xsf, src, k)
    o = moe.quantize_sort_mx(dev(xb), dev(ids), E)
    assert moe.device_error() == 0
    assert np.array_equal(host(o["sorted_src"]), src) and np.array_equal(host(o["pos"]), pos)
    assert np.array_equal(host(o["group_sizes"]), sizes) and np.array_equal(host(o["group_offsets"]), offsets)
    assert np.array_equal(host(o["xs_q"]), xs_q)
    assert np.array_equal(sf_rows(o["xs_scale"]), xs_sf)


@pytest.mark.parametrize("R,F", [(1, 128), (300, 128), (77, 2048), (16, 14336)])
def test_swiglu_quant_mx_bit_exact(R, F):
    rng = np.random.default_rng(R + F)
    a = rng.standard_normal((R, 2 * F)).astype(np.float32) * 3
    a[rng.random((R, 2 * F)) < 0.05] = 0.0
    a[:, :32] *= np.float32(1e-3)
    ab = bf16(a)
    hq_ref, hsf_ref, _ = oracle.swiglu_quant_mx(ab)
    hq, hsf = moe.swiglu_quant_mx(dev(ab))
    assert np.array_equal(host(hq), hq_ref)
    assert np.array_equal(sf_rows(hsf), hsf_ref)


# ------------------------------------------------------------------ gmm ----

def mx_args(a, asf, w, wsf, sizes):
    """Device arguments of gmm_mx from the oracle-layout case."""
    El, N, K = w.shape
    return (dev(a), dev(sf_kmajor(asf)), dev(w), dev(sf_kmajor(wsf.reshape(El * N, K // 32))), dev(sizes))


def make_mx_case(seed, M, K, N, E, zero_frac=0.25):
    rng = np.random.default_rng(seed)
    sizes = ragged_sizes(rng, E, M, zero_frac)
    a = rand_codes(rng, (M, K))
    w = rand_codes(rng, (E, N, K))
    # E8M0 codes around 2^-8 (lhs) and 2^-8 / sqrt(K) (rhs), so outputs are O(1)
    ka = int(round(np.log2(np.sqrt(K))))
    asf = rng.integers(116, 123, (M, K // 32)).astype(np.uint8)
    wsf = rng.integers(116 - ka, 123 - ka, (E, N, K // 32)).astype(np.uint8)
    return sizes, a, asf, w, wsf


@pytest.mark.parametrize("M,K,N,E", [
    (128, 128, 256, 1),       # one tile, one stage
    (1, 128, 256, 1),         # a single row
    (200, 256, 512, 3),       # ragged groups, several tiles
    (300, 128, 144, 4),       # N not a multiple of the tile
    (1000, 1024, 272, 7),     # an N tail of 16 past the 256-column tile
    (600, 7168, 512, 3),      # K = 7168: 56 stages, the stage ring wraps many times
    (700, 4096, 512, 5),
    (2048, 2048, 1536, 128),  # E = 128 experts, many empty or short groups
    (129, 384, 256, 2),       # a group of 1 row past a full tile
    (129, 3072, 272, 2),      # a one-row group, an N tail
    (1, 4096, 256, 1),
    (3000, 3072, 768, 24),    # many groups, several tiles per group
])
def test_gmm_mx_matches_oracle(M, K, N, E):
    sizes, a, asf, w, wsf = make_mx_case(M * 31 + K + N + E, M, K, N, E)
    ref = oracle.gmm_mx(a, asf, w, wsf, sizes)
    out = moe.gmm_mx(*mx_args(a, asf, w, wsf, sizes))
    assert moe.device_error() == 0
    assert_close(host(out), ref, f"gmm_mx M={M} K={K} N={N} E={E}")


def test_gmm_mx_block_scales_are_per_32_columns():
    # one lhs block scaled by 2^20 and one rhs block by 2^-20 in different
    # K blocks: a scale applied to the wrong block changes the output by far
    # more than the tolerance
    sizes, a, asf, w, wsf = make_mx_case(5, 256, 512, 256, 2, zero_frac=0)
    asf[:, 5] = np.minimum(asf[:, 5].astype(int) + 20, 254).astype(np.uint8)
    wsf[:, :, 9] = np.maximum(wsf[:, :, 9].astype(int) - 20, 1).astype(np.uint8)
    ref = oracle.gmm_mx(a, asf, w, wsf, sizes)
    out = moe.gmm_mx(*mx_args(a, asf, w, wsf, sizes))
    assert moe.device_error() == 0
    assert_close(host(out), ref, "gmm_mx with outlier blocks")


@pytest.mark.parametrize("K", [512, 4096])
def test_gmm_mx_expert_parallel_shard(K):
    M, N, E = 1000, 384, 9
    sizes, a, asf, w, wsf = make_mx_case(17 + K, M, K, N, E, zero_frac=0.2)
    g0, El = 2, 4
    w, wsf = np.ascontiguousarray(w[g0:g0 + El]), np.ascontiguousarray(wsf[g0:g0 + El])
    ref = oracle.gmm_mx(a, asf, w, wsf, sizes, group_offset=g0, E_local=El)
    out = host(moe.gmm_mx(*mx_args(a, asf, w, wsf, sizes), group_offset=g0, E_local=El))
    assert moe.device_error() == 0
    starts = np.concatenate([[0], np.cumsum(sizes)])
    lo, hi = starts[g0], starts[g0 + El]
    assert not out[:lo].any() and not out[hi:].any()
    assert_close(out[lo:hi], ref[lo:hi], "gmm_mx shard")


@pytest.mark.parametrize("M,K,F,E,shard", [
    (256, 256, 128, 2, None),
    (700, 512, 384, 5, None),
    (1000, 7168, 256, 8, None),
    (1, 128, 128, 1, None),
    (1000, 512, 384, 9, (3, 5)),
    (700, 4096, 256, 5, None),
    (1000, 3072, 384, 9, (2, 4)),
    (1, 4096, 128, 1, None),
])
def test_gmm_mx_swiglu_stagewise(M, K, F, E, shard):
    """a against the oracle's MX gmm; h codes and E8M0 codes bit-exact
    against the oracle's MX SwiGLU requantisation of the GPU's own a, and
    bit-identical to gmm_mx followed by swiglu_quant_mx on the GPU."""
    sizes, a, asf, w, wsf = make_mx_case(M + K + F + E, M, K, 2 * F, E, zero_frac=0.2)
    asf = (asf.astype(int) + 2).astype(np.uint8)  # a0, a1 of O(1..5): exercises silu's range
    g0, El = shard if shard else (0, E)
    w, wsf = np.ascontiguousarray(w[g0:g0 + El]), np.ascontiguousarray(wsf[g0:g0 + El])
    args = mx_args(a, asf, w, wsf, sizes)
    hq, hsf, a_out = moe.gmm_mx_swiglu(*args, group_offset=g0, E_local=El, keep_a=True)
    assert moe.device_error() == 0
    starts = np.concatenate([[0], np.cumsum(sizes)])
    lo, hi = starts[g0], starts[g0 + El]
    a_gpu = host(a_out)[lo:hi]
    a_or = oracle.gmm_mx(a, asf, w, wsf, sizes, group_offset=g0, E_local=El)
    assert_close(a_gpu, a_or[lo:hi], "gmm_mx_swiglu a")
    hq_ref, hsf_ref, _ = oracle.swiglu_quant_mx(a_gpu)
    hq_h, hsf_h = host(hq), sf_rows(hsf)
    assert np.array_equal(hq_h[lo:hi], hq_ref)
    assert np.array_equal(hsf_h[lo:hi], hsf_ref)
    # rows outside the local groups: zero codes, E8M0 code 0
    assert not hq_h[:lo].any() and not hq_h[hi:].any()
    assert not hsf_h[:lo].any() and not hsf_h[hi:].any()
    # the unfused path on the GPU gives the same bytes
    a_unf = moe.gmm_mx(*args, group_offset=g0, E_local=El)
    hq_u, hsf_u = moe.swiglu_quant_mx(a_unf)
    assert np.array_equal(host(a_unf)[lo:hi], a_gpu)
    assert np.array_equal(host(hq_u), hq_h) and np.array_equal(sf_rows(hsf_u), hsf_h)


def test_gmm_mx_bounded_wait_timeout_reports_and_recovers():
    """The failure path of the block-scaled kernel: with the epilogue held on
    a barrier nothing arrives on (200 us limit), the scale gatherer, the
    producer and the MMA issuer stop, every copy in flight lands, tensor
    memory is freed and MOE_DEVERR_TIMEOUT is raised; the next call is exact."""
    lib = moe.lib()
    for M, K, N, E in [(4096, 512, 1024, 8), (2048, 4096, 512, 4)]:  # short and long K loops
        sizes, a, asf, w, wsf = make_mx_case(23 + K, M, K, N, E)
        args = mx_args(a, asf, w, wsf, sizes)
        assert moe.device_error() == 0
        lib.moe_test_stall_epilogue(200_000)
        try:
            moe.gmm_mx(*args)
            assert moe.device_error() == 0x4  # MOE_DEVERR_TIMEOUT
        finally:
            lib.moe_test_stall_epilogue(0)
        out = moe.gmm_mx(*args)
        assert moe.device_error() == 0
        assert_close(host(out), oracle.gmm_mx(a, asf, w, wsf, sizes), f"gmm_mx after a timed-out call (K={K})")


# ------------------------------------------------------------------ FFN ----

def test_ffn_mx_small_matches_oracle():
    """Every stage against the oracle fed the GPU's previous-stage output;
    the composed chain within 5e-3."""
    cfg = synth.scaled(synth.CONFIGS["dsv3_mx"], T=256, D=384, E=16, k=4, F=256)
    x_t = synth.activations(cfg, 0)
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    xb, wib, wob = (oracle.bf16_bits(t) for t in (x_t, w_in, w_out))
    wq = oracle.prepare_weights_mx(wib, wob)
    ref = oracle.ffn_forward_mx(xb, ids, w, wq, cfg.E)
    W = moe.prepare_weights(dev(wib), dev(wob), synth.MX32)
    assert np.array_equal(host(W.w_in), wq[0]) and np.array_equal(sf_rows(W.s_in), wq[1].reshape(-1, cfg.D // 32))
    assert np.array_equal(host(W.w_out), wq[2]) and np.array_equal(sf_rows(W.s_out), wq[3].reshape(-1, cfg.F // 32))
    buf = moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, synth.MX32, "cuda")
    buf.keep_a = True
    y = moe.ffn_forward(dev(xb), dev(ids), dev(w), W, synth.MX32, buf)
    assert moe.device_error() == 0
    s = buf.sort
    assert np.array_equal(host(s["xs_q"]), ref["xs_q"]) and np.array_equal(sf_rows(s["xs_scale"]), ref["xs_sf"])
    sizes = ref["sizes"]
    a_gpu = host(buf.a)
    assert_close(a_gpu, ref["a"], "a")
    hq_ref, hsf_ref, _ = oracle.swiglu_quant_mx(a_gpu)
    assert np.array_equal(host(buf.h_q), hq_ref) and np.array_equal(sf_rows(buf.h_s), hsf_ref)
    o_stage = oracle.gmm_mx(host(buf.h_q), sf_rows(buf.h_s), wq[2], wq[3], sizes)
    assert_close(host(buf.o), o_stage, "o (stage)")
    y_stage = oracle.combine(host(buf.o), ref["pos"], w, cfg.k)
    assert_close(host(y), y_stage, "y (stage)")
    assert_close(host(y), ref["y"], "y (composed)", rel_fro=5e-3)


@pytest.mark.parametrize("name", ["dsv3_mx", "mixtral_mx"])
def test_ffn_mx_full_size_sampled_tokens(name):
    """The full-size MXFP8 layers in the benchmark's launch configuration, on
    sampled tokens that the oracle evaluates one by one: the token's codes
    bit-exact, a within 2e-3, h codes of the GPU's a bit-exact, o of the
    GPU's h and y of the GPU's o within 2e-3, the composed y within 5e-3."""
    cfg = synth.CONFIGS[name]
    x_t = synth.activations(cfg, 0, device="cuda")
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0, device="cuda")
    W = moe.prepare_weights(w_in, w_out, synth.MX32)
    buf = moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, synth.MX32, "cuda")
    buf.keep_a = True
    y = moe.ffn_forward(x_t, dev(ids), dev(w), W, synth.MX32, buf)
    assert moe.device_error() == 0
    yh, xb, pos = host(y), host(x_t), host(buf.sort["pos"])
    rng = np.random.default_rng(2)
    tokens = rng.choice(cfg.T, 3, replace=False)
    ys, ys_stage = [], []
    one = np.array([1], np.int32)
    for t in tokens:
        xq, xsf = oracle.quantize_rows_mx(xb[t:t + 1])
        acc = np.zeros(cfg.D)
        o_rows = []
        for j in range(cfg.k):
            e = int(ids[t, j])
            r = int(pos[t * cfg.k + j])
            assert np.array_equal(host(buf.sort["xs_q"][r:r + 1]), xq)
            assert np.array_equal(host(buf.sort["xs_scale"][:, r]).reshape(1, -1), xsf)
            qin, sin, qo, so = oracle.prepare_weights_mx(host(w_in[e:e + 1]), host(w_out[e:e + 1]))
            a = oracle.gmm_mx(xq, xsf, qin, sin, one)
            a_gpu = host(buf.a[r:r + 1])
            assert_close(a_gpu, a, f"{name}: a[t={t}, j={j}]")
            hq_ref, hsf_ref, _ = oracle.swiglu_quant_mx(a_gpu)
            hq_gpu, hsf_gpu = host(buf.h_q[r:r + 1]), host(buf.h_s[:, r]).reshape(1, -1)
            assert np.array_equal(hq_gpu, hq_ref) and np.array_equal(hsf_gpu, hsf_ref)
            o_stage = oracle.gmm_mx(hq_gpu, hsf_gpu, qo, so, one)
            o_gpu = host(buf.o[r:r + 1])
            assert_close(o_gpu, o_stage, f"{name}: o[t={t}, j={j}] (stage)")
            hq_c, hsf_c, _ = oracle.swiglu_quant_mx(a)
            o_c = oracle.gmm_mx(hq_c, hsf_c, qo, so, one)
            acc += float(w[t, j]) * oracle.bf16_to_f64(o_c)[0]
            o_rows.append(o_gpu[0])
        ys.append(oracle.f64_to_bf16(acc))
        ys_stage.append(oracle.combine(np.stack(o_rows), np.arange(cfg.k, dtype=np.int32), w[t:t + 1], cfg.k)[0])
    assert_close(yh[tokens], np.stack(ys_stage), f"{name}: y sampled (stage)")
    assert_close(yh[tokens], np.stack(ys), f"{name}: y sampled (composed)", rel_fro=5e-3)
