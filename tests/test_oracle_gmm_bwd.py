"""Pins of the oracle's grouped matmuls, combine, SwiGLU and backward pass
(CPU only): dense-matmul special cases, brute force without the sort,
adjoint identities and central finite differences."""

import numpy as np
import pytest
import torch

import oracle
import synth


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def deq_rows(q, s, mode):
    v = oracle.e4m3_to_f64(q)
    if mode == synth.PER_ROW:
        return v * s.astype(np.float64)[:, None]
    if mode == synth.PER_ROW_BLOCK128:
        return v * np.repeat(s.astype(np.float64), 128, axis=1)[:, : v.shape[1]]
    return v * float(s[0])


def deq_weights(q, s, mode):
    v = oracle.e4m3_to_f64(q)  # [E, N, K]
    if mode == synth.PER_ROW:
        return v * s.astype(np.float64)[:, :, None]
    if mode == synth.PER_ROW_BLOCK128:
        sb = np.repeat(s.astype(np.float64).transpose(0, 2, 1), 128, axis=2)[:, :, : v.shape[2]]
        return v * sb
    return v * float(s[0])


def rand_codes(rng, shape):
    c = rng.integers(0, 0x7F, shape).astype(np.uint8)
    return c | (rng.integers(0, 2, shape).astype(np.uint8) << 7)


# ---------------------------------------------------------------- gmm ------

@pytest.mark.parametrize("amode,wmode", [(0, 0), (1, 1), (0, 1), (2, 2), (1, 0)])
def test_gmm_single_group_is_dense_matmul(amode, wmode):
    rng = np.random.default_rng(10 + amode * 3 + wmode)
    M, K, N = 37, 384, 48
    a = rand_codes(rng, (M, K))
    w = rand_codes(rng, (1, N, K))
    sa = {0: rng.uniform(0.5, 2, M), 1: rng.uniform(0.5, 2, (M, 3)), 2: [0.75]}[amode]
    sw = {0: rng.uniform(0.5, 2, (1, N)), 1: rng.uniform(0.5, 2, (1, 3, N)), 2: [1.25]}[wmode]
    sa = np.asarray(sa, np.float32)
    sw = np.asarray(sw, np.float32)
    out = oracle.gmm(a, sa, amode, w, sw, wmode, np.array([M], np.int32), want="f64")
    ref = deq_rows(a, sa, amode) @ deq_weights(w, sw, wmode)[0].T  # numpy dense matmul
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    ob = oracle.gmm(a, sa, amode, w, sw, wmode, np.array([M], np.int32))
    assert np.array_equal(ob, oracle.f64_to_bf16(out))


def test_gmm_groups_offset_and_zero_groups():
    rng = np.random.default_rng(20)
    K, N = 256, 32
    sizes = np.array([5, 0, 17, 9, 0, 3], np.int32)
    M = int(sizes.sum())
    a = rand_codes(rng, (M, K))
    sa = rng.uniform(0.5, 2, M).astype(np.float32)
    w = rand_codes(rng, (6, N, K))
    sw = rng.uniform(0.5, 2, (6, N)).astype(np.float32)
    out = oracle.gmm(a, sa, 0, w, sw, 0, sizes, want="f64")
    A = deq_rows(a, sa, 0)
    W = deq_weights(w, sw, 0)
    start = 0
    for e, sz in enumerate(sizes):
        mag = np.abs(A[start:start + sz]) @ np.abs(W[e]).T  # sum of |terms| bounds the rounding
        assert np.all(np.abs(out[start:start + sz] - A[start:start + sz] @ W[e].T) <= 1e-13 * mag)
        start += sz
    # expert-parallel shard: groups [2, 5) only; rows of other groups are zero
    part = oracle.gmm(a, sa, 0, w[2:5], sw[2:5], 0, sizes, group_offset=2, E_local=3, want="f64")
    lo, hi = 5, 5 + 17 + 9
    assert np.all(part[:lo] == 0) and np.all(part[hi:] == 0)
    np.testing.assert_allclose(part[lo:hi], out[lo:hi], rtol=0, atol=0)
    # removing a zero-token group changes no row
    keep = [0, 2, 3, 4, 5]
    out2 = oracle.gmm(a, sa, 0, w[keep], sw[keep], 0, sizes[keep], want="f64")
    assert np.array_equal(out2, out)
    # row sampling returns the same rows
    rows = np.array([30, 0, 7, 22], np.int64)
    samp = oracle.gmm(a, sa, 0, w, sw, 0, sizes, rows=rows, want="f64")
    assert np.array_equal(samp, out[rows])


# ----------------------------------------------------------- whole FFN -----

def brute_force_ffn(x_bits, ids, topw, wq, act_mode, static):
    """Per token, a dense FFN over its k experts with no sort and no gather."""
    qin, sin, min_, qo, so, mo = wq
    Win = deq_weights(qin, sin, min_)
    Wout = deq_weights(qo, so, mo)
    T, D = x_bits.shape
    k = ids.shape[1]
    sx = static["x"] if static else 1.0
    sh = static["h"] if static else 1.0
    y = np.empty((T, D), np.uint16)
    for t in range(T):
        xq, xs = oracle.quantize_rows(x_bits[t:t + 1], act_mode, sx)
        xd = deq_rows(xq, xs, act_mode)
        acc = np.zeros(D)
        for j in range(k):
            e = ids[t, j]
            a = oracle.f64_to_bf16(xd @ Win[e].T)
            hq, hs, _ = oracle.swiglu_quant(a, act_mode, sh)
            o = oracle.f64_to_bf16(deq_rows(hq, hs, act_mode) @ Wout[e].T)
            acc += float(topw[t, j]) * oracle.bf16_to_f64(o)[0]
        y[t] = oracle.f64_to_bf16(acc)
    return y


@pytest.mark.parametrize("name", ["tiny", "dsv3", "prefill", "fwdbwd"])
def test_ffn_forward_equals_brute_force(name):
    base = synth.CONFIGS[name]
    cfg = synth.scaled(base, T=24, D=256, E=min(base.E, 6), F=256)
    x = oracle.bf16_bits(synth.activations(cfg, 0))
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode, static)
    fwd = oracle.ffn_forward(x, ids, w, wq, cfg.E, cfg.act_mode, static)
    ref = brute_force_ffn(x, ids, w, wq, cfg.act_mode, static)
    assert np.array_equal(fwd["y"], ref)
    # token-sampled forward agrees with the full forward
    toks = np.array([3, 0, 17], np.int64)
    samp = oracle.ffn_forward(x, ids, w, wq, cfg.E, cfg.act_mode, static, tokens=toks)
    assert np.array_equal(samp["y"], fwd["y"][toks])


def test_fp8_output_error_is_plausible_against_bf16_dense():
    """Context only: the pages report a relative-norm gap of ~0.064 between an
    fp8_dynamic MoE layer and bf16 dense (shape unstated).  The oracle's
    fp8 forward must sit in the same order of magnitude against its own fp64
    unquantised forward."""
    cfg = synth.scaled(synth.CONFIGS["tiny"], T=64)
    x = oracle.bf16_bits(synth.activations(cfg, 0))
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode)
    y = oracle.bf16_to_f64(oracle.ffn_forward(x, ids, w, wq, cfg.E, cfg.act_mode)["y"])
    src, pos, sizes, _ = oracle.ragged_sort(ids, cfg.E)
    xs = oracle.bf16_to_f64(x)[src // cfg.k]
    a = oracle.gmm_f64(xs, oracle.bf16_to_f64(oracle.bf16_bits(w_in)), sizes)
    h = oracle.swiglu_f64(a)
    o = oracle.gmm_f64(h, oracle.bf16_to_f64(oracle.bf16_bits(w_out)), sizes)
    y64 = oracle.combine_f64(o, pos, w, cfg.k)
    rel = np.linalg.norm(y - y64) / np.linalg.norm(y64)
    assert 0.005 < rel < 0.2, rel


# ------------------------------------------------------------- combine -----

def test_combine_k1_unit_weight_is_inverse_permutation():
    rng = np.random.default_rng(30)
    T, D = 40, 64
    ids = rng.integers(0, 5, (T, 1)).astype(np.int32)
    src, pos, _, _ = oracle.ragged_sort(ids, 5)
    o = bf16(rng.standard_normal((T, D)))
    y = oracle.combine(o, pos, None, 1)
    assert np.array_equal(y, o[pos])
    y1 = oracle.combine(o, pos, np.ones((T, 1), np.float32), 1)
    assert np.array_equal(y1, o[pos])


def test_combine_weighted_sum_and_token_sampling():
    rng = np.random.default_rng(31)
    T, k, D = 16, 3, 32
    ids = rng.integers(0, 4, (T, k)).astype(np.int32)
    src, pos, _, _ = oracle.ragged_sort(ids, 4)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    o = bf16(rng.standard_normal((T * k, D)))
    y = oracle.combine(o, pos, w, k, want="f64")
    ov = oracle.bf16_to_f64(o)
    ref = np.stack([sum(float(w[t, j]) * ov[pos[t * k + j]] for j in range(k)) for t in range(T)])
    np.testing.assert_allclose(y, ref, rtol=1e-14)
    toks = np.array([5, 1], np.int64)
    assert np.array_equal(oracle.combine(o, pos, w, k, tokens=toks), oracle.combine(o, pos, w, k)[toks])


# ---------------------------------------------------- adjoint identities ---

def _routing(rng, T, k, E):
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[:, 0] = rng.integers(0, E - 1, T)  # expert E-1 gets few rows
    return ids


def test_combine_adjoint_is_gather_scale():
    rng = np.random.default_rng(40)
    T, k, D, E = 20, 3, 16, 5
    ids = _routing(rng, T, k, E)
    src, pos, _, _ = oracle.ragged_sort(ids, E)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    o = rng.standard_normal((T * k, D))
    G = rng.standard_normal((T, D))
    lhs = np.sum(oracle.combine_f64(o, pos, w, k) * G)
    rhs = np.sum(o * oracle.gather_scale_f64(G, w, src, k))
    assert abs(lhs - rhs) <= 1e-12 * abs(lhs)


def test_gmm_adjoints_dx_and_tgmm():
    rng = np.random.default_rng(41)
    sizes = np.array([6, 0, 11, 4], np.int32)
    M, K, N = int(sizes.sum()), 24, 10
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((4, N, K))
    dY = rng.standard_normal((M, N))
    Y = oracle.gmm_f64(X, W, sizes)
    inner = np.sum(Y * dY)
    # input gradient: gmm of dY with the transposed weights
    dX = oracle.gmm_f64(dY, np.ascontiguousarray(W.transpose(0, 2, 1)), sizes)
    assert abs(np.sum(X * dX) - inner) <= 1e-12 * abs(inner)
    # weight gradient: tgmm, out[e, k, n] pairs with W[e, n, k]
    dW = oracle.tgmm_f64(X, dY, sizes)
    assert abs(np.sum(dW * W.transpose(0, 2, 1)) - inner) <= 1e-12 * abs(inner)
    assert np.all(dW[1] == 0)  # zero-token expert


def test_tgmm_sum_over_experts_is_dense_xt_dy():
    rng = np.random.default_rng(42)
    sizes = np.array([9, 0, 13, 2, 7], np.int32)
    M, K, N = int(sizes.sum()), 48, 40
    x = rand_codes(rng, (M, K))
    g = rand_codes(rng, (M, N))
    sx, sg = 0.37, 1.7
    out = oracle.tgmm(x, np.array([sx], np.float32), synth.PER_TENSOR, g, np.array([sg], np.float32),
                      synth.PER_TENSOR, sizes, want="f64")
    Xd = oracle.e4m3_to_f64(x) * np.float64(np.float32(sx))
    Gd = oracle.e4m3_to_f64(g) * np.float64(np.float32(sg))
    np.testing.assert_allclose(out.sum(axis=0), Xd.T @ Gd, rtol=1e-12, atol=1e-12)
    assert np.all(out[1] == 0)
    # per-(expert, column) scales agree with the dequantised double path
    sgc = rng.uniform(0.5, 2, (5, N)).astype(np.float32)
    sxc = rng.uniform(0.5, 2, (5, K)).astype(np.float32)
    out2 = oracle.tgmm(x, sxc, oracle.PER_GROUP_COL, g, sgc, oracle.PER_GROUP_COL, sizes, want="f64")
    starts = np.concatenate([[0], np.cumsum(sizes)])
    rows_e = np.repeat(np.arange(5), sizes)
    Xe = oracle.e4m3_to_f64(x) * sxc[rows_e].astype(np.float64)
    Ge = oracle.e4m3_to_f64(g) * sgc[rows_e].astype(np.float64)
    np.testing.assert_allclose(out2, oracle.tgmm_f64(Xe, Ge, sizes), rtol=1e-12, atol=1e-300)
    # sampled outputs equal the full tensor
    samp = np.array([0, 5 * K * N - 1, 2 * K * N + 17], np.int64)
    s_out = oracle.tgmm(x, sxc, oracle.PER_GROUP_COL, g, sgc, oracle.PER_GROUP_COL, sizes, samples=samp,
                        want="f64")
    assert np.array_equal(s_out, out2.reshape(-1)[samp])
    del starts


def test_quantize_group_cols():
    rng = np.random.default_rng(43)
    sizes = np.array([4, 0, 7], np.int32)
    M, N = 11, 20
    g = bf16(rng.standard_normal((M, N)) * np.exp(rng.uniform(-2, 2, (1, N))))
    q, s = oracle.quantize_group_cols(g, sizes)
    gv = oracle.bf16_to_f64(g).astype(np.float32)
    assert np.all(s[1] == 1.0)  # zero-token expert
    for e, (lo, hi) in enumerate([(0, 4), (4, 4), (4, 11)]):
        if hi == lo:
            continue
        amax = np.abs(gv[lo:hi]).max(axis=0)
        assert np.array_equal(s[e], (amax / np.float32(448.0)).astype(np.float32))
        qq, _ = oracle.quantize_rows(np.ascontiguousarray(g[lo:hi].T), synth.PER_ROW)
        assert np.array_equal(q[lo:hi], qq.T)


# ------------------------------------------------------ SwiGLU backward ----

def test_swiglu_bwd_f64_matches_finite_differences():
    rng = np.random.default_rng(50)
    R, F = 6, 9
    a = rng.standard_normal((R, 2 * F)) * 2
    dH = rng.standard_normal((R, F))
    dA = oracle.swiglu_bwd_f64(dH, a)
    eps = 1e-6
    num = np.empty_like(a)
    for idx in np.ndindex(a.shape):
        ap, am = a.copy(), a.copy()
        ap[idx] += eps
        am[idx] -= eps
        num[idx] = (np.sum(oracle.swiglu_f64(ap) * dH) - np.sum(oracle.swiglu_f64(am) * dH)) / (2 * eps)
    np.testing.assert_allclose(dA, num, rtol=1e-6, atol=1e-8)


def test_swiglu_fp32_paths_match_f64_within_bf16_rounding():
    rng = np.random.default_rng(51)
    R, F = 16, 64
    a = bf16(rng.standard_normal((R, 2 * F)) * 3)
    dH = bf16(rng.standard_normal((R, F)))
    av = oracle.bf16_to_f64(a)
    dA = oracle.bf16_to_f64(oracle.swiglu_bwd(dH, a))
    ref = oracle.swiglu_bwd_f64(oracle.bf16_to_f64(dH), av)
    assert np.all(np.abs(dA - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)
    _, _, hb = oracle.swiglu_quant(a, synth.PER_ROW)
    h = oracle.bf16_to_f64(hb)
    href = oracle.swiglu_f64(av)
    assert np.all(np.abs(h - href) <= 2.0 ** -8 * np.abs(href) + 1e-30)


def _ffn_loss_f64(x, W_in, W_out, ids, w, G, E):
    """Unquantised fp64 forward composed from the oracle's double helpers."""
    k = ids.shape[1]
    src, pos, sizes, _ = oracle.ragged_sort(ids, E)
    xs = x[src // k]
    a = oracle.gmm_f64(xs, W_in, sizes)
    h = oracle.swiglu_f64(a)
    o = oracle.gmm_f64(h, W_out, sizes)
    y = oracle.combine_f64(o, pos, w, k)
    return np.sum(y * G), (src, pos, sizes, xs, a, h)


def _ffn_grads_f64(x, W_in, W_out, ids, w, G, E):
    """The backward pass in the same composition as oracle.ffn_backward, on
    doubles: dO = gather-scale, dH = gmm(dO, wo^T), SwiGLU bwd,
    dXs = gmm(dA, w_in^T), dX = combine(dXs, w = 1), dW = tgmm."""
    k = ids.shape[1]
    _, (src, pos, sizes, xs, a, h) = _ffn_loss_f64(x, W_in, W_out, ids, w, G, E)
    dO = oracle.gather_scale_f64(G, w, src, k)
    dH = oracle.gmm_f64(dO, np.ascontiguousarray(W_out.transpose(0, 2, 1)), sizes)
    dA = oracle.swiglu_bwd_f64(dH, a)
    dXs = oracle.gmm_f64(dA, np.ascontiguousarray(W_in.transpose(0, 2, 1)), sizes)
    dX = oracle.combine_f64(dXs, pos, None, k)
    dW_in = oracle.tgmm_f64(xs, dA, sizes)   # [E, D, 2F]
    dW_out = oracle.tgmm_f64(h, dO, sizes)   # [E, F, D]
    return dX, dW_in, dW_out


def test_ffn_backward_matches_finite_differences():
    rng = np.random.default_rng(52)
    T, D, E, k, F = 6, 8, 3, 2, 5
    x = rng.standard_normal((T, D))
    W_in = rng.standard_normal((E, 2 * F, D)) * 0.5
    W_out = rng.standard_normal((E, D, F)) * 0.5
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1, (T, k)).astype(np.float32)
    G = rng.standard_normal((T, D))
    dX, dW_in, dW_out = _ffn_grads_f64(x, W_in, W_out, ids, w, G, E)
    eps = 1e-6

    def fd(arr, idx):
        p, m = arr.copy(), arr.copy()
        p[idx] += eps
        m[idx] -= eps
        return p, m

    for idx in [(0, 0), (3, 5), (5, 7)]:
        p, m = fd(x, idx)
        num = (_ffn_loss_f64(p, W_in, W_out, ids, w, G, E)[0] - _ffn_loss_f64(m, W_in, W_out, ids, w, G, E)[0])
        assert abs(num / (2 * eps) - dX[idx]) <= 1e-6 * max(1, abs(dX[idx]))
    for (e, c, d) in [(0, 0, 0), (1, 7, 3), (2, 9, 7)]:
        p, m = fd(W_in, (e, c, d))
        num = (_ffn_loss_f64(x, p, W_out, ids, w, G, E)[0] - _ffn_loss_f64(x, m, W_out, ids, w, G, E)[0])
        assert abs(num / (2 * eps) - dW_in[e, d, c]) <= 1e-6 * max(1, abs(dW_in[e, d, c]))
    for (e, d, f) in [(0, 0, 0), (1, 3, 4), (2, 7, 2)]:
        p, m = fd(W_out, (e, d, f))
        num = (_ffn_loss_f64(x, W_in, p, ids, w, G, E)[0] - _ffn_loss_f64(x, W_in, m, ids, w, G, E)[0])
        assert abs(num / (2 * eps) - dW_out[e, f, d]) <= 1e-6 * max(1, abs(dW_out[e, f, d]))


def test_ffn_backward_quantised_tracks_f64_gradients():
    """The quantised backward of the static scheme stays close to the exact
    gradients of the dequantised forward (loose: fp8 gradients)."""
    cfg = synth.scaled(synth.CONFIGS["fwdbwd"], T=48, D=128, E=12, F=128)
    x = oracle.bf16_bits(synth.activations(cfg, 0))
    ids, w = synth.routing(cfg, 0)
    G = oracle.bf16_bits(synth.output_grad(cfg, 0))
    w_in, w_out = synth.expert_weights(cfg, 0)
    static = synth.calibration_scales(cfg, 0)
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode, static)
    fwd = oracle.ffn_forward(x, ids, w, wq, cfg.E, cfg.act_mode, static)
    bwd = oracle.ffn_backward(fwd, G, w, wq, cfg.k, static)
    qin, sin, min_, qo, so, mo = wq
    dX64, dWin64, dWout64 = _ffn_grads_f64(oracle.bf16_to_f64(x), deq_weights(qin, sin, min_),
                                           deq_weights(qo, so, mo), ids, w, oracle.bf16_to_f64(G), cfg.E)
    for got, ref in [(oracle.bf16_to_f64(bwd["dX"]), dX64), (bwd["dW_in"], dWin64), (bwd["dW_out"], dWout64)]:
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 0.25, rel


def test_ffn_backward_composition_against_dense_numpy():
    """Pins every contraction of oracle.ffn_backward against dense numpy
    products of the oracle's own codes and scales ("Support quantization for
    tokamax gmm v2", fp8_static_wa: fixed weight and activation scales,
    absmax-quantised gradients).  wi_0 and wi_1 get static scales a factor
    4.7 apart, so putting s_w0 on the wrong half of the [dA0 | dA1]
    contraction, swapping the two, or splitting at the wrong K block changes
    dXs grossly (the negative controls below check that it would)."""
    cfg = synth.scaled(synth.CONFIGS["fwdbwd"], T=40, D=128, E=10, F=256)
    x = oracle.bf16_bits(synth.activations(cfg, 3))
    ids, w = synth.routing(cfg, 3)
    G = oracle.bf16_bits(synth.output_grad(cfg, 3))
    w_in, w_out = synth.expert_weights(cfg, 3)
    static = dict(synth.calibration_scales(cfg, 3))
    static["w1"] = float(np.float32(4.7 * static["w0"]))
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode, static)
    fwd = oracle.ffn_forward(x, ids, w, wq, cfg.E, cfg.act_mode, static)
    bwd = oracle.ffn_backward(fwd, G, w, wq, cfg.k, static)
    qin, _, _, qo, _, _ = wq
    F, D, k = cfg.F, cfg.D, cfg.k
    s0, s1, so = np.float64(np.float32(static["w0"])), np.float64(np.float32(static["w1"])), \
        np.float64(np.float32(static["wo"]))
    sx, sh = np.float64(np.float32(static["x"])), np.float64(np.float32(static["h"]))
    sizes = fwd["sizes"]
    starts = np.concatenate([[0], np.cumsum(sizes)])
    expert = np.repeat(np.arange(cfg.E), sizes)  # expert of each sorted row
    W0 = oracle.e4m3_to_f64(qin[:, :F, :])  # [E, F, D] codes of wi_0
    W1 = oracle.e4m3_to_f64(qin[:, F:, :])
    Wo = oracle.e4m3_to_f64(qo)             # [E, D, F]

    def close_bf16(got_bits, ref_f64, what):
        ref = oracle.bf16_to_f64(bf16(ref_f64))
        got = oracle.bf16_to_f64(got_bits)
        diff = got != ref
        # products of e4m3 codes sum exactly in fp64; only the order of the
        # scale multiplications may move a value across a bf16 rounding edge
        assert diff.mean() < 1e-3, (what, diff.mean())
        assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30), what

    # dH = dO @ wo: per-row dO scale, static wo scale
    dOq = oracle.e4m3_to_f64(bwd["dO_q"]) * bwd["dO_s"].astype(np.float64)[:, None]
    dH = np.stack([dOq[r] @ Wo[expert[r]] for r in range(len(expert))]) * so
    close_bf16(bwd["dH"], dH, "dH")
    # dXs = dA0 @ wi_0^T-side (s_w0) + dA1 @ wi_1 (s_w1), per-row dA scale
    dAq = oracle.e4m3_to_f64(bwd["dA_q"])
    dAs = bwd["dA_s"].astype(np.float64)
    part0 = np.stack([dAq[r, :F] @ W0[expert[r]] for r in range(len(expert))])
    part1 = np.stack([dAq[r, F:] @ W1[expert[r]] for r in range(len(expert))])
    dXs = (s0 * part0 + s1 * part1) * dAs[:, None]
    close_bf16(bwd["dXs"], dXs, "dXs")
    got = oracle.bf16_to_f64(bwd["dXs"])
    for wrong in ((s1 * part0 + s0 * part1) * dAs[:, None],   # scales swapped
                  (s0 * (part0 + part1)) * dAs[:, None],      # one scale for both halves
                  (s0 * np.stack([dAq[r, :F - 128] @ W0[expert[r], :F - 128] for r in range(len(expert))])
                   + s1 * (part1 + np.stack([dAq[r, F - 128:F] @ W0[expert[r], F - 128:] for r in
                                             range(len(expert))]))) * dAs[:, None]):  # split one block early
        assert np.linalg.norm(got - wrong) / np.linalg.norm(wrong) > 0.05
    # dX = the combine's adjoint with unit weights: sum of a token's k rows
    dX = np.zeros((cfg.T, D))
    for i in range(cfg.T * k):
        dX[i // k] += oracle.bf16_to_f64(bwd["dXs"][fwd["pos"][i]])
    close_bf16(bwd["dX"], dX, "dX")
    # weight gradients: per-(expert, column) gradient codes, static x / h scales
    xs = oracle.e4m3_to_f64(fwd["xs_q"]) * sx
    hq = oracle.e4m3_to_f64(fwd["h_q"]) * sh
    dAg = oracle.e4m3_to_f64(bwd["dAg_q"])
    dOg = oracle.e4m3_to_f64(bwd["dOg_q"])
    for e in range(cfg.E):
        rows = slice(starts[e], starts[e + 1])
        ref_in = xs[rows].T @ (dAg[rows] * bwd["dAg_s"][e].astype(np.float64)[None, :])
        ref_out = hq[rows].T @ (dOg[rows] * bwd["dOg_s"][e].astype(np.float64)[None, :])
        np.testing.assert_allclose(bwd["dW_in"][e], ref_in, rtol=2e-7, atol=1e-7 * max(np.abs(ref_in).max(), 1e-30))
        np.testing.assert_allclose(bwd["dW_out"][e], ref_out, rtol=2e-7,
                                   atol=1e-7 * max(np.abs(ref_out).max(), 1e-30))
    # the per-(expert, column) gradient codes are the absmax codes of dA / dO over the expert's rows
    for g_bits, gq, gs in ((bwd["dA"], bwd["dAg_q"], bwd["dAg_s"]), (bwd["dO"], bwd["dOg_q"], bwd["dOg_s"])):
        gv = oracle.bf16_to_f64(g_bits)
        for e in range(cfg.E):
            rows = slice(starts[e], starts[e + 1])
            if starts[e + 1] == starts[e]:
                assert np.all(gs[e] == 1.0)
                continue
            amax = np.abs(gv[rows]).max(axis=0)
            exp_s = np.where(amax > 0, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32), 1.0)
            assert np.array_equal(gs[e], exp_s.astype(np.float32))
