"""Pins of the oracle's router (CPU only): the gate layer against a numpy
dense matmul, the fp32 softmax / top-k against an fp64 softmax and its
invariants (ties to the lower expert index, masked experts, k = E), the
softmax backward against central finite differences, and the gate gradients
against numpy products and against finite differences of the composed
routing loss ("Support quantization for tokamax gmm v2", table 1:
grad_gate-kernel and state_grad)."""

import numpy as np
import torch

import oracle


def bf16(a) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def dec(b) -> np.ndarray:
    return oracle.bf16_to_f64(b)


def softmax64(l):
    l = np.asarray(l, np.float64)
    m = np.max(l, axis=1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=1, keepdims=True)


def test_router_logits_is_dense_matmul():
    rng = np.random.default_rng(0)
    x = bf16(rng.standard_normal((37, 96)))
    wg = bf16(rng.standard_normal((24, 96)) * 0.1)
    got = oracle.router_logits(x, wg)
    np.testing.assert_allclose(got, dec(x) @ dec(wg).T, rtol=1e-12, atol=1e-12)


def test_router_topk_matches_fp64_softmax_and_invariants():
    rng = np.random.default_rng(1)
    T, E, k = 300, 64, 6
    l = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    ids, w, p = oracle.router_topk(l, k, want_p=True)
    p64 = softmax64(l)
    # probabilities: fp32 values of the softmax (a few roundings each)
    np.testing.assert_allclose(p, p64, rtol=2e-6, atol=1e-12)
    assert np.allclose(p.sum(axis=1, dtype=np.float64), 1.0, atol=1e-5)
    for t in range(T):
        assert len(set(ids[t])) == k
        assert np.array_equal(w[t], p[t, ids[t]])
        assert np.all(np.diff(w[t]) <= 0)  # descending
        order = np.argsort(-p64[t], kind="stable")
        kth, nxt = p64[t, order[k - 1]], p64[t, order[k]]
        if kth - nxt > 1e-5 * kth:  # no near-tie at the cut: the same set as the fp64 softmax
            assert set(ids[t]) == set(order[:k])


def test_router_topk_ties_go_to_the_lower_index():
    T, E, k = 4, 16, 5
    l = np.zeros((T, E), np.float32)
    ids, w = oracle.router_topk(l, k)
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    assert np.all(w == np.float32(1.0 / 16))
    l[1, [3, 9, 12]] = 2.0  # three equal maxima, then equal rest
    ids, _ = oracle.router_topk(l, k)
    assert list(ids[1]) == [3, 9, 12, 0, 1]


def test_router_topk_masked_experts_and_k_equals_e():
    rng = np.random.default_rng(2)
    T, E = 50, 12
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[:, [2, 7]] = -np.inf
    ids, w, p = oracle.router_topk(l, 10, want_p=True)
    assert np.all(p[:, [2, 7]] == 0)
    assert not np.isin(ids, [2, 7]).any()
    ids_all, w_all = oracle.router_topk(l, E)
    for t in range(T):
        assert sorted(ids_all[t]) == list(range(E))
        assert set(ids_all[t, -2:]) == {2, 7} and np.all(w_all[t, -2:] == 0)


def _route_loss64(l, ids, dw):
    p = softmax64(l)
    return np.sum(np.take_along_axis(p, ids, axis=1) * dw)


def test_router_dlogits_match_finite_differences():
    rng = np.random.default_rng(3)
    T, E, k = 6, 10, 3
    l = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = oracle.router_topk(l, k)
    dw = rng.standard_normal((T, k)).astype(np.float32)
    got = dec(oracle.router_dlogits(l, ids, dw))
    eps = 1e-6
    fd = np.zeros((T, E))
    l64 = l.astype(np.float64)
    for t in range(T):
        for i in range(E):
            a, b = l64.copy(), l64.copy()
            a[t, i] += eps
            b[t, i] -= eps
            fd[t, i] = (_route_loss64(a, ids, dw) - _route_loss64(b, ids, dw)) / (2 * eps)
    scale = np.abs(fd).max()
    assert np.all(np.abs(got - fd) <= 2.0 ** -7 * np.abs(fd) + 1e-5 * scale)
    # the test tells the softmax backward from plausible mistakes
    p = softmax64(l)
    g = np.zeros((T, E))
    np.put_along_axis(g, ids, dw.astype(np.float64), axis=1)
    s = np.sum(np.take_along_axis(p, ids, axis=1) * dw, axis=1, keepdims=True)
    for wrong in (p * g, p * (g + s), g - s):
        assert np.linalg.norm(wrong - fd) > 0.05 * np.linalg.norm(fd)


def test_router_dw_and_gate_gradients_are_dense_products():
    rng = np.random.default_rng(4)
    T, D, E, k = 40, 64, 12, 3
    x = bf16(rng.standard_normal((T, D)))
    wg = bf16(rng.standard_normal((E, D)) * 0.1)
    G = bf16(rng.standard_normal((T, D)))
    o = bf16(rng.standard_normal((T * k, D)))
    pos = rng.permutation(T * k).astype(np.int32)
    dw = oracle.router_dw(G, o, pos, k)
    ref = np.einsum("td,tjd->tj", dec(G), dec(o)[pos.reshape(T, k)])
    np.testing.assert_allclose(dw, ref, rtol=1e-12, atol=1e-10)
    dl = bf16(rng.standard_normal((T, E)) * 0.01)
    gg, sg = oracle.router_grads(x, wg, dl)
    np.testing.assert_allclose(gg, dec(dl).T @ dec(x), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(sg, dec(dl) @ dec(wg), rtol=1e-12, atol=1e-12)


def test_router_chain_matches_finite_differences():
    """grad_gate and state_grad of L(x, W_gate) = sum_{t,j} dw[t, j] p[t, id_j]
    with p = softmax(x W_gate^T) and the routing ids held fixed."""
    rng = np.random.default_rng(5)
    T, D, E, k = 8, 16, 6, 2
    x = bf16(rng.standard_normal((T, D)))
    wg = bf16(rng.standard_normal((E, D)) * 0.3)
    l = oracle.router_logits(x, wg).astype(np.float32)
    ids, _ = oracle.router_topk(l, k)
    dw = rng.standard_normal((T, k)).astype(np.float32)
    dl = oracle.router_dlogits(l, ids, dw)
    gg, sg = oracle.router_grads(x, wg, dl)
    X, W = dec(x), dec(wg)

    def loss(X, W):
        return _route_loss64(X @ W.T, ids, dw)

    eps = 1e-6
    fd_w = np.zeros_like(W)
    for e in range(E):
        for d in range(D):
            a, b = W.copy(), W.copy()
            a[e, d] += eps
            b[e, d] -= eps
            fd_w[e, d] = (loss(X, a) - loss(X, b)) / (2 * eps)
    fd_x = np.zeros_like(X)
    for t in range(T):
        for d in range(D):
            a, b = X.copy(), X.copy()
            a[t, d] += eps
            b[t, d] -= eps
            fd_x[t, d] = (loss(a, W) - loss(b, W)) / (2 * eps)
    # bf16 dlogits: about 2^-9 relative per element
    assert np.linalg.norm(gg - fd_w) <= 1e-2 * np.linalg.norm(fd_w)
    assert np.linalg.norm(sg - fd_x) <= 1e-2 * np.linalg.norm(fd_x)
