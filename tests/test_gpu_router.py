"""GPU parity of the router ("Support quantization for tokamax gmm v2",
table 1: grad_gate-kernel and state_grad) against the oracle: the gate's
logits within relative Frobenius 2e-3, the softmax / top-k decisions and
weights bit-exact against the oracle fed the GPU's logits, the softmax
backward bit-exact against the oracle fed the GPU's inputs, and the gate's
two gradient contractions within 2e-3."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import assert_close, dev, host

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("fp8_quantized_moe_gb300")


def bf16_rand(rng, shape, std=1.0):
    return oracle.bf16_bits(torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16))


def router_case(T, D, E, seed):
    rng = np.random.default_rng(seed)
    x = bf16_rand(rng, (T, D))
    wg = bf16_rand(rng, (E, D), 1.5 / np.sqrt(D))  # logits of O(1)
    return rng, x, wg


@pytest.mark.parametrize("T,D,E,k", [
    (256, 128, 4, 2),      # the tiny layer's shape
    (1000, 4096, 8, 2),    # Mixtral-shaped gate
    (513, 7168, 256, 8),   # DeepSeek-V3-shaped gate, a ragged last tile
    (300, 2048, 128, 8),   # prefill chunk
    (200, 4096, 64, 6),
    (128, 64, 16, 8),      # one K block
    (77, 136, 24, 3),      # a K tail of 8 columns
    (1, 128, 1, 1),
])
def test_router_topk_matches_oracle(T, D, E, k):
    _, x, wg = router_case(T, D, E, T + D + E + k)
    logits, ids, w = moe.router_topk(dev(x), dev(wg), k)
    assert moe.device_error() == 0
    ref = oracle.router_logits(x, wg)
    assert_close(host(logits), ref.astype(np.float32), f"logits T={T} D={D} E={E}")
    # the routing decision from the GPU's logits: bit-exact
    ids_ref, w_ref = oracle.router_topk(host(logits), k)
    assert np.array_equal(host(ids), ids_ref)
    assert np.array_equal(host(w).view(np.uint32), w_ref.view(np.uint32))


def test_router_topk_ties_go_to_the_lower_index():
    T, D, E, k = 130, 64, 32, 8
    x = np.zeros((T, D), np.uint16)  # every logit 0: all experts tie
    rng = np.random.default_rng(0)
    wg = bf16_rand(rng, (E, D))
    logits, ids, w = moe.router_topk(dev(x), dev(wg), k)
    assert moe.device_error() == 0
    assert np.all(host(logits) == 0)
    assert np.array_equal(host(ids), np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    assert np.all(host(w) == np.float32(1.0 / E))


@pytest.mark.parametrize("T,D,E,k", [(256, 128, 4, 2), (600, 1024, 64, 6), (300, 2048, 128, 8), (129, 256, 24, 3)])
def test_router_backward_matches_oracle(T, D, E, k):
    rng, x, wg = router_case(T, D, E, 7 * T + D + E)
    logits, ids, w = moe.router_topk(dev(x), dev(wg), k)
    ids_h = host(ids)
    src, pos, _, _ = oracle.ragged_sort(ids_h, E)
    G = bf16_rand(rng, (T, D))
    o = bf16_rand(rng, (T * k, D))
    dw, dl, gg, sg = moe.router_backward(dev(G), dev(o), dev(pos), dev(x), dev(wg), logits, ids)
    assert moe.device_error() == 0
    assert_close(host(dw), oracle.router_dw(G, o, pos, k).astype(np.float32), "dw")
    # the softmax backward of the GPU's logits, ids and dw: bit-exact
    dl_ref = oracle.router_dlogits(host(logits), ids_h, host(dw))
    assert np.array_equal(host(dl), dl_ref)
    gg_ref, sg_ref = oracle.router_grads(x, wg, host(dl))
    assert_close(host(gg), gg_ref.astype(np.float32), "grad_gate")
    assert_close(host(sg), oracle.f64_to_bf16(sg_ref), "state_grad")


def test_router_full_size_deepseek_v3_gate():
    """The DeepSeek-V3-shaped gate (T=16384, D=7168, E=256, k=8): the routing
    decision of every token bit-exact from the GPU's logits, and the logits
    of sampled tokens against the oracle."""
    cfg = synth.CONFIGS["dsv3"]
    T, D, E, k = cfg.T, cfg.D, cfg.E, cfg.k
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    x = torch.randn(T, D, generator=g, device="cuda").to(torch.bfloat16)
    wg = (torch.randn(E, D, generator=g, device="cuda") * (1.5 / np.sqrt(D))).to(torch.bfloat16)
    logits, ids, w = moe.router_topk(x, wg, k)
    assert moe.device_error() == 0
    ids_ref, w_ref = oracle.router_topk(host(logits), k)
    assert np.array_equal(host(ids), ids_ref)
    assert np.array_equal(host(w).view(np.uint32), w_ref.view(np.uint32))
    rows = np.random.default_rng(1).choice(T, 16, replace=False)
    ref = oracle.router_logits(host(x)[rows], host(wg))
    assert_close(host(logits)[rows], ref.astype(np.float32), "dsv3 logits sampled")
