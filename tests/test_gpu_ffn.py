"""End-to-end GPU parity of the expert FFN (forward, and backward for the
static scheme) against the oracle on seeded synthetic inputs.

Small cases run the whole oracle; the full-size workloads compare sampled
tokens, which the oracle evaluates one by one (y[t] depends only on x[t]).
Quantised bytes and indices produced from the inputs directly are bit-exact;
every output downstream of a contraction is compared with the tolerance."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_helpers import assert_close, dev, host

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("fp8_quantized_moe_gb300")


def run_gpu_forward(cfg, x, ids, w, W, static):
    sx = sh = None
    if cfg.act_mode == synth.PER_TENSOR:
        sx = torch.tensor([static["x"]], dtype=torch.float32, device="cuda")
        sh = torch.tensor([static["h"]], dtype=torch.float32, device="cuda")
    buf = moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, cfg.act_mode, "cuda", backward=cfg.backward)
    buf.keep_a = True  # the tests compare the wi_0 | wi_1 product too
    y = moe.ffn_forward(x, ids, w, W, cfg.act_mode, buf, sx, sh)
    assert moe.device_error() == 0
    return y, buf, sx, sh


SMALL = {
    "tiny": synth.CONFIGS["tiny"],
    "mixtral": synth.scaled(synth.CONFIGS["mixtral"], T=384, D=256, F=512),
    "dsv3": synth.scaled(synth.CONFIGS["dsv3"], T=256, D=384, E=32, F=256),
    "prefill": synth.scaled(synth.CONFIGS["prefill"], T=512, D=256, E=32, F=384),
    "fwdbwd": synth.scaled(synth.CONFIGS["fwdbwd"], T=512, D=256, E=24, F=384),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_ffn_small_matches_oracle(name):
    cfg = SMALL[name]
    x_t = synth.activations(cfg, 0)
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    xb = oracle.bf16_bits(x_t)
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode, static)
    ref = oracle.ffn_forward(xb, ids, w, wq, cfg.E, cfg.act_mode, static)

    W = moe.prepare_weights(w_in.cuda(), w_out.cuda(), cfg.w_mode, static, for_backward=cfg.backward)
    # weight quantisation is bit-exact
    assert np.array_equal(host(W.w_in), wq[0]) and np.array_equal(host(W.w_out), wq[3])
    assert np.array_equal(host(W.s_in), wq[1])
    if cfg.w_mode != synth.PER_TENSOR:
        assert np.array_equal(host(W.s_out), wq[4])
    y, buf, sx, sh = run_gpu_forward(cfg, x_t.cuda(), dev(ids), dev(w), W, static)
    # steps computed from the inputs directly (quantise + sort + gather, fused): bit-exact
    for key in ("sorted_src", "pos", "group_sizes", "group_offsets", "xs_q"):
        assert np.array_equal(host(buf.sort[key]), ref[{"group_sizes": "sizes", "group_offsets": "offsets"}.get(key, key)]), key
    if cfg.act_mode != synth.PER_TENSOR:
        _, xss_ref = oracle.gather_rows(ref["x_q"], ref["x_s"], cfg.act_mode, ref["sorted_src"], cfg.k)
        assert np.array_equal(host(buf.sort["xs_scale"]).view(np.uint32), xss_ref.view(np.uint32))
    # downstream of the contractions: tolerance
    assert_close(host(buf.a), ref["a"], f"{name}: a")
    assert_close(host(buf.o), ref["o"], f"{name}: o", rel_fro=5e-3)
    assert_close(host(y), ref["y"], f"{name}: y", rel_fro=5e-3)
    # h: dequantised values agree (codes may differ where a differs)
    h_ref = oracle.e4m3_to_f64(ref["h_q"])
    h_gpu = oracle.e4m3_to_f64(host(buf.h_q))
    if cfg.act_mode == synth.PER_ROW:
        h_ref *= ref["h_s"][:, None]
        h_gpu *= host(buf.h_s)[:, None]
    mism = np.mean(host(buf.h_q) != ref["h_q"])
    assert mism < 2e-3, f"{name}: {mism:.2e} of the h codes differ"

    if cfg.backward:
        G_t = synth.output_grad(cfg, 0)
        bref = oracle.ffn_backward(ref, oracle.bf16_bits(G_t), w, wq, cfg.k, static)
        dX, dW_in, dW_out = moe.ffn_backward(G_t.cuda(), dev(w.reshape(-1)), W, buf, sx, sh)
        assert moe.device_error() == 0
        assert_close(host(buf.dH), bref["dH"], f"{name}: dH")
        assert_close(host(buf.dXs), bref["dXs"], f"{name}: dXs", rel_fro=5e-3)
        assert_close(host(dX), bref["dX"], f"{name}: dX", rel_fro=5e-3)
        assert_close(host(dW_in), bref["dW_in"], f"{name}: dW_in", rel_fro=5e-3)
        assert_close(host(dW_out), bref["dW_out"], f"{name}: dW_out", rel_fro=5e-3)


def oracle_token(xq_row, xs_row, cfg, e, wq_e, static):
    """Oracle forward of one (token, expert) pair: returns (a, h_q, o) rows."""
    qin, sin, min_, qo, so, mo = wq_e
    sizes = np.array([1], np.int32)
    a = oracle.gmm(xq_row, xs_row, cfg.act_mode, qin, sin, min_, sizes)
    sh = static["h"] if static else 1.0
    hq, hs, _ = oracle.swiglu_quant(a, cfg.act_mode, sh)
    o = oracle.gmm(hq, hs, cfg.act_mode, qo, so, mo, sizes)
    return a, o


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "prefill", "fwdbwd"])
def test_ffn_full_size_sampled_tokens(name):
    cfg = synth.CONFIGS[name]
    torch.manual_seed(0)
    x_t = synth.activations(cfg, 0, device="cuda")
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0, device="cuda")
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    W = moe.prepare_weights(w_in, w_out, cfg.w_mode, static)
    y, buf, _, _ = run_gpu_forward(cfg, x_t, dev(ids), dev(w), W, static)
    yh = host(y)
    xb = host(x_t)
    rng = np.random.default_rng(1)
    tokens = rng.choice(cfg.T, 4, replace=False)
    sx = static["x"] if static else 1.0
    ys = []
    F = cfg.F
    for t in tokens:
        xq, xs = oracle.quantize_rows(xb[t:t + 1], cfg.act_mode, sx)
        acc = np.zeros(cfg.D)
        for j in range(cfg.k):
            e = int(ids[t, j])
            w_in_e = host(w_in[e:e + 1])
            w_out_e = host(w_out[e:e + 1])
            wq_e = oracle.prepare_weights(w_in_e, w_out_e, cfg.w_mode, static)
            a, o = oracle_token(xq, xs, cfg, e, wq_e, static)
            r = int(host(buf.sort["pos"])[t * cfg.k + j])
            assert_close(host(buf.a[r:r + 1]), a, f"{name}: a[t={t}, j={j}]")
            acc += float(w[t, j]) * oracle.bf16_to_f64(o)[0]
        ys.append(oracle.f64_to_bf16(acc))
    assert_close(yh[tokens], np.stack(ys), f"{name}: y sampled", rel_fro=5e-3)
    del F


@pytest.mark.parametrize("name", ["tiny", "mixtral", "fwdbwd"])
def test_fused_and_unfused_forward_are_identical(name):
    cfg = SMALL[name]
    x_t = synth.activations(cfg, 0).cuda()
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    W = moe.prepare_weights(w_in.cuda(), w_out.cuda(), cfg.w_mode, static)
    assert moe.swiglu_fusable(cfg.act_mode, W.in_mode, cfg.F)
    sx = sh = None
    if static:
        sx = torch.tensor([static["x"]], dtype=torch.float32, device="cuda")
        sh = torch.tensor([static["h"]], dtype=torch.float32, device="cuda")
    outs = []
    for fuse in (True, False):
        buf = moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, cfg.act_mode, "cuda")
        y = moe.ffn_forward(x_t, dev(ids), dev(w), W, cfg.act_mode, buf, sx, sh, fuse_swiglu=fuse,
                            fuse_quant_sort=fuse)
        outs.append((host(y), host(buf.h_q), host(buf.sort["xs_q"])))
    assert moe.device_error() == 0
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
