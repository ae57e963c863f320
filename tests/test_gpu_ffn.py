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


def _h_scales_equal(got, ref, mode):
    if mode == synth.PER_TENSOR:
        return True
    return np.array_equal(np.asarray(got).view(np.uint32), np.asarray(ref).view(np.uint32))


@pytest.mark.parametrize("name", list(SMALL))
def test_ffn_small_matches_oracle(name):
    """Every stage against the oracle fed the GPU's own previous-stage output
    (stagewise parity): requantised codes and scales bit-exact, every
    contraction and the combine within relative Frobenius 2e-3 and
    max |delta| <= 1e-2 max|ref|.  The composed chain (the oracle run from the
    inputs alone) is held to 5e-3 on outputs downstream of a contraction and a
    requantisation: where fp32 and fp64 sums round a gmm output to
    neighbouring bf16 values, a requantised code moves by one e4m3 step."""
    cfg = SMALL[name]
    x_t = synth.activations(cfg, 0)
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0)
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    xb = oracle.bf16_bits(x_t)
    wq = oracle.prepare_weights(oracle.bf16_bits(w_in), oracle.bf16_bits(w_out), cfg.w_mode, static)
    qin, sin, min_, qo, so, mo = wq
    ref = oracle.ffn_forward(xb, ids, w, wq, cfg.E, cfg.act_mode, static)

    W = moe.prepare_weights(w_in.cuda(), w_out.cuda(), cfg.w_mode, static, for_backward=cfg.backward)
    # weight quantisation is bit-exact
    assert np.array_equal(host(W.w_in), qin) and np.array_equal(host(W.w_out), qo)
    assert np.array_equal(host(W.s_in), sin)
    if cfg.w_mode != synth.PER_TENSOR:
        assert np.array_equal(host(W.s_out), so)
    y, buf, sx, sh = run_gpu_forward(cfg, x_t.cuda(), dev(ids), dev(w), W, static)
    # steps computed from the inputs directly (quantise + sort + gather, fused): bit-exact
    for key in ("sorted_src", "pos", "group_sizes", "group_offsets", "xs_q"):
        assert np.array_equal(host(buf.sort[key]), ref[{"group_sizes": "sizes", "group_offsets": "offsets"}.get(key, key)]), key
    if cfg.act_mode != synth.PER_TENSOR:
        _, xss_ref = oracle.gather_rows(ref["x_q"], ref["x_s"], cfg.act_mode, ref["sorted_src"], cfg.k)
        assert np.array_equal(host(buf.sort["xs_scale"]).view(np.uint32), xss_ref.view(np.uint32))
    sizes = ref["sizes"]
    sh_f = static["h"] if static else 1.0
    # stage 3 (gmm wi_0 | wi_1): its inputs are bit-exact, so the oracle's own a is the reference
    assert_close(host(buf.a), ref["a"], f"{name}: a")
    # stage 4 (SwiGLU + requantisation) of the GPU's a: bit-exact codes and scales
    hq_ref, hs_ref, _ = oracle.swiglu_quant(host(buf.a), cfg.act_mode, sh_f)
    assert np.array_equal(host(buf.h_q), hq_ref), f"{name}: h codes"
    if cfg.act_mode != synth.PER_TENSOR:
        assert _h_scales_equal(host(buf.h_s), hs_ref, cfg.act_mode), f"{name}: h scales"
    # stage 5 (gmm wo) of the GPU's h
    h_s_gpu = host(buf.h_s) if cfg.act_mode != synth.PER_TENSOR else np.array([sh_f], np.float32)
    o_stage = oracle.gmm(host(buf.h_q), h_s_gpu, cfg.act_mode, qo, so, mo, sizes)
    assert_close(host(buf.o), o_stage, f"{name}: o (stage)")
    # stage 6 (combine) of the GPU's o
    y_stage = oracle.combine(host(buf.o), ref["pos"], w, cfg.k)
    assert_close(host(y), y_stage, f"{name}: y (stage)")
    # the composed chain from the inputs alone
    assert_close(host(buf.o), ref["o"], f"{name}: o (composed)", rel_fro=5e-3)
    assert_close(host(y), ref["y"], f"{name}: y (composed)", rel_fro=5e-3)
    mism = np.mean(host(buf.h_q) != ref["h_q"])
    assert mism < 2e-3, f"{name}: {mism:.2e} of the composed h codes differ"

    if cfg.backward:
        G_t = synth.output_grad(cfg, 0)
        Gb = oracle.bf16_bits(G_t)
        bref = oracle.ffn_backward(ref, Gb, w, wq, cfg.k, static)
        keep = {}
        dX, dW_in, dW_out = moe.ffn_backward(G_t.cuda(), dev(w.reshape(-1)), W, buf, sx, sh, keep=keep)
        assert moe.device_error() == 0
        src, pos = ref["sorted_src"], ref["pos"]
        # dO = w G[src] and its per-row codes: bit-exact (inputs only)
        assert np.array_equal(host(keep["dO"]), bref["dO"])
        assert np.array_equal(host(keep["dO_q"]), bref["dO_q"])
        assert np.array_equal(host(keep["dO_s"]).view(np.uint32), bref["dO_s"].view(np.uint32))
        # dH = gmm(dO_q, wo^T): inputs bit-exact, the oracle's dH is the stage reference
        assert_close(host(buf.dH), bref["dH"], f"{name}: dH")
        # SwiGLU backward of the GPU's dH and a, and its per-row codes: bit-exact
        dA_stage = oracle.swiglu_bwd(host(buf.dH), host(buf.a))
        assert np.array_equal(host(keep["dA"]), dA_stage), f"{name}: dA"
        dAq_stage, dAs_stage = oracle.quantize_rows(dA_stage, synth.PER_ROW)
        assert np.array_equal(host(keep["dA_q"]), dAq_stage), f"{name}: dA codes"
        assert np.array_equal(host(keep["dA_s"]).view(np.uint32), dAs_stage.view(np.uint32))
        # dXs = [dA0 | dA1] w_in^T with s_w0 on the first F columns of K, s_w1 on the rest
        F2, D = 2 * cfg.F, cfg.D
        qinT = np.ascontiguousarray(np.transpose(qin, (0, 2, 1)))
        sinT = np.empty((cfg.E, F2 // 128, D), np.float32)
        sinT[:, : cfg.F // 128] = np.float32(static["w0"])
        sinT[:, cfg.F // 128:] = np.float32(static["w1"])
        dXs_stage = oracle.gmm(dAq_stage, dAs_stage, synth.PER_ROW, qinT, sinT, synth.PER_ROW_BLOCK128, sizes)
        assert_close(host(buf.dXs), dXs_stage, f"{name}: dXs (stage)")
        dX_stage = oracle.combine(host(buf.dXs), pos, None, cfg.k)
        assert_close(host(dX), dX_stage, f"{name}: dX (stage)")
        # weight gradients of the GPU's gradients: per-(expert, column) scales bit-exact, tgmm at 2e-3
        dAg_q, dAg_s = oracle.quantize_group_cols(dA_stage, sizes)
        dOg_q, dOg_s = oracle.quantize_group_cols(bref["dO"], sizes)
        assert np.array_equal(host(keep["dAg_s"]).view(np.uint32), dAg_s.view(np.uint32))
        assert np.array_equal(host(keep["dOg_s"]).view(np.uint32), dOg_s.view(np.uint32))
        sxa = np.array([static["x"]], np.float32)
        sha = np.array([static["h"]], np.float32)
        dWin_stage = oracle.tgmm(host(buf.sort["xs_q"]), sxa, synth.PER_TENSOR, dAg_q, dAg_s,
                                 synth.PER_GROUP_COL, sizes)
        dWout_stage = oracle.tgmm(host(buf.h_q), sha, synth.PER_TENSOR, dOg_q, dOg_s, synth.PER_GROUP_COL, sizes)
        assert_close(host(dW_in), dWin_stage, f"{name}: dW_in (stage)")
        assert_close(host(dW_out), dWout_stage, f"{name}: dW_out (stage)")
        # the composed chain
        assert_close(host(buf.dXs), bref["dXs"], f"{name}: dXs (composed)", rel_fro=5e-3)
        assert_close(host(dX), bref["dX"], f"{name}: dX (composed)", rel_fro=5e-3)
        assert_close(host(dW_in), bref["dW_in"], f"{name}: dW_in (composed)", rel_fro=5e-3)
        assert_close(host(dW_out), bref["dW_out"], f"{name}: dW_out (composed)", rel_fro=5e-3)


def oracle_token(xq_row, xs_row, cfg, e, wq_e, static):
    """Oracle forward of one (token, expert) pair: returns (a, o) rows."""
    qin, sin, min_, qo, so, mo = wq_e
    sizes = np.array([1], np.int32)
    a = oracle.gmm(xq_row, xs_row, cfg.act_mode, qin, sin, min_, sizes)
    sh = static["h"] if static else 1.0
    hq, hs, _ = oracle.swiglu_quant(a, cfg.act_mode, sh)
    o = oracle.gmm(hq, hs, cfg.act_mode, qo, so, mo, sizes)
    return a, o


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "prefill", "fwdbwd"])
def test_ffn_full_size_sampled_tokens(name):
    """The full-size layers in the launch configuration of the benchmark, on
    sampled tokens the oracle evaluates one by one (y[t] depends only on
    x[t]).  Stagewise: a from the oracle, h codes and scales of the GPU's a
    bit-exact, o of the GPU's h and y of the GPU's o within 2e-3; the
    composed y within 5e-3."""
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
    pos = host(buf.sort["pos"])
    rng = np.random.default_rng(1)
    tokens = rng.choice(cfg.T, 4, replace=False)
    sx = static["x"] if static else 1.0
    sh = static["h"] if static else 1.0
    ys, ys_stage = [], []
    for t in tokens:
        xq, xs = oracle.quantize_rows(xb[t:t + 1], cfg.act_mode, sx)
        acc = np.zeros(cfg.D)
        o_rows, w_rows = [], []
        for j in range(cfg.k):
            e = int(ids[t, j])
            w_in_e = host(w_in[e:e + 1])
            w_out_e = host(w_out[e:e + 1])
            wq_e = oracle.prepare_weights(w_in_e, w_out_e, cfg.w_mode, static)
            a, o = oracle_token(xq, xs, cfg, e, wq_e, static)
            r = int(pos[t * cfg.k + j])
            a_gpu = host(buf.a[r:r + 1])
            assert_close(a_gpu, a, f"{name}: a[t={t}, j={j}]")
            # SwiGLU + requantisation of the GPU's a row: bit-exact
            hq_ref, hs_ref, _ = oracle.swiglu_quant(a_gpu, cfg.act_mode, sh)
            hq_gpu = host(buf.h_q[r:r + 1])
            assert np.array_equal(hq_gpu, hq_ref), f"{name}: h codes of row {r}"
            if cfg.act_mode != synth.PER_TENSOR:
                hs_gpu = host(buf.h_s[r:r + 1])
                assert _h_scales_equal(hs_gpu, hs_ref, cfg.act_mode), f"{name}: h scales of row {r}"
            else:
                hs_gpu = np.array([sh], np.float32)
            # wo gmm of the GPU's h row
            qin, sin, min_, qo, so, mo = wq_e
            o_stage = oracle.gmm(hq_gpu, hs_gpu, cfg.act_mode, qo, so, mo, np.array([1], np.int32))
            o_gpu = host(buf.o[r:r + 1])
            assert_close(o_gpu, o_stage, f"{name}: o[t={t}, j={j}] (stage)")
            acc += float(w[t, j]) * oracle.bf16_to_f64(o)[0]
            o_rows.append(o_gpu[0])
        ys.append(oracle.f64_to_bf16(acc))
        # combine of the GPU's o rows of this token (a one-token combine, k rows in order)
        ys_stage.append(oracle.combine(np.stack(o_rows), np.arange(cfg.k, dtype=np.int32),
                                       w[t:t + 1], cfg.k)[0])
    assert_close(yh[tokens], np.stack(ys_stage), f"{name}: y sampled (stage)")
    assert_close(yh[tokens], np.stack(ys), f"{name}: y sampled (composed)", rel_fro=5e-3)


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
